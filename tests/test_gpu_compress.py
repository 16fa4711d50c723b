"""GPU parity of snap_compress (prefill compression) against the CPU oracle.

SnapStream episode companion page, "Fixed-Size Cache Layout": sinks + SnapKV
top-K middle + recent window, built once at prefill.  Each case runs the CUDA
library through its C ABI and the oracle on the same seeded inputs, then checks
the meta exactly, the selection up to ties within 1e-6 relative, and every cache
row bit-exactly.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from fixed_size_kv_gb300 import inputs, snap
from parity import (check_cache_rows, check_selection, gpu_meta, oracle_cfg, snap_cfg)

pytestmark = pytest.mark.gpu


def run_compress(wl, S, seed, slot=0, max_batch=2, want_pool=True, strided=False):
    pre = inputs.gen_prefill(wl, S, seed=seed)
    cache = snap.SnapCache(snap_cfg(wl), max_batch=max_batch, max_prompt=S)
    K, V = pre.K.cuda(), (pre.V.cuda() if pre.V is not None else None)
    if strided:
        # K and V as views into one [S][2][H_kv][d] prefill buffer (non-contiguous tokens)
        kv = torch.stack([K, V], dim=1)
        K, V = kv[:, 0], kv[:, 1]
    cache.compress(slot, K, V, pre.Q.cuda())
    torch.cuda.synchronize()
    assert cache.check_device() == snap.SNAP_OK
    ocache = oracle.compress(oracle_cfg(wl), pre.K, pre.V, pre.Q, want_pool=want_pool)
    return pre, cache, ocache


def check_all(wl, pre, cache, ocache, slot=0, where=""):
    swaps = 0
    if ocache.pool is not None and ocache.meta.n_mid == wl.K and wl.K > 0 and \
            ocache.meta.R0 - ocache.meta.n_sink > wl.K:
        gsel = cache.selected()[slot].cpu().numpy()
        for h in range(wl.n_kv_heads):
            swaps += check_selection(gsel[h], ocache.sel[h], ocache.pool[h], f"{where} head {h}")
    else:
        if wl.K > 0:
            np.testing.assert_array_equal(cache.selected()[slot].cpu().numpy(), ocache.sel)
    check_cache_rows(cache, slot, ocache, pre.K, pre.V, where)
    return swaps


def small_gqa(**kw):
    base = dict(name="small", layout=0, n_q_heads=32, n_kv_heads=8, d_qk=128, d_v=128,
                L_sink=4, K=60, L_recent=64, W=16, P=7, batch=1, prompt_min=0, prompt_max=0,
                decode_steps=0, sm_scale=1 / math.sqrt(128))
    base.update(kw)
    return inputs.Workload(**base)


def test_compress_tiny_config_exact():
    """Llama-3.1-8B shape, 2048-token prompt, cache 4 + 252 + 256 (the smallest workload)."""
    wl = inputs.WORKLOADS["gqa_2k_tiny"]
    pre, cache, ocache = run_compress(wl, 2048, seed=0, slot=1)
    swaps = check_all(wl, pre, cache, ocache, slot=1, where="gqa_2k_tiny")
    assert swaps <= 2


@pytest.mark.parametrize("S", [2048 + 37, 1000, 777])
def test_compress_ragged_lengths(S):
    """Prompt lengths that are not a multiple of any tile (ragged tails)."""
    wl = inputs.WORKLOADS["gqa_2k_tiny"]
    pre, cache, ocache = run_compress(wl, S, seed=S)
    check_all(wl, pre, cache, ocache, where=f"S={S}")


@pytest.mark.parametrize("case", [
    dict(S=3),                                # shorter than the sinks
    dict(S=4),                                # exactly the sinks
    dict(S=50),                               # sinks + ring, no middle
    dict(S=68),                               # ring just full, no middle
    dict(S=128),                              # middle holds exactly K = 60
    dict(S=129),                              # one too many: scoring runs
    dict(S=300, K=0),                         # StreamingLLM only (no middle)
    dict(S=300, P=1),                         # no pooling
    dict(S=300, W=1),                         # one observation query
    dict(S=300, L_sink=0),                    # no sinks
    dict(S=513, W=64, L_recent=64, K=100),    # window fills the whole ring
])
def test_compress_edge_cases(case):
    case = dict(case)
    S = case.pop("S")
    wl = small_gqa(**case)
    pre, cache, ocache = run_compress(wl, S, seed=7 + S)
    check_all(wl, pre, cache, ocache, where=str(case))


@pytest.mark.parametrize("case", [
    dict(S=3000, n_q_heads=32, n_kv_heads=16),   # more heads than 12-CTA select clusters fit at once
    dict(S=3001, P=9),                           # pooling radius 4: the widest four-position path
    dict(S=2999, P=11),                          # pooling radius 5: one position per thread
])
def test_compress_select_paths(case):
    """The select kernel's cluster sizes and pooling paths, each against the oracle."""
    case = dict(case)
    S = case.pop("S")
    wl = small_gqa(**case)
    pre, cache, ocache = run_compress(wl, S, seed=S)
    check_all(wl, pre, cache, ocache, where=str(case))


def test_compress_select_slices_in_workspace():
    """A 400k-token prompt on one KV head: each select CTA's slice outgrows shared memory, so
    the pooled scores go through the workspace."""
    wl = small_gqa(n_q_heads=2, n_kv_heads=1, W=4, K=5000, L_recent=1024)
    pre, cache, ocache = run_compress(wl, 400_000, seed=11)
    check_all(wl, pre, cache, ocache, where="400k one head")


def test_compress_group_of_eight_and_strided_inputs():
    """G = 8 query heads per KV head; K and V passed as strided views."""
    wl = small_gqa(n_q_heads=16, n_kv_heads=2, W=8)
    pre, cache, ocache = run_compress(wl, 900, seed=5, strided=True)
    check_all(wl, pre, cache, ocache, where="G=8 strided")


def test_compress_mla_small():
    """DeepSeek MLA latent layout (576-wide key row, value = first 512 columns)."""
    wl = inputs.Workload("mla_small", 1, 128, 1, 576, 512, 4, 40, 64, 4, 5, 1, 0, 0, 0,
                         1 / math.sqrt(192))
    pre, cache, ocache = run_compress(wl, 700, seed=11)
    check_all(wl, pre, cache, ocache, where="mla small")


def test_compress_reuses_slot_cleanly():
    """A slot compressed twice holds only the second prompt (unused slots zeroed)."""
    wl = small_gqa()
    pre1 = inputs.gen_prefill(wl, 400, seed=1)
    pre2 = inputs.gen_prefill(wl, 30, seed=2)
    cache = snap.SnapCache(snap_cfg(wl), max_batch=1, max_prompt=400)
    cache.compress(0, pre1.K.cuda(), pre1.V.cuda(), pre1.Q.cuda())
    cache.compress(0, pre2.K.cuda(), pre2.V.cuda(), pre2.Q.cuda())
    torch.cuda.synchronize()
    ocache = oracle.compress(oracle_cfg(wl), pre2.K, pre2.V, pre2.Q)
    check_cache_rows(cache, 0, ocache, pre2.K, pre2.V, "reused slot")
    v = cache.k_cache()[0].float()
    pos = ocache.slot_positions()
    assert float(v[torch.from_numpy(pos < 0)].abs().sum()) == 0.0


def _window_lse(wl, K, Q):
    """Natural-log LSE of every observation row over its causal keys, [W][H_q] (float64)."""
    S = K.shape[0]
    Kd = K.double().cuda()
    Qd = Q.double().cuda()
    out = torch.empty((wl.W, wl.n_q_heads), dtype=torch.float64, device="cuda")
    for i in range(wl.n_q_heads):
        h = i // wl.G
        s = wl.sm_scale * (Qd[:, i, :] @ Kd[:, h, :].T)            # [W][S]
        pos = torch.arange(S - wl.W, S, device="cuda").view(-1, 1)
        s = s.masked_fill(torch.arange(S, device="cuda").view(1, -1) > pos, float("-inf"))
        out[:, i] = torch.logsumexp(s, dim=1)
    return out.float().contiguous()


@pytest.mark.parametrize("mla", [False, True])
def test_compress_with_supplied_lse_matches_oracle(mla):
    """snap_compress_lse: the prefill's row log-sum-exp replaces the row pass."""
    if mla:
        wl = inputs.Workload("mla_small", 1, 128, 1, 576, 512, 4, 40, 64, 4, 5, 1, 0, 0, 0,
                             1 / math.sqrt(192))
        S = 700
    else:
        wl = inputs.WORKLOADS["gqa_2k_tiny"]
        S = 2048 + 37
    pre = inputs.gen_prefill(wl, S, seed=31)
    cache = snap.SnapCache(snap_cfg(wl), max_batch=1, max_prompt=S)
    lse = _window_lse(wl, pre.K, pre.Q)
    cache.compress_lse(0, pre.K.cuda(), pre.V.cuda() if pre.V is not None else None, pre.Q.cuda(), lse)
    torch.cuda.synchronize()
    assert cache.check_device() == snap.SNAP_OK
    ocache = oracle.compress(oracle_cfg(wl), pre.K, pre.V, pre.Q, want_pool=True)
    check_all(wl, pre, cache, ocache, where="supplied lse")


@pytest.mark.parametrize("mla", [False, True])
def test_compress_stage_by_stage_equals_one_call(mla):
    """snap_compress_stages: the four stages run as four calls on one stream give the
    one-call result bit for bit (selection, every cache row, meta); a call without the
    write stage leaves the cache untouched."""
    if mla:
        wl = inputs.Workload("mla_small", 1, 128, 1, 576, 512, 4, 40, 64, 4, 5, 1, 0, 0, 0,
                             1 / math.sqrt(192))
        S = 900
    else:
        wl = small_gqa(K=124, L_recent=128)
        S = 3000
    pre = inputs.gen_prefill(wl, S, seed=41)
    K, V, Q = pre.K.cuda(), (pre.V.cuda() if pre.V is not None else None), pre.Q.cuda()
    one = snap.SnapCache(snap_cfg(wl), max_batch=1, max_prompt=S)
    one.compress(0, K, V, Q)
    staged = snap.SnapCache(snap_cfg(wl), max_batch=1, max_prompt=S)
    staged.compress_stages(0, K, V, Q, snap.STAGE_ROWS | snap.STAGE_COLUMNS | snap.STAGE_SELECT)
    torch.cuda.synchronize()
    assert float(staged.k_cache().float().abs().sum()) == 0.0      # nothing written yet
    for st in (snap.STAGE_ROWS, snap.STAGE_COLUMNS, snap.STAGE_SELECT, snap.STAGE_WRITE):
        staged.compress_stages(0, K, V, Q, st)
    torch.cuda.synchronize()
    assert one.check_device() == snap.SNAP_OK and staged.check_device() == snap.SNAP_OK
    assert torch.equal(one.selected(), staged.selected())
    assert torch.equal(one.k_cache(), staged.k_cache())
    if V is not None:
        assert torch.equal(one.v_cache(), staged.v_cache())
    assert torch.equal(one.meta(), staged.meta())
    ocache = oracle.compress(oracle_cfg(wl), pre.K, pre.V, pre.Q, want_pool=True)
    check_all(wl, pre, staged, ocache, where="staged")
