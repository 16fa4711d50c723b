"""GPU parity of snap_prefill_attn: causal prefill attention on the tensor cores, and
the log-sum-exp of the observation rows it hands to snap_compress_lse.

SnapStream episode companion page, headline figure "2-5% extra prefill latency": the
compression runs at prefill, next to the prefill's attention, whose per-row
log-sum-exp is the softmax denominator of the window rows.  The oracle is the plain
fp64 causal attention (pinned against torch SDPA).  Outputs are bf16, compared within
2e-2 max-abs and 5e-3 mean-abs; the log-sum-exp (fp32, natural log) within 1e-4.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from fixed_size_kv_gb300 import inputs, snap
from parity import MAX_ABS, MEAN_ABS, check_cache_rows, oracle_cfg, snap_cfg

pytestmark = pytest.mark.gpu

LSE_ABS = 1e-4


def gqa(Hq, Hkv, W=16, L_sink=4, K=60, L_recent=64):
    return inputs.Workload("prefill", 0, Hq, Hkv, 128, 128, L_sink, K, L_recent, W, 7, 1, 0, 0, 0,
                           1 / math.sqrt(128))


def run(wl, S, seed):
    pre = inputs.gen_prefill(wl, S, seed=seed)
    Q = inputs.gen_prompt_queries(wl, pre, seed=seed)
    cache = snap.SnapCache(snap_cfg(wl), max_batch=1, max_prompt=S)
    lse = torch.full((wl.W, wl.n_q_heads), float("nan"), dtype=torch.float32, device="cuda") if S >= wl.W else None
    O = cache.prefill_attn(Q.cuda(), pre.K.cuda(), pre.V.cuda(), lse_obs=lse)
    torch.cuda.synchronize()
    assert cache.check_device() == snap.SNAP_OK
    out, olse = oracle.prefill_attn(oracle_cfg(wl), Q, pre.K, pre.V)
    return pre, Q, cache, O, lse, out, olse


@pytest.mark.parametrize("S,Hq,Hkv", [(1, 8, 2), (77, 8, 2), (128, 8, 2), (300, 32, 8), (513, 8, 8),
                                      (700, 8, 2)])
def test_prefill_matches_oracle(S, Hq, Hkv):
    """Ragged lengths: shorter than one 128-row tile, exactly one, several with a ragged
    last tile, an odd number of tiles (the last pair holds one); G = 4 and G = 1."""
    wl = gqa(Hq, Hkv, W=16 if S >= 16 else 1)
    pre, Q, cache, O, lse, out, olse = run(wl, S, seed=S + Hq)
    d = np.abs(O.float().cpu().numpy().astype(np.float64) - out)
    assert d.max() <= MAX_ABS and d.mean() <= MEAN_ABS, (d.max(), d.mean())
    if lse is not None:
        dl = np.abs(lse.cpu().numpy().astype(np.float64) - olse[S - wl.W:])
        assert np.isfinite(lse.cpu().numpy()).all()
        assert dl.max() <= LSE_ABS, dl.max()


def test_prefill_lse_feeds_compression():
    """The prefill's log-sum-exp of the window rows replaces the compression's row pass
    (snap_compress_lse).  An LSE error e (natural log) scales every probability of its
    row by exp(-e), so each column score moves by at most a factor exp(max|e|); the
    selection may therefore differ from the oracle's only where the oracle's pooled
    scores of the swapped positions are within that factor (|e| <= 1e-4 here, checked),
    and every cache row is a bit copy of the prompt row the layout assigns."""
    wl = gqa(32, 8, W=32, L_sink=4, K=252, L_recent=256)
    S = 2048 + 37
    pre, Q, cache, O, lse, out, olse = run(wl, S, seed=61)
    err = float(np.abs(lse.cpu().numpy().astype(np.float64) - olse[S - wl.W:]).max())
    assert err <= LSE_ABS, err
    cache.compress_lse(0, pre.K.cuda(), pre.V.cuda(), pre.Q.cuda(), lse)
    torch.cuda.synchronize()
    assert cache.check_device() == snap.SNAP_OK
    ocache = oracle.compress(oracle_cfg(wl), pre.K, pre.V, pre.Q, want_pool=True)
    gsel = cache.selected()[0].cpu().numpy()
    rel = math.expm1(2 * err) + 1e-6          # both ends of a swap may move, plus the kernel's own rounding
    swaps = 0
    for h in range(wl.n_kv_heads):
        g, o = set(gsel[h].tolist()), set(ocache.sel[h].tolist())
        tau = float(min(ocache.pool[h][list(o)]))
        for j in g ^ o:
            assert abs(float(ocache.pool[h][j]) - tau) <= rel * abs(tau), (h, j, ocache.pool[h][j], tau)
        swaps += len(g ^ o) // 2
    check_cache_rows(cache, 0, ocache, pre.K, pre.V, "prefill-lse compression")
    assert swaps <= 4, swaps


def test_prefill_rejects_mla_and_short_prompts():
    """MLA has no prefill kernel here; with lse_obs the prompt must hold W rows."""
    mla = inputs.Workload("m", 1, 128, 1, 576, 512, 4, 40, 64, 4, 5, 1, 0, 0, 0, 1 / math.sqrt(192))
    cache = snap.SnapCache(snap_cfg(mla), max_batch=1, max_prompt=64)
    x = torch.zeros((64, 128, 576), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((64, 1, 576), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(snap.SnapError) as e:
        cache.prefill_attn(x, k, k)
    assert e.value.status == snap.SNAP_ERR_UNSUPPORTED
    wl = gqa(8, 2, W=16)
    c2 = snap.SnapCache(snap_cfg(wl), max_batch=1, max_prompt=8)
    q = torch.zeros((8, 8, 128), dtype=torch.bfloat16, device="cuda")
    kv = torch.zeros((8, 2, 128), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((16, 8), dtype=torch.float32, device="cuda")
    with pytest.raises(snap.SnapError) as e:
        c2.prefill_attn(q, kv, kv, lse_obs=lse)
    assert e.value.status == snap.SNAP_ERR_SHAPE
