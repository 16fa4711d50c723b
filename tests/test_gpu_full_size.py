"""Parity at the full workload sizes, in the launch configuration the benchmark uses.

The CUDA path runs the whole workload; the oracle, which would take hours at 128k
context, checks sampled outputs it can compute one by one (one KV head's
selection, one sequence's decode outputs fed the GPU's own cache) and the
properties that hold at any size (the ring holds exactly the last L_recent
positions, sinks and selected rows are bit copies of the prompt rows, the
selection is strictly ascending inside the middle, planted heavy hitters are
kept).  Workloads: Llama-3.1-8B GQA with prompts U[16k,32k] (batch 8) and at
128k (batch 16); DeepSeek-R1 MLA latent at 128k (batch 8).
"""
import numpy as np
import pytest
import torch

import oracle
from fixed_size_kv_gb300 import inputs, snap
from parity import (bits, check_outputs, check_selection, oracle_cache_from_gpu, oracle_cfg,
                    snap_cfg)

pytestmark = pytest.mark.gpu


def oracle_head_selection(wl, pre, h):
    """The oracle's selection and pooled scores for KV head h alone (a one-head problem
    with the same rows: KV head h and its G query heads)."""
    G = wl.G
    one = wl.replace(n_q_heads=G, n_kv_heads=1)
    ocfg = oracle_cfg(one)
    K1 = pre.K[:, h:h + 1].contiguous()
    Q1 = pre.Q[:, h * G:(h + 1) * G].contiguous()
    S = K1.shape[0]
    _, col = oracle.window_scores(ocfg, K1, Q1)
    pooled = oracle.maxpool(col[0, :S - wl.W], wl.P)
    m = oracle.plan(ocfg, S)
    sel = oracle.select(pooled, m.n_sink, m.R0, wl.K)
    return sel, pooled


def check_properties(wl, cache, slot, pre, K_tail=None, V_tail=None):
    """Layout properties of one sequence's cache after compression (+ appended tail)."""
    meta = cache.meta()[slot].cpu().tolist()
    S, T, R0, n_sink, n_mid = meta[:5]
    assert S == pre.K.shape[0]
    kc = cache.k_cache()[slot]
    vc = cache.v_cache()[slot] if cache.v_cache() is not None else None
    sel = cache.selected()[slot].cpu()
    Kd = pre.K.cuda()
    Vd = pre.V.cuda() if pre.V is not None else None
    kept_total, heavy_total = 0, 0
    for h in range(wl.n_kv_heads):
        s = sel[h, :n_mid].long()
        assert bool((s[1:] > s[:-1]).all()), "selection not ascending"
        assert int(s.min()) >= wl.L_sink and int(s.max()) < R0
        assert torch.equal(kc[h, :n_sink], Kd[:n_sink, h])
        assert torch.equal(kc[h, wl.L_sink:wl.L_sink + n_mid], Kd[s.cuda(), h])
        if vc is not None:
            assert torch.equal(vc[h, wl.L_sink:wl.L_sink + n_mid], Vd[s.cuda(), h])
        # planted heavy hitters: pooling gives each one's score to its P - 1 neighbours,
        # so about K / P of them fit; most of those must be kept
        hh = pre.heavy[h].cpu()
        hh = hh[(hh >= wl.L_sink + wl.P) & (hh < R0 - wl.P)]
        kept = set(s.tolist())
        kept_total += sum(int(p) in kept for p in hh.tolist())
        heavy_total += min(len(hh), n_mid // wl.P)
    assert kept_total >= 0.8 * heavy_total, (kept_total, heavy_total)
    # ring: positions [max(R0, T - L_recent), T) at slot L_sink + K + p mod L_recent
    lo = max(R0, T - wl.L_recent)
    allK = Kd if K_tail is None else torch.cat([Kd, K_tail.cuda()])
    pos = torch.arange(lo, T, device="cuda")
    ring_slots = wl.L_sink + wl.K + pos % wl.L_recent
    for h in range(wl.n_kv_heads):
        assert torch.equal(kc[h, ring_slots], allK[pos, h])


@pytest.mark.parametrize("name", ["gqa_16k32k_b8", "gqa_128k_b16"])
def test_gqa_full_size(name):
    wl = inputs.WORKLOADS[name]
    seed = 0
    lengths = inputs.prompt_lengths(wl, seed)
    cache = snap.SnapCache(snap_cfg(wl), max_batch=wl.batch, max_prompt=max(lengths))
    sample_seq = wl.batch - 1
    sample = None
    for b, S in enumerate(lengths):
        pre = inputs.gen_prefill(wl, S, seed=seed, seq=b, device="cuda")
        cache.compress(b, pre.K, pre.V, pre.Q)
        if b == sample_seq:
            sample = inputs.Prefill(pre.K.cpu(), pre.V.cpu(), pre.Q.cpu(), pre.heavy.cpu())
        else:
            torch.cuda.synchronize()
            check_properties(wl, cache, b, pre)
        del pre
    torch.cuda.synchronize()
    assert cache.check_device() == snap.SNAP_OK
    # one KV head's selection against the oracle
    h = 3
    osel, opool = oracle_head_selection(wl, sample, h)
    gsel = cache.selected()[sample_seq, h].cpu().numpy()
    check_selection(gsel, osel, opool, f"{name} seq {sample_seq} head {h}")
    # decode steps for the whole batch; sampled outputs against the oracle fed the GPU cache
    slots = torch.arange(wl.batch, dtype=torch.int32, device="cuda")
    steps = 24 if name == "gqa_128k_b16" else 40
    ktail = []
    for t in range(steps):
        tok = inputs.gen_decode(wl, wl.batch, step=t, seed=seed, device="cuda")
        cache.decode_append(slots, tok.k, tok.v)
        out = cache.decode_attn(slots, tok.q)
        ktail.append(tok.k[sample_seq:sample_seq + 1].cpu())
        if t in (0, steps - 1):
            torch.cuda.synchronize()
            oc = oracle_cache_from_gpu(cache, sample_seq, oracle_cfg(wl))
            check_outputs(out[sample_seq], oracle.decode_attn(oc, tok.q[sample_seq].cpu()),
                          f"{name} step {t}")
    torch.cuda.synchronize()
    assert cache.check_device() == snap.SNAP_OK
    check_properties(wl, cache, sample_seq, sample, K_tail=torch.cat(ktail))


def test_mla_full_size():
    wl = inputs.WORKLOADS["mla_128k_b8"]
    seed = 0
    S = wl.prompt_max
    cache = snap.SnapCache(snap_cfg(wl), max_batch=wl.batch, max_prompt=S)
    keep = None
    for b in range(wl.batch):
        pre = inputs.gen_prefill(wl, S, seed=seed, seq=b, device="cuda")
        cache.compress(b, pre.K, None, pre.Q)
        torch.cuda.synchronize()
        check_properties(wl, cache, b, pre)
        if b == 0:
            keep = inputs.Prefill(pre.K.cpu(), None, pre.Q.cpu(), pre.heavy.cpu())
        del pre
    assert cache.check_device() == snap.SNAP_OK
    slots = torch.arange(wl.batch, dtype=torch.int32, device="cuda")
    ktail = []
    for t in range(8):
        tok = inputs.gen_decode(wl, wl.batch, step=t, seed=seed, device="cuda")
        cache.decode_append(slots, tok.k, None)
        out = cache.decode_attn(slots, tok.q)
        ktail.append(tok.k[0:1].cpu())
        if t == 7:
            torch.cuda.synchronize()
            oc = oracle_cache_from_gpu(cache, 0, oracle_cfg(wl))
            check_outputs(out[0], oracle.decode_attn(oc, tok.q[0].cpu()), "mla step 7")
    torch.cuda.synchronize()
    check_properties(wl, cache, 0, keep, K_tail=torch.cat(ktail))
