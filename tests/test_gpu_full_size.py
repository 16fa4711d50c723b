"""Parity at the full workload sizes, in the launch configuration the benchmark uses.

The CUDA path runs each whole workload.  The oracle, which would take hours on every
head at 128k context, builds its own cache of one sampled KV head per sequence from
the same seeded prompt (every step of the method is independent across KV heads), on
several threads; that head's selection and its query heads' decode outputs are
compared with the GPU's.  Properties that hold at any size are checked on every
sequence: sinks and selected rows are bit copies of the prompt rows, the selection is
strictly ascending inside the middle, planted heavy hitters are kept, and the ring
holds exactly the last L_recent positions.

Workloads (Llama-3.1-8B GQA, 32/8 heads of 128; DeepSeek-R1 MLA latent, 128 heads over
512 + 64): prompts U[16k,32k] (batch 8, cache 4096), 128k (batch 16, cache 32768), the
mixed continuous batch's cache shape (4 + 4092 + 4096) with prompts drawn from
U[4k,128k], MLA at 128k (batch 8, cache 64 + 960 + 31744), and MLA compression at the
full observation height (128 heads x W = 64 = 8192 rows).
"""
from concurrent.futures import ThreadPoolExecutor

import pytest
import torch

import oracle
from fixed_size_kv_gb300 import inputs, snap
from parity import (check_outputs, check_selection, oracle_head_cache, oracle_workers, snap_cfg)

pytestmark = pytest.mark.gpu


def check_properties(wl, cache, slot, pre, K_tail=None):
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
        if n_mid:
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


def run_sampled(wl, lengths, seed, sample_heads, steps, check_steps, slot_of=None, mla_group=0):
    """Compresses every prompt on the GPU, builds the oracle's cache of the sampled KV
    heads of every sequence on a thread pool while the GPU works, compares selections,
    then decodes `steps` steps of the whole batch and compares the sampled heads'
    outputs at `check_steps`.  sample_heads(b) -> KV heads of sequence b."""
    B = len(lengths)
    slot_of = slot_of or list(range(B))
    cache = snap.SnapCache(snap_cfg(wl), max_batch=max(slot_of) + 1, max_prompt=max(lengths))
    workers = oracle_workers()
    # GQA: one oracle job per sampled head, run side by side; MLA: one job at a time,
    # each scoring its 128 query heads in groups of mla_group on every thread
    pool = ThreadPoolExecutor(1 if mla_group else workers)
    jobs = {}
    for b, S in enumerate(lengths):
        pre = inputs.gen_prefill(wl, S, seed=seed, seq=b, device="cuda")
        cache.compress(slot_of[b], pre.K, pre.V, pre.Q)
        heads = sample_heads(b)
        Kc = pre.K[:, heads].cpu()
        Vc = pre.V[:, heads].cpu() if pre.V is not None else None
        Qc = torch.cat([pre.Q[:, h * wl.G:(h + 1) * wl.G] for h in heads], dim=1).cpu()
        for i, h in enumerate(heads):
            jobs[(b, h)] = pool.submit(oracle_head_cache, wl.replace(n_kv_heads=len(heads),
                                                                    n_q_heads=len(heads) * wl.G),
                                       Kc, Vc, Qc, i, workers if mla_group else 1, mla_group)
        torch.cuda.synchronize()
        check_properties(wl, cache, slot_of[b], pre)
        del pre
    assert cache.check_device() == snap.SNAP_OK
    ocs = {key: f.result() for key, f in jobs.items()}
    pool.shutdown()
    sel = cache.selected().cpu().numpy()
    meta = cache.meta().cpu().tolist()
    n_swaps = 0
    for (b, h), oc in ocs.items():
        om = oc.meta
        assert tuple(meta[slot_of[b]][:5]) == (om.S, om.T, om.R0, om.n_sink, om.n_mid), (b, meta[slot_of[b]], om)
        n_mid = om.n_mid
        n_swaps += check_selection(sel[slot_of[b], h, :n_mid], oc.sel[0, :n_mid], oc.pool[0],
                                   f"{wl.name} seq {b} head {h}")
    slots = torch.tensor(slot_of, dtype=torch.int32, device="cuda")
    G = wl.G
    for t in range(steps):
        tok = inputs.gen_decode(wl, B, step=t, seed=seed, device="cuda")
        cache.decode_append(slots, tok.k, tok.v)
        out = cache.decode_attn(slots, tok.q)
        kk, vv, qq = tok.k.cpu(), tok.v.cpu() if tok.v is not None else None, tok.q.cpu()
        for (b, h), oc in ocs.items():
            oracle.append(oc, kk[b, h:h + 1], vv[b, h:h + 1] if vv is not None else None)
        if t in check_steps:
            torch.cuda.synchronize()
            o = out.cpu()
            for (b, h), oc in ocs.items():
                check_outputs(o[b, h * G:(h + 1) * G], oracle.decode_attn(oc, qq[b, h * G:(h + 1) * G]),
                              f"{wl.name} step {t} seq {b} head {h}")
    torch.cuda.synchronize()
    assert cache.check_device() == snap.SNAP_OK
    return cache, n_swaps


@pytest.mark.parametrize("name", ["gqa_16k32k_b8", "gqa_128k_b16"])
def test_gqa_full_size(name):
    """Every sequence: one KV head (rotating over the 8) checked against the oracle's
    own cache of it, selection and decode outputs at the first and last checked steps."""
    wl = inputs.WORKLOADS[name]
    lengths = inputs.prompt_lengths(wl, 0)
    steps = 24 if name == "gqa_128k_b16" else 40
    run_sampled(wl, lengths, 0, lambda b: [b % wl.n_kv_heads], steps, (0, steps // 2, steps - 1))


def test_mixed_cache_shape_prompts_4k_to_128k():
    """The 64-slot mixed batch's cache (4 + 4092 + 4096) with prompts drawn from its
    U[4k,128k] length distribution, one of them at least 64k; the sequences sit in
    scattered slots at different ring offsets; two KV heads of each are checked."""
    wl = inputs.WORKLOADS["gqa_mixed_b64"]
    drawn = inputs.prompt_lengths(wl, 0)
    long_one = next(S for S in drawn if S >= 65536)
    short = [S for S in drawn if S < 65536][:3]
    lengths = [short[0], long_one, short[1], short[2]]
    run_sampled(wl, lengths, 0, lambda b: [b % wl.n_kv_heads, (b + 5) % wl.n_kv_heads], 40, (0, 39),
                slot_of=[41, 3, 17, 60])


def test_mla_compression_full_observation_height():
    """DeepSeek-R1 MLA shape at the full observation height: 128 query heads x W = 64
    window rows = 8192 rows per KV head.  At S = 6144 the row pass splits the keys in two
    (64 row tiles x 2 key splits on a 152-SM GPU) and the column pass streams all 32
    blocks of 256 rows.  L_recent is 1024 (the workload's 31744 would leave no middle to
    select at this length).  Selection and decode outputs against the oracle."""
    wl = inputs.WORKLOADS["mla_128k_b8"].replace(L_recent=1024, name="mla_rows8192")
    run_sampled(wl, [6144, 5000], 3, lambda b: [0], 6, (0, 5), mla_group=8)


def test_mla_full_size():
    """8 x 128k MLA (cache 64 + 960 + 31744): sequence 0's selection and decode outputs
    against the oracle's own cache (scored on every host thread); layout properties of
    every sequence."""
    wl = inputs.WORKLOADS["mla_128k_b8"]
    S = wl.prompt_max
    B = wl.batch
    cache = snap.SnapCache(snap_cfg(wl), max_batch=B, max_prompt=S)
    keep = None
    job = None
    pool = ThreadPoolExecutor(1)
    for b in range(B):
        pre = inputs.gen_prefill(wl, S, seed=0, seq=b, device="cuda")
        cache.compress(b, pre.K, None, pre.Q)
        if b == 0:
            keep = inputs.Prefill(pre.K.cpu(), None, pre.Q.cpu(), pre.heavy.cpu())
            job = pool.submit(oracle_head_cache, wl, keep.K, None, keep.Q, 0, oracle_workers(), 8)
        torch.cuda.synchronize()
        check_properties(wl, cache, b, pre)
        del pre
    assert cache.check_device() == snap.SNAP_OK
    oc = job.result()
    pool.shutdown()
    n_mid = oc.meta.n_mid
    check_selection(cache.selected()[0, 0, :n_mid].cpu().numpy(), oc.sel[0, :n_mid], oc.pool[0], "mla 128k seq 0")
    slots = torch.arange(B, dtype=torch.int32, device="cuda")
    ktail = []
    for t in range(8):
        tok = inputs.gen_decode(wl, B, step=t, seed=0, device="cuda")
        cache.decode_append(slots, tok.k, None)
        out = cache.decode_attn(slots, tok.q)
        ktail.append(tok.k[0:1].cpu())
        oracle.append(oc, tok.k[0].cpu())
        if t in (0, 7):
            torch.cuda.synchronize()
            check_outputs(out[0], oracle.decode_attn(oc, tok.q[0].cpu()), f"mla step {t}")
    torch.cuda.synchronize()
    check_properties(wl, cache, 0, keep, K_tail=torch.cat(ktail))
