"""GPU parity of snap_decode_append + snap_decode_attn against the CPU oracle.

SnapStream episode companion page, "Ring Buffer vs. Naive Slicing": decode only
rotates the recent window, scattering each new token into a fixed ring index;
"Prefill / Decode Pipeline": decode streams the cache once per token.  Cases
cover a continuous batch whose sequences sit at different ring offsets, partly
filled caches, permuted slots, the full-KV baseline and the MLA latent layout.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from fixed_size_kv_gb300 import inputs, snap
from parity import check_cache_rows, check_outputs, oracle_cfg, snap_cfg

pytestmark = pytest.mark.gpu


class Batch:
    """Runs the GPU cache and the oracle caches side by side."""

    def __init__(self, wl, lengths, slots, seed, max_batch=None):
        self.wl = wl
        self.slots = list(slots)
        self.cache = snap.SnapCache(snap_cfg(wl), max_batch=max_batch or (max(slots) + 1),
                                    max_prompt=max(lengths))
        self.ocaches, self.K, self.V = [], [], []
        for i, (S, slot) in enumerate(zip(lengths, slots)):
            pre = inputs.gen_prefill(wl, S, seed=seed, seq=i)
            self.cache.compress(slot, pre.K.cuda(), pre.V.cuda() if pre.V is not None else None,
                                pre.Q.cuda())
            self.ocaches.append(oracle.compress(oracle_cfg(wl), pre.K, pre.V, pre.Q))
            self.K.append(pre.K)
            self.V.append(pre.V)
        torch.cuda.synchronize()
        self.dslots = torch.tensor(self.slots, dtype=torch.int32, device="cuda")
        self.seed = seed

    def step(self, t, append=True, fused=False):
        wl, n = self.wl, len(self.slots)
        tok = inputs.gen_decode(wl, n, step=t, seed=self.seed)
        if fused:
            out = self.cache.decode_step(self.dslots, tok.q.cuda(), tok.k.cuda(),
                                         tok.v.cuda() if tok.v is not None else None)
        else:
            if append:
                self.cache.decode_append(self.dslots, tok.k.cuda(), tok.v.cuda() if tok.v is not None else None)
            out = self.cache.decode_attn(self.dslots, tok.q.cuda())
        torch.cuda.synchronize()
        assert self.cache.check_device() == snap.SNAP_OK
        for i in range(n):
            if append:
                oracle.append(self.ocaches[i], tok.k[i], tok.v[i] if tok.v is not None else None)
                self.K[i] = torch.cat([self.K[i], tok.k[i:i + 1]])
                if tok.v is not None:
                    self.V[i] = torch.cat([self.V[i], tok.v[i:i + 1]])
            check_outputs(out[i], oracle.decode_attn(self.ocaches[i], tok.q[i]), f"step {t} seq {i}")
        return out

    def check_rows(self):
        for i, slot in enumerate(self.slots):
            check_cache_rows(self.cache, slot, self.ocaches[i], self.K[i], self.V[i], f"seq {i}")


def test_decode_tiny_config_64_steps():
    """The 2048-token workload: 64 decode steps, every output and the final ring checked."""
    wl = inputs.WORKLOADS["gqa_2k_tiny"]
    b = Batch(wl, [2048], [0], seed=3)
    b.step(0, append=False)  # attention right after compression
    for t in range(1, 65):
        b.step(t)
    b.check_rows()


def test_decode_continuous_batch_ring_offsets():
    """Sequences of different lengths (different ring offsets, some partly filled),
    in permuted slots; several steps wrap the ring of the longest."""
    wl = inputs.Workload("cb", 0, 32, 8, 128, 128, 4, 60, 64, 16, 7, 5, 0, 0, 0, 1 / math.sqrt(128))
    lengths = [300, 37, 129, 2, 1000]
    b = Batch(wl, lengths, slots=[3, 0, 6, 1, 4], seed=9, max_batch=8)
    for t in range(80):
        b.step(t)
    b.check_rows()


def test_fused_decode_step_continuous_batch():
    """snap_decode_step (for GQA one kernel: ring append, attention, split merge) over a
    continuous batch at different ring offsets, with splits (cache 4096) and without
    (cache 128); every output against the oracle and the ring bit-exact afterwards."""
    for C_parts, lengths in (((4, 2044, 2048), [6000, 300, 2100, 4500]), ((4, 60, 64), [300, 37, 129, 2])):
        wl = inputs.Workload("fused", 0, 32, 8, 128, 128, *C_parts, 16, 7, 4, 0, 0, 0, 1 / math.sqrt(128))
        b = Batch(wl, lengths, slots=[2, 0, 3, 1], seed=17, max_batch=4)
        for t in range(70):
            b.step(t, fused=True)
        b.check_rows()


def test_decode_subset_of_slots():
    """Only some sequences of the cache decode in a step; the others do not move."""
    wl = inputs.Workload("cb", 0, 32, 8, 128, 128, 4, 60, 64, 16, 7, 5, 0, 0, 0, 1 / math.sqrt(128))
    b = Batch(wl, [300, 200, 150], slots=[0, 1, 2], seed=4)
    T_before = b.cache.meta()[:, 1].cpu().tolist()
    sub = torch.tensor([2, 0], dtype=torch.int32, device="cuda")
    tok = inputs.gen_decode(wl, 2, step=0, seed=1)
    b.cache.decode_append(sub, tok.k.cuda(), tok.v.cuda())
    out = b.cache.decode_attn(sub, tok.q.cuda())
    torch.cuda.synchronize()
    T_after = b.cache.meta()[:, 1].cpu().tolist()
    assert T_after == [T_before[0] + 1, T_before[1], T_before[2] + 1]
    for j, seq in enumerate([2, 0]):
        oracle.append(b.ocaches[seq], tok.k[j], tok.v[j])
        check_outputs(out[j], oracle.decode_attn(b.ocaches[seq], tok.q[j]), f"subset {seq}")


def test_decode_attn_is_bitwise_repeatable():
    """Splits are merged in a fixed order by whichever CTA finishes last: repeated calls
    on the same cache give bit-identical outputs (a plan with three or more splits)."""
    wl = inputs.Workload("rep", 0, 32, 8, 128, 128, 4, 508, 512, 16, 7, 6, 0, 0, 0, 1 / math.sqrt(128))
    b = Batch(wl, [5000, 3000, 700, 4096, 1200, 2500], slots=list(range(6)), seed=31)
    assert b.cache.decode_attn_plan(6)[0] >= 3
    q = inputs.gen_decode(wl, 6, step=0, seed=31).q.cuda()
    outs = [b.cache.decode_attn(b.dslots, q) for _ in range(5)]
    torch.cuda.synchronize()
    for o in outs[1:]:
        assert torch.equal(o, outs[0])


def test_decode_eight_split_cluster():
    """Two sequences on a 4096-slot cache: the plan has 5-8 splits, so each (sequence, KV
    head) is one cluster of that many CTAs merging through distributed shared memory.
    Fused steps against the oracle; repeated calls bitwise equal."""
    wl = inputs.Workload("c8", 0, 32, 8, 128, 128, 4, 2044, 2048, 16, 7, 2, 0, 0, 0, 1 / math.sqrt(128))
    b = Batch(wl, [6000, 3500], [0, 1], seed=41)
    assert 5 <= b.cache.decode_attn_plan(2)[0] <= 8
    for t in range(3):
        b.step(t, fused=True)
    q = inputs.gen_decode(wl, 2, step=9, seed=41).q.cuda()
    outs = [b.cache.decode_attn(b.dslots, q) for _ in range(3)]
    torch.cuda.synchronize()
    assert all(torch.equal(o, outs[0]) for o in outs[1:])
    b.check_rows()


def test_decode_splits_beyond_a_cluster():
    """One sequence on a 32768-slot cache: the plan has more than eight splits, so the
    splits merge through the global partials (the last CTA to finish folds them), not
    within a cluster.  Fused steps against the oracle."""
    wl = inputs.Workload("wide", 0, 32, 8, 128, 128, 4, 16380, 16384, 16, 7, 1, 0, 0, 0, 1 / math.sqrt(128))
    b = Batch(wl, [20000], [0], seed=37)
    assert b.cache.decode_attn_plan(1)[0] > 8
    for t in range(4):
        b.step(t, fused=True)
    b.check_rows()


def test_decode_full_kv_baseline_equals_full_attention():
    """A cache with L_sink = 0, K = 0 and a ring as long as the whole sequence is the
    uncompressed baseline: it must equal attention over every token (torch SDPA)."""
    S, steps = 3000, 5
    wl = inputs.Workload("full", 0, 32, 8, 128, 128, 0, 0, S + steps, 16, 7, 1, 0, 0, 0,
                         1 / math.sqrt(128))
    b = Batch(wl, [S], [0], seed=5)
    for t in range(steps):
        out = b.step(t)
        q = inputs.gen_decode(wl, 1, step=t, seed=b.seed).q[0].float().cuda()
        k = b.K[0].float().cuda().permute(1, 0, 2).repeat_interleave(4, 0)
        v = b.V[0].float().cuda().permute(1, 0, 2).repeat_interleave(4, 0)
        ref = torch.nn.functional.scaled_dot_product_attention(q.unsqueeze(1), k, v, scale=wl.sm_scale)
        assert (out[0].float() - ref.squeeze(1)).abs().max().item() < 2e-2


def test_decode_compressed_equals_full_when_cache_covers():
    """L_sink + K + L_recent >= S with no eviction yet: compressed attention equals
    attention over the whole prompt."""
    S = 500
    wl = inputs.Workload("cover", 0, 32, 8, 128, 128, 4, 100, 512, 16, 7, 1, 0, 0, 0,
                         1 / math.sqrt(128))
    b = Batch(wl, [S], [0], seed=6)
    out = b.step(0, append=False)
    q = inputs.gen_decode(wl, 1, step=0, seed=b.seed).q[0].float().cuda()
    k = b.K[0].float().cuda().permute(1, 0, 2).repeat_interleave(4, 0)
    v = b.V[0].float().cuda().permute(1, 0, 2).repeat_interleave(4, 0)
    ref = torch.nn.functional.scaled_dot_product_attention(q.unsqueeze(1), k, v, scale=wl.sm_scale)
    assert (out[0].float() - ref.squeeze(1)).abs().max().item() < 2e-2


def test_decode_mla_small():
    """MLA latent layout: 576-wide keys, values = first 512 columns, 128 query heads;
    ragged cache (C = 4 + 40 + 100, not a multiple of the 64-key tile), one sequence
    shorter than the cache, enough steps to wrap the ring."""
    wl = inputs.Workload("mla_small", 1, 128, 1, 576, 512, 4, 40, 100, 4, 5, 1, 0, 0, 0,
                         1 / math.sqrt(192))
    b = Batch(wl, [700, 90], [1, 0], seed=12)
    for t in range(110):
        b.step(t)
    b.check_rows()


def test_decode_mla_long_cache_splits():
    """MLA over a 4096-slot cache (many 64-key tiles, several splits, merge)."""
    wl = inputs.Workload("mla_mid", 1, 128, 1, 576, 512, 64, 960, 3072, 8, 7, 1, 0, 0, 0,
                         1 / math.sqrt(192))
    b = Batch(wl, [6000, 2500, 4100], [0, 1, 2], seed=13)
    for t in range(3):
        b.step(t)


def test_decode_out_of_range_slot_reports_without_fault():
    """A slot index past max_batch is rejected by the kernels through the status word
    (the call itself returns OK: the index lives on the device)."""
    wl = inputs.Workload("cb", 0, 32, 8, 128, 128, 4, 60, 64, 16, 7, 1, 0, 0, 0, 1 / math.sqrt(128))
    b = Batch(wl, [100], [0], seed=1, max_batch=2)
    bad = torch.tensor([5], dtype=torch.int32, device="cuda")
    tok = inputs.gen_decode(wl, 1, step=0, seed=1)
    b.cache.decode_append(bad, tok.k.cuda(), tok.v.cuda())
    assert b.cache.check_device() == snap.SNAP_ERR_DEVICE_CHECK
    out = b.cache.decode_attn(bad, tok.q.cuda())
    assert b.cache.check_device() == snap.SNAP_ERR_DEVICE_CHECK
    assert float(out.float().abs().sum()) == 0.0
    assert b.cache.check_device() == snap.SNAP_OK  # cleared by the previous read


@pytest.mark.parametrize("mla", [False, True])
def test_decode_plan_covers_every_tile(mla):
    """snap_decode_attn_plan: splits x tiles per split covers the cache, every split is
    non-empty, and a wave holds at least one CTA."""
    if mla:
        wl = inputs.Workload("mla_mid", 1, 128, 1, 576, 512, 64, 960, 3072, 8, 7, 1, 0, 0, 0, 1 / math.sqrt(192))
    else:
        wl = inputs.Workload("cb", 0, 32, 8, 128, 128, 4, 2044, 2048, 16, 7, 5, 0, 0, 0, 1 / math.sqrt(128))
    cache = snap.SnapCache(snap_cfg(wl), max_batch=8, max_prompt=64)
    tiles = -(-cache.C // (64 if mla else 32))    # key tile of the MLA / GQA kernel
    for n in (1, 3, 8):
        splits, per, wave = cache.decode_attn_plan(n)
        assert 1 <= splits <= 32 and wave >= 1
        assert splits * per >= tiles and (splits - 1) * per < tiles


def test_graph_replayed_decode_steps_match_oracle():
    """The benchmark's launch form: snap_decode_step (append, attention with
    programmatic dependent launch, merge) for several steps captured once as a CUDA
    graph and replayed; every step's output against the oracle."""
    wl = inputs.Workload("graph", 0, 32, 8, 128, 128, 4, 2044, 2048, 16, 7, 4, 0, 0, 0, 1 / math.sqrt(128))
    b = Batch(wl, [6000, 300, 2100, 4500], slots=[0, 1, 2, 3], seed=23, max_batch=4)
    b.step(0, fused=True)            # one eager step first (one-time launch set-up), as the bench warms up
    steps = 6
    toks = [inputs.gen_decode(wl, 4, step=1 + t, seed=23) for t in range(steps)]
    q = [t.q.cuda() for t in toks]
    k = [t.k.cuda() for t in toks]
    v = [t.v.cuda() for t in toks]
    outs = [torch.empty((4, wl.n_q_heads, wl.d_v), dtype=torch.float32, device="cuda") for _ in range(steps)]
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for t in range(steps):
            b.cache.decode_step(b.dslots, q[t], k[t], v[t], out=outs[t], stream=stream)
    with torch.cuda.stream(stream):
        graph.replay()
    stream.synchronize()
    assert b.cache.check_device() == snap.SNAP_OK
    for t in range(steps):
        for i in range(4):
            oracle.append(b.ocaches[i], toks[t].k[i], toks[t].v[i])
            check_outputs(outs[t][i], oracle.decode_attn(b.ocaches[i], toks[t].q[i]), f"graph step {t} seq {i}")


def test_compress_on_second_stream_while_decoding():
    """The mixed workload's lifecycle: a new request is compressed into a free slot on a
    second stream while the other slots keep decoding on the first; afterwards all of
    them decode together.  Every output against the oracle."""
    wl = inputs.Workload("mix", 0, 32, 8, 128, 128, 4, 1020, 1024, 16, 7, 4, 0, 0, 0, 1 / math.sqrt(128))
    b = Batch(wl, [3000, 1500, 2500], slots=[0, 1, 2], seed=29, max_batch=4)
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    sa.wait_stream(torch.cuda.current_stream())
    sb.wait_stream(torch.cuda.current_stream())
    new = inputs.gen_prefill(wl, 2800, seed=29, seq=9)
    nK, nV, nQ = new.K.cuda(), new.V.cuda(), new.Q.cuda()
    torch.cuda.synchronize()
    b.cache.compress(3, nK, nV, nQ, stream=sb)                 # the arrival, on stream B
    for t in range(8):                                         # the others decode on stream A
        tok = inputs.gen_decode(wl, 3, step=t, seed=29)
        out = b.cache.decode_step(b.dslots, tok.q.cuda(), tok.k.cuda(), tok.v.cuda(), stream=sa)
        sa.synchronize()
        for i in range(3):
            oracle.append(b.ocaches[i], tok.k[i], tok.v[i])
            check_outputs(out[i], oracle.decode_attn(b.ocaches[i], tok.q[i]), f"while compressing, step {t} seq {i}")
    sb.synchronize()
    assert b.cache.check_device() == snap.SNAP_OK
    onew = oracle.compress(oracle_cfg(wl), new.K, new.V, new.Q)
    slots = torch.tensor([0, 1, 2, 3], dtype=torch.int32, device="cuda")
    ocs = b.ocaches + [onew]
    for t in range(8, 12):                                     # the arrival has joined the batch
        tok = inputs.gen_decode(wl, 4, step=t, seed=29)
        out = b.cache.decode_step(slots, tok.q.cuda(), tok.k.cuda(), tok.v.cuda())
        torch.cuda.synchronize()
        for i in range(4):
            oracle.append(ocs[i], tok.k[i], tok.v[i])
            check_outputs(out[i], oracle.decode_attn(ocs[i], tok.q[i]), f"joined, step {t} seq {i}")
    assert b.cache.check_device() == snap.SNAP_OK


def test_fused_decode_step_mla():
    """The MLA layout's snap_decode_step (append fused into the attention kernel, merge
    kernel after) over a ragged cache whose ring wraps, against the oracle."""
    wl = inputs.Workload("mla_fused", 1, 128, 1, 576, 512, 4, 40, 100, 4, 5, 1, 0, 0, 0,
                         1 / math.sqrt(192))
    b = Batch(wl, [700, 90, 260], [2, 0, 1], seed=15, max_batch=3)
    for t in range(105):
        b.step(t, fused=True)
    b.check_rows()


def _kernels_of(fn):
    """Names of the GPU kernels one call launches (torch profiler)."""
    from torch.profiler import ProfilerActivity, profile
    torch.cuda.synchronize()
    with profile(activities=[ProfilerActivity.CUDA]) as prof:
        fn()
        torch.cuda.synchronize()
    names = []
    for e in prof.events():
        dt = str(getattr(e, "device_type", ""))
        if "CUDA" in dt and ("kernel" in e.name or "decode" in e.name or "append" in e.name):
            names.append(e.name)
    return names


@pytest.mark.parametrize("C_parts,lengths", [((4, 2044, 2048), [6000, 300, 2100, 4500]),
                                             ((4, 16380, 16384), [20000, 9000])])
def test_gqa_decode_step_is_one_launch(C_parts, lengths):
    """A GQA decode step is one kernel launch whatever the split plan (the ring append
    and the split merge run inside the attention kernel)."""
    wl = inputs.Workload("one", 0, 32, 8, 128, 128, *C_parts, 16, 7, len(lengths), 0, 0, 0, 1 / math.sqrt(128))
    b = Batch(wl, lengths, slots=list(range(len(lengths))), seed=19)
    splits = b.cache.decode_attn_plan(len(lengths))[0]
    tok = inputs.gen_decode(wl, len(lengths), step=0, seed=19)
    q, k, v = tok.q.cuda(), tok.k.cuda(), tok.v.cuda()
    b.cache.decode_step(b.dslots, q, k, v)         # first call: one-time set-up outside the profile
    _kernels_of(lambda: torch.zeros(1, device="cuda").add_(1))   # the profiler's own first-use set-up
    names = _kernels_of(lambda: [b.cache.decode_step(b.dslots, q, k, v) for _ in range(3)])
    if not names:
        pytest.skip("the profiler reported no kernels on this box")
    assert len(names) == 3 and all("gqa_decode_kernel" in n for n in names), (splits, names)
