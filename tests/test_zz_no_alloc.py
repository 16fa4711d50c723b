"""snap_decode_attn_noalloc: decode attention for callers that cannot allocate.

Some callers (a real-time thread that must not block in the allocator, a stream
under graph capture, a runtime that owns every device allocation) cannot provide the
device workspace that snap_decode_attn needs for its split-KV partial results.  The no-alloc entry point
keeps those partials in a fixed scratch array inside the library.  These tests call
it through the C ABI and check it against the workspace entry point on the same
cache, on two calls in a row (the scratch keeps the previous call's contents, which
must not leak into the next result), and check that an oversized batch is refused.

This file is collected last on purpose; it also passes alone in a fresh process.
"""
import math

import pytest
import torch

from fixed_size_kv_gb300 import inputs, snap

pytestmark = pytest.mark.gpu

def _cfg(wl):
    return snap.make_config(**wl.config_kwargs())


def _batch(wl, lengths, seed):
    snap.load(build_if_missing=True)
    cache = snap.SnapCache(_cfg(wl), max_batch=len(lengths), max_prompt=max(lengths))
    for i, S in enumerate(lengths):
        pre = inputs.gen_prefill(wl, S, seed=seed, seq=i, device="cuda")
        cache.compress(i, pre.K, pre.V, pre.Q)
    return cache


@pytest.mark.parametrize("layout", ["gqa", "mla"])
def test_noalloc_matches_workspace_entry_point_twice(layout):
    if layout == "gqa":
        wl = inputs.Workload("na", 0, 32, 8, 128, 128, 4, 508, 512, 32, 7, 6, 0, 0, 0, 1 / math.sqrt(128))
        lengths = [5000, 3000, 700, 4096, 1200, 2500]
    else:
        wl = inputs.Workload("na_mla", 1, 128, 1, 576, 512, 16, 240, 768, 16, 7, 3, 0, 0, 0,
                             1 / math.sqrt(192))
        lengths = [3000, 1500, 900]
    cache = _batch(wl, lengths, seed=21)
    slots = torch.tensor(list(range(len(lengths)))[::-1], dtype=torch.int32, device="cuda")
    n = slots.numel()
    for step in range(2):
        tok = inputs.gen_decode(wl, n, step=step, seed=21, device="cuda")
        cache.decode_append(slots, tok.k, tok.v)
        ref = cache.decode_attn(slots, tok.q)
        out = torch.full_like(ref, float("nan"))
        status = cache.decode_attn_noalloc(slots, tok.q, out)
        assert status == snap.SNAP_OK, snap.status_string(status)
        torch.cuda.synchronize()
        assert cache.check_device() == snap.SNAP_OK
        assert bool(torch.isfinite(out).all())
        # the same kernels with the same split plan: a stale partial would show as a difference
        assert torch.equal(out, ref), (step, (out - ref).abs().max().item())


def _scratch_need(n, heads, splits, d_v):
    """Bytes of split partials one call needs: O rounded up to 256 B, then (max, sum)."""
    parts = n * heads * splits
    return -(-parts * 4 * d_v // 256) * 256 + parts * 4 * 2


def test_noalloc_refuses_batches_beyond_its_scratch():
    """128-head MLA at a 32768-slot cache: the first batch size whose split partials
    (per the library's own launch plan) exceed the fixed scratch is refused before
    any launch, and nothing is written."""
    wl = inputs.WORKLOADS["mla_128k_b8"]
    snap.load(build_if_missing=True)
    cache = snap.SnapCache(_cfg(wl), max_batch=64, max_prompt=1)
    limit = 32 << 20    # SNAP_NOALLOC_SCRATCH_BYTES in include/snap.h
    n = next((n for n in range(1, 65)
              if _scratch_need(n, wl.n_q_heads, cache.decode_attn_plan(n)[0], wl.d_v) > limit
              and cache.decode_attn_plan(n)[0] > 1), None)
    assert n is not None, "no batch of up to 64 sequences overflows the scratch"
    slots = torch.arange(n, dtype=torch.int32, device="cuda")
    q = torch.zeros((n, wl.n_q_heads, wl.d_qk), dtype=torch.bfloat16, device="cuda")
    out = torch.full((n, wl.n_q_heads, wl.d_v), 7.0, dtype=torch.float32, device="cuda")
    assert cache.decode_attn_noalloc(slots, q, out) == snap.SNAP_ERR_SHAPE
    torch.cuda.synchronize()
    assert bool((out == 7.0).all())
