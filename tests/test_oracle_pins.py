"""Pins of the CPU oracle to facts that do not come from the oracle itself.

Method: SnapStream: Efficient Long Sequence Decoding on Dataflow Accelerators,
episode companion page -- "Fixed-Size Cache Layout" (sinks + SnapKV top-K middle
+ recent window, built once at prefill), "Ring Buffer vs. Naive Slicing" (decode
writes into a fixed ring index), "Infinity-Bench KV Retrieval" (pooling-based
top-K), headline figure "4.0x lower KV memory".

Each pin is a closed form, an invariant, a special case that reduces to a
library routine (scipy / numpy / torch SDPA in float64), a hand-worked fixture
under tests/golden/, or a brute force on tiny inputs along an independent code
path.  A dropped term, a wrong sign or index, or a transposed operand in the
oracle fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch
from scipy import ndimage, special

import oracle
from fixed_size_kv_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def cfg_of(layout=0, Hq=4, Hkv=2, dk=8, dv=8, L_sink=2, K=4, L_recent=6, W=2, P=3, scale=None):
    if scale is None:
        scale = 1.0 / math.sqrt(dk)
    return oracle.Config(layout, Hq, Hkv, dk, dv, L_sink, K, L_recent, W, P, scale)


def bf16(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * scale).to(torch.bfloat16)


# ----------------------------------------------------------------------------- plan

@pytest.mark.parametrize("S,exp", [
    # (n_sink, R0, n_mid) by hand for L_sink=4, K=252, L_recent=256
    (2048, (4, 1792, 252)),   # middle [4,1792) has 1788 > 252 -> 252 kept
    (100, (4, 4, 0)),         # everything fits in sinks + ring
    (3, (3, 3, 0)),           # shorter than the sinks
    (512, (4, 256, 252)),     # middle holds exactly K
    (513, (4, 257, 252)),     # one too many: scoring needed
])
def test_plan_by_hand(oracle_lib, S, exp):
    c = cfg_of(Hq=32, Hkv=8, dk=128, dv=128, L_sink=4, K=252, L_recent=256, W=32, P=7)
    m = oracle.plan(c, S)
    assert (m.n_sink, m.R0, m.n_mid) == exp
    assert m.S == S and m.T == S


def test_config_rejections(oracle_lib):
    assert oracle.check_config(cfg_of())
    assert not oracle.check_config(cfg_of(P=4))           # P must be odd
    assert not oracle.check_config(cfg_of(W=7, L_recent=6))  # window inside the ring
    assert not oracle.check_config(cfg_of(Hq=5, Hkv=2))   # whole groups
    assert not oracle.check_config(cfg_of(layout=1, Hkv=2))  # MLA has one latent head


# ------------------------------------------------------------------- window scores

def test_scores_sum_to_rows(oracle_lib):
    """Each causal softmax row sums to 1, so every head's column mass is G*W."""
    c = cfg_of(Hq=6, Hkv=2, dk=16, W=5)
    S = 23
    K, Q = bf16((S, 2, 16), 1, 2.0), bf16((5, 6, 16), 2, 2.0)
    _, col = oracle.window_scores(c, K, Q)
    np.testing.assert_allclose(col.sum(axis=1), [c.G * c.W] * 2, rtol=1e-12)
    assert (col >= 0).all()


def test_scores_single_row_is_softmax(oracle_lib):
    """W = 1, G = 1: the column score is one textbook softmax row over all S keys."""
    c = cfg_of(Hq=1, Hkv=1, dk=16, W=1, scale=0.37)
    S = 40
    K, Q = bf16((S, 1, 16), 3), bf16((1, 1, 16), 4)
    lse, col = oracle.window_scores(c, K, Q)
    s = 0.37 * (K.double()[:, 0, :] @ Q.double()[0, 0, :]).numpy()
    np.testing.assert_allclose(col[0], special.softmax(s), rtol=1e-12)
    np.testing.assert_allclose(lse[0, 0, 0], special.logsumexp(s), rtol=1e-13)


def test_scores_zero_keys_closed_form(oracle_lib):
    """All-zero keys: each row is uniform over its causal prefix, p = 1/(pos+1)."""
    c = cfg_of(Hq=4, Hkv=2, dk=8, W=3)
    S = 10
    K = torch.zeros((S, 2, 8), dtype=torch.bfloat16)
    Q = bf16((3, 4, 8), 5)
    lse, col = oracle.window_scores(c, K, Q)
    expect = np.zeros(S)
    for w in range(3):
        pos = S - 3 + w
        expect[: pos + 1] += c.G / (pos + 1)
        np.testing.assert_allclose(lse[:, w, :], math.log(pos + 1), rtol=1e-14)
    np.testing.assert_allclose(col, np.stack([expect, expect]), rtol=1e-13)


def test_scores_brute_force_tiny(oracle_lib):
    """Independent dense path: full score matrix, causal mask, softmax, sums."""
    c = cfg_of(Hq=6, Hkv=3, dk=12, W=4, scale=0.21)
    S = 17
    K, Q = bf16((S, 3, 12), 6, 1.5), bf16((4, 6, 12), 7, 1.5)
    lse, col = oracle.window_scores(c, K, Q)
    Kd, Qd = K.double(), Q.double()
    for h in range(3):
        q = Qd[:, 2 * h:2 * h + 2, :]                    # [W][G][d]
        s = 0.21 * torch.einsum("wgd,jd->wgj", q, Kd[:, h, :])
        pos = torch.arange(S - 4, S).view(4, 1, 1)
        s = s.masked_fill(torch.arange(S).view(1, 1, S) > pos, float("-inf"))
        p = torch.softmax(s, dim=-1)
        np.testing.assert_allclose(col[h], p.sum(dim=(0, 1)).numpy(), rtol=1e-12, atol=1e-300)
        np.testing.assert_allclose(lse[h], torch.logsumexp(s, -1).numpy(), rtol=1e-13)


def test_scores_group_mapping(oracle_lib):
    """Query heads h*G..h*G+G-1 read KV head h: a key aligned with the queries of head
    group 1 only stands out in KV head 1's scores."""
    c = cfg_of(Hq=8, Hkv=2, dk=8, W=2, scale=1.0)
    S = 12
    Q = torch.zeros((2, 8, 8))
    Q[:, 4:8, 0] = 4.0             # group 1 queries point along e0
    Q[:, 0:4, 1] = 4.0             # group 0 queries point along e1
    K = torch.zeros((S, 2, 8))
    K[5, 1, 0] = 4.0               # aligned with group 1 in KV head 1
    K[7, 0, 0] = 4.0               # along e0 in KV head 0: orthogonal to group 0
    _, col = oracle.window_scores(c, K.to(torch.bfloat16), Q.to(torch.bfloat16))
    assert col[1].argmax() == 5 and col[1, 5] > 0.99 * c.G * c.W
    np.testing.assert_allclose(col[0, 7], col[0, 6], rtol=1e-14)


# ------------------------------------------------------------------ pool and select

def test_pool_select_hand_fixture(oracle_lib):
    with open(os.path.join(GOLDEN, "pool_select_hand.json")) as f:
        cases = json.load(f)["cases"]
    for case in cases:
        y = oracle.maxpool(np.array(case["x"], float), case["P"])
        np.testing.assert_array_equal(y, case["pooled"])
        for s in case["select"]:
            got = oracle.select(y, s["lo"], s["hi"], s["K"])
            assert got.tolist() == s["sel"], s["why"]


def test_pool_special_cases(oracle_lib):
    x = np.random.default_rng(0).random(101)
    np.testing.assert_array_equal(oracle.maxpool(x, 1), x)
    np.testing.assert_array_equal(oracle.maxpool(x, 203), np.full(101, x.max()))
    for P in (3, 7, 31):
        ref = ndimage.maximum_filter1d(x, size=P, mode="constant", cval=-np.inf)
        np.testing.assert_array_equal(oracle.maxpool(x, P), ref)


def test_select_brute_force(oracle_lib):
    rng = np.random.default_rng(1)
    for trial in range(50):
        n = int(rng.integers(1, 60))
        x = rng.integers(0, 6, n).astype(float)   # many ties
        lo = int(rng.integers(0, n))
        hi = int(rng.integers(lo, n + 1))
        K = int(rng.integers(0, n + 2))
        got = oracle.select(x, lo, hi, K)
        idx = np.arange(lo, hi)
        order = idx[np.lexsort((idx, -x[lo:hi]))]
        expect = np.sort(order[:K])
        assert got.tolist() == expect.tolist()


# ------------------------------------------------------------------------ compress

def test_compress_keeps_everything_when_it_fits(oracle_lib):
    """M <= K: no scoring, the middle is the whole middle, rows are bit copies."""
    c = cfg_of(Hq=4, Hkv=2, dk=8, L_sink=2, K=5, L_recent=6, W=2)
    S = 11                               # middle [2, 5) has 3 <= 5 positions
    K, V, Q = bf16((S, 2, 8), 8), bf16((S, 2, 8), 9), bf16((2, 4, 8), 10)
    cache = oracle.compress(c, K, V, Q)
    m = cache.meta
    assert (m.n_sink, m.R0, m.n_mid) == (2, 5, 3)
    pos = cache.slot_positions()
    kb = K.view(torch.int16).numpy().view(np.uint16)
    vb = V.view(torch.int16).numpy().view(np.uint16)
    for h in range(2):
        held = sorted(p for p in pos[h] if p >= 0)
        assert held == list(range(S))
        for s, p in enumerate(pos[h]):
            if p >= 0:
                np.testing.assert_array_equal(cache.k[h, s], kb[p, h])
                np.testing.assert_array_equal(cache.v[h, s], vb[p, h])
            else:
                assert not cache.k[h, s].any() and not cache.v[h, s].any()


def test_compress_selects_planted_heavy_hitters(oracle_lib):
    """Strong heavy hitters aligned with the window queries are all kept: without
    pooling when their count is <= K, and with a width-P pool when P * count <= K
    (pooling copies each one's score to its P-1 neighbours, which tie with it)."""
    for P, K in ((1, 12), (3, 30)):
        wl = inputs.Workload("t", 0, 8, 2, 32, 32, 2, K, 16, 4, P, 1, 300, 300, 0,
                             1 / math.sqrt(32))
        pre = inputs.gen_prefill(wl, 300, seed=3, heavy_fraction=0.03, gamma=8.0)
        c = oracle.Config(**wl.config_kwargs())
        cache = oracle.compress(c, pre.K, pre.V, pre.Q)
        for h in range(2):
            planted = set(p for p in pre.heavy[h].tolist() if c.L_sink <= p < cache.meta.R0)
            assert 0 < P * len(planted) <= c.K
            assert planted <= set(cache.sel[h].tolist())


def test_compress_selection_matches_scores(oracle_lib):
    """The kept middle is the top-K of the max-pooled window scores."""
    c = cfg_of(Hq=4, Hkv=2, dk=16, L_sink=3, K=7, L_recent=8, W=4, P=5)
    S = 60
    K, V, Q = bf16((S, 2, 16), 11), bf16((S, 2, 16), 12), bf16((4, 4, 16), 13)
    cache = oracle.compress(c, K, V, Q, want_pool=True)
    _, col = oracle.window_scores(c, K, Q)
    for h in range(2):
        pooled = ndimage.maximum_filter1d(col[h, :S - 4], size=5, mode="constant",
                                          cval=-np.inf)
        np.testing.assert_array_equal(cache.pool[h], pooled)
        lo, hi = 3, cache.meta.R0
        idx = np.arange(lo, hi)
        expect = np.sort(idx[np.lexsort((idx, -pooled[lo:hi]))][:7])
        assert cache.sel[h].tolist() == expect.tolist()


def test_compress_from_supplied_scores_is_the_same_compression(oracle_lib):
    """Compression with the column scores supplied (the path the large parity tests use
    to score on several threads) is bit-identical to compression from the queries."""
    c = cfg_of(Hq=8, Hkv=2, dk=16, L_sink=3, K=7, L_recent=8, W=4, P=5)
    S = 80
    K, V, Q = bf16((S, 2, 16), 21), bf16((S, 2, 16), 22), bf16((4, 8, 16), 23)
    ref = oracle.compress(c, K, V, Q, want_pool=True)
    _, col = oracle.window_scores(c, K, Q)
    got = oracle.compress(c, K, V, None, want_pool=True, col=col)
    np.testing.assert_array_equal(got.sel, ref.sel)
    np.testing.assert_array_equal(got.k, ref.k)
    np.testing.assert_array_equal(got.v, ref.v)
    np.testing.assert_array_equal(got.pool, ref.pool)
    assert got.meta == ref.meta


@pytest.mark.parametrize("layout,Hq,Hkv,group", [(0, 8, 2, 2), (0, 8, 2, 0), (1, 16, 1, 4)])
def test_window_columns_by_head_groups(oracle_lib, layout, Hq, Hkv, group):
    """Column scores summed over disjoint groups of query heads, scored on several
    threads, equal the one-call scores up to the order of the double additions; the
    MLA case checks the per-head mass as well (each query head's W rows sum to W)."""
    dk = 24 if layout == 1 else 16
    dv = 16
    c = cfg_of(layout=layout, Hq=Hq, Hkv=Hkv, dk=dk, dv=dv, L_sink=2, K=5, L_recent=8, W=4, P=3)
    S = 50
    K, Q = bf16((S, Hkv, dk), 31), bf16((4, Hq, dk), 32)
    _, col = oracle.window_scores(c, K, Q)
    got = oracle.window_columns(c, K, Q, threads=3, group=group)
    np.testing.assert_allclose(got, col, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(got.sum(axis=1), np.full(Hkv, c.G * c.W), rtol=1e-12)


def test_cache_is_four_times_smaller(oracle_lib):
    """The page's 4.0x lower KV memory at 128K context with a 32k cache."""
    with open(os.path.join(GOLDEN, "pages_figures.json")) as f:
        pages = json.load(f)
    for name in ("gqa_128k_b16", "mla_128k_b8"):
        wl = inputs.WORKLOADS[name]
        assert wl.C == pages["cache_tokens"]["value"]
        assert wl.prompt_max / wl.C == pages["kv_memory_reduction"]["value"]
    assert inputs.WORKLOADS["mla_128k_b8"].L_recent == pages["deepseek_L_recent"]["value"]


# ------------------------------------------------------------------ append and ring

def test_ring_holds_last_window(oracle_lib):
    """After N appends the ring holds exactly positions [max(R0, T-L_recent), T), each
    at slot L_sink + K + (p mod L_recent), bit-exact."""
    c = cfg_of(Hq=4, Hkv=2, dk=8, L_sink=2, K=3, L_recent=5, W=2)
    S = 20
    K, V, Q = bf16((S, 2, 8), 14), bf16((S, 2, 8), 15), bf16((2, 4, 8), 16)
    cache = oracle.compress(c, K, V, Q)
    allk = [K[p] for p in range(S)]
    for step in range(13):
        kn, vn = bf16((2, 8), 100 + step), bf16((2, 8), 200 + step)
        oracle.append(cache, kn, vn)
        allk.append(kn)
        T = S + step + 1
        assert cache.meta.T == T
        pos = cache.slot_positions()
        ring = pos[:, c.L_sink + c.K:]
        lo = max(cache.meta.R0, T - c.L_recent)
        for h in range(2):
            assert sorted(ring[h].tolist()) == list(range(lo, T))
            for p in range(lo, T):
                s = c.L_sink + c.K + p % c.L_recent
                assert pos[h, s] == p
                np.testing.assert_array_equal(
                    cache.k[h, s], allk[p][h].view(torch.int16).numpy().view(np.uint16))


# -------------------------------------------------------------------------- attention

def _sdpa(q, k, v, scale):
    """torch SDPA in float64 for one query per head: q [H][d], k [H][T][d], v [H][T][dv]."""
    out = torch.nn.functional.scaled_dot_product_attention(
        q.unsqueeze(1), k, v, scale=scale)
    return out.squeeze(1).numpy()


def test_attention_equals_full_when_cache_covers_prompt(oracle_lib):
    """L_sink + K + L_recent >= S and no eviction yet: compressed == full attention."""
    c = cfg_of(Hq=8, Hkv=2, dk=16, dv=16, L_sink=2, K=4, L_recent=16, W=2)
    S = 15
    K, V, Q = bf16((S, 2, 16), 17), bf16((S, 2, 16), 18), bf16((2, 8, 16), 19)
    cache = oracle.compress(c, K, V, Q)
    q = bf16((8, 16), 20)
    out = oracle.decode_attn(cache, q)
    kf = K.double().permute(1, 0, 2).repeat_interleave(4, dim=0)
    vf = V.double().permute(1, 0, 2).repeat_interleave(4, dim=0)
    np.testing.assert_allclose(out, _sdpa(q.double(), kf, vf, c.sm_scale), rtol=1e-12, atol=1e-13)
    # and after appends that keep T - R0 <= L_recent
    ks, vs = [K], [V]
    for step in range(2):
        kn, vn = bf16((1, 2, 16), 30 + step), bf16((1, 2, 16), 40 + step)
        oracle.append(cache, kn[0], vn[0])
        ks.append(kn), vs.append(vn)
    Kall, Vall = torch.cat(ks), torch.cat(vs)
    out = oracle.decode_attn(cache, q)
    kf = Kall.double().permute(1, 0, 2).repeat_interleave(4, dim=0)
    vf = Vall.double().permute(1, 0, 2).repeat_interleave(4, dim=0)
    np.testing.assert_allclose(out, _sdpa(q.double(), kf, vf, c.sm_scale), rtol=1e-12, atol=1e-13)


def test_attention_over_held_positions_after_eviction(oracle_lib):
    """With evictions, attention equals full attention restricted to the positions the
    cache holds (sinks, the selected middle, the ring window)."""
    c = cfg_of(Hq=4, Hkv=2, dk=16, dv=16, L_sink=2, K=3, L_recent=5, W=2, P=3)
    S = 30
    K, V, Q = bf16((S, 2, 16), 21), bf16((S, 2, 16), 22), bf16((2, 4, 16), 23)
    cache = oracle.compress(c, K, V, Q)
    ks, vs = [K], [V]
    for step in range(7):
        kn, vn = bf16((1, 2, 16), 50 + step), bf16((1, 2, 16), 60 + step)
        oracle.append(cache, kn[0], vn[0])
        ks.append(kn), vs.append(vn)
    Kall, Vall = torch.cat(ks).double(), torch.cat(vs).double()
    T = cache.meta.T
    lo = max(cache.meta.R0, T - c.L_recent)
    q = bf16((4, 16), 24)
    out = oracle.decode_attn(cache, q)
    for i in range(4):
        h = i // c.G
        held = list(range(min(c.L_sink, S))) + cache.sel[h].tolist() + list(range(lo, T))
        held = [p for p in held if p >= 0]
        ref = _sdpa(q[i:i + 1].double(), Kall[held, h].unsqueeze(0), Vall[held, h].unsqueeze(0),
                    c.sm_scale)
        np.testing.assert_allclose(out[i], ref[0], rtol=1e-12, atol=1e-13)


def test_mla_attention_is_mqa_with_latent_values(oracle_lib):
    """MLA absorbed attention = MQA with a d_qk-wide key and the first d_v key columns
    as the value."""
    c = cfg_of(layout=1, Hq=16, Hkv=1, dk=24, dv=16, L_sink=2, K=4, L_recent=20, W=2,
               scale=0.3)
    S = 18
    K, Q = bf16((S, 1, 24), 25), bf16((2, 16, 24), 26)
    cache = oracle.compress(c, K, None, Q)
    q = bf16((16, 24), 27)
    out = oracle.decode_attn(cache, q)
    kf = K.double()[:, 0, :].unsqueeze(0).expand(16, S, 24)
    ref = _sdpa(q.double(), kf, kf[..., :16], 0.3)
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-13)


# -------------------------------------------------------------------- prefill attention

def test_prefill_attention_equals_causal_sdpa(oracle_lib):
    """Causal prefill attention with grouped KV heads equals torch SDPA (float64,
    is_causal) over the same rows, and its log-sum-exp equals torch.logsumexp of the
    scaled, causally masked scores."""
    c = cfg_of(Hq=8, Hkv=2, dk=16, dv=16)
    S = 37
    Q, K, V = bf16((S, 8, 16), 51), bf16((S, 2, 16), 52), bf16((S, 2, 16), 53)
    out, lse = oracle.prefill_attn(c, Q, K, V)
    q = Q.double().permute(1, 0, 2)                                   # [H][S][d]
    k = K.double().permute(1, 0, 2).repeat_interleave(4, dim=0)
    v = V.double().permute(1, 0, 2).repeat_interleave(4, dim=0)
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True, scale=c.sm_scale)
    np.testing.assert_allclose(out, ref.permute(1, 0, 2).numpy(), rtol=1e-12, atol=1e-13)
    s = c.sm_scale * (q @ k.transpose(1, 2))
    s = s.masked_fill(torch.ones(S, S, dtype=torch.bool).triu(1), float("-inf"))
    np.testing.assert_allclose(lse, torch.logsumexp(s, dim=2).T.numpy(), rtol=1e-13, atol=1e-13)


def test_prefill_lse_of_window_rows_equals_window_scores_lse(oracle_lib):
    """The last W rows' prefill log-sum-exp is the window scoring's row normaliser (two
    separate loops of the oracle): the quantity snap_compress_lse takes from a prefill."""
    c = cfg_of(Hq=8, Hkv=2, dk=16, dv=16, W=5)
    S = 41
    Q, K, V = bf16((S, 8, 16), 54), bf16((S, 2, 16), 55), bf16((S, 2, 16), 56)
    _, lse = oracle.prefill_attn(c, Q, K, V)
    lse_w, _ = oracle.window_scores(c, K, Q[S - c.W:].contiguous())       # [H_kv][W][G]
    for w in range(c.W):
        for hq in range(8):
            assert abs(lse[S - c.W + w, hq] - lse_w[hq // 4, w, hq % 4]) <= 1e-13 * max(1.0, abs(lse_w[hq // 4, w, hq % 4]))


def test_prefill_zero_keys_closed_form(oracle_lib):
    """With all-zero keys every causal row is uniform: row i averages values 0..i and its
    log-sum-exp is log(i + 1)."""
    c = cfg_of(Hq=4, Hkv=1, dk=8, dv=8)
    S = 19
    Q, V = bf16((S, 4, 8), 57), bf16((S, 1, 8), 58)
    K = torch.zeros((S, 1, 8), dtype=torch.bfloat16)
    out, lse = oracle.prefill_attn(c, Q, K, V)
    vd = V.double()[:, 0]
    for i in range(S):
        np.testing.assert_allclose(out[i], vd[:i + 1].mean(dim=0).numpy()[None].repeat(4, 0), rtol=1e-13,
                                   atol=1e-14)
        np.testing.assert_allclose(lse[i], np.full(4, math.log(i + 1)), rtol=1e-14, atol=1e-14)
