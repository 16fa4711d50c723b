"""The algorithmic byte and FLOP counts behind the bench's roofline fractions, pinned to
closed forms written out from the workload shapes (no GPU).

The decode step reads every valid cache row once: 16 sequences x 32768 slots x 8 KV heads x
(128 + 128) bf16 = 2^31 bytes at 128k GQA, plus the queries (bf16) and outputs (fp32).  One
score GEMM pass is 2 R d S per KV head with R = G W observation rows.  A compression call
reads the prompt's keys once per score pass and reads and writes every kept cache row.
"""
import bench
from fixed_size_kv_gb300 import inputs


def full_meta(wl, S):
    """(S, T, R0, n_sink, n_mid) of a sequence compressed from an S-token prompt."""
    R0 = max(wl.L_sink, S - wl.L_recent)
    return (S, S, R0, wl.L_sink, min(wl.K, R0 - wl.L_sink))


def test_decode_bytes_and_flop_gqa_128k():
    wl = inputs.WORKLOADS["gqa_128k_b16"]
    metas = [full_meta(wl, 131072)] * 16
    rows = 16 * 32768 * 8 * (128 + 128) * 2                     # every valid K and V row once
    io = 16 * 32 * (128 * 2 + 128 * 4)                          # bf16 queries in, fp32 outputs out
    assert bench.algorithmic_decode_bytes(wl, metas) == rows + io == 2147876864
    # per valid row and query head: q.k (2 d_qk) and p v (2 d_v)
    assert bench.algorithmic_decode_flop(wl, metas) == 16 * 32768 * 32 * 2 * (128 + 128)


def test_decode_bytes_and_flop_mla_128k():
    wl = inputs.WORKLOADS["mla_128k_b8"]
    metas = [full_meta(wl, 131072)] * 8
    rows = 8 * 32768 * 576 * 2                                  # one latent row holds K and V
    io = 8 * 128 * (576 * 2 + 512 * 4)
    assert bench.algorithmic_decode_bytes(wl, metas) == rows + io == 305266688
    flop = bench.algorithmic_decode_flop(wl, metas)
    assert flop == 8 * 32768 * 128 * 2 * (576 + 512)
    assert abs(flop / 1e9 - 73.0) < 0.1                         # the ~73 GFLOP of one MLA step
    # issued: each CTA of a pair computes the whole 576-wide score, and each half of P V
    issued = bench.issued_decode_flop(wl, metas)
    assert issued == 8 * 32768 * 128 * (2 * 2 * 576 + 2 * 512)
    assert abs(issued / flop - (2 * 576 + 512) / (576 + 512)) < 1e-12         # 1.53x the algorithmic work
    gqa = inputs.WORKLOADS["gqa_128k_b16"]
    gm = [full_meta(gqa, 131072)] * 16
    assert bench.issued_decode_flop(gqa, gm) == bench.algorithmic_decode_flop(gqa, gm)


def test_ring_not_yet_full_counts_only_valid_rows():
    """A 300-token prompt in a 4 + 60 + 64 cache: the sinks, 60 selected rows and the ring
    window [R0, S) of 64 rows; after 10 more tokens the ring still holds 64."""
    wl = inputs.Workload(name="t", layout=0, n_q_heads=8, n_kv_heads=2, d_qk=128, d_v=128, L_sink=4, K=60,
                         L_recent=64, W=16, P=7, batch=1, prompt_min=0, prompt_max=0, decode_steps=0,
                         sm_scale=1.0)
    S = 300
    m = full_meta(wl, S)
    assert m == (300, 300, 236, 4, 60)
    row = 2 * 256 * 2
    assert bench.algorithmic_decode_bytes(wl, [m]) == (4 + 60 + 64) * row + 8 * (256 + 512)
    m2 = (S, S + 10, 236, 4, 60)
    assert bench.algorithmic_decode_bytes(wl, [m2]) == (4 + 60 + 64) * row + 8 * (256 + 512)
    short = (50, 50, 4, 4, 0)                                   # sinks + a 46-token ring, no middle
    assert bench.algorithmic_decode_bytes(wl, [short]) == (4 + 46) * row + 8 * (256 + 512)


def test_score_pass_flop():
    gqa = inputs.WORKLOADS["gqa_128k_b16"]
    assert bench.score_pass_flop(gqa, [131072]) == 2 * (4 * 64) * 128 * 131072 * 8     # 68.7 GFLOP
    mla = inputs.WORKLOADS["mla_128k_b8"]
    f = bench.score_pass_flop(mla, [131072])
    assert f == 2 * (128 * 64) * 576 * 131072                                          # 1.24 TFLOP
    assert abs(f * 8 / 1e12 - 9.90) < 0.01                                              # per 8-prompt batch
    assert bench.score_pass_flop(gqa, [1000, 3000]) == 2 * 256 * 128 * 2000 * 8         # mean over lengths


def test_compress_call_bytes():
    gqa = inputs.WORKLOADS["gqa_128k_b16"]
    keys = 131072 * 8 * 128 * 2                                  # the prompt's keys, read once per pass
    kept = 2 * 32768 * 8 * (128 + 128) * 2                       # kept rows read, then written
    assert bench.compress_hbm_bytes(gqa, [131072], 1) == keys + kept == 536870912
    assert bench.compress_hbm_bytes(gqa, [131072], 2) == 2 * keys + kept
    mla = inputs.WORKLOADS["mla_128k_b8"]
    assert bench.compress_hbm_bytes(mla, [131072], 1) == 131072 * 576 * 2 + 2 * 32768 * 576 * 2
