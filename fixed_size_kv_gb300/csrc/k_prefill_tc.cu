// k_prefill_tc.cu -- causal prefill attention of one prompt on the 5th-generation
// tensor cores, handing the observation rows' log-sum-exp to the compression.
//
// SnapStream episode companion page, headline figure "2-5% extra prefill latency":
// the SnapKV scoring runs once at prefill, next to the prefill's own attention.  A
// flash-attention prefill already holds, for every query row, the log-sum-exp of its
// causal softmax row; the compression's row pass (the softmax denominators of the last
// W rows) is exactly that quantity.  This kernel computes the prefill attention
// O = softmax(scale Q K^T, causal) V of one GQA layer (head_dim 128, query head i reads
// KV head i / G) and writes, for the last W rows, lse_obs[w][i] in the layout
// snap_compress_lse() takes, so the compression skips its row pass.
//
// One CTA per (query head, pair of 128-row query tiles), the heaviest pairs first.
// The two query tiles share every K/V tile load and ping-pong on the tensor core: while
// one softmax group exponentiates its scores, the other tile's scores or P V run.
//   S_t = Q_t K_j^T    M = 128 rows, N = 128 keys, 8 MMAs over d (A, B in shared memory)
//   O_t += P_t V_j     M = 128 rows, N = 128 (d), 8 MMAs over keys (P in TMEM, V MN-major)
// TMEM (512 columns): S_0 | S_1 | O_0 | O_1, 128 each; P_t (bf16) is written over S_t.
// Roles (384 threads, three warpgroups): warp 0 TMA, warp 1 TMEM + MMA issue (warps 2, 3
// idle), warps 4..7 softmax of tile 0, warps 8..11 softmax of tile 1 (thread = query row).  The running max moves
// lazily (only when a tile's max exceeds it by more than 8 in log2 units; O is then
// rescaled in TMEM), so most tiles skip the rescale.  P is rounded to bf16 for the
// MMA and the output's normaliser sums those rounded weights; the log-sum-exp sums the
// unrounded ones.  Every wait is bounded.
#include "kernels.cuh"
#include "tc.cuh"

namespace snap {

namespace {

constexpr float NEG_INF = -__builtin_huge_valf();
constexpr int D = 128;                        // head dim
constexpr int BM = 128;                       // query rows per tile
constexpr int BN = 128;                       // keys per tile
constexpr int CHB = 128 * 128;                // one 64-column chunk of a 128-row tile: 16 KB
constexpr int THREADS = 384;                  // three warpgroups
// Registers: the launch gives 168 per thread (384 threads); the load / MMA warpgroup
// gives back all but SETUP_REGS and each softmax warpgroup takes SOFTMAX_REGS, within
// the launch's total (80 * 128 + 208 * 256 = 63,488 <= 168 * 384 = 64,512), so the
// softmax keeps a tile's 128 scores in registers without spilling.
constexpr int SETUP_REGS = 80;
constexpr int SOFTMAX_REGS = 208;
static_assert(SETUP_REGS * 128 + SOFTMAX_REGS * 256 <= 168 * THREADS, "register split within the launch's");
constexpr float RESCALE_GAP = 8.f;

constexpr int OFF_Q = 0;                      // 2 tiles x 2 chunks
constexpr int OFF_KV = OFF_Q + 4 * CHB;       // 2 stages x (K 2 chunks + V 2 chunks)
constexpr int STAGE_B = 4 * CHB;
constexpr int OFF_BAR = OFF_KV + 2 * STAGE_B;
constexpr int SMEM = OFF_BAR + 256 + 1024;

enum {
    B_Q_FULL = 0,
    B_KV_FULL = 1,     // + 2
    B_KV_EMPTY = 3,    // + 2
    B_S_FULL = 5,      // + 2
    B_P_FULL = 7,      // + 2
    B_PV_DONE = 9,     // + 2
    N_BARS = 11
};
static_assert(SMEM <= 232448, "shared memory");

__device__ __forceinline__ bool waitb(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
    return mbar_wait_bounded(bar, parity, abort_flag);
}

__global__ void __launch_bounds__(THREADS, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, PrefillArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int hq = blockIdx.x;
    const int p = (int)gridDim.y - 1 - (int)blockIdx.y;      // heaviest query-tile pairs first
    const int h = hq / a.G;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t s_base = smem_u32(smem);
    const uint32_t s_q = s_base + OFF_Q, s_kv = s_base + OFF_KV;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
    auto bar = [&](int i) { return smem_u32(bars + i); };
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + N_BARS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

    // query tiles 2p and 2p+1; tile t attends to key tiles 0..qt[t]
    const int qt0 = 2 * p, qt1 = 2 * p + 1;
    const bool valid1 = qt1 * BM < a.S;
    const int J = valid1 ? qt1 : qt0;                        // last key tile of the CTA

    if (threadIdx.x == 0) {
        mbar_init(bar(B_Q_FULL), 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(B_KV_FULL + i), 1);
            mbar_init(bar(B_KV_EMPTY + i), 1);
            mbar_init(bar(B_S_FULL + i), 1);
            mbar_init(bar(B_P_FULL + i), 4);
            mbar_init(bar(B_PV_DONE + i), 1);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_holder), 512);
        tmem_relinquish();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    int cur = -1;
    auto fail = [&](int role) {
        *abort_flag = 1;
        report_error(a.status, SNAP_ERR_TIMEOUT, 500, role, cur);
    };

    // warpgroup 0 (warps 0-3: TMA, MMA, two idle) hands registers to the two softmax
    // warpgroups (warps 4-7, 8-11)
    if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(SETUP_REGS));
    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            tma_prefetch(&tmQ);
            tma_prefetch(&tmK);
            tma_prefetch(&tmV);
            const int ntq = valid1 ? 2 : 1;
            mbar_expect_tx(bar(B_Q_FULL), ntq * 2 * CHB);
            for (int t = 0; t < ntq; ++t)
                for (int c = 0; c < 2; ++c)
                    tma_load_3d(s_q + (t * 2 + c) * CHB, &tmQ, bar(B_Q_FULL), 64 * c, (qt0 + t) * BM, hq);
            for (int j = 0; j <= J; ++j) {
                cur = j;
                const int st = j & 1;
                if (!waitb(bar(B_KV_EMPTY + st), ((j >> 1) & 1) ^ 1, abort_flag)) { fail(0); break; }
                mbar_expect_tx(bar(B_KV_FULL + st), STAGE_B);
                const uint32_t sb = s_kv + st * STAGE_B;
                for (int c = 0; c < 2; ++c) {
                    tma_load_3d(sb + c * CHB, &tmK, bar(B_KV_FULL + st), 64 * c, j * BN, h);
                    tma_load_3d(sb + (2 + c) * CHB, &tmV, bar(B_KV_FULL + st), 64 * c, j * BN, h);
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t id_s = idesc_bf16(BM, BN);
            constexpr uint32_t id_pv = idesc_bf16_bmn(BM, D);
            const uint64_t q_desc = desc_sw128(s_q);
            const uint64_t k_desc = desc_sw128(s_kv);
            const uint64_t v_desc = desc_sw128_mn(s_kv + 2 * CHB, CHB);
            constexpr uint64_t CH16 = CHB >> 4, ST16 = STAGE_B >> 4;
            bool ok = waitb(bar(B_Q_FULL), 0, abort_flag);
            if (!ok) fail(10);
            // Issue order (ping-pong of the two query tiles): S_0(0) S_1(0), then per key
            // tile j: P V_0(j), S_0(j+1), P V_1(j), S_1(j+1).  Each score MMA group goes in
            // as soon as its tile's previous weights are consumed, so one group's softmax
            // overlaps the other group's MMAs.
            // The S buffer holds P of the previous key tile, read by that tile's P V; the
            // next S is issued after that P V on the same thread, and tcgen05.mma operations
            // of one thread execute in issue order, so it writes the buffer only after the
            // P V has read it.  (The softmax had finished reading the previous scores before
            // it signalled their weights.)
            auto active_at = [&](int t, int j) { return j <= qt0 + t && (t == 0 || valid1) && j <= J; };
            auto issue_s = [&](int t, int j) {
                const int st = j & 1;
                const uint32_t d = tmem + t * 128;
                const uint64_t qa = q_desc + (uint64_t)(t * 2) * CH16;
                const uint64_t kb = k_desc + (uint64_t)st * ST16;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    tc_mma(d, qa + (uint64_t)((kk >> 2) * CH16 + (kk & 3) * 2),
                           kb + (uint64_t)((kk >> 2) * CH16 + (kk & 3) * 2), id_s, kk > 0 ? 1u : 0u);
                tc_commit(bar(B_S_FULL + t));
            };
            auto issue_pv = [&](int t, int j) {
                const int st = j & 1;
                const uint32_t pa = tmem + t * 128;
                const uint32_t o = tmem + 256 + t * 128;
                const uint64_t vb = v_desc + (uint64_t)st * ST16;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)      // 16 keys (8 TMEM columns of P) per MMA
                    tc_mma_ta(o, pa + kk * 8, vb + (uint64_t)kk * (2048 >> 4), id_pv, (j > 0 || kk > 0) ? 1u : 0u);
                tc_commit(bar(B_PV_DONE + t));
            };
            if (ok) {
                if (!waitb(bar(B_KV_FULL + 0), 0, abort_flag)) {
                    fail(11);
                    ok = false;
                } else {
                    tc_fence_after();
                    issue_s(0, 0);
                    if (active_at(1, 0)) issue_s(1, 0);
                }
            }
            for (int j = 0; ok && j <= J; ++j) {
                cur = j;
                const int st = j & 1;
                // the next key tile (its scores follow each P V below)
                const bool next = j + 1 <= J;
                bool next_ready = false;
                for (int t = 0; t < 2 && ok; ++t) {
                    if (active_at(t, j)) {
                        if (!waitb(bar(B_P_FULL + t), j & 1, abort_flag)) { fail(13); ok = false; break; }
                        tc_fence_after();
                        issue_pv(t, j);
                    }
                    if (next && active_at(t, j + 1)) {
                        if (!next_ready) {
                            if (!waitb(bar(B_KV_FULL + ((j + 1) & 1)), ((j + 1) >> 1) & 1, abort_flag)) {
                                fail(11);
                                ok = false;
                                break;
                            }
                            next_ready = true;
                            tc_fence_after();
                        }
                        issue_s(t, j + 1);
                    }
                }
                tc_commit(bar(B_KV_EMPTY + st));    // after both P V of key tile j
            }
        }
    }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;\n" ::"n"(SOFTMAX_REGS));
        // ------------------------------------------------------------ softmax groups
        const int t = (warp - 4) >> 2;                   // query tile of this group
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;               // row within the tile (TMEM lane)
        const int qt = qt0 + t;
        const int row = qt * BM + r;
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const uint32_t tS = tmem + t * 128 + lane_off;
        const uint32_t tO = tmem + 256 + t * 128 + lane_off;
        const float sl2 = a.sl2;
        const bool active = t == 0 || valid1;
        // the unrounded sum feeds only the log-sum-exp of the last W rows
        const bool need_lse = a.lse_obs != nullptr && __any_sync(0xffffffffu, row >= a.S - a.W && row < a.S);
        float m_used = NEG_INF, l_bf = 0.f, l_ex = 0.f;
        bool ok = true;
        for (int j = 0; active && ok && j <= qt; ++j) {
            cur = j;
            if (!__all_sync(0xffffffffu, waitb(bar(B_S_FULL + t), j & 1, abort_flag))) {
                fail(3);
                ok = false;
                break;
            }
            tc_fence_after();
            const bool diag = j == qt;                   // keys j*BN .. may pass the row
            const int key0 = j * BN;
            // the tile's 128 scores of this row, all in registers (one TMEM round trip)
            float v[4][32];
#pragma unroll
            for (int c = 0; c < 4; ++c) tmem_ld32(tS + c * 32, v[c]);
#pragma unroll
            for (int c = 0; c < 4; ++c) tmem_ld_wait(v[c]);
            if (diag) {                                  // the tile that crosses the causal limit
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        if (key0 + c * 32 + e > row) v[c][e] = NEG_INF;
            }
            // the row max: eight independent chains, three operands per instruction
            float mq[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) mq[k] = fmaxf(v[0][2 * k], v[0][2 * k + 1]);
#pragma unroll
            for (int i = 16; i < 128; i += 16)
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    mq[k] = fmax3(mq[k], v[(i + 2 * k) >> 5][(i + 2 * k) & 31], v[(i + 2 * k + 1) >> 5][(i + 2 * k + 1) & 31]);
            float mx = fmax3(fmax3(mq[0], mq[1], mq[2]), fmax3(mq[3], mq[4], mq[5]), fmaxf(mq[6], mq[7]));
            mx *= sl2;                                   // sl2 > 0: the max of the scaled scores
            // lazy running max; O is rescaled (warp-wide, tcgen05 is warp-collective) when
            // a lane's max moves and its old max was finite, after P V of the last tile
            const bool move = mx > m_used + RESCALE_GAP || (m_used == NEG_INF && mx != NEG_INF);
            const float m_new = move ? fmaxf(mx, m_used) : m_used;
            const bool rescale = move && m_used != NEG_INF;
            if (__any_sync(0xffffffffu, rescale)) {
                if (!__all_sync(0xffffffffu, waitb(bar(B_PV_DONE + t), (j - 1) & 1, abort_flag))) {
                    fail(5);
                    ok = false;
                    break;
                }
                tc_fence_after();
                const float alpha = rescale ? ex2(m_used - m_new) : 1.f;
#pragma unroll 1
                for (int c = 0; c < 4; ++c) {
                    float o[32];
                    tmem_ld32(tO + c * 32, o);
                    tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] *= alpha;
                    tmem_st32(tO + c * 32, o);
                }
                tmem_st_wait();
            }
            if (m_new != m_used) {
                const float alpha = m_used == NEG_INF ? 0.f : ex2(m_used - m_new);
                l_bf *= alpha;
                l_ex *= alpha;
                m_used = m_new;
            }
            // weights, bf16 pairs written over the scores (64 columns)
#pragma unroll
            for (int c2 = 0; c2 < 2; ++c2) {
                float (&lo)[32] = v[2 * c2];
                float (&hi)[32] = v[2 * c2 + 1];
                float w[32];
                const float nm = -m_used;
                // sums of the bf16 weights (and, for the log-sum-exp rows, of the unrounded
                // ones) as packed f32x2 accumulators, two weights per add
                uint64_t sb2[2] = {0ull, 0ull}, se2[2] = {0ull, 0ull};
                const uint64_t sl2x2 = f32x2_splat(sl2), nmx2 = f32x2_splat(nm);
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    float a0, a1;
                    fma_f32x2(a0, a1, lo[2 * e], lo[2 * e + 1], sl2x2, nmx2);
                    const float p0 = ex2(a0), p1 = ex2(a1);
                    const uint32_t pk = pack_bf16(p0, p1);   // the weights P V uses
                    add_f32x2(sb2[e & 1], pk << 16, pk & 0xffff0000u);
                    if (need_lse) add_f32x2(se2[e & 1], __float_as_uint(p0), __float_as_uint(p1));
                    w[e] = __uint_as_float(pk);
                }
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    float a0, a1;
                    fma_f32x2(a0, a1, hi[2 * e], hi[2 * e + 1], sl2x2, nmx2);
                    const float p0 = ex2(a0), p1 = ex2(a1);
                    const uint32_t pk = pack_bf16(p0, p1);
                    add_f32x2(sb2[e & 1], pk << 16, pk & 0xffff0000u);
                    if (need_lse) add_f32x2(se2[e & 1], __float_as_uint(p0), __float_as_uint(p1));
                    w[16 + e] = __uint_as_float(pk);
                }
                l_bf += f32x2_sum(sb2[0]) + f32x2_sum(sb2[1]);
                l_ex += f32x2_sum(se2[0]) + f32x2_sum(se2[1]);
                tmem_st32(tS + c2 * 32, w);
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_P_FULL + t));
        }
        // output: O / l (bf16) and the log-sum-exp of the observation rows
        if (active && ok) {
            if (!__all_sync(0xffffffffu, waitb(bar(B_PV_DONE + t), qt & 1, abort_flag))) {
                fail(8);
                ok = false;
            }
        }
        if (active && ok) {
            tc_fence_after();
            const float inv = l_bf > 0.f ? 1.f / l_bf : 0.f;
            bf16* orow = a.O + (size_t)row * a.o_tok_stride + (size_t)hq * D;
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
                float o[32];
                tmem_ld32(tO + c * 32, o);
                tmem_ld_wait();
                if (row < a.S) {
#pragma unroll
                    for (int e = 0; e < 32; e += 8) {
                        uint4 u;
                        u.x = pack_bf16(o[e] * inv, o[e + 1] * inv);
                        u.y = pack_bf16(o[e + 2] * inv, o[e + 3] * inv);
                        u.z = pack_bf16(o[e + 4] * inv, o[e + 5] * inv);
                        u.w = pack_bf16(o[e + 6] * inv, o[e + 7] * inv);
                        *reinterpret_cast<uint4*>(orow + c * 32 + e) = u;
                    }
                }
            }
            if (a.lse_obs && row < a.S && row >= a.S - a.W)
                a.lse_obs[(size_t)(row - (a.S - a.W)) * a.Hq + hq] = (m_used + log2f(l_ex)) * 0.6931471805599453f;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace

cudaError_t launch_prefill_tc(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                              const PrefillArgs& a, cudaStream_t st) {
    static std::atomic<uint64_t> smem_set{0};
    if (cudaError_t e = opt_in_smem(prefill_tc_kernel, SMEM, smem_set); e != cudaSuccess) return e;
    const int pairs = (a.S + 2 * BM - 1) / (2 * BM);
    dim3 grid(a.Hq, pairs);
    prefill_tc_kernel<<<grid, THREADS, SMEM, st>>>(tq, tk, tv, a);
    return cudaGetLastError();
}

}  // namespace snap
