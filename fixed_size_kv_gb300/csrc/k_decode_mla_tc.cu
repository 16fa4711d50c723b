// k_decode_mla_tc.cu -- absorbed-query MLA decode attention over the fixed-size
// cache on the 5th-generation tensor cores.
//
// DeepSeek-R1 shape (SnapStream episode companion page, "16-Socket Deployment:
// Prefill vs. Decode Parallelism"): 128 query heads read one latent KV row
// [latent 512 | rope 64] per cached token; the value is the latent.  The 128 heads
// of one sequence form the M = 128 side of every MMA.
//
// Two CTAs handle one (sequence, split) and divide the output: CTA `half` accumulates
// O[:, 256 half .. 256 half + 255] = P V over its 256 value columns (256 fp32 TMEM
// columns; all 512 would fill TMEM).  Each computes the whole score S = Q K^T over
// all 576 columns itself, so the pair needs no exchange and no cluster: the scores
// are computed twice (the cheap part of the step at this size), and the pair's two
// reads of every cache tile start together, so the second is served by L2.
//
// Per 64-key tile: S into TMEM with N = 64 score MMAs (q's four chunks 0..3 from
// TMEM, chunks 4..8 from shared memory), the softmax, the bf16 weights P written
// over their scores in TMEM, then O += P V as one N = 256 MMA per 16 keys (the
// CTA's four 64-column value chunks, 8 KB apart in the stage).  Measured on GB300
// with back-to-back issue: an M = 128 tcgen05.mma takes ~45 cycles at any N <= 64,
// 64 at N = 128 and 128 at N = 256 (4096 MAC/clk), so the 36 N = 64 score MMAs of a
// tile run at about 70% of the tensor rate.  TMEM columns: scores / weights 0..127
// (one 64-column buffer per softmax group), q 128..255, O 256..511.
//
// Roles (320 threads per CTA): warp 0 issues TMA loads (and L2 prefetches ahead),
// warp 1 owns TMEM and one thread issues tcgen05.mma from two queues (scores of the
// next tile, P V of the oldest tile with weights), warps 2..9 run the softmax as two
// groups of four warps (one TMEM lane quarter each; thread = head) that take
// alternate tiles.  Both groups accumulate into the one O, so they share one running
// max, handed from the group of tile i-1 to the group of tile i (per lane quarter,
// through an mbarrier).  It moves lazily: only when a tile's max exceeds it by more
// than 32 in log2 units, and then O is rescaled in TMEM after P V of the previous
// tile.  Each group keeps its own sum of weights, rescaled when the shared max
// moves; the two sums are added at the end.  Every wait is bounded.
#include "kernels.cuh"
#include "tc.cuh"

namespace snap {

namespace {

constexpr float NEG_INF = -__builtin_huge_valf();
constexpr int MV = 512;                     // value (latent) width
constexpr int HEADS = 128;                  // M of every MMA
constexpr int TK = 64;                      // keys per tile
constexpr int NCH = 9;                      // 64-column chunks of a key row (8 latent + rope)
constexpr int QT_CH = 4;                    // chunks of q held in TMEM (the rest in shared memory)
constexpr int CH_B = TK * 128;              // one 64-column chunk of a KV tile: 8 KB
constexpr int QCH_B = HEADS * 128;          // one 64-column chunk of q: 16 KB
constexpr int KST = 2;                      // KV tile stages (L2 prefetch runs further ahead)
constexpr int NG = 2;                       // softmax groups (tile i goes to group i % 2)
constexpr int THREADS = 64 + NG * 128;
constexpr float RESCALE_GAP = 32.f;         // weights up to 2^32 stay exact in fp32 O and l

constexpr int OFF_Q = 0;                                  // q chunks 4..8: 80 KB
constexpr int OFF_KV = OFF_Q + (NCH - QT_CH) * QCH_B;     // + KST x 72 KB
constexpr int OFF_ML = OFF_KV + KST * NCH * CH_B;         // running max [128] and group sums [2][128]
constexpr int OFF_BAR = OFF_ML + 1536;
constexpr int SMEM = OFF_BAR + 256 + 1024;                // barriers + alignment slack

enum {
    B_Q_FULL = 0,                // q chunks 0..3 moved into TMEM (and 4..8 in place)
    B_KV_FULL = 1,               // + KST
    B_KV_EMPTY = 1 + KST,        // + KST
    B_S_FULL = 1 + 2 * KST,      // + NG: scores of the group's tile are in TMEM
    B_SP_EMPTY = 3 + 2 * KST,    // + NG: P V of the group's previous tile done (buffer free)
    B_P_FULL = 5 + 2 * KST,      // + NG: weights of the group's tile are in TMEM
    B_M_READY = 7 + 2 * KST,     // + 4 (one per lane quarter)
    B_Q_LOAD = 11 + 2 * KST,     // the TMA load of q (all nine chunks) has landed
    N_BARS = 12 + 2 * KST
};
static_assert((N_BARS + 1) * 8 <= 256, "barrier area");
static_assert(SMEM <= 232448, "shared memory");
static_assert(TK == 64, "the mask below takes two 32-key ballots");
static_assert(TK == MLA_KEYS, "the host plans splits and the cache tensor map in MLA_KEYS tiles");

constexpr int SOFTMAX_BAR_ID = 1;           // named barrier of the softmax warps (bar 0 = __syncthreads)

__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
    return mbar_wait_bounded(bar, parity, abort_flag);
}

__global__ void __launch_bounds__(THREADS, 1)
    mla_decode_tc_kernel(const __grid_constant__ CUtensorMap tmKV, const __grid_constant__ CUtensorMap tmQ,
                         DecodeArgs a) {
    pdl_launch_dependents();    // the merge may launch once the last wave has started
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const DevConfig& c = a.cfg;
    const int half = blockIdx.x & 1;            // which 256 value columns this CTA accumulates
    const int split = blockIdx.x >> 1, b = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const uint32_t s_base = smem_u32(smem);
    const uint32_t s_q = s_base + OFF_Q, s_kv = s_base + OFF_KV;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
    auto bar = [&](int i) { return smem_u32(bars + i); };
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + N_BARS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
    float* m_sh = reinterpret_cast<float*>(smem + OFF_ML);         // running max handed between groups
    float* l_sh = m_sh + HEADS;                                    // [NG][HEADS] group sums at the end

    if (threadIdx.x == 0) {
        mbar_init(bar(B_Q_LOAD), 1);
        mbar_init(bar(B_Q_FULL), NG * 4);      // the softmax warps, after storing q
        for (int i = 0; i < KST; ++i) {
            mbar_init(bar(B_KV_FULL + i), 1);
            mbar_init(bar(B_KV_EMPTY + i), 1);
        }
        for (int g = 0; g < NG; ++g) {
            mbar_init(bar(B_S_FULL + g), 1);
            mbar_init(bar(B_SP_EMPTY + g), 1);
            mbar_init(bar(B_P_FULL + g), 4);
        }
        for (int q = 0; q < 4; ++q) mbar_init(bar(B_M_READY + q), 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_holder), 512);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch(&tmKV);
        tma_prefetch(&tmQ);
    }
    __syncthreads();
    tc_fence_after();
    // set-up above overlaps the previous kernel; from here on this kernel reads what
    // earlier kernels wrote (the cache, its meta, q)
    pdl_wait();
    const int slot = a.slots[b];
    const bool slot_ok = slot >= 0 && slot < c.max_batch;
    const uint32_t tmem = *tmem_holder;
    // TMEM: scores, then weights (one 64-column buffer per group), q chunks 0..3, O
    const uint32_t T_S = tmem, T_Q = tmem + 128, T_O = tmem + 256;

    // status detail: 300 + half, the wait that gave up, the tile index reached
    int cur_tile = -1;
    auto fail = [&](int role) {
        *abort_flag = 1;
        report_error(a.status, SNAP_ERR_TIMEOUT, 300 + half, role, cur_tile);
    };

    SlotValidity sv;
    snap_seq_meta m{};
    if (slot_ok) {
        m = a.meta[slot];
    } else if (threadIdx.x == 0 && split == 0 && half == 0) {
        report_error(a.status, SNAP_ERR_DEVICE_CHECK, 1, b, slot);
    }
    const int ntiles = (c.C + TK - 1) / TK;
    const int t_begin = split * a.tiles_per_split;
    const int t_end = slot_ok ? min(ntiles, t_begin + a.tiles_per_split) : t_begin;
    if (slot_ok && a.k_new) {
        // fused ring append: both CTAs of the split whose key range holds the new token's
        // ring slot write its row (the same bytes) before their own TMA reads of the cache
        const int s_app = c.L_sink + c.K + m.T % c.L_recent;
        if (s_app >= t_begin * TK && s_app < t_end * TK && threadIdx.x < c.dqk / 8) {
            const uint4* src = reinterpret_cast<const uint4*>(a.k_new + (size_t)b * c.dqk);
            bf16* dst = const_cast<bf16*>(a.kc) + ((size_t)slot * c.C + s_app) * c.dqk;
            reinterpret_cast<uint4*>(dst)[threadIdx.x] = src[threadIdx.x];
            asm volatile("fence.proxy.async.global;\n" ::: "memory");   // visible to this CTA's TMA
        }
        m.T += 1;
        __syncthreads();            // every thread has read the meta; the row is written
        if (threadIdx.x == 33) {    // an idle lane of the MMA warp (not the TMA or MMA thread)
            __threadfence();
            if (atomicAdd(&a.meta_rw[slot].pad[0], 1) == (int)gridDim.x - 1) {   // 2 x splits CTAs
                a.meta_rw[slot].T = m.T;
                a.meta_rw[slot].pad[0] = 0;
            }
        }
    }
    if (slot_ok) sv.init(m, c);
    auto next_tile = [&](int t) {
        while (t < t_end && !sv.any_valid(t * TK, min(c.C, (t + 1) * TK))) ++t;
        return t;
    };

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0 && t_begin < t_end) {
            // q, one TMA box per 64-column chunk: chunks 4..8 straight to their place, chunks
            // 0..3 staged in the second KV stage until the softmax warps move them to TMEM
            mbar_expect_tx(bar(B_Q_LOAD), NCH * QCH_B);
            for (int j = 0; j < NCH; ++j) {
                const uint32_t dst = j < QT_CH ? s_kv + NCH * CH_B + j * QCH_B : s_q + (j - QT_CH) * QCH_B;
                tma_load_3d(dst, &tmQ, bar(B_Q_LOAD), 64 * j, 0, b);
            }
            constexpr int AHEAD = 2;    // tiles on their way to L2 ahead of the loads (0-2 time the same; 4: +1.4%)
            int i = 0;
            for (int t = next_tile(t_begin); t < t_end; t = next_tile(t + 1), ++i) {
                cur_tile = t;
                // the first stages' loads go out before any L2 prefetch; then the prefetch
                // runs AHEAD tiles in front of the loads
                if (i == KST)
                    for (int u = t; u < min(t_end, t + AHEAD); ++u)
                        for (int j = 0; j < NCH; ++j) tma_prefetch_3d(&tmKV, 64 * j, u * TK, slot);
                if (i >= KST && t + AHEAD < t_end)
                    for (int j = 0; j < NCH; ++j) tma_prefetch_3d(&tmKV, 64 * j, (t + AHEAD) * TK, slot);
                const int st = i % KST;
                const uint32_t n = i / KST;
                // the second stage holds q's staged chunks until they are in TMEM
                if (i == 1 && !wait_bar(bar(B_Q_FULL), 0, abort_flag)) { fail(0); break; }
                if (!wait_bar(bar(B_KV_EMPTY + st), (n & 1) ^ 1, abort_flag)) { fail(0); break; }
                mbar_expect_tx(bar(B_KV_FULL + st), NCH * CH_B);
                for (int j = 0; j < NCH; ++j)
                    tma_load_3d(s_kv + (st * NCH + j) * CH_B, &tmKV, bar(B_KV_FULL + st), 64 * j, t * TK, slot);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0 && t_begin < t_end) {
            const uint32_t id_qk = idesc_bf16(HEADS, TK);
            const uint32_t id_pv = idesc_bf16_bmn(HEADS, 256);   // this CTA's four value chunks per MMA
            // Descriptors are formed once; the MMAs of a tile add compile-time offsets to
            // their start-address field (16-byte units), so the issuing thread spends a
            // few instructions per MMA (a tcgen05.mma takes ~45 cycles at N = 64).
            const uint64_t q_desc = desc_sw128(s_q);
            const uint64_t kv_desc0 = desc_sw128(s_kv);
            const uint64_t v_desc0 = desc_sw128_mn(s_kv + 4 * half * CH_B, CH_B);
            constexpr uint64_t CH16 = CH_B >> 4, QCH16 = QCH_B >> 4, ST16 = (NCH * CH_B) >> 4;
            bool ok = wait_bar(bar(B_Q_FULL), 0, abort_flag);
            if (!ok) fail(10);
            // Two queues: P V of the oldest tile with weights ready (first: it frees a
            // KV stage for the next load), else the scores of the next tile (needs its
            // KV and its group's buffer back from P V two tiles ago).
            int n_t = 0;
            for (int t = next_tile(t_begin); t < t_end; t = next_tile(t + 1)) ++n_t;
            int qk = 0, pv = 0;
            uint64_t t_idle = 0;
            // P V of the oldest tile whose weights are ready, first (it frees a KV stage for
            // the next load), else the scores of the next tile
            auto try_pv = [&]() -> bool {
                if (!(pv < qk && mbar_test_wait(bar(B_P_FULL + (pv & 1)), (pv >> 1) & 1))) return false;
                tc_fence_after();
                const int stp = pv % KST;
                const uint32_t pa = T_S + (pv & 1) * TK;  // the weights, written over the scores
                const uint64_t vd = v_desc0 + (uint64_t)stp * ST16;
                tc_mma_ta(T_O, pa, vd, id_pv, pv > 0 ? 1u : 0u);
#pragma unroll
                for (int k = 1; k < TK / 16; ++k)       // 16 keys (8 TMEM columns of P) per step
                    tc_mma_ta(T_O, pa + k * 8, vd + (uint64_t)k * (2048 >> 4), id_pv, 1u);
                tc_commit(bar(B_SP_EMPTY + (pv & 1)));
                tc_commit(bar(B_KV_EMPTY + stp));
                ++pv;
                return true;
            };
            while (ok && pv < n_t) {
                bool progressed = try_pv();
                if (!progressed && qk < n_t && mbar_test_wait(bar(B_SP_EMPTY + (qk & 1)), ((qk >> 1) & 1) ^ 1) &&
                    mbar_test_wait(bar(B_KV_FULL + qk % KST), (qk / KST) & 1)) {
                    tc_fence_after();
                    const int st = qk % KST, sb = qk & 1;
                    const uint32_t d = T_S + sb * TK;
                    const uint64_t kd = kv_desc0 + (uint64_t)st * ST16;
                    tc_mma_ta(d, T_Q, kd, id_qk, 0u);
#pragma unroll
                    for (int i = 1; i < 4 * QT_CH; ++i) {    // q chunks 0..3 from TMEM; 16 columns
                        tc_mma_ta(d, T_Q + (i >> 2) * 32 + (i & 3) * 8,   // (8 TMEM columns of q) per step
                                  kd + (uint64_t)((i >> 2) * CH16 + (i & 3) * 2), id_qk, 1u);
                    }
#pragma unroll
                    for (int i = 4 * QT_CH; i < 4 * NCH; ++i) { // q chunks 4..8 from shared memory
                        tc_mma(d, q_desc + (uint64_t)(((i >> 2) - QT_CH) * QCH16 + (i & 3) * 2),
                               kd + (uint64_t)((i >> 2) * CH16 + (i & 3) * 2), id_qk, 1u);
                    }
                    tc_commit(bar(B_S_FULL + sb));
                    ++qk;
                    progressed = true;
                }
                if (progressed) {
                    t_idle = 0;
                } else if (t_idle == 0) {
                    t_idle = globaltimer_ns();
                } else if (__nanosleep(20), globaltimer_ns() - t_idle > WAIT_NS || *abort_flag) {
                    cur_tile = pv;
                    fail(qk < n_t ? 11 : 13);
                    ok = false;
                }
            }
        }
    } else {
        // ------------------------------------------------------------ softmax groups
        const int g = (warp - 2) >> 2;          // group: takes the tiles i with i % NG == g
        const int quarter = warp & 3;           // TMEM lane quarter this warp may access
        const int row = quarter * 32 + lane;    // query head
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const uint32_t t_buf = T_S + lane_off + g * TK;    // this group's score / weight buffer
        const float sl2 = c.scale_log2;
        const uint32_t m_ready = bar(B_M_READY + quarter);
        bool ok = true;

        // q: the TMA load put chunks 4..8 in place (128-byte swizzled K-major tiles) and
        // staged chunks 0..3 in the second KV stage; each lane moves its head's row of a
        // staged chunk into TMEM (the two groups take alternate chunks)
        {
            bool qok = true;
            if (t_begin < t_end)
                qok = __all_sync(0xffffffffu, wait_bar(bar(B_Q_LOAD), 0, abort_flag));
            if (!qok) {
                fail(2);
                ok = false;
            }
            for (int j = g; qok && t_begin < t_end && j < QT_CH; j += NG) {
                const uint32_t src = s_kv + NCH * CH_B + j * QCH_B + (row >> 3) * 1024 + (row & 7) * 128;
                float v[32];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    uint32_t x, y, z, w;
                    asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];\n"
                                 : "=r"(x), "=r"(y), "=r"(z), "=r"(w)
                                 : "r"(src + ((e ^ (row & 7)) << 4))
                                 : "memory");
                    v[4 * e] = __uint_as_float(x);
                    v[4 * e + 1] = __uint_as_float(y);
                    v[4 * e + 2] = __uint_as_float(z);
                    v[4 * e + 3] = __uint_as_float(w);
                }
                tmem_st32(T_Q + lane_off + 32 * j, v);
            }
            fence_proxy_async();    // the staged chunks were read before the stage is reloaded
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_Q_FULL));
        }

        float m_used = NEG_INF;     // the running max this group's sum l_g is relative to
        float l_g = 0.f;
        int i = 0;
        for (int t = next_tile(t_begin); t < t_end; t = next_tile(t + 1), ++i) {
            if ((i & 1) != g || !ok) continue;
            cur_tile = t;
            const int k_g = i >> 1;             // this group's k-th tile: barrier phase parity k_g & 1
            // 0. which of the tile's 64 slots are valid (two ballots), before its scores exist
            const uint32_t v0 = __ballot_sync(0xffffffffu, t * TK + lane < c.C && sv.valid(t * TK + lane));
            const uint32_t v1 =
                __ballot_sync(0xffffffffu, t * TK + 32 + lane < c.C && sv.valid(t * TK + 32 + lane));
            // 1. the scores of tile i, out of TMEM
            float s[TK];
            if (!__all_sync(0xffffffffu, wait_bar(bar(B_S_FULL + g), k_g & 1, abort_flag))) {
                fail(3);
                ok = false;
                continue;
            }
            tc_fence_after();
            {
                float lo[32], hi[32];
                tmem_ld32(t_buf, lo);
                tmem_ld32(t_buf + 32, hi);
                tmem_ld_wait(lo);
                tmem_ld_wait(hi);
#pragma unroll
                for (int k = 0; k < 32; ++k) {
                    s[k] = lo[k];
                    s[32 + k] = hi[k];
                }
            }
            // 2. mask, scale, tile max
            float mt = NEG_INF;
#pragma unroll
            for (int k = 0; k < 32; ++k) {
                s[k] = ((v0 >> k) & 1u) ? s[k] * sl2 : NEG_INF;
                s[32 + k] = ((v1 >> k) & 1u) ? s[32 + k] * sl2 : NEG_INF;
                mt = fmaxf(mt, fmaxf(s[k], s[32 + k]));
            }
            // 3. the running max as left by tile i-1 (the other group)
            float m_prev = NEG_INF;
            if (i > 0) {
                if (!__all_sync(0xffffffffu, wait_bar(m_ready, (i - 1) & 1, abort_flag))) {
                    fail(9);
                    ok = false;
                    continue;
                }
                m_prev = m_sh[row];
            }
            // lazy max: each lane (head) decides whether its max moves; the TMEM rescale
            // of O is done by the whole warp (tcgen05.ld/st are warp-collective), with
            // factor 1 on the lanes whose max stays, once P V of tile i-1 is complete
            // (P V of tile i is not issued before this tile's weights exist).
            const bool move = mt > m_prev + RESCALE_GAP || (m_prev == NEG_INF && mt != NEG_INF);
            const float m_new = move ? fmaxf(mt, m_prev) : m_prev;
            const bool rescale_lane = move && m_prev != NEG_INF;
            if (__any_sync(0xffffffffu, rescale_lane)) {
                // a lane with a finite running max saw weights in an earlier tile: i >= 1.
                // (The scores of tile i-1 waited for P V of tile i-3, so the other
                // group's buffer barrier is at most one phase behind this wait.)
                if (!__all_sync(0xffffffffu,
                                wait_bar(bar(B_SP_EMPTY + ((i - 1) & 1)), ((i - 1) >> 1) & 1, abort_flag))) {
                    fail(5);
                    ok = false;
                    continue;
                }
                tc_fence_after();
                const float alpha = rescale_lane ? ex2(m_prev - m_new) : 1.f;
#pragma unroll 1
                for (int j = 0; j < 8; ++j) {
                    float o[32];
                    tmem_ld32(T_O + lane_off + j * 32, o);
                    tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] *= alpha;
                    tmem_st32(T_O + lane_off + j * 32, o);
                }
                tmem_st_wait();
                tc_fence_before();
            }
            // 4. hand the running max to tile i+1
            m_sh[row] = m_new;
            __syncwarp();
            if (lane == 0) mbar_arrive(m_ready);
            if (m_used != m_new) {
                l_g = m_used == NEG_INF ? l_g : l_g * ex2(m_used - m_new);
                m_used = m_new;
            }
            // 5. weights (bf16, two keys per TMEM column) over this group's scores (read
            //    above, so the buffer is free until P V of this tile releases it)
            float w[32];
            float ps[4] = {0.f, 0.f, 0.f, 0.f};     // independent partial sums
            const float m_sub = m_new == NEG_INF ? 0.f : m_new;   // all scores -inf then: weights 0
#pragma unroll
            for (int e = 0; e < TK / 2; ++e) {
                // one conversion per pair; the sum takes the rounded weights back out of
                // the packed word with integer ops
                const uint32_t pk = pack_bf16(ex2(s[2 * e] - m_sub), ex2(s[2 * e + 1] - m_sub));
                ps[e & 3] += __uint_as_float(pk << 16) + __uint_as_float(pk & 0xffff0000u);
                w[e] = __uint_as_float(pk);
            }
            tmem_st32(t_buf, w);
            tmem_st_wait();
            tc_fence_before();
            l_g += (ps[0] + ps[1]) + (ps[2] + ps[3]);
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_P_FULL + g));
        }
        const int n_t = i;

        // 6. the final running max (from the group of the last tile) and P V of the
        //    last tile done (its commit covers every earlier MMA too)
        float m_fin = NEG_INF;
        if (ok && n_t > 0) {
            if (((n_t - 1) & 1) != g &&
                !__all_sync(0xffffffffu, wait_bar(m_ready, (n_t - 1) & 1, abort_flag))) {
                fail(8);
                ok = false;
            }
            if (ok && !__all_sync(0xffffffffu, wait_bar(bar(B_SP_EMPTY + ((n_t - 1) & 1)), ((n_t - 1) >> 1) & 1,
                                                        abort_flag))) {
                fail(8);
                ok = false;
            }
            if (ok) m_fin = m_sh[row];
            tc_fence_after();
        }
        if (l_g > 0.f && m_used != m_fin) l_g = m_fin == NEG_INF ? 0.f : l_g * ex2(m_used - m_fin);
        l_sh[g * HEADS + row] = l_g;
        asm volatile("bar.sync %0, %1;\n" ::"n"(SOFTMAX_BAR_ID), "n"(NG * 128) : "memory");
        const float l_run = l_sh[row] + l_sh[HEADS + row];

        // 7. this CTA's half of the output; group g writes TMEM columns 128 g .. 128 g + 127
        if (ok && row < c.Hq) {
            const int head = row;
            const int d0 = 256 * half;
            for (int j = 4 * g; j < 4 * g + 4; ++j) {
                float o[32];
                if (n_t > 0) {
                    tmem_ld32(T_O + lane_off + j * 32, o);
                    tmem_ld_wait();
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] = 0.f;
                }
                float* dst;
                float scale = 1.f;
                if (a.splits == 1) {
                    dst = a.out + ((size_t)b * c.Hq + head) * MV + d0 + j * 32;
                    scale = l_run > 0.f ? 1.f / l_run : 0.f;
                } else {
                    const size_t pi = ((size_t)b * a.splits + split) * c.Hq + head;
                    dst = a.part_o + pi * MV + d0 + j * 32;
                }
#pragma unroll
                for (int e = 0; e < 32; e += 4)
                    *reinterpret_cast<float4*>(dst + e) =
                        make_float4(o[e] * scale, o[e + 1] * scale, o[e + 2] * scale, o[e + 3] * scale);
            }
            if (a.splits > 1 && half == 0 && g == 0) {
                const size_t pi = ((size_t)b * a.splits + split) * c.Hq + head;
                a.part_ml[pi * 2 + 0] = m_fin;
                a.part_ml[pi * 2 + 1] = l_run;
            }
        }
    }

    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace

static std::atomic<uint64_t> mla_smem_set{0};

int mla_decode_wave_ctas() {
    static std::atomic<int> cached[64];     // zero-initialised (static storage)
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    const bool cacheable = dev >= 0 && dev < 64;
    if (cacheable) {
        const int c = cached[dev].load(std::memory_order_relaxed);
        if (c > 0) return c;
    }
    if (opt_in_smem(mla_decode_tc_kernel, SMEM, mla_smem_set) != cudaSuccess) return 0;
    int per_sm = 0, sms = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, mla_decode_tc_kernel, THREADS, SMEM) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || per_sm <= 0)
        return 0;
    if (cacheable) cached[dev].store(per_sm * sms, std::memory_order_relaxed);
    return per_sm * sms;
}

cudaError_t launch_decode_mla_tc(const DecodeArgs& a, const CUtensorMap& tkv, const CUtensorMap& tq,
                                 cudaStream_t st) {
    if (cudaError_t e = opt_in_smem(mla_decode_tc_kernel, SMEM, mla_smem_set); e != cudaSuccess) return e;
    dim3 grid(2 * a.splits, a.n);
    return launch_dependent(mla_decode_tc_kernel, grid, dim3(THREADS), SMEM, st, tkv, tq, a);
}

}  // namespace snap
