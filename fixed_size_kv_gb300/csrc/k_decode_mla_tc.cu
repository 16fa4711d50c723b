// k_decode_mla_tc.cu -- absorbed-query MLA decode attention over the fixed-size
// cache on the 5th-generation tensor cores.
//
// DeepSeek-R1 shape (SnapStream episode companion page, "16-Socket Deployment:
// Prefill vs. Decode Parallelism"): 128 query heads read one latent KV row
// [latent 512 | rope 64] per cached token; the value is the latent.  The 128 heads
// of one sequence form the M = 128 side of every MMA.
//
// A cluster of two CTAs handles one (sequence, split) and divides the 576 columns:
//   rank 0 owns columns   0..255 (4 chunks of 64): its part of q.k and values 0..255
//   rank 1 owns columns 256..575 (5 chunks):       its part of q.k and values 256..511
// Per 32-key tile, each CTA computes its partial scores S_r = Q_r K_r^T into TMEM,
// the two exchange their partials through distributed shared memory (both then hold
// the same S = S_0 + S_1), run the same online softmax (same max, same rounded
// weights), and each accumulates its half of O = P V in TMEM (256 fp32 columns).
// No score is computed twice and each cache byte is read by one CTA only.
//
// Roles (192 threads per CTA): warp 0 issues TMA loads (and L2 prefetches ahead),
// warp 1 owns TMEM and one thread issues tcgen05.mma from two queues (scores of the
// next tile, P V of the oldest ready tile), warps 2..5 (one TMEM lane quarter each;
// thread = head) run the softmax.  The softmax loop is software-pipelined: the
// TMEM load of tile i+1's partial scores is issued before tile i's exchange and max,
// and those partials go to the peer before tile i's weights are computed, so the
// exchange travels while the math runs.  Exchange buffers and the weight buffer P
// are double-buffered (P's two tiles share each 128-byte swizzled row), so the
// weights of tile i are written while P V of tile i-1 still runs.
// The running max is updated lazily (only when a tile's max exceeds it by more than
// 32 in log2 units), so O in TMEM is rescaled rarely.  Every wait is bounded.
#include "kernels.cuh"
#include "tc.cuh"

namespace snap {

namespace {

constexpr float NEG_INF = -__builtin_huge_valf();
constexpr int MV = 512;                     // value (latent) width
constexpr int HEADS = 128;                  // M of every MMA
constexpr int TK = 32;                      // keys per tile
constexpr int CH_B = TK * 128;              // one 64-column chunk of a KV tile: 4 KB
constexpr int QCH_B = HEADS * 128;          // one 64-column chunk of Q: 16 KB
constexpr int MAXCH = 5;                    // chunks owned by rank 1
constexpr int KST = 4;                      // KV tile stages
constexpr int THREADS = 192;
constexpr float RESCALE_GAP = 32.f;         // weights up to 2^32 stay exact in fp32 O and l
constexpr int XROW_B = TK * 4;              // one head's partial scores: 128 B

constexpr int OFF_Q = 0;
constexpr int OFF_KV = OFF_Q + MAXCH * QCH_B;             // 80 KB
constexpr int OFF_P = OFF_KV + KST * MAXCH * CH_B;        // + 80 KB
constexpr int OFF_X = OFF_P + HEADS * 128;                // + 16 KB (P: 128-byte rows, two 32-key tiles)
constexpr int OFF_BAR = OFF_X + 2 * HEADS * XROW_B;       // + 32 KB (two exchange buffers)
constexpr int SMEM = OFF_BAR + 256 + 1024;                // barriers + alignment slack

enum {
    B_Q_FULL = 0,
    B_KV_FULL = 1,               // + KST
    B_KV_EMPTY = 1 + KST,        // + KST
    B_S_FULL = 1 + 2 * KST,      // + 2
    B_S_EMPTY = 3 + 2 * KST,     // + 2
    B_P_FULL = 5 + 2 * KST,      // + 2
    B_P_EMPTY = 7 + 2 * KST,     // + 2
    B_X_FULL = 9 + 2 * KST,      // + 2
    B_X_EMPTY = 11 + 2 * KST,    // + 2
    N_BARS = 13 + 2 * KST
};

__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag, bool cluster) {
    return mbar_wait_bounded(bar, parity, abort_flag, cluster);
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(THREADS, 1)
    mla_decode_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmKV,
                         DecodeArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const DevConfig& c = a.cfg;
    const uint32_t rank = cluster_rank();
    const uint32_t peer = rank ^ 1u;
    const int split = blockIdx.x >> 1, b = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nch = rank == 0 ? 4 : 5;          // chunks owned
    const int c0 = rank == 0 ? 0 : 4;           // first owned chunk

    const uint32_t s_base = smem_u32(smem);
    const uint32_t s_q = s_base + OFF_Q, s_kv = s_base + OFF_KV, s_p = s_base + OFF_P, s_x = s_base + OFF_X;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
    auto bar = [&](int i) { return smem_u32(bars + i); };
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + N_BARS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

    const int slot = a.slots[b];
    const bool slot_ok = slot >= 0 && slot < c.max_batch;

    if (threadIdx.x == 0) {
        mbar_init(bar(B_Q_FULL), 1);
        for (int i = 0; i < KST; ++i) {
            mbar_init(bar(B_KV_FULL + i), 1);
            mbar_init(bar(B_KV_EMPTY + i), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(B_S_FULL + i), 1);
            mbar_init(bar(B_S_EMPTY + i), 4);
            mbar_init(bar(B_X_FULL + i), 1);    // this CTA's expect_tx + the peer's st.async bytes
            mbar_init(bar(B_X_EMPTY + i), 4);   // the peer's four softmax warps
            mbar_init(bar(B_P_FULL + i), 4);
            mbar_init(bar(B_P_EMPTY + i), 1);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_holder), 512);
        tmem_relinquish();
    }
    __syncthreads();
    cluster_sync_all();                 // both CTAs' barriers exist before any remote arrive
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    // TMEM: scores (two buffers) at columns 0 and 32; this CTA's half of O at 256..511
    const uint32_t T_S = tmem, T_O = tmem + 256;

    // status detail: 300 + rank, the wait that gave up, the tile index reached
    int cur_tile = -1;
    auto fail = [&](int role) {
        *abort_flag = 1;
        report_error(a.status, SNAP_ERR_TIMEOUT, 300 + (int)rank, role, cur_tile);
    };

    SlotValidity sv;
    snap_seq_meta m{};
    if (slot_ok) {
        m = a.meta[slot];
        sv.init(m, c);
    } else if (threadIdx.x == 0 && split == 0 && rank == 0) {
        report_error(a.status, SNAP_ERR_DEVICE_CHECK, 1, b, slot);
    }
    const int ntiles = (c.C + TK - 1) / TK;
    const int t_begin = split * a.tiles_per_split;
    const int t_end = slot_ok ? min(ntiles, t_begin + a.tiles_per_split) : t_begin;
    auto next_tile = [&](int t) {
        while (t < t_end && !sv.any_valid(t * TK, min(c.C, (t + 1) * TK))) ++t;
        return t;
    };

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0 && t_begin < t_end) {
            tma_prefetch(&tmQ);
            tma_prefetch(&tmKV);
            mbar_expect_tx(bar(B_Q_FULL), nch * QCH_B);
            for (int j = 0; j < nch; ++j) tma_load_3d(s_q + j * QCH_B, &tmQ, bar(B_Q_FULL), 64 * (c0 + j), 0, b);
            constexpr int AHEAD = 8;    // tiles on their way to L2 ahead of the loads
            for (int t = t_begin; t < min(t_end, t_begin + AHEAD); ++t)
                for (int j = 0; j < nch; ++j) tma_prefetch_3d(&tmKV, 64 * (c0 + j), t * TK, slot);
            int i = 0;
            for (int t = next_tile(t_begin); t < t_end; t = next_tile(t + 1), ++i) {
                cur_tile = t;
                if (t + AHEAD < t_end)
                    for (int j = 0; j < nch; ++j) tma_prefetch_3d(&tmKV, 64 * (c0 + j), (t + AHEAD) * TK, slot);
                const int st = i % KST;
                const uint32_t n = i / KST;
                if (!wait_bar(bar(B_KV_EMPTY + st), (n & 1) ^ 1, abort_flag, false)) { fail(0); break; }
                mbar_expect_tx(bar(B_KV_FULL + st), nch * CH_B);
                for (int j = 0; j < nch; ++j)
                    tma_load_3d(s_kv + (st * MAXCH + j) * CH_B, &tmKV, bar(B_KV_FULL + st), 64 * (c0 + j), t * TK,
                                slot);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0 && t_begin < t_end) {
            const uint32_t id_qk = idesc_bf16(HEADS, TK);
            const uint32_t id_pv = idesc_bf16_bmn(HEADS, 64);
            bool ok = wait_bar(bar(B_Q_FULL), 0, abort_flag, false);
            if (!ok) fail(10);
            // Two queues: the scores of the next tile (needs its KV and a free score
            // buffer) and P V of the oldest tile with weights ready.  Issue whichever is
            // ready, so P V never waits behind the next tile's data.
            int n_t = 0;
            for (int t = next_tile(t_begin); t < t_end; t = next_tile(t + 1)) ++n_t;
            int qk = 0, pv = 0;
            uint64_t t_idle = 0;
            while (ok && pv < n_t) {
                bool progressed = false;
                if (qk < n_t && mbar_test_wait(bar(B_S_EMPTY + (qk & 1)), ((qk >> 1) & 1) ^ 1) &&
                    mbar_test_wait(bar(B_KV_FULL + qk % KST), (qk / KST) & 1)) {
                    tc_fence_after();
                    const int st = qk % KST, sb = qk & 1;
                    for (int j = 0; j < nch; ++j)
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            tc_mma(T_S + sb * TK, desc_sw128(s_q + j * QCH_B + k * 32),
                                   desc_sw128(s_kv + (st * MAXCH + j) * CH_B + k * 32), id_qk, (j | k) ? 1u : 0u);
                    tc_commit(bar(B_S_FULL + sb));
                    ++qk;
                    progressed = true;
                }
                if (pv < qk && mbar_test_wait(bar(B_P_FULL + (pv & 1)), (pv >> 1) & 1)) {
                    tc_fence_after();
                    const int stp = pv % KST;
                    const uint32_t pa = s_p + (pv & 1) * 64;   // this tile's half of the P rows
#pragma unroll
                    for (int j = 0; j < 4; ++j)             // this CTA's four value chunks
#pragma unroll
                        for (int k = 0; k < TK / 16; ++k)   // 16 keys per step
                            tc_mma(T_O + j * 64, desc_sw128(pa + k * 32),
                                   desc_sw128_mn(s_kv + (stp * MAXCH + j) * CH_B + k * 2048), id_pv,
                                   (pv > 0 || k > 0) ? 1u : 0u);
                    tc_commit(bar(B_P_EMPTY + (pv & 1)));
                    tc_commit(bar(B_KV_EMPTY + stp));
                    ++pv;
                    progressed = true;
                }
                if (progressed) {
                    t_idle = 0;
                } else if (t_idle == 0) {
                    t_idle = globaltimer_ns();
                } else if (globaltimer_ns() - t_idle > WAIT_NS || *abort_flag) {
                    cur_tile = pv;
                    fail(qk < n_t ? 11 : 13);
                    ok = false;
                }
            }
        }
    } else {
        // ------------------------------------------------------------ softmax warps
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;    // query head
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const float sl2 = c.scale_log2;
        int n_t = 0;
        for (int t = next_tile(t_begin); t < t_end; t = next_tile(t + 1)) ++n_t;
        bool ok = true;
        // Sends tile j's partial scores (in registers) into the peer's exchange buffer
        // j & 1; the 16-byte chunks of a 128-byte row are XOR-swizzled by row so that a
        // warp reading chunk k of 32 rows hits distinct banks.
        auto send = [&](int j, const float (&s)[TK]) -> bool {
            const int xb = j & 1;
            // the peer has consumed what this CTA sent two tiles ago into that buffer
            if (!__all_sync(0xffffffffu, wait_bar(bar(B_X_EMPTY + xb), ((j >> 1) & 1) ^ 1, abort_flag, true)))
                return false;
            // the peer's scores of tile j will land in this CTA's buffer xb: announce the bytes
            if (quarter == 0 && lane == 0) mbar_expect_tx(bar(B_X_FULL + xb), HEADS * XROW_B);
            const uint32_t dst = mapa(s_x + xb * HEADS * XROW_B + row * XROW_B, peer);
            const uint32_t xfull_peer = mapa(bar(B_X_FULL + xb), peer);
#pragma unroll
            for (int k = 0; k < TK / 4; ++k)
                st_async_v4(dst + 16 * (k ^ (row & 7)), s[4 * k], s[4 * k + 1], s[4 * k + 2], s[4 * k + 3], xfull_peer);
            return true;
        };
        // Issues the TMEM load of tile j's partial scores (completed by finish_scores).
        auto start_scores = [&](int j, float (&s)[TK]) -> bool {
            const int sb = j & 1;
            if (!__all_sync(0xffffffffu, wait_bar(bar(B_S_FULL + sb), (j >> 1) & 1, abort_flag, false))) return false;
            tc_fence_after();
            tmem_ld32(T_S + lane_off + sb * TK, s);
            return true;
        };
        // Waits for that load and frees the score buffer for the scores of tile j + 2.
        auto finish_scores = [&](int j, float (&s)[TK]) {
            tmem_ld_wait(s);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_S_EMPTY + (j & 1)));
        };

        float m_run = NEG_INF, l_run = 0.f;
        float s_next[TK];
        if (n_t > 0) {
            if (start_scores(0, s_next)) {
                finish_scores(0, s_next);
                if (!send(0, s_next)) ok = false;
            } else {
                ok = false;
            }
            if (!ok) fail(2);
        }
        int i = 0;
        for (int t = next_tile(t_begin); ok && t < t_end; t = next_tile(t + 1), ++i) {
            cur_tile = t;
            float s[TK];
#pragma unroll
            for (int k = 0; k < TK; ++k) s[k] = s_next[k];
            // 1. the TMEM load of the next tile's partial scores runs during steps 2-3
            const bool has_next = i + 1 < n_t;
            if (has_next && !start_scores(i + 1, s_next)) {
                fail(3);
                ok = false;
                break;
            }
            // 2. the peer's partial scores of this tile
            const int xb = i & 1;
            if (!__all_sync(0xffffffffu, wait_bar(bar(B_X_FULL + xb), (i >> 1) & 1, abort_flag, true))) {
                fail(4);
                ok = false;
                break;
            }
            const float4* xr = reinterpret_cast<const float4*>(smem + OFF_X + xb * HEADS * XROW_B + row * XROW_B);
#pragma unroll
            for (int k = 0; k < TK / 4; ++k) {
                const float4 v = xr[k ^ (row & 7)];
                // rank 0 adds S_0 + S_1 and rank 1 S_1 + S_0: the same value in both CTAs
                s[4 * k] += v.x;
                s[4 * k + 1] += v.y;
                s[4 * k + 2] += v.z;
                s[4 * k + 3] += v.w;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(mapa(bar(B_X_EMPTY + xb), peer));
            // 3. mask (one ballot for the tile's 32 slots), scale, tile max
            const uint32_t vmask = __ballot_sync(0xffffffffu, t * TK + lane < c.C && sv.valid(t * TK + lane));
            float mt = NEG_INF;
#pragma unroll
            for (int k = 0; k < TK; ++k) {
                s[k] = ((vmask >> k) & 1u) ? s[k] * sl2 : NEG_INF;
                mt = fmaxf(mt, s[k]);
            }
            // 4. the next tile's partial scores go to the peer before this tile's weights
            if (has_next) {
                finish_scores(i + 1, s_next);
                if (!send(i + 1, s_next)) {
                    fail(6);
                    ok = false;
                    break;
                }
            }
            // 5. lazy max: each lane (head) decides whether its max moved; the TMEM
            //    rescale of O is done by the whole warp (tcgen05.ld/st are
            //    warp-collective), with factor 1 on the lanes whose max stays, once P V
            //    of tile i-1 (the last one issued) is complete.
            const bool move = mt > m_run + RESCALE_GAP || (m_run == NEG_INF && mt != NEG_INF);
            const float m_new = move ? fmaxf(mt, m_run) : m_run;
            const bool rescale_lane = move && m_run != NEG_INF;
            if (__any_sync(0xffffffffu, rescale_lane)) {
                // a lane with a finite running max had weights in an earlier tile: i >= 1
                if (!__all_sync(0xffffffffu,
                                wait_bar(bar(B_P_EMPTY + ((i - 1) & 1)), ((i - 1) >> 1) & 1, abort_flag, false))) {
                    fail(5);
                    ok = false;
                    break;
                }
                tc_fence_after();
                const float alpha = rescale_lane ? ex2(m_run - m_new) : 1.f;
                l_run *= alpha;
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
            m_run = m_new;
            // 6. weights (bf16) into this tile's half of the P rows (128-byte swizzled
            //    K-major rows: tile i uses 16-byte chunks 4 (i & 1) .. 4 (i & 1) + 3),
            //    once P V of tile i-2 has released that half
            if (!__all_sync(0xffffffffu, wait_bar(bar(B_P_EMPTY + (i & 1)), ((i >> 1) & 1) ^ 1, abort_flag, false))) {
                fail(7);
                ok = false;
                break;
            }
            const uint32_t prow = s_p + (row >> 3) * 1024 + (row & 7) * 128;
            float psum = 0.f;
#pragma unroll
            for (int ch = 0; ch < TK / 8; ++ch) {
                uint32_t w[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float p0 = m_run == NEG_INF ? 0.f : bf16_round(ex2(s[ch * 8 + 2 * e] - m_run));
                    const float p1 = m_run == NEG_INF ? 0.f : bf16_round(ex2(s[ch * 8 + 2 * e + 1] - m_run));
                    psum += p0 + p1;
                    w[e] = pack_bf16(p0, p1);
                }
                const uint32_t dst = prow + ((((i & 1) * 4 + ch) ^ (row & 7)) << 4);
                asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};\n" ::"r"(dst), "r"(w[0]), "r"(w[1]), "r"(w[2]),
                             "r"(w[3])
                             : "memory");
            }
            l_run += psum;
            fence_proxy_async();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_P_FULL + (i & 1)));
        }
        // 6. this CTA's half of the output (once P V of the last tile is done)
        if (ok && i >= 1) {
            // the commit after P V of the last tile covers every earlier MMA too
            if (!__all_sync(0xffffffffu,
                            wait_bar(bar(B_P_EMPTY + ((i - 1) & 1)), ((i - 1) >> 1) & 1, abort_flag, false))) {
                fail(8);
                ok = false;
            }
            tc_fence_after();
        }
        if (ok && row < c.Hq) {
            const int head = row;
            const int d0 = rank == 0 ? 0 : 256;
            for (int j = 0; j < 8; ++j) {
                float o[32];
                if (i >= 1) {
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
            if (a.splits > 1 && rank == 0) {
                const size_t pi = ((size_t)b * a.splits + split) * c.Hq + head;
                a.part_ml[pi * 2 + 0] = m_run;
                a.part_ml[pi * 2 + 1] = l_run;
            }
        }
    }

    __syncthreads();
    cluster_sync_all();                 // no CTA leaves while its peer may still write to it
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace

cudaError_t launch_decode_mla_tc(const DecodeArgs& a, const CUtensorMap& tq, const CUtensorMap& tkv, cudaStream_t st) {
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(mla_decode_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    dim3 grid(2 * a.splits, a.n);
    mla_decode_tc_kernel<<<grid, THREADS, SMEM, st>>>(tq, tkv, a);
    return cudaGetLastError();
}

}  // namespace snap
