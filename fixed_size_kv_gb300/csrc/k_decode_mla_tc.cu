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
// Per 64-key tile, each CTA computes its partial scores S_r = Q_r K_r^T into TMEM,
// the two exchange their partials through distributed shared memory (both then hold
// the same S = S_0 + S_1), run the same online softmax (same max, same rounded
// weights), and each accumulates its half of O = P V in TMEM (256 fp32 columns).
// No score is computed twice and each cache byte is read by one CTA only.
//
// Roles (192 threads per CTA): warp 0 issues TMA loads (and L2 prefetches two
// tiles ahead), warp 1 owns TMEM and one thread issues tcgen05.mma, warps 2..5
// (one TMEM lane quarter each; thread = head) run the softmax.  The running max
// is updated lazily (only when a tile's max exceeds it by more than 8 in log2
// units), so O in TMEM is rescaled rarely.  Every wait is bounded.
#include "kernels.cuh"
#include "tc.cuh"

namespace snap {

namespace {

constexpr float NEG_INF = -__builtin_huge_valf();
constexpr int MV = 512;                     // value (latent) width
constexpr int HEADS = 128;                  // M of every MMA
constexpr int TK = 64;                      // keys per tile
constexpr int CH_B = TK * 128;              // one 64-column chunk of a KV tile: 8 KB
constexpr int QCH_B = HEADS * 128;          // one 64-column chunk of Q: 16 KB
constexpr int MAXCH = 5;                    // chunks owned by rank 1
constexpr int KST = 2;                      // KV tile stages
constexpr int THREADS = 192;
constexpr float RESCALE_GAP = 8.f;

constexpr int OFF_Q = 0;
constexpr int OFF_KV = OFF_Q + MAXCH * QCH_B;             // 80 KB
constexpr int OFF_P = OFF_KV + KST * MAXCH * CH_B;        // + 80 KB
constexpr int OFF_X = OFF_P + 2 * HEADS * 128;            // + 32 KB (two P buffers)
constexpr int OFF_BAR = OFF_X + HEADS * TK * 4;           // + 32 KB (score exchange)
constexpr int SMEM = OFF_BAR + 256 + 1024;                // barriers + alignment slack

enum {
    B_Q_FULL = 0,
    B_KV_FULL = 1,               // + KST
    B_KV_EMPTY = 1 + KST,        // + KST
    B_S_FULL = 1 + 2 * KST,      // + 2
    B_S_EMPTY = 3 + 2 * KST,     // + 2
    B_P_FULL = 5 + 2 * KST,      // + 2
    B_P_EMPTY = 7 + 2 * KST,     // + 2
    B_X_FULL = 9 + 2 * KST,
    B_X_EMPTY = 10 + 2 * KST,
    N_BARS = 11 + 2 * KST
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
            mbar_init(bar(B_P_FULL + i), 4);
            mbar_init(bar(B_P_EMPTY + i), 1);
        }
        mbar_init(bar(B_X_FULL), 4);    // the peer's four softmax warps
        mbar_init(bar(B_X_EMPTY), 4);
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
    // TMEM: scores (two buffers) at columns 0 and 64; this CTA's half of O at 256..511
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
            int i = 0;
            for (int t = next_tile(t_begin); t < t_end; t = next_tile(t + 1), ++i) {
                cur_tile = t;
                if (t + 2 < t_end)
                    for (int j = 0; j < nch; ++j) tma_prefetch_3d(&tmKV, 64 * (c0 + j), (t + 2) * TK, slot);
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
            auto issue_pv = [&](int ip) -> bool {
                const int pb = ip & 1, stp = ip % KST;
                if (!wait_bar(bar(B_P_FULL + pb), (ip >> 1) & 1, abort_flag, false)) return false;
                tc_fence_after();
                const uint32_t pa = s_p + pb * HEADS * 128;
#pragma unroll
                for (int j = 0; j < 4; ++j)             // this CTA's four value chunks
#pragma unroll
                    for (int k = 0; k < 4; ++k)         // 16 keys per step
                        tc_mma(T_O + j * 64, desc_sw128(pa + k * 32),
                               desc_sw128_mn(s_kv + (stp * MAXCH + j) * CH_B + k * 2048), id_pv,
                               (ip > 0 || k > 0) ? 1u : 0u);
                tc_commit(bar(B_P_EMPTY + pb));
                tc_commit(bar(B_KV_EMPTY + stp));
                return true;
            };
            int i = 0;
            for (int t = next_tile(t_begin); ok && t < t_end; t = next_tile(t + 1), ++i) {
                cur_tile = t;
                const int st = i % KST, sb = i & 1;
                if (!wait_bar(bar(B_S_EMPTY + sb), ((i >> 1) & 1) ^ 1, abort_flag, false)) {
                    fail(11);
                    ok = false;
                    break;
                }
                if (!wait_bar(bar(B_KV_FULL + st), (i / KST) & 1, abort_flag, false)) {
                    fail(12);
                    ok = false;
                    break;
                }
                tc_fence_after();
                for (int j = 0; j < nch; ++j)
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        tc_mma(T_S + sb * 64, desc_sw128(s_q + j * QCH_B + k * 32),
                               desc_sw128(s_kv + (st * MAXCH + j) * CH_B + k * 32), id_qk, (j | k) ? 1u : 0u);
                tc_commit(bar(B_S_FULL + sb));
                if (i >= 1 && !issue_pv(i - 1)) {
                    fail(13);
                    ok = false;
                    break;
                }
            }
            if (ok && i >= 1 && !issue_pv(i - 1)) fail(14);
        }
    } else {
        // ------------------------------------------------------------ softmax warps
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;    // query head
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const uint32_t x_peer_row = mapa(s_x + row * (TK * 4), peer);
        const uint32_t x_full_peer = mapa(bar(B_X_FULL), peer);
        const uint32_t x_empty_peer = mapa(bar(B_X_EMPTY), peer);
        const float sl2 = c.scale_log2;
        float m_run = NEG_INF, l_run = 0.f;
        int i = 0;
        bool ok = true;
        for (int t = next_tile(t_begin); t < t_end; t = next_tile(t + 1), ++i) {
            cur_tile = t;
            const int sb = i & 1, pb = i & 1;
            // 1. this CTA's partial scores
            if (!__all_sync(0xffffffffu, wait_bar(bar(B_S_FULL + sb), (i >> 1) & 1, abort_flag, false))) {
                fail(2);
                ok = false;
                break;
            }
            tc_fence_after();
            float s[64];
            tmem_ld32(T_S + lane_off + sb * 64, *reinterpret_cast<float(*)[32]>(&s[0]));
            tmem_ld32(T_S + lane_off + sb * 64 + 32, *reinterpret_cast<float(*)[32]>(&s[32]));
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_S_EMPTY + sb));
            // 2. exchange partials with the peer CTA
            if (!__all_sync(0xffffffffu, wait_bar(bar(B_X_EMPTY), (i & 1) ^ 1, abort_flag, true))) {
                fail(3);
                ok = false;
                break;
            }
#pragma unroll
            for (int k = 0; k < 16; ++k)
                st_cluster_v4(x_peer_row + 16 * k, s[4 * k], s[4 * k + 1], s[4 * k + 2], s[4 * k + 3]);
            fence_acq_rel_cluster();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(x_full_peer);
            if (!__all_sync(0xffffffffu, wait_bar(bar(B_X_FULL), i & 1, abort_flag, true))) {
                fail(4);
                ok = false;
                break;
            }
            const float4* xr = reinterpret_cast<const float4*>(smem + OFF_X + row * (TK * 4));
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                const float4 v = xr[k];
                // rank 0 adds S_0 + S_1 and rank 1 S_1 + S_0: the same value in both CTAs
                s[4 * k] += v.x;
                s[4 * k + 1] += v.y;
                s[4 * k + 2] += v.z;
                s[4 * k + 3] += v.w;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(x_empty_peer);
            // 3. the P buffer this tile writes is free once the P V of tile i-2 is done
            if (!__all_sync(0xffffffffu, wait_bar(bar(B_P_EMPTY + pb), ((i >> 1) & 1) ^ 1, abort_flag, false))) {
                fail(5);
                ok = false;
                break;
            }
            // 4. mask, scale, lazy max
            float mt = NEG_INF;
#pragma unroll
            for (int k = 0; k < 64; ++k) {
                const int key = t * TK + k;
                s[k] = (key < c.C && sv.valid(key)) ? s[k] * sl2 : NEG_INF;
                mt = fmaxf(mt, s[k]);
            }
            // Each lane (head) decides whether its max moved; the TMEM rescale of O is
            // done by the whole warp (tcgen05.ld/st are warp-collective), with factor 1
            // on the lanes whose max stays.
            const bool move = mt > m_run + RESCALE_GAP || (m_run == NEG_INF && mt != NEG_INF);
            const float m_new = move ? fmaxf(mt, m_run) : m_run;
            const bool rescale_lane = move && m_run != NEG_INF;
            if (__any_sync(0xffffffffu, rescale_lane)) {
                // O holds sums against the old max: wait for the P V of tile i-1, rescale
                const int ip = i - 1;
                const bool w = wait_bar(bar(B_P_EMPTY + (ip & 1)), (ip >> 1) & 1, abort_flag, false);
                if (!__all_sync(0xffffffffu, w)) {
                    fail(6);
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
            // 5. weights (bf16) into this tile's P buffer (128-byte swizzled K-major rows)
            const uint32_t prow = s_p + pb * HEADS * 128 + (row >> 3) * 1024 + (row & 7) * 128;
            float psum = 0.f;
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) {
                uint32_t w[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float p0 = m_run == NEG_INF ? 0.f : bf16_round(ex2(s[ch * 8 + 2 * e] - m_run));
                    const float p1 = m_run == NEG_INF ? 0.f : bf16_round(ex2(s[ch * 8 + 2 * e + 1] - m_run));
                    psum += p0 + p1;
                    w[e] = pack_bf16(p0, p1);
                }
                const uint32_t dst = prow + ((ch ^ (row & 7)) << 4);
                asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};\n" ::"r"(dst), "r"(w[0]), "r"(w[1]), "r"(w[2]),
                             "r"(w[3])
                             : "memory");
            }
            l_run += psum;
            fence_proxy_async();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_P_FULL + pb));
        }
        // 6. this CTA's half of the output
        if (ok && i >= 1) {
            const int ip = i - 1;
            if (!__all_sync(0xffffffffu, wait_bar(bar(B_P_EMPTY + (ip & 1)), (ip >> 1) & 1, abort_flag, false))) {
                fail(7);
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
