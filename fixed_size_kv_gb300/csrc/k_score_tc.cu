// k_score_tc.cu -- the observation-window score GEMM on the 5th-generation tensor
// cores (tcgen05 + TMEM), fed by TMA.
//
// SnapStream episode companion page, "Fixed-Size Cache Layout": the middle of the
// cache holds the SnapKV top-K tokens chosen at prefill.  The scores come from the
// window queries' softmax over the prompt keys: for KV head h, observation row
// r = (w, g) (query head h*G+g at position S-W+w) against key j, the logit is
// s = sm_scale * log2(e) * q.k (base-2 domain).  This GEMM, R x d by d x S per KV
// head, is the dense contraction of the compression step.
//
// One persistent kernel template, three epilogues:
//   ROWSTAT  X = 128 observation rows (resident), Y = 256-key tiles (streamed);
//            TMEM lane = row; per row a partial (max, sum 2^(s-max)) over its keys,
//            with the causal limit j <= S-W+w.
//   COLSUM   X = 128-key tiles, Y = observation rows; TMEM lane = key; per key the
//            sum over rows of 2^(s - lse2(row)) for keys j < S-W (which every
//            window row sees, so no causal limit applies).
//   LOGITS   as ROWSTAT, writing the raw base-2 logits (inspection / GEMM checks).
//
// Roles (576 threads): warp 0 issues TMA loads, warp 1 owns TMEM and one thread
// issues tcgen05.mma, warps 2..17 read TMEM (warp w reads lanes 32*(w%4).. of part
// (w-2)/4 of the columns: four epilogue warps per SM sub-partition, so that the
// latency of one warp's ex2 / add chains is hidden by the others).  The accumulator is double-buffered in TMEM (2 x 256
// columns) so the epilogue of one tile overlaps the MMAs of the next.  Every wait
// is bounded; on expiry the kernel records SNAP_ERR_TIMEOUT, drains and exits.
#include "kernels.cuh"
#include "tc.cuh"

namespace snap {

namespace {

constexpr float NEG_INF = -__builtin_huge_valf();

enum { ROWSTAT = SCORE_ROWSTAT, COLSUM = SCORE_COLSUM, LOGITS = SCORE_LOGITS };

constexpr int XROWS = 128;                 // rows of the X operand per MMA (M)
constexpr int CHUNK_B = 128;               // bytes per swizzled row (64 bf16)
constexpr int SMEM_BUDGET = 216 * 1024;    // operand bytes per CTA
constexpr int EPI_WARPS = 4 * SCORE_PARTS;  // epilogue warps: one per (TMEM lane quarter, column part)
constexpr int THREADS = 64 + 32 * EPI_WARPS;

template <int D, bool XRES>
struct Layout {
    static constexpr int KCH = D / 64;                           // 64-column chunks
    static constexpr int XB = XROWS * CHUNK_B;                   // one X chunk: 16 KB
    static constexpr int YB = 256 * CHUNK_B;                     // one Y chunk (max rows): 32 KB
    static constexpr int RES_CH = XRES ? XB : YB;
    static constexpr int STG = XRES ? YB : XB;
    static constexpr int RES_BYTES = KCH * RES_CH;
    static constexpr int ST_RAW = (SMEM_BUDGET - RES_BYTES) / STG;
    static constexpr int STAGES = ST_RAW > 8 ? 8 : ST_RAW;
    static constexpr int BAR_OFF = RES_BYTES + STAGES * STG;
    static constexpr int TOTAL = BAR_OFF + 1024 + 1024;                      // + alignment slack
};

__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
    return mbar_wait_bounded(bar, parity, abort_flag);
}

// sum_i 2^(v_i * a + b) over 32 values: the arguments two at a time (packed f32x2 FMA),
// the sums in four packed f32x2 accumulators
__device__ __forceinline__ float sum32_ex2(const float (&v)[32], float a, float b) {
    const uint64_t a2 = f32x2_splat(a), b2 = f32x2_splat(b);
    uint64_t t[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        float x0, x1;
        fma_f32x2(x0, x1, v[2 * k], v[2 * k + 1], a2, b2);
        add_f32x2(t[k & 3], __float_as_uint(ex2(x0)), __float_as_uint(ex2(x1)));
    }
    return (f32x2_sum(t[0]) + f32x2_sum(t[1])) + (f32x2_sum(t[2]) + f32x2_sum(t[3]));
}

// max of 32 values: four chains of three-operand max
__device__ __forceinline__ float max32(const float (&v)[32]) {
    float t[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) t[k] = fmax3(v[3 * k], v[3 * k + 1], v[3 * k + 2]);   // 0..11
#pragma unroll
    for (int i = 12; i < 28; i += 8)
#pragma unroll
        for (int k = 0; k < 4; ++k) t[k] = fmax3(t[k], v[i + 2 * k], v[i + 2 * k + 1]);   // 12..27
#pragma unroll
    for (int k = 0; k < 4; ++k) t[k] = fmaxf(t[k], v[28 + k]);                           // 28..31
    return fmaxf(fmaxf(t[0], t[1]), fmaxf(t[2], t[3]));
}

struct Unit {
    int h;
    int xt;        // X tile (fixed for XRES)
    int yt0;       // first Y tile (XRES) / Y tile (resident Y)
    int xt0;       // first X tile (!XRES)
    int nsteps;
    int split;
};

template <int MODE, bool XRES>
__device__ __forceinline__ Unit decode_unit(int u, const ScoreParams& p) {
    Unit U;
    if (MODE != COLSUM) {
        // (h, split, x tile) over row tiles; Y = key tiles up to the tile's causal limit.
        // The row tiles of one key split are neighbours in u, so the CTAs running at the
        // same time stream the same key range and share it in L2.
        const int per_h = p.x_tiles * p.splits;
        U.h = u / per_h;
        const int rem = u % per_h;
        U.split = rem / p.x_tiles;
        U.xt = rem % p.x_tiles;
        const int row_last = min(p.R, (U.xt + 1) * XROWS) - 1;
        const int kmax = min(p.S, p.S - p.W + row_last / p.G + 1);
        const int ny = (kmax + p.Ny - 1) / p.Ny;
        const int per = (ny + p.splits - 1) / p.splits;
        U.yt0 = U.split * per;
        U.nsteps = max(0, min(ny, U.yt0 + per) - U.yt0);
        U.xt0 = U.xt;
    } else if (!XRES) {
        // (h, split) over key tiles; Y = all observation rows, resident
        U.h = u / p.splits;
        U.split = u % p.splits;
        const int nx = (p.n_sc + XROWS - 1) / XROWS;
        const int per = (nx + p.splits - 1) / p.splits;
        U.xt0 = U.split * per;
        U.nsteps = max(0, min(nx, U.xt0 + per) - U.xt0);
        U.xt = U.xt0;
        U.yt0 = 0;
    } else {
        // (h, key tile); Y = observation-row tiles, streamed
        const int nx = (p.n_sc + XROWS - 1) / XROWS;
        U.h = u / nx;
        U.xt = u % nx;
        U.xt0 = U.xt;
        U.yt0 = 0;
        U.split = 0;
        U.nsteps = (p.R + p.Ny - 1) / p.Ny;
    }
    return U;
}

// Loads chunk c of `rows` rows starting at tile row0 of operand Q or K.
__device__ __forceinline__ void load_q(uint32_t dst, const CUtensorMap* m, uint32_t bar, int c, int row0, int G,
                                       int h) {
    tma_load_4d(dst, m, bar, c * 64, 0, row0 / G, h);
}
__device__ __forceinline__ void load_k(uint32_t dst, const CUtensorMap* m, uint32_t bar, int c, int key0, int h) {
    tma_load_3d(dst, m, bar, c * 64, key0, h);
}

template <int MODE, int D, bool XQ, bool XRES>
__global__ void __launch_bounds__(THREADS, 1)
    score_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmY,
                    ScoreParams p) {
    using L = Layout<D, XRES>;
    constexpr int KCH = L::KCH;
    constexpr int STAGES = L::STAGES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t s_base = smem_u32(smem);
    const uint32_t s_res = s_base;
    const uint32_t s_stg = s_base + L::RES_BYTES;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);
    auto bar = [&](int i) { return smem_u32(bars + i); };
    // barrier indices
    const int B_FULL = 0, B_EMPTY = STAGES, B_RES_FULL = 2 * STAGES, B_RES_EMPTY = 2 * STAGES + 1,
              B_ACC_FULL = 2 * STAGES + 2, B_ACC_EMPTY = 2 * STAGES + 4;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 6);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int Ny = p.Ny;
    const uint32_t x_bytes = XROWS * CHUNK_B;
    const uint32_t y_bytes = (uint32_t)Ny * CHUNK_B;

    if (threadIdx.x == 0) {
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(bar(B_FULL + i), 1);
            mbar_init(bar(B_EMPTY + i), 1);
        }
        mbar_init(bar(B_RES_FULL), 1);
        mbar_init(bar(B_RES_EMPTY), 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar(B_ACC_FULL + b), 1);
            mbar_init(bar(B_ACC_EMPTY + b), EPI_WARPS);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_holder), 512);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch(&tmX);
        tma_prefetch(&tmY);
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    // the next kernel (the selection after a column pass) may launch and wait for this grid
    pdl_launch_dependents();

    auto fail = [&](int role, int u) {
        *abort_flag = 1;
        report_error(p.status, SNAP_ERR_TIMEOUT, 100 + MODE, role, u);
    };

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            uint32_t it = 0, nu = 0;
            for (int u = blockIdx.x; u < p.n_units; u += gridDim.x) {
                const Unit U = decode_unit<MODE, XRES>(u, p);
                if (U.nsteps == 0) continue;
                if (!wait_or_abort(bar(B_RES_EMPTY), (nu & 1) ^ 1, abort_flag)) { fail(0, u); break; }
                mbar_expect_tx(bar(B_RES_FULL), KCH * (XRES ? x_bytes : y_bytes));
                for (int c = 0; c < KCH; ++c) {
                    const uint32_t dst = s_res + c * L::RES_CH;
                    if (XRES) {
                        if (XQ) load_q(dst, &tmX, bar(B_RES_FULL), c, U.xt * XROWS, p.G, U.h);
                        else load_k(dst, &tmX, bar(B_RES_FULL), c, U.xt * XROWS, U.h);
                    } else {
                        // resident Y: all observation rows
                        load_q(dst, &tmY, bar(B_RES_FULL), c, 0, p.G, U.h);
                    }
                }
                for (int s = 0; s < U.nsteps; ++s) {
                    for (int c = 0; c < KCH; ++c, ++it) {
                        const int slot = it % STAGES;
                        const uint32_t n = it / STAGES;
                        if (!wait_or_abort(bar(B_EMPTY + slot), (n & 1) ^ 1, abort_flag)) { fail(0, u); goto prod_done; }
                        mbar_expect_tx(bar(B_FULL + slot), XRES ? y_bytes : x_bytes);
                        const uint32_t dst = s_stg + slot * L::STG;
                        if (XRES) {
                            const int row0 = (U.yt0 + s) * Ny;
                            if (XQ) load_k(dst, &tmY, bar(B_FULL + slot), c, row0, U.h);
                            else load_q(dst, &tmY, bar(B_FULL + slot), c, row0, p.G, U.h);
                        } else {
                            load_k(dst, &tmX, bar(B_FULL + slot), c, (U.xt0 + s) * XROWS, U.h);
                        }
                    }
                }
                ++nu;
            }
        prod_done:;
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16(XROWS, Ny);
            uint32_t it = 0, acc_it = 0, nu = 0;
            for (int u = blockIdx.x; u < p.n_units; u += gridDim.x) {
                const Unit U = decode_unit<MODE, XRES>(u, p);
                if (U.nsteps == 0) continue;
                if (!wait_or_abort(bar(B_RES_FULL), nu & 1, abort_flag)) { fail(1, u); break; }
                tc_fence_after();
                for (int s = 0; s < U.nsteps; ++s, ++acc_it) {
                    const int buf = acc_it & 1;
                    const uint32_t na = acc_it >> 1;
                    if (!wait_or_abort(bar(B_ACC_EMPTY + buf), (na & 1) ^ 1, abort_flag)) { fail(1, u); goto mma_done; }
                    tc_fence_after();
                    const uint32_t d_tmem = tmem + buf * 256;
                    for (int c = 0; c < KCH; ++c, ++it) {
                        const int slot = it % STAGES;
                        const uint32_t n = it / STAGES;
                        if (!wait_or_abort(bar(B_FULL + slot), n & 1, abort_flag)) { fail(1, u); goto mma_done; }
                        tc_fence_after();
                        const uint32_t xa = XRES ? s_res + c * L::RES_CH : s_stg + slot * L::STG;
                        const uint32_t ya = XRES ? s_stg + slot * L::STG : s_res + c * L::RES_CH;
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            tc_mma(d_tmem, desc_sw128(xa + k * 32), desc_sw128(ya + k * 32), idesc,
                                   (c | k) != 0 ? 1u : 0u);
                        tc_commit(bar(B_EMPTY + slot));
                    }
                    tc_commit(bar(B_ACC_FULL + buf));
                }
                tc_commit(bar(B_RES_EMPTY));
                ++nu;
            }
        mma_done:;
        }
    } else {
        // ------------------------------------------------------------ epilogue
        // launched behind the row statistics' merge (column pass): -lse2 is read from here
        // on; the loads and MMAs above read only the caller's K and Q
        pdl_wait();
        const int ew = warp - 2;
        const int quarter = warp & 3;
        const int part = ew >> 2;
        const int trow = quarter * 32 + lane;     // TMEM lane = X row within the tile
        // this part's accumulator columns: Ny / SCORE_PARTS rounded up to whole 32-column
        // chunks (the last parts get none when Ny is small)
        const int pcols = ((Ny / SCORE_PARTS + 31) / 32) * 32;
        const int cbeg = min(Ny, part * pcols);
        const int ncol = min(Ny, cbeg + pcols) - cbeg;
        const float sl2 = p.sl2;
        // COLSUM: the column sums stay in L2 for the selection that reads them next,
        // past the key tiles streaming through it
        const uint64_t keep_l2 = l2_policy_evict_last();
        uint32_t acc_it = 0;
        for (int u = blockIdx.x; u < p.n_units; u += gridDim.x) {
            const Unit U = decode_unit<MODE, XRES>(u, p);
            float m = NEG_INF, l = 0.f, acc = 0.f;
            const int r = U.xt * XROWS + trow;    // observation row (ROWSTAT/LOGITS)
            const int pos = (r < p.R) ? p.S - p.W + r / p.G : -1;
            for (int s = 0; s < U.nsteps; ++s, ++acc_it) {
                const int buf = acc_it & 1;
                const uint32_t na = acc_it >> 1;
                // warp-uniform exit: the TMEM loads below are warp-collective
                if (!__all_sync(0xffffffffu, wait_or_abort(bar(B_ACC_FULL + buf), na & 1, abort_flag))) {
                    fail(2, u);
                    goto epi_done;
                }
                tc_fence_after();
                const int y0 = (XRES ? (U.yt0 + s) : U.yt0) * Ny;   // first column's key / row index
                // -lse2 of the observation rows on this tile's columns (same for every lane)
                const float* nl = (MODE == COLSUM) ? p.nlse2 + (size_t)U.h * p.R_pad + y0 : nullptr;
                for (int cc = 0; cc < ncol; cc += 32) {
                    const int col0 = cbeg + cc;
                    float v[32];
                    tmem_ld32(tmem + ((uint32_t)(quarter * 32) << 16) + buf * 256 + col0, v);
                    tmem_ld_wait();
                    if (MODE == ROWSTAT) {
                        const int key0 = y0 + col0;
                        if (key0 + 31 > p.S - p.W) {  // near the causal limit: mask
#pragma unroll
                            for (int i = 0; i < 32; ++i)
                                if (key0 + i > pos) v[i] = NEG_INF;
                        }
                        // The reference m is kept lazily: it is set from a chunk's true
                        // maximum only when it is still -inf or when the chunk's sum against
                        // it leaves [0, 2^32] (a logit more than ~27 above m, or overflow).
                        // l * 2^m is exact either way.
                        float sum = 0.f;
                        bool redo = (m == NEG_INF);
                        if (!redo) {
                            sum = sum32_ex2(v, sl2, -m);
                            redo = !(sum <= 4294967296.f);
                        }
                        if (redo) {
                            float mx = max32(v) * sl2;
                            const float mn = fmaxf(m, mx);
                            if (mn != NEG_INF) {
                                sum = sum32_ex2(v, sl2, -mn);
                                l = l * ex2(m - mn);
                                m = mn;
                            } else {
                                sum = 0.f;
                            }
                        }
                        l += sum;
                    } else if (MODE == COLSUM) {
                        const float4* nl4 = reinterpret_cast<const float4*>(nl + col0);
                        const uint64_t sl2x2 = f32x2_splat(sl2);
                        uint64_t s2[2] = {0ull, 0ull};   // packed f32x2 accumulators
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const float4 b = __ldg(nl4 + i);
                            float x0, x1, x2, x3;
                            fma_f32x2(x0, x1, v[4 * i + 0], v[4 * i + 1], sl2x2, f32x2_pack(b.x, b.y));
                            fma_f32x2(x2, x3, v[4 * i + 2], v[4 * i + 3], sl2x2, f32x2_pack(b.z, b.w));
                            add_f32x2(s2[0], __float_as_uint(ex2(x0)), __float_as_uint(ex2(x1)));
                            add_f32x2(s2[1], __float_as_uint(ex2(x2)), __float_as_uint(ex2(x3)));
                        }
                        acc += f32x2_sum(s2[0]) + f32x2_sum(s2[1]);
                    } else {  // LOGITS
                        if (r < p.R) {
                            float* o = p.logits + ((size_t)U.h * p.R + r) * p.S;
#pragma unroll
                            for (int i = 0; i < 32; ++i)
                                if (y0 + col0 + i < p.S) o[y0 + col0 + i] = v[i] * sl2;
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_ACC_EMPTY + buf));
                if (MODE == COLSUM) {
                    if (!XRES) {  // a new key tile each step: write its partial column sums
                        const int key = (U.xt0 + s) * XROWS + trow;
                        if (key < p.n_sc) st_global_policy(p.col + ((size_t)part * p.Hkv + U.h) * p.S_pad + key, acc, keep_l2);
                        acc = 0.f;
                    }
                }
            }
            if (MODE == ROWSTAT && r < p.R) {
                float* o = p.part_ml + (((size_t)U.h * p.R + r) * (SCORE_PARTS * p.splits) + SCORE_PARTS * U.split + part) * 2;
                o[0] = m;
                o[1] = l;
            }
            if (MODE == COLSUM && XRES && U.nsteps > 0) {
                const int key = U.xt * XROWS + trow;
                if (key < p.n_sc) st_global_policy(p.col + ((size_t)part * p.Hkv + U.h) * p.S_pad + key, acc, keep_l2);
            }
        }
    epi_done:;
    }

    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template <int MODE, int D, bool XQ, bool XRES>
cudaError_t launch_inst(const CUtensorMap& tx, const CUtensorMap& ty, const ScoreParams& p, int num_sms, bool pdl,
                        cudaStream_t st) {
    using L = Layout<D, XRES>;
    static std::atomic<uint64_t> smem_set{0};
    if (cudaError_t e = opt_in_smem(score_tc_kernel<MODE, D, XQ, XRES>, L::TOTAL, smem_set); e != cudaSuccess)
        return e;
    const int grid = p.n_units < num_sms ? p.n_units : num_sms;
    if (grid <= 0) return cudaSuccess;
    if (pdl) return launch_dependent(score_tc_kernel<MODE, D, XQ, XRES>, dim3(grid), dim3(THREADS), L::TOTAL, st, tx, ty, p);
    score_tc_kernel<MODE, D, XQ, XRES><<<grid, THREADS, L::TOTAL, st>>>(tx, ty, p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_score_tc(int mode, const CUtensorMap& tx, const CUtensorMap& ty, const ScoreParams& p,
                            int D, bool x_is_q, bool x_resident, int num_sms, bool pdl, cudaStream_t st) {
    if (mode == ROWSTAT && D == 128 && x_is_q && x_resident)
        return launch_inst<ROWSTAT, 128, true, true>(tx, ty, p, num_sms, pdl, st);
    if (mode == ROWSTAT && D == 576 && x_is_q && x_resident)
        return launch_inst<ROWSTAT, 576, true, true>(tx, ty, p, num_sms, pdl, st);
    if (mode == LOGITS && D == 128 && x_is_q && x_resident)
        return launch_inst<LOGITS, 128, true, true>(tx, ty, p, num_sms, pdl, st);
    if (mode == LOGITS && D == 576 && x_is_q && x_resident)
        return launch_inst<LOGITS, 576, true, true>(tx, ty, p, num_sms, pdl, st);
    if (mode == COLSUM && D == 128 && !x_is_q && !x_resident)
        return launch_inst<COLSUM, 128, false, false>(tx, ty, p, num_sms, pdl, st);
    if (mode == COLSUM && D == 128 && !x_is_q && x_resident)
        return launch_inst<COLSUM, 128, false, true>(tx, ty, p, num_sms, pdl, st);
    if (mode == COLSUM && D == 576 && !x_is_q && x_resident)
        return launch_inst<COLSUM, 576, false, true>(tx, ty, p, num_sms, pdl, st);
    return cudaErrorInvalidValue;
}

}  // namespace snap
