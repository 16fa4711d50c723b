// k_compress.cu -- SnapKV-style observation-window scoring, pooling and top-K.
//
// SnapStream episode companion page, "Fixed-Size Cache Layout": the middle of
// the cache holds the SnapKV top-K tokens, chosen once at prefill;
// "Infinity-Bench KV Retrieval": selection is pooling-based top-K.  Scoring rule:
// for KV head h, observation row r = (w, g) is query head h*G+g at prompt
// position S-W+w; its causal softmax over keys 0..S-W+w gives p_r(j); the score
// of prefix position j < S-W is col(j) = sum_r p_r(j).  The scores are max-pooled
// (width P, edges clipped) and the K largest middle positions are kept, ties to
// the lower position.
//
// Three passes:
//   rowstat  per observation row: partial (max, sum of 2^(s - max)) over a key range
//   lse      merge of the partials: lse2(r) = log2 sum_j 2^(s_rj)
//   colsum   per key: col(j) = sum_r 2^(s_rj - lse2(r))
// followed by select (pool + radix top-K + ordered compaction).  Scores s are kept
// in the base-2 domain: s = sm_scale * log2(e) * q.k.
#include "kernels.cuh"

namespace snap {

namespace {

constexpr float NEG_INF = -__builtin_huge_valf();
constexpr float POS_INF = __builtin_huge_valf();

template <int D>
struct Geo {
    static constexpr int ROWB = D * 2;        // bytes per row
    static constexpr int CH = D / 8;          // 16-byte chunks per row
    static constexpr int KS = D / 16;         // k16 steps
};

// Loads rows [0, nrows) of a [64][D] tile through cp.async; row_ptr(r) gives the
// source row or nullptr (zero fill).
template <int D, typename F>
__device__ __forceinline__ void load_rows(uint32_t dst, int nrows, F row_ptr) {
    using Gm = Geo<D>;
    for (int i = threadIdx.x; i < nrows * Gm::CH; i += blockDim.x) {
        const int r = i / Gm::CH, ch = i % Gm::CH;
        const bf16* src = row_ptr(r);
        if (src)
            cp_async16(dst + swz(r, ch, Gm::ROWB), src + ch * 8, 16);
        else
            cp_async16(dst + swz(r, ch, Gm::ROWB), row_ptr(-1), 0);
    }
}

// acc[8][4] = A(16 rows at a_row0 of tile a) x B(64 rows of tile b)^T over D.
template <int D>
__device__ __forceinline__ void mma_16x64(float (&acc)[8][4], uint32_t a, int a_row0, uint32_t b,
                                          int lane) {
    using Gm = Geo<D>;
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
#pragma unroll 4
    for (int ks = 0; ks < Gm::KS; ++ks) {
        uint32_t af[4];
        ldsm_x4(a + swz(a_row0 + (lane & 7) + (((lane >> 3) & 1) << 3), ks * 2 + (lane >> 4), Gm::ROWB),
                af[0], af[1], af[2], af[3]);
#pragma unroll
        for (int np = 0; np < 4; ++np) {
            uint32_t bfr[4];
            ldsm_x4(b + swz(np * 16 + (lane & 7) + ((lane >> 4) << 3), ks * 2 + ((lane >> 3) & 1), Gm::ROWB),
                    bfr[0], bfr[1], bfr[2], bfr[3]);
            mma_bf16(acc[2 * np], af, bfr[0], bfr[1]);
            mma_bf16(acc[2 * np + 1], af, bfr[2], bfr[3]);
        }
    }
}

// ------------------------------------------------------------------ rowstat
// grid (row_splits, row blocks of 64, Hkv); 4 warps x 16 observation rows.
template <int D>
__global__ void __launch_bounds__(128, 1) rowstat_kernel(CompressArgs a) {
    using Gm = Geo<D>;
    extern __shared__ __align__(1024) uint8_t smem[];
    const DevConfig& c = a.cfg;
    const int split = blockIdx.x, rb = blockIdx.y, h = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g4 = lane >> 2, t4 = lane & 3;
    const uint32_t s_q = smem_u32(smem);
    const uint32_t s_k = s_q + CMP_ROWS * Gm::ROWB;
    const int R = a.R, S = a.S;

    load_rows<D>(s_q, CMP_ROWS, [&](int r) -> const bf16* {
        if (r < 0) return a.Q;
        const int row = rb * CMP_ROWS + r;
        if (row >= R) return nullptr;
        const int w = row / c.G, g = row % c.G;
        return a.Q + ((size_t)w * c.Hq + (size_t)h * c.G + g) * D;
    });
    cp_async_commit();

    const int row_last = min(R, (rb + 1) * CMP_ROWS) - 1;
    const int pos_last = S - c.W + row_last / c.G;
    const int nkt = min((S + CMP_KEYS - 1) / CMP_KEYS, pos_last / CMP_KEYS + 1);
    const int per = (nkt + a.row_splits - 1) / a.row_splits;
    const int kt0 = split * per, kt1 = min(nkt, kt0 + per);
    auto load_k = [&](int kt, int st) {
        load_rows<D>(s_k + st * CMP_KEYS * Gm::ROWB, CMP_KEYS, [&](int r) -> const bf16* {
            if (r < 0) return a.K;
            const int key = kt * CMP_KEYS + r;
            if (key >= S) return nullptr;
            return a.K + (size_t)key * a.tok_stride + (size_t)h * a.head_stride;
        });
    };

    const int r0 = rb * CMP_ROWS + warp * 16 + g4;
    const int pos[2] = {r0 < R ? S - c.W + r0 / c.G : -1, r0 + 8 < R ? S - c.W + (r0 + 8) / c.G : -1};
    float m[2] = {NEG_INF, NEG_INF}, l[2] = {0.f, 0.f};
    const float sl2 = c.scale_log2;

    if (kt0 < kt1) load_k(kt0, 0);
    cp_async_commit();
    for (int kt = kt0, st = 0; kt < kt1; ++kt, st ^= 1) {
        if (kt + 1 < kt1) load_k(kt + 1, st ^ 1);
        cp_async_commit();
        cp_async_wait<1>();
        __syncthreads();
        float acc[8][4];
        mma_16x64<D>(acc, s_q, warp * 16, s_k + st * CMP_KEYS * Gm::ROWB, lane);
#pragma unroll
        for (int rh = 0; rh < 2; ++rh) {
            float mx = NEG_INF;
#pragma unroll
            for (int nt = 0; nt < 8; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int key = kt * CMP_KEYS + nt * 8 + 2 * t4 + e;
                    const float v = key <= pos[rh] ? acc[nt][2 * rh + e] * sl2 : NEG_INF;
                    acc[nt][2 * rh + e] = v;
                    mx = fmaxf(mx, v);
                }
            const float mn = fmaxf(m[rh], mx);
            if (mn == NEG_INF) continue;
            float sum = 0.f;
#pragma unroll
            for (int nt = 0; nt < 8; ++nt) sum += ex2(acc[nt][2 * rh] - mn) + ex2(acc[nt][2 * rh + 1] - mn);
            l[rh] = l[rh] * ex2(m[rh] - mn) + sum;
            m[rh] = mn;
        }
        __syncthreads();
    }
    cp_async_wait<0>();
#pragma unroll
    for (int rh = 0; rh < 2; ++rh) {
#pragma unroll
        for (int x = 1; x < 4; x <<= 1) {
            const float mo = __shfl_xor_sync(0xffffffffu, m[rh], x);
            const float lo = __shfl_xor_sync(0xffffffffu, l[rh], x);
            const float M = fmaxf(m[rh], mo);
            l[rh] = M == NEG_INF ? 0.f : l[rh] * ex2(m[rh] - M) + lo * ex2(mo - M);
            m[rh] = M;
        }
        const int row = r0 + 8 * rh;
        if (t4 == 0 && row < R) {
            float* p = a.part_ml + (((size_t)h * R + row) * a.row_splits + split) * 2;
            p[0] = m[rh];
            p[1] = l[rh];
        }
    }
}

// --------------------------------------------------------------------- lse
__global__ void lse_merge_kernel(CompressArgs a) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    const int total = a.cfg.Hkv * a.R;
    if (i >= total) return;
    const float* p = a.part_ml + (size_t)i * a.row_splits * 2;
    float M = NEG_INF;
    for (int s = 0; s < a.row_splits; ++s) M = fmaxf(M, p[2 * s]);
    float L = 0.f;
    if (M != NEG_INF)
        for (int s = 0; s < a.row_splits; ++s) L += p[2 * s + 1] * ex2(p[2 * s] - M);
    a.lse2[i] = (L > 0.f) ? M + log2f(L) : POS_INF;
}

// ------------------------------------------------------- colsum, Q resident
// GQA: all R <= 256 observation rows of the head stay in shared memory; key
// tiles of 64 stream through 3 stages.  Warp w owns keys 16w..16w+15 of a tile.
constexpr int CQ_STAGES = 3;
constexpr int CQ_MAXR = 256;

__global__ void __launch_bounds__(128, 1) colsum_qres_kernel(CompressArgs a) {
    constexpr int D = 128;
    using Gm = Geo<D>;
    extern __shared__ __align__(1024) uint8_t smem[];
    const DevConfig& c = a.cfg;
    const int split = blockIdx.x, h = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g4 = lane >> 2, t4 = lane & 3;
    const int R = a.R, S = a.S;
    const int R_pad = (R + CMP_ROWS - 1) / CMP_ROWS * CMP_ROWS;
    const uint32_t s_q = smem_u32(smem);
    float* lse_s = reinterpret_cast<float*>(smem + CQ_MAXR * Gm::ROWB);
    const uint32_t s_k = s_q + CQ_MAXR * Gm::ROWB + CQ_MAXR * 4;

    load_rows<D>(s_q, R_pad, [&](int r) -> const bf16* {
        if (r < 0) return a.Q;
        if (r >= R) return nullptr;
        const int w = r / c.G, g = r % c.G;
        return a.Q + ((size_t)w * c.Hq + (size_t)h * c.G + g) * D;
    });
    for (int r = threadIdx.x; r < R_pad; r += blockDim.x)
        lse_s[r] = r < R ? a.lse2[(size_t)h * R + r] : POS_INF;
    cp_async_commit();

    const int n_sc = S - c.W;
    const int nkt = (n_sc + CMP_KEYS - 1) / CMP_KEYS;
    const int per = (nkt + gridDim.x - 1) / gridDim.x;
    const int kt0 = split * per, kt1 = min(nkt, kt0 + per);
    auto load_k = [&](int kt, int st) {
        load_rows<D>(s_k + st * CMP_KEYS * Gm::ROWB, CMP_KEYS, [&](int r) -> const bf16* {
            if (r < 0) return a.K;
            const int key = kt * CMP_KEYS + r;
            if (key >= n_sc) return nullptr;
            return a.K + (size_t)key * a.tok_stride + (size_t)h * a.head_stride;
        });
    };
#pragma unroll
    for (int i = 0; i < CQ_STAGES - 1; ++i) {
        if (kt0 + i < kt1) load_k(kt0 + i, i);
        cp_async_commit();
    }
    const float sl2 = c.scale_log2;
    for (int kt = kt0, st = 0; kt < kt1; ++kt, st = (st + 1) % CQ_STAGES) {
        if (kt + CQ_STAGES - 1 < kt1) load_k(kt + CQ_STAGES - 1, (st + CQ_STAGES - 1) % CQ_STAGES);
        cp_async_commit();
        cp_async_wait<CQ_STAGES - 1>();
        __syncthreads();
        const uint32_t kb = s_k + st * CMP_KEYS * Gm::ROWB;
        float sum[2] = {0.f, 0.f};
        for (int rc = 0; rc < R_pad / CMP_ROWS; ++rc) {
            float acc[8][4];
            // keys on M (tile kb), observation rows on N (rows rc*64.. of s_q)
            mma_16x64<D>(acc, kb, warp * 16, s_q + rc * CMP_ROWS * Gm::ROWB, lane);
#pragma unroll
            for (int nt = 0; nt < 8; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int row = rc * CMP_ROWS + nt * 8 + 2 * t4 + (i & 1);
                    sum[i >> 1] += ex2(acc[nt][i] * sl2 - lse_s[row]);
                }
        }
#pragma unroll
        for (int kh = 0; kh < 2; ++kh) {
            sum[kh] += __shfl_xor_sync(0xffffffffu, sum[kh], 1);
            sum[kh] += __shfl_xor_sync(0xffffffffu, sum[kh], 2);
            const int key = kt * CMP_KEYS + warp * 16 + g4 + 8 * kh;
            if (t4 == 0 && key < n_sc) a.col[(size_t)h * a.S_pad + key] = sum[kh];
        }
        __syncthreads();
    }
    cp_async_wait<0>();
}

// ------------------------------------------------------- colsum, K resident
// MLA (R = G*W up to thousands of rows): one 64-key tile stays in shared memory
// while the observation rows stream through 2 stages.
template <int D>
__global__ void __launch_bounds__(128, 1) colsum_kres_kernel(CompressArgs a) {
    using Gm = Geo<D>;
    extern __shared__ __align__(1024) uint8_t smem[];
    const DevConfig& c = a.cfg;
    const int split = blockIdx.x, h = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g4 = lane >> 2, t4 = lane & 3;
    const int R = a.R, S = a.S;
    const uint32_t s_k = smem_u32(smem);
    const uint32_t s_q = s_k + CMP_KEYS * Gm::ROWB;
    const int n_sc = S - c.W;
    const int nkt = (n_sc + CMP_KEYS - 1) / CMP_KEYS;
    const int nrt = (R + CMP_ROWS - 1) / CMP_ROWS;
    const int per = (nkt + gridDim.x - 1) / gridDim.x;
    const int kt0 = split * per, kt1 = min(nkt, kt0 + per);
    const float* lse = a.lse2 + (size_t)h * R;
    auto load_q = [&](int rt, int st) {
        load_rows<D>(s_q + st * CMP_ROWS * Gm::ROWB, CMP_ROWS, [&](int r) -> const bf16* {
            if (r < 0) return a.Q;
            const int row = rt * CMP_ROWS + r;
            if (row >= R) return nullptr;
            const int w = row / c.G, g = row % c.G;
            return a.Q + ((size_t)w * c.Hq + (size_t)h * c.G + g) * D;
        });
    };
    const float sl2 = c.scale_log2;
    for (int kt = kt0; kt < kt1; ++kt) {
        load_rows<D>(s_k, CMP_KEYS, [&](int r) -> const bf16* {
            if (r < 0) return a.K;
            const int key = kt * CMP_KEYS + r;
            if (key >= n_sc) return nullptr;
            return a.K + (size_t)key * a.tok_stride + (size_t)h * a.head_stride;
        });
        cp_async_commit();
        load_q(0, 0);
        cp_async_commit();
        float sum[2] = {0.f, 0.f};
        for (int rt = 0, st = 0; rt < nrt; ++rt, st ^= 1) {
            if (rt + 1 < nrt) load_q(rt + 1, st ^ 1);
            cp_async_commit();
            cp_async_wait<1>();
            __syncthreads();
            float acc[8][4];
            mma_16x64<D>(acc, s_k, warp * 16, s_q + st * CMP_ROWS * Gm::ROWB, lane);
#pragma unroll
            for (int nt = 0; nt < 8; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int row = rt * CMP_ROWS + nt * 8 + 2 * t4 + (i & 1);
                    if (row < R) sum[i >> 1] += ex2(acc[nt][i] * sl2 - __ldg(lse + row));
                }
            __syncthreads();
        }
#pragma unroll
        for (int kh = 0; kh < 2; ++kh) {
            sum[kh] += __shfl_xor_sync(0xffffffffu, sum[kh], 1);
            sum[kh] += __shfl_xor_sync(0xffffffffu, sum[kh], 2);
            const int key = kt * CMP_KEYS + warp * 16 + g4 + 8 * kh;
            if (t4 == 0 && key < n_sc) a.col[(size_t)h * a.S_pad + key] = sum[kh];
        }
    }
    cp_async_wait<0>();
}

// ------------------------------------------------------------------- select
// One CTA of 1024 threads per KV head.  Pooled scores (non-negative floats,
// compared as their IEEE bit patterns, which order them) of the middle
// positions; the K-th largest found by a 4 x 8-bit radix descent; then an
// ordered compaction keeps every score above it and the lowest-position ties.
constexpr int SEL_THREADS = 1024;

__device__ __forceinline__ int block_excl_scan(int x, int* warp_tot, int& total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int v = lane < (SEL_THREADS / 32) ? warp_tot[lane] : 0;
        int vi = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, vi, o);
            if (lane >= o) vi += y;
        }
        warp_tot[lane] = vi - v;        // exclusive prefix of warp totals
        if (lane == 31) warp_tot[32] = vi;
    }
    __syncthreads();
    const int r = warp_tot[warp] + incl - x;
    total = warp_tot[32];
    __syncthreads();
    return r;
}

__global__ void __launch_bounds__(SEL_THREADS, 1) select_kernel(CompressArgs a) {
    __shared__ int hist[256];
    __shared__ int warp_tot[33];
    __shared__ uint32_t sh_prefix;
    __shared__ int sh_kk;
    const DevConfig& c = a.cfg;
    const int h = blockIdx.x;
    const int n_sc = a.S - c.W;
    const int M = a.R0 - c.L_sink;        // middle candidates [L_sink, R0)
    const int r = c.P / 2;
    const float* colh = a.col + (size_t)h * a.S_pad;
    uint32_t* pool = a.pool + (size_t)h * a.S_pad;

    for (int i = threadIdx.x; i < M; i += SEL_THREADS) {
        const int j = c.L_sink + i;
        const int lo = max(0, j - r), hi = min(n_sc - 1, j + r);
        float mx = colh[lo];
        for (int k = lo + 1; k <= hi; ++k) mx = fmaxf(mx, colh[k]);
        pool[i] = __float_as_uint(mx);
    }
    if (threadIdx.x == 0) {
        sh_prefix = 0u;
        sh_kk = c.K;
    }
    __syncthreads();

    uint32_t mask = 0u;
    for (int pass = 0; pass < 4; ++pass) {
        const int shift = 24 - 8 * pass;
        for (int i = threadIdx.x; i < 256; i += SEL_THREADS) hist[i] = 0;
        __syncthreads();
        const uint32_t prefix = sh_prefix;
        for (int i = threadIdx.x; i < M; i += SEL_THREADS) {
            const uint32_t v = pool[i];
            if ((v & mask) == prefix) atomicAdd(&hist[(v >> shift) & 255u], 1);
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            int kk = sh_kk, cum = 0, d = 255;
            for (; d > 0; --d) {
                if (cum + hist[d] >= kk) break;
                cum += hist[d];
            }
            sh_kk = kk - cum;
            sh_prefix = prefix | ((uint32_t)d << shift);
        }
        mask |= 255u << shift;
        __syncthreads();
    }
    const uint32_t tau = sh_prefix;
    const int kk = sh_kk;                 // how many scores equal to tau are kept

    int32_t* out = a.sel + ((size_t)a.slot * c.Hkv + h) * c.K;
    int eq_before = 0, taken_before = 0;
    for (int base = 0; base < M; base += SEL_THREADS) {
        const int i = base + threadIdx.x;
        const uint32_t v = i < M ? pool[i] : 0u;
        const int gt = (i < M && v > tau) ? 1 : 0;
        const int eq = (i < M && v == tau) ? 1 : 0;
        int eq_tot;
        const int eq_rank = block_excl_scan(eq, warp_tot, eq_tot);
        const int take = gt | (eq && (eq_before + eq_rank) < kk);
        int take_tot;
        const int pos = block_excl_scan(take, warp_tot, take_tot);
        if (take) out[taken_before + pos] = c.L_sink + i;
        eq_before += eq_tot;
        taken_before += take_tot;
    }
}

}  // namespace

template <int D>
static cudaError_t launch_rowstat_d(const CompressArgs& a, cudaStream_t st) {
    constexpr int smem = CMP_ROWS * D * 2 + 2 * CMP_KEYS * D * 2;
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(rowstat_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    dim3 grid(a.row_splits, (a.R + CMP_ROWS - 1) / CMP_ROWS, a.cfg.Hkv);
    rowstat_kernel<D><<<grid, 128, smem, st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_rowstat(const CompressArgs& a, int, cudaStream_t st) {
    if (a.cfg.dqk == 128) return launch_rowstat_d<128>(a, st);
    if (a.cfg.dqk == 576) return launch_rowstat_d<576>(a, st);
    return cudaErrorInvalidValue;
}

cudaError_t launch_lse_merge(const CompressArgs& a, cudaStream_t st) {
    const int total = a.cfg.Hkv * a.R;
    lse_merge_kernel<<<(total + 255) / 256, 256, 0, st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_colsum(const CompressArgs& a, int num_sms, cudaStream_t st) {
    const int n_sc = a.S - a.cfg.W;
    const int nkt = (n_sc + CMP_KEYS - 1) / CMP_KEYS;
    if (a.cfg.dqk == 128 && a.R <= CQ_MAXR) {
        constexpr int smem = CQ_MAXR * 256 + CQ_MAXR * 4 + CQ_STAGES * CMP_KEYS * 256;
        static bool attr = false;
        if (!attr) {
            cudaError_t e = cudaFuncSetAttribute(colsum_qres_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
            if (e != cudaSuccess) return e;
            attr = true;
        }
        int splits = (num_sms + a.cfg.Hkv - 1) / a.cfg.Hkv;
        if (splits > nkt) splits = nkt;
        if (splits < 1) splits = 1;
        dim3 grid(splits, a.cfg.Hkv);
        colsum_qres_kernel<<<grid, 128, smem, st>>>(a);
        return cudaGetLastError();
    }
    if (a.cfg.dqk == 576) {
        constexpr int smem = CMP_KEYS * 1152 + 2 * CMP_ROWS * 1152;
        static bool attr = false;
        if (!attr) {
            cudaError_t e = cudaFuncSetAttribute(colsum_kres_kernel<576>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
            if (e != cudaSuccess) return e;
            attr = true;
        }
        int splits = nkt < num_sms * 4 ? nkt : num_sms * 4;
        if (splits < 1) splits = 1;
        dim3 grid(splits, a.cfg.Hkv);
        colsum_kres_kernel<576><<<grid, 128, smem, st>>>(a);
        return cudaGetLastError();
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_select(const CompressArgs& a, cudaStream_t st) {
    select_kernel<<<a.cfg.Hkv, SEL_THREADS, 0, st>>>(a);
    return cudaGetLastError();
}

}  // namespace snap
