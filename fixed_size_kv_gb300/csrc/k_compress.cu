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
// The score GEMM (k_score_tc.cu) runs twice: a row pass leaves per observation
// row partial (max, sum of 2^(s - max)) over key ranges; lse_merge (here) turns
// them into -lse2(r) = -log2 sum_j 2^(s_rj); a column pass then gives per key
// col(j) = sum_r 2^(s_rj - lse2(r)).  select (here) pools, finds the K-th largest
// by radix descent and compacts the kept positions in order.  Scores s are in the
// base-2 domain: s = sm_scale * log2(e) * q.k.
#include "kernels.cuh"

namespace snap {

namespace {

constexpr float NEG_INF = -__builtin_huge_valf();

// --------------------------------------------------------------------- lse
__global__ void lse_merge_kernel(CompressArgs a) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;   // over Hkv * R_pad
    const int total = a.cfg.Hkv * a.R_pad;
    if (i >= total) return;
    const int h = i / a.R_pad, r = i % a.R_pad;
    if (r >= a.R) {
        a.nlse2[i] = NEG_INF;  // padding rows contribute 2^-inf = 0
        return;
    }
    const float* p = a.part_ml + ((size_t)h * a.R + r) * a.row_splits * 2;
    float M = NEG_INF;
    for (int s = 0; s < a.row_splits; ++s) M = fmaxf(M, p[2 * s]);
    float L = 0.f;
    if (M != NEG_INF)
        for (int s = 0; s < a.row_splits; ++s) L += p[2 * s + 1] * ex2(p[2 * s] - M);
    a.nlse2[i] = (L > 0.f) ? -(M + log2f(L)) : NEG_INF;
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
    // the score GEMM leaves each column sum as two halves (two groups of rows)
    const float* c0 = a.col + (size_t)h * a.S_pad;
    const float* c1 = a.col + ((size_t)c.Hkv + h) * a.S_pad;
    uint32_t* pool = a.pool + (size_t)h * a.S_pad;

    for (int i = threadIdx.x; i < M; i += SEL_THREADS) {
        const int j = c.L_sink + i;
        const int lo = max(0, j - r), hi = min(n_sc - 1, j + r);
        float mx = c0[lo] + c1[lo];
        for (int k = lo + 1; k <= hi; ++k) mx = fmaxf(mx, c0[k] + c1[k]);
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

cudaError_t launch_lse_merge(const CompressArgs& a, cudaStream_t st) {
    const int total = a.cfg.Hkv * a.R_pad;
    lse_merge_kernel<<<(total + 255) / 256, 256, 0, st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_select(const CompressArgs& a, cudaStream_t st) {
    select_kernel<<<a.cfg.Hkv, SEL_THREADS, 0, st>>>(a);
    return cudaGetLastError();
}

}  // namespace snap
