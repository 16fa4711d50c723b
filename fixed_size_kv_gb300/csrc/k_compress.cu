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
#include <cooperative_groups.h>

#include "kernels.cuh"

namespace snap {

namespace {

constexpr float NEG_INF = -__builtin_huge_valf();

// --------------------------------------------------------------------- lse
// One warp per observation row: the lanes merge the row's key-split partials
// (max, sum) in parallel, then across the warp.
__device__ __forceinline__ void ml_merge(float& M, float& L, float m, float l) {
    const float Mn = fmaxf(M, m);
    if (Mn == NEG_INF) return;
    L = L * ex2(M - Mn) + l * ex2(m - Mn);
    M = Mn;
}

__global__ void lse_merge_kernel(CompressArgs a) {
    const int i = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;   // over Hkv * R_pad
    const int lane = threadIdx.x & 31;
    const int total = a.cfg.Hkv * a.R_pad;
    if (i >= total) return;
    const int h = i / a.R_pad, r = i % a.R_pad;
    if (r >= a.R) {
        if (lane == 0) a.nlse2[i] = NEG_INF;  // padding rows contribute 2^-inf = 0
        return;
    }
    const float* p = a.part_ml + ((size_t)h * a.R + r) * a.row_splits * 2;
    float M = NEG_INF, L = 0.f;
    for (int s = lane; s < a.row_splits; s += 32) ml_merge(M, L, p[2 * s], p[2 * s + 1]);
#pragma unroll
    for (int x = 16; x > 0; x >>= 1) {
        const float m = __shfl_xor_sync(0xffffffffu, M, x), l = __shfl_xor_sync(0xffffffffu, L, x);
        ml_merge(M, L, m, l);
    }
    if (lane == 0) a.nlse2[i] = (L > 0.f) ? -(M + log2f(L)) : NEG_INF;
}

// ------------------------------------------------------------------- select
// One cluster of SEL_CLUSTER CTAs per KV head; CTA r owns a contiguous slice of
// the middle positions.  The slice's column sums (plus the pooling halo) are read
// once into shared memory and max-pooled there; the pooled scores (non-negative
// floats, compared as their IEEE bit patterns, which order them) stay in shared
// memory for the rest of the kernel (the workspace takes them when a slice is too
// long).  The K-th largest is found by a 4 x 8-bit radix descent whose per-CTA
// histograms are summed through distributed shared memory, the digit of each pass
// picked by one warp's scan; an ordered compaction then keeps every score above it
// and, among the scores equal to it, the lowest positions.
constexpr int SEL_THREADS = 1024;
constexpr int SEL_WARPS = SEL_THREADS / 32;
constexpr int SEL_CLUSTER = 8;

// Exclusive prefix sum over the block; *total receives the block sum.
__device__ __forceinline__ int block_excl_scan(int x, int* warp_tot, int* total) {
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
        const int v = warp_tot[lane];
        int vi = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, vi, o);
            if (lane >= o) vi += y;
        }
        warp_tot[lane] = vi - v;
        if (lane == 31) warp_tot[32] = vi;
    }
    __syncthreads();
    const int r = warp_tot[warp] + incl - x;
    *total = warp_tot[32];
    __syncthreads();
    return r;
}

// Digit of this radix pass that holds the kk-th largest value: the largest d with
// (count of digits > d) < kk <= (count of digits >= d).  Warp 0; lane l scans digits
// 255 - 8l .. 248 - 8l after an exclusive scan of the lanes' totals.
__device__ __forceinline__ void find_digit(const int* hist, int kk, int* digit, int* kk_left) {
    const int lane = threadIdx.x & 31;
    int v[8], tot = 0;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        v[e] = hist[255 - (8 * lane + e)];
        tot += v[e];
    }
    int incl = tot;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    int cum = incl - tot;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        if (cum < kk && cum + v[e] >= kk) {
            *digit = 255 - (8 * lane + e);
            *kk_left = kk - cum;
        }
        cum += v[e];
    }
}

__global__ void __cluster_dims__(SEL_CLUSTER, 1, 1) __launch_bounds__(SEL_THREADS, 1)
    select_kernel(CompressArgs a, int in_smem) {
    namespace cg = cooperative_groups;
    cg::cluster_group cluster = cg::this_cluster();
    extern __shared__ uint32_t sel_dyn[];         // [per] pooled bits, then [per + 2 rad] raw sums
    __shared__ int hist_w[SEL_WARPS][256];       // per-warp private histograms
    __shared__ int hist_cta[2][256];             // this CTA's histogram, double-buffered by pass
    __shared__ int hist_all[256];
    __shared__ int warp_tot[33];
    __shared__ int counts[2];                    // this CTA's (greater, equal) counts
    __shared__ uint32_t sh_prefix;
    __shared__ int sh_kk;
    __shared__ int sh_done;                      // the descent stopped early
    __shared__ int peer_counts[SEL_CLUSTER][2];
    const DevConfig& c = a.cfg;
    const int h = blockIdx.y;
    const int rank = (int)cluster.block_rank();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int n_sc = a.S - c.W;
    const int M = a.R0 - c.L_sink;               // middle candidates [L_sink, R0)
    const int rad = c.P / 2;
    const int per = (M + SEL_CLUSTER - 1) / SEL_CLUSTER;
    const int i0 = min(M, rank * per), i1 = min(M, i0 + per);
    // column sum of position k: the score kernel's SCORE_PARTS parts, added in order
    auto colsum = [&](int k) {
        float t = __ldcg(a.col + (size_t)h * a.S_pad + k);
#pragma unroll
        for (int q = 1; q < SCORE_PARTS; ++q) t += __ldcg(a.col + ((size_t)q * c.Hkv + h) * a.S_pad + k);
        return t;
    };
    // this CTA's pooled values: shared memory when they fit, else the workspace
    uint32_t* vals = in_smem ? sel_dyn - i0 : a.pool + (size_t)h * a.S_pad;

    // per-warp histogram of one radix digit (shared-memory atomics; lanes that hit the
    // same bin are serialised by the hardware)
    auto hist_add = [&](bool match, uint32_t d) {
        if (match) atomicAdd(&hist_w[warp][d], 1);
    };
    for (int i = lane; i < 256; i += 32) hist_w[warp][i] = 0;
    __syncwarp();

    // 0. pooled scores of this slice (the score GEMM leaves each column sum in two
    //    halves), with the histogram of their top 8 bits (the first radix pass)
    if (in_smem) {
        // the column sums of positions L_sink + i0 - rad .. L_sink + i1 - 1 + rad, once;
        // eight positions per thread in flight
        float* raw = reinterpret_cast<float*>(sel_dyn + per);
        const int k0 = c.L_sink + i0 - rad;
        const int nk = (i1 - i0) + 2 * rad;
        for (int t0 = 0; t0 < nk; t0 += 8 * SEL_THREADS) {
            float x[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int t = t0 + e * SEL_THREADS + tid, k = k0 + t;
                x[e] = (t < nk && k >= 0 && k < n_sc) ? colsum(k) : -__builtin_huge_valf();
            }
#pragma unroll
            for (int e = 0; e < 8; ++e)
                if (t0 + e * SEL_THREADS + tid < nk) raw[t0 + e * SEL_THREADS + tid] = x[e];
        }
        __syncthreads();
        for (int base = i0; base < i1; base += SEL_THREADS) {
            const int i = base + tid;
            const bool in = i < i1;
            uint32_t v = 0u;
            if (in) {
                const int t = i - i0 + rad;          // raw index of position L_sink + i
                float mx = raw[t - rad];
                for (int d = -rad + 1; d <= rad; ++d) mx = fmaxf(mx, raw[t + d]);
                v = __float_as_uint(mx);
                vals[i] = v;
            }
            hist_add(in, v >> 24);
        }
    } else {
        for (int base = i0; base < i1; base += SEL_THREADS) {
            const int i = base + tid;
            const bool in = i < i1;
            uint32_t v = 0u;
            if (in) {
                const int j = c.L_sink + i;
                const int lo = max(0, j - rad), hi = min(n_sc - 1, j + rad);
                float mx = colsum(lo);
                for (int k = lo + 1; k <= hi; ++k) mx = fmaxf(mx, colsum(k));
                v = __float_as_uint(mx);
                vals[i] = v;
            }
            hist_add(in, v >> 24);
        }
    }
    if (tid == 0) {
        sh_prefix = 0u;
        sh_kk = c.K;
        sh_done = 0;
    }
    __syncthreads();

    // 1-4. radix descent over the whole middle, 8 bits at a time.  It stops early when
    //      the digit's bucket holds exactly the positions still to take: they are all
    //      kept, so the threshold becomes "at least the bucket's prefix".
    uint32_t mask = 0u;
    for (int pass = 0; pass < 4; ++pass) {
        const int shift = 24 - 8 * pass;
        const uint32_t prefix = sh_prefix;
        if (pass > 0) {
            for (int i = lane; i < 256; i += 32) hist_w[warp][i] = 0;
            __syncwarp();
            for (int base = i0; base < i1; base += SEL_THREADS) {
                const int i = base + tid;
                const bool in = i < i1;
                const uint32_t v = in ? vals[i] : 0u;
                hist_add(in && (v & mask) == prefix, (v >> shift) & 255u);
            }
            __syncthreads();
        }
        int* hc = hist_cta[pass & 1];
        if (tid < 256) {
            int t = 0;
#pragma unroll 8
            for (int w = 0; w < SEL_WARPS; ++w) t += hist_w[w][tid];
            hc[tid] = t;
        }
        cluster.sync();                          // every CTA's histogram of this pass is ready
        if (tid < 256) {
            int t = 0;
#pragma unroll
            for (int r = 0; r < SEL_CLUSTER; ++r) t += cluster.map_shared_rank(hc, r)[tid];
            hist_all[tid] = t;
        }
        __syncthreads();
        if (warp == 0) {
            int d = 0, kk = 0;
            find_digit(hist_all, sh_kk, &d, &kk);
            // exactly one lane found the digit; hand it to the block
            const unsigned who = __ballot_sync(0xffffffffu, kk > 0);
            const int src = who ? __ffs(who) - 1 : 0;
            d = __shfl_sync(0xffffffffu, d, src);
            kk = __shfl_sync(0xffffffffu, kk, src);
            if (lane == 0) {
                const uint32_t p = prefix | ((uint32_t)d << shift);
                if (pass < 3 && kk == hist_all[d] && p != 0u) {
                    // the whole bucket is kept: keep every value >= p, no ties
                    sh_prefix = p - 1u;
                    sh_kk = 0;
                    sh_done = 1;
                } else {
                    sh_kk = kk;
                    sh_prefix = p;
                }
            }
        }
        mask |= 255u << shift;
        __syncthreads();
        if (sh_done) break;
    }
    const uint32_t tau = sh_prefix;
    const int kk = sh_kk;                        // how many scores equal to tau are kept

    // 5. ordered compaction: thread t scans a contiguous run of this slice
    const int run = (i1 - i0 + SEL_THREADS - 1) / SEL_THREADS;
    const int r0 = min(i1, i0 + tid * run), r1 = min(i1, r0 + run);
    int gt = 0, eq = 0;
    for (int i = r0; i < r1; ++i) {
        const uint32_t v = vals[i];
        gt += v > tau;
        eq += v == tau;
    }
    int gt_before, eq_before, gt_cta, eq_cta;
    if (per < 32768) {
        // one scan of both counts, packed 15 + 16 bits
        int both_cta;
        const int both_before = block_excl_scan((gt << 16) | eq, warp_tot, &both_cta);
        gt_before = both_before >> 16;
        eq_before = both_before & 0xffff;
        gt_cta = both_cta >> 16;
        eq_cta = both_cta & 0xffff;
    } else {
        gt_before = block_excl_scan(gt, warp_tot, &gt_cta);
        eq_before = block_excl_scan(eq, warp_tot, &eq_cta);
    }
    if (tid == 0) {
        counts[0] = gt_cta;
        counts[1] = eq_cta;
    }
    cluster.sync();
    // the lower-ranked CTAs' counts, read in parallel
    if (tid < rank) {
        const int* cr = cluster.map_shared_rank(counts, tid);
        peer_counts[tid][0] = cr[0];
        peer_counts[tid][1] = cr[1];
    }
    __syncthreads();
    // positions kept by lower-ranked CTAs, and equal scores met before this slice
    int taken_prev = 0, eq_prev = 0;
    for (int r = 0; r < rank; ++r) {
        const int g = peer_counts[r][0], e = peer_counts[r][1];
        taken_prev += g + min(max(kk - eq_prev, 0), e);
        eq_prev += e;
    }
    int32_t* out = a.sel + ((size_t)a.slot * c.Hkv + h) * c.K;
    // this thread's first output index: greater ones before it in the slice, plus the
    // equal ones before it that are kept
    const int eq_g = eq_prev + eq_before;       // equal scores before this thread's run
    int pos = taken_prev + gt_before + min(max(kk - eq_prev, 0), eq_before);
    int e_seen = eq_g;
    for (int i = r0; i < r1; ++i) {
        const uint32_t v = vals[i];
        bool take = v > tau;
        if (v == tau) {
            take = e_seen < kk;
            ++e_seen;
        }
        if (take) out[pos++] = c.L_sink + i;
    }
    cluster.sync();                              // peers may still read this CTA's counters
}

}  // namespace

namespace {
// Row r = w*G + g of KV head h is query head h*G + g at window position w; the
// caller's LSE is natural-log: -lse2 = -lse * log2(e).
__global__ void lse_import_kernel(CompressArgs a, const float* lse_obs) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;   // over Hkv * R_pad
    if (i >= a.cfg.Hkv * a.R_pad) return;
    const int h = i / a.R_pad, r = i % a.R_pad;
    if (r >= a.R) {
        a.nlse2[i] = NEG_INF;
        return;
    }
    const int w = r / a.cfg.G, g = r % a.cfg.G;
    a.nlse2[i] = -lse_obs[(size_t)w * a.cfg.Hq + (size_t)h * a.cfg.G + g] * 1.4426950408889634f;
}
}  // namespace

cudaError_t launch_lse_import(const CompressArgs& a, const float* lse_obs, cudaStream_t st) {
    const int total = a.cfg.Hkv * a.R_pad;
    lse_import_kernel<<<(total + 255) / 256, 256, 0, st>>>(a, lse_obs);
    return cudaGetLastError();
}

cudaError_t launch_lse_merge(const CompressArgs& a, cudaStream_t st) {
    const int total = a.cfg.Hkv * a.R_pad;   // rows, one warp each
    lse_merge_kernel<<<(total + 7) / 8, 256, 0, st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_select(const CompressArgs& a, cudaStream_t st) {
    // pooled values (and the raw column sums they come from) of one CTA's slice in
    // shared memory when they fit next to the histograms, else in the workspace
    constexpr int DYN_MAX = 150 * 1024;
    static std::atomic<uint64_t> smem_set{0};
    const int M = a.R0 - a.cfg.L_sink;
    const int per = (M + SEL_CLUSTER - 1) / SEL_CLUSTER;
    const long long bytes = 4ll * (2ll * per + 2 * (a.cfg.P / 2));
    const int in_smem = bytes <= DYN_MAX;
    if (cudaError_t e = opt_in_smem(select_kernel, DYN_MAX, smem_set); e != cudaSuccess) return e;
    dim3 grid(SEL_CLUSTER, a.cfg.Hkv);
    select_kernel<<<grid, SEL_THREADS, in_smem ? (size_t)bytes : 0, st>>>(a, in_smem);
    return cudaGetLastError();
}

}  // namespace snap
