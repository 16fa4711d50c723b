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
    pdl_wait();                 // the row pass's partials are complete and visible
    pdl_launch_dependents();    // the column pass may launch (it waits for this grid)
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
// One cluster of CL CTAs per KV head (16 or 12 where the device can hold every head's
// cluster at once, else 8); CTA r owns a contiguous slice of
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

// In-place exclusive prefix sum of v[0..31] by one warp; returns the total.
__device__ __forceinline__ int warp_excl_scan32(int* v) {
    const int lane = threadIdx.x & 31;
    const int x = v[lane];
    int incl = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    v[lane] = incl - x;
    return __shfl_sync(0xffffffffu, incl, 31);
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

// Max-pool of four consecutive positions with radius RAD <= 4: w[m] holds the raw sum of
// the position 4 - m places before the first output.
template <int RAD>
__device__ __forceinline__ void pool4(const float (&w)[12], float (&o)[4]) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        float mx = w[4 + j - RAD];
#pragma unroll
        for (int d = -RAD + 1; d <= RAD; ++d) mx = fmaxf(mx, w[4 + j + d]);
        o[j] = mx;
    }
}

// Raw column sums held per side of a select CTA's slice: the pooling radius, at least 4
// so that the four-position path reads whole 16-byte groups.
__host__ __device__ __forceinline__ int select_pad(int P) { return P / 2 > 4 ? P / 2 : 4; }
// Raw column sums read for a slice of n positions: with the four-position path (radius
// <= 4) whole groups of four plus the two groups its last loads reach, else the slice
// and its halo.
__host__ __device__ __forceinline__ int select_raw_words(int n, int P) {
    return P / 2 <= 4 ? 4 * ((n + 3) / 4) + 12 : n + 2 * select_pad(P);
}

template <int CL>
__global__ void __launch_bounds__(SEL_THREADS, 1) select_kernel(CompressArgs a, int in_smem) {
    namespace cg = cooperative_groups;
    cg::cluster_group cluster = cg::this_cluster();
    extern __shared__ uint4 sel_dyn4[];           // [per] pooled bits, then [per + 2 pad] raw sums
    uint32_t* sel_dyn = reinterpret_cast<uint32_t*>(sel_dyn4);
    __shared__ int hist_w[SEL_WARPS][256];       // per-warp private histograms
    __shared__ int hist_cta[2][256];             // this CTA's histogram, double-buffered by pass
    __shared__ int hist_all[256];
    __shared__ int warp_gt[SEL_WARPS], warp_eq[SEL_WARPS];   // per-warp counts, then their scans
    __shared__ int counts[2];                    // this CTA's (greater, equal) counts
    __shared__ uint32_t sh_prefix;
    __shared__ int sh_kk;
    __shared__ int sh_done;                      // the descent stopped early
    __shared__ int sh_digit;                     // the digit picked by the last pass
    __shared__ int peer_counts[CL][2];
    pdl_wait();                 // the column sums are complete and visible
    pdl_launch_dependents();    // the cache write may launch (it waits for this grid)
    const DevConfig& c = a.cfg;
    const int h = blockIdx.y;
    const int rank = (int)cluster.block_rank();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int n_sc = a.S - c.W;
    const int M = a.R0 - c.L_sink;               // middle candidates [L_sink, R0)
    const int rad = c.P / 2;
    const int per = (M + CL - 1) / CL;
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
    // warp w owns positions [w0, w1) of the slice (whole groups of four, the pooling's
    // quads), its lanes taking consecutive positions: every loop over positions uses this
    // split, so a warp's histograms count exactly the block it compacts
    const int nq_all = (i1 - i0 + 3) / 4;
    const int nqw = (nq_all + SEL_WARPS - 1) / SEL_WARPS;
    const int qw0 = min(nq_all, warp * nqw), qw1 = min(nq_all, qw0 + nqw);
    const int w0 = min(i1, i0 + 4 * qw0), w1 = min(i1, i0 + 4 * qw1);

    // per-warp histogram of one radix digit (shared-memory atomics; lanes that hit the
    // same bin are serialised by the hardware)
    auto hist_add = [&](bool match, uint32_t d) {
        if (match) atomicAdd(&hist_w[warp][d], 1);
    };
    for (int i = lane; i < 256; i += 32) hist_w[warp][i] = 0;
    __syncwarp();

    // 0. pooled scores of this slice, with the histogram of their top 8 bits (the first
    //    radix pass)
    if (in_smem) {
        // the column sums of positions L_sink + i0 - pad .. (at least L_sink + i1 - 1 +
        // pad), once (outside the scored range: -inf); eight positions per thread in flight
        const int pad = select_pad(c.P);
        float* raw = reinterpret_cast<float*>(sel_dyn + ((per + 3) & ~3));   // 16-byte aligned
        const int k0 = c.L_sink + i0 - pad;
        const int nk = select_raw_words(i1 - i0, c.P);
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
        if (rad <= 4) {
            // four consecutive positions per thread from three 16-byte loads
            const float4* raw4 = reinterpret_cast<const float4*>(raw);
            uint4* out4 = reinterpret_cast<uint4*>(sel_dyn);                  // position i0 + 4q.. at q
            const int nq = nq_all;
            for (int q = qw0 + lane; q < qw1; q += 32) {
                float o[4] = {0.f, 0.f, 0.f, 0.f};
                {
                    const float4 A = raw4[q], B = raw4[q + 1], C = raw4[q + 2];
                    const float w[12] = {A.x, A.y, A.z, A.w, B.x, B.y, B.z, B.w, C.x, C.y, C.z, C.w};
                    switch (rad) {
                        case 0: pool4<0>(w, o); break;
                        case 1: pool4<1>(w, o); break;
                        case 2: pool4<2>(w, o); break;
                        case 3: pool4<3>(w, o); break;
                        default: pool4<4>(w, o); break;
                    }
                    // positions past the slice keep 0 (never read as candidates)
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        if (i0 + 4 * q + j >= i1) o[j] = 0.f;
                    out4[q] = make_uint4(__float_as_uint(o[0]), __float_as_uint(o[1]), __float_as_uint(o[2]),
                                         __float_as_uint(o[3]));
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) hist_add(q < nq && i0 + 4 * q + j < i1, __float_as_uint(o[j]) >> 24);
            }
        } else {
            for (int i = w0 + lane; i < w1; i += 32) {
                const int t = i - i0 + pad;              // raw index of position L_sink + i
                float mx = raw[t - rad];
                for (int d = -rad + 1; d <= rad; ++d) mx = fmaxf(mx, raw[t + d]);
                const uint32_t v = __float_as_uint(mx);
                vals[i] = v;
                hist_add(true, v >> 24);
            }
        }
    } else {
        for (int i = w0 + lane; i < w1; i += 32) {
            const int j = c.L_sink + i;
            const int lo = max(0, j - rad), hi = min(n_sc - 1, j + rad);
            float mx = colsum(lo);
            for (int k = lo + 1; k <= hi; ++k) mx = fmaxf(mx, colsum(k));
            const uint32_t v = __float_as_uint(mx);
            vals[i] = v;
            hist_add(true, v >> 24);
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
    //      Each warp also counts, from its own histogram of each pass, the positions of
    //      its block above the final threshold (a larger digit than the pass's) and, after
    //      the last pass, those equal to it.
    uint32_t mask = 0u;
    int my_gt = 0, my_eq = 0;
    for (int pass = 0; pass < 4; ++pass) {
        const int shift = 24 - 8 * pass;
        const uint32_t prefix = sh_prefix;
        if (pass > 0) {
            for (int i = lane; i < 256; i += 32) hist_w[warp][i] = 0;
            __syncwarp();
            for (int i = w0 + lane; i < w1; i += 32) {
                const uint32_t v = vals[i];
                hist_add((v & mask) == prefix, (v >> shift) & 255u);
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
            for (int r = 0; r < CL; ++r) t += cluster.map_shared_rank(hc, r)[tid];
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
                sh_digit = d;
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
        {
            // stopping early keeps the whole digit's bucket: it counts as greater
            const int d = sh_digit;
            const bool done = sh_done != 0;
            int g = 0;
            for (int b = lane; b < 256; b += 32) g += (b > d || (done && b == d)) ? hist_w[warp][b] : 0;
            my_gt += __reduce_add_sync(0xffffffffu, g);
            if (pass == 3 && !done) my_eq = hist_w[warp][d];
        }
        if (sh_done) break;
    }
    const uint32_t tau = sh_prefix;
    const int kk = sh_kk;                        // how many scores equal to tau are kept

    // 5. ordered compaction of each warp's block [w0, w1), its lanes reading consecutive
    //    positions; ballots order the kept positions within each group of 32
    if (lane == 0) {
        warp_gt[warp] = my_gt;
        warp_eq[warp] = my_eq;
    }
    __syncthreads();
    if (warp == 0) {
        const int gt_cta = warp_excl_scan32(warp_gt);
        const int eq_cta = warp_excl_scan32(warp_eq);
        if (lane == 0) {
            counts[0] = gt_cta;
            counts[1] = eq_cta;
        }
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
    // this warp's first output index: greater ones before its block, plus the equal
    // ones before it that are kept
    const int eq_before = warp_eq[warp];
    int pos = taken_prev + warp_gt[warp] + min(max(kk - eq_prev, 0), eq_before);
    int e_seen = eq_prev + eq_before;           // equal scores before the current group
    const unsigned lt = (1u << lane) - 1u;
    for (int base = w0; base < w1; base += 32) {
        const int i = base + lane;
        const uint32_t v = (i < w1) ? vals[i] : 0u;
        const bool ise = i < w1 && v == tau;
        const unsigned be = __ballot_sync(0xffffffffu, ise);
        const bool take = (i < w1 && v > tau) || (ise && e_seen + __popc(be & lt) < kk);
        const unsigned bt = __ballot_sync(0xffffffffu, take);
        if (take) out[pos + __popc(bt & lt)] = c.L_sink + i;
        pos += __popc(bt);
        e_seen += __popc(be);
    }
    cluster.sync();                              // peers may still read this CTA's counters
}

}  // namespace

namespace {
// Row r = w*G + g of KV head h is query head h*G + g at window position w; the
// caller's LSE is natural-log: -lse2 = -lse * log2(e).
__global__ void lse_import_kernel(CompressArgs a, const float* lse_obs) {
    pdl_launch_dependents();    // the column pass may launch (it waits for this grid)
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
    return launch_dependent(lse_merge_kernel, dim3((total + 7) / 8), dim3(256), 0, st, a);
}

namespace {
constexpr int SEL_DYN_MAX = 150 * 1024;

// Dynamic shared memory of one select CTA holding its slice (pooled values and the
// raw column sums with the pooling halo); 0 when the slice goes to the workspace.
long long select_slice_bytes(const CompressArgs& a, int cl) {
    const int M = a.R0 - a.cfg.L_sink;
    const int per = (M + cl - 1) / cl;
    const long long bytes = 4ll * (((per + 3) & ~3) + (long long)select_raw_words(per, a.cfg.P));
    return bytes <= SEL_DYN_MAX ? bytes : 0;
}

// Clusters of CL select CTAs that can be resident at once on this device (0 if the
// device refuses that size); the kernel's attributes are set on the way.  Cached per
// device.
template <int CL>
int select_active_clusters() {
    static std::atomic<int> cached[64];        // zero-initialised; -1 = refused
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    const bool cacheable = dev >= 0 && dev < 64;
    if (cacheable) {
        const int v = cached[dev].load(std::memory_order_relaxed);
        if (v != 0) return v > 0 ? v : 0;
    }
    int n = 0;
    if ((CL <= 8 || cudaFuncSetAttribute(select_kernel<CL>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
                        cudaSuccess) &&
        cudaFuncSetAttribute(select_kernel<CL>, cudaFuncAttributeMaxDynamicSharedMemorySize, SEL_DYN_MAX) ==
            cudaSuccess) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(CL, 1, 1);
        cfg.blockDim = dim3(SEL_THREADS);
        cfg.dynamicSmemBytes = SEL_DYN_MAX;
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeClusterDimension;
        at[0].val.clusterDim.x = CL;
        at[0].val.clusterDim.y = 1;
        at[0].val.clusterDim.z = 1;
        cfg.attrs = at;
        cfg.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(&n, select_kernel<CL>, &cfg) != cudaSuccess) n = 0;
    }
    cudaGetLastError();                          // a refusal above is an answer, not an error
    if (cacheable) cached[dev].store(n > 0 ? n : -1, std::memory_order_relaxed);
    return n;
}

template <int CL>
cudaError_t launch_select_cl(const CompressArgs& a, cudaStream_t st) {
    const long long bytes = select_slice_bytes(a, CL);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(CL, a.cfg.Hkv, 1);
    cfg.blockDim = dim3(SEL_THREADS);
    cfg.dynamicSmemBytes = (size_t)bytes;
    cfg.stream = st;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = CL;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    // the kernel waits for the previous grid before its first read
    at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, select_kernel<CL>, a, bytes > 0 ? 1 : 0);
}
}  // namespace

cudaError_t launch_select(const CompressArgs& a, cudaStream_t st) {
    // the largest cluster (shortest slices) with every head's cluster resident at once
    // (a cluster stays within one GPC); the portable 8 otherwise
    if (a.cfg.Hkv <= select_active_clusters<16>()) return launch_select_cl<16>(a, st);
    if (a.cfg.Hkv <= select_active_clusters<12>()) return launch_select_cl<12>(a, st);
    if (select_active_clusters<8>() == 0) {
        static std::atomic<uint64_t> smem_set{0};
        if (cudaError_t e = opt_in_smem(select_kernel<8>, SEL_DYN_MAX, smem_set); e != cudaSuccess) return e;
    }
    return launch_select_cl<8>(a, st);
}

}  // namespace snap
