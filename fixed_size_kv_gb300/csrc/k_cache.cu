// k_cache.cu -- writes into the fixed-size cache: the prefill cache build and
// the decode-step ring append.
//
// SnapStream episode companion page:
//  - "Fixed-Size Cache Layout": the cache is built once at prefill as
//    [L_sink sinks | K selected middle | L_recent recent].
//  - "Ring Buffer vs. Naive Slicing": decode only rotates the recent window;
//    each new token is scattered into a fixed index, with no gather and no
//    concatenation.  Position p lives in ring slot L_sink + K + (p mod L_recent).
#include "kernels.cuh"

namespace snap {

namespace {

// One CTA per sequence of the batch.  Copies the new token's rows into the ring
// slot of position T, then advances T.
__global__ void append_kernel(AppendArgs a) {
    pdl_launch_dependents();    // the attention that follows may set up (it waits for this grid)
    const DevConfig& c = a.cfg;
    const int b = blockIdx.x;
    const int slot = a.slots[b];
    if (slot < 0 || slot >= c.max_batch) {
        if (threadIdx.x == 0) report_error(a.status, SNAP_ERR_DEVICE_CHECK, 2, b, slot);
        return;
    }
    const int T = a.meta[slot].T;
    const int s = c.L_sink + c.K + T % c.L_recent;
    const int ck = c.dqk / 8, cv = (c.layout == SNAP_LAYOUT_GQA) ? c.dv / 8 : 0;
    const int per_head = ck + cv;
    for (int i = threadIdx.x; i < c.Hkv * per_head; i += blockDim.x) {
        const int h = i / per_head, ch = i % per_head;
        const size_t row = ((size_t)slot * c.Hkv + h) * (size_t)c.C + s;
        if (ch < ck) {
            const uint4 v = reinterpret_cast<const uint4*>(a.k_new + ((size_t)b * c.Hkv + h) * c.dqk)[ch];
            reinterpret_cast<uint4*>(a.kc + row * c.dqk)[ch] = v;
        } else {
            const int cc = ch - ck;
            const uint4 v = reinterpret_cast<const uint4*>(a.v_new + ((size_t)b * c.Hkv + h) * c.dv)[cc];
            reinterpret_cast<uint4*>(a.vc + row * c.dv)[cc] = v;
        }
    }
    __syncthreads();  // every thread has read T before it moves
    if (threadIdx.x == 0) a.meta[slot].T = T + 1;
}

// Prefill cache build: every slot of the sequence is written, with the row of
// the position it holds, or zeros when it holds nothing (so a reused cache slot
// never carries a previous request's rows).  One warp per cache row (KV head h,
// slot s), four rows in flight per warp: the lanes copy the row's 16-byte chunks (a GQA
// row is 16 K chunks + 16 V chunks, one per lane; an MLA row 72 key chunks).
constexpr int CW_ROWS = 4;

__device__ __forceinline__ int cache_row_position(const CompressArgs& a, const int32_t* sel_h, int s) {
    const DevConfig& c = a.cfg;
    const int ring0 = c.L_sink + c.K;
    if (s < c.L_sink) return s < a.n_sink ? s : -1;
    if (s < ring0) {
        const int i = s - c.L_sink;
        if (i >= a.n_mid) return -1;
        return a.scored ? __ldg(sel_h + i) : c.L_sink + i;
    }
    int off = (s - ring0) - a.R0 % c.L_recent;
    if (off < 0) off += c.L_recent;
    const int q = a.R0 + off;   // the position congruent to this ring slot in [R0, R0 + L_recent)
    return q < a.S ? q : -1;
}

__global__ void __launch_bounds__(256) cache_write_kernel(CompressArgs a) {
    const DevConfig& c = a.cfg;
    const int lane = threadIdx.x & 31;
    const int ck = c.dqk / 8, cv = (c.layout == SNAP_LAYOUT_GQA) ? c.dv / 8 : 0;
    const int per_row = ck + cv;
    const int64_t rows = (int64_t)c.Hkv * c.C;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    const int64_t w0 = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    for (int64_t r0 = w0 * CW_ROWS; r0 < rows; r0 += warps * CW_ROWS) {
        int pos[CW_ROWS];
#pragma unroll
        for (int u = 0; u < CW_ROWS; ++u) {
            const int64_t r = r0 + u;
            pos[u] = -1;
            if (r < rows) {
                const int h = (int)(r / c.C), s = (int)(r % c.C);
                pos[u] = cache_row_position(a, a.sel + ((size_t)a.slot * c.Hkv + h) * c.K, s);
            }
        }
        for (int ch = lane; ch < per_row; ch += 32) {
            uint4 v[CW_ROWS];
#pragma unroll
            for (int u = 0; u < CW_ROWS; ++u) {
                const int64_t r = r0 + u;
                v[u] = make_uint4(0u, 0u, 0u, 0u);
                if (r < rows && pos[u] >= 0) {
                    const int h = (int)(r / c.C);
                    const size_t src = (size_t)pos[u] * a.tok_stride + (size_t)h * a.head_stride;
                    v[u] = ch < ck ? __ldg(reinterpret_cast<const uint4*>(a.K + src) + ch)
                                   : __ldg(reinterpret_cast<const uint4*>(a.V + src) + (ch - ck));
                }
            }
#pragma unroll
            for (int u = 0; u < CW_ROWS; ++u) {
                const int64_t r = r0 + u;
                if (r >= rows) continue;
                const size_t row = (size_t)a.slot * rows + r;      // [slot][h][s]
                if (ch < ck) reinterpret_cast<uint4*>(a.kc + row * c.dqk)[ch] = v[u];
                else reinterpret_cast<uint4*>(a.vc + row * c.dv)[ch - ck] = v[u];
            }
        }
    }
    // selected-position list for sequences that needed no scoring
    if (!a.scored && blockIdx.x < c.Hkv) {
        const int h = blockIdx.x;
        int32_t* out = a.sel + ((size_t)a.slot * c.Hkv + h) * c.K;
        for (int i = threadIdx.x; i < c.K; i += blockDim.x) out[i] = i < a.n_mid ? c.L_sink + i : -1;
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        snap_seq_meta m;
        m.S = a.S;
        m.T = a.S;
        m.R0 = a.R0;
        m.n_sink = a.n_sink;
        m.n_mid = a.n_mid;
        m.pad[0] = m.pad[1] = m.pad[2] = 0;
        a.meta[a.slot] = m;
    }
}

}  // namespace

cudaError_t launch_append(const AppendArgs& a, cudaStream_t st) {
    append_kernel<<<a.n, 256, 0, st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_cache_write(const CompressArgs& a, int num_sms, cudaStream_t st) {
    // one wave of 8 CTAs (64 warps) per SM, fewer when the cache has fewer row groups
    const long long groups = ((long long)a.cfg.Hkv * a.cfg.C + CW_ROWS - 1) / CW_ROWS;
    long long blocks = (groups + 7) / 8;
    const long long cap = (long long)num_sms * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < a.cfg.Hkv) blocks = a.cfg.Hkv;       // the unscored selection list: one CTA per head
    cache_write_kernel<<<(unsigned)blocks, 256, 0, st>>>(a);
    return cudaGetLastError();
}

}  // namespace snap
