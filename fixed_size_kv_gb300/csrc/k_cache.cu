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
// never carries a previous request's rows).
__global__ void cache_write_kernel(CompressArgs a) {
    const DevConfig& c = a.cfg;
    const int h = blockIdx.y;
    const int ck = c.dqk / 8, cv = (c.layout == SNAP_LAYOUT_GQA) ? c.dv / 8 : 0;
    const int per_slot = ck + cv;
    const int32_t* sel_h = a.sel + ((size_t)a.slot * c.Hkv + h) * c.K;
    const int ring0 = c.L_sink + c.K;
    const int R0m = a.R0 % c.L_recent;
    const size_t total = (size_t)c.C * per_slot;
    for (size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (size_t)gridDim.x * blockDim.x) {
        const int s = (int)(idx / per_slot), ch = (int)(idx % per_slot);
        int p = -1;
        if (s < c.L_sink) {
            p = s < a.n_sink ? s : -1;
        } else if (s < ring0) {
            const int i = s - c.L_sink;
            if (i < a.n_mid) p = a.scored ? sel_h[i] : c.L_sink + i;
        } else {
            int off = (s - ring0) - R0m;
            if (off < 0) off += c.L_recent;
            const int q = a.R0 + off;  // the position congruent to this ring slot in [R0, R0+L_recent)
            p = q < a.S ? q : -1;
        }
        const size_t row = ((size_t)a.slot * c.Hkv + h) * (size_t)c.C + s;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (ch < ck) {
            if (p >= 0)
                v = reinterpret_cast<const uint4*>(a.K + (size_t)p * a.tok_stride + (size_t)h * a.head_stride)[ch];
            reinterpret_cast<uint4*>(a.kc + row * c.dqk)[ch] = v;
        } else {
            const int cc = ch - ck;
            if (p >= 0)
                v = reinterpret_cast<const uint4*>(a.V + (size_t)p * a.tok_stride + (size_t)h * a.head_stride)[cc];
            reinterpret_cast<uint4*>(a.vc + row * c.dv)[cc] = v;
        }
    }
    // selected-position list for sequences that needed no scoring
    if (!a.scored && blockIdx.x == 0) {
        int32_t* out = a.sel + ((size_t)a.slot * c.Hkv + h) * c.K;
        for (int i = threadIdx.x; i < c.K; i += blockDim.x) out[i] = i < a.n_mid ? c.L_sink + i : -1;
    }
    if (blockIdx.x == 0 && h == 0 && threadIdx.x == 0) {
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
    const int per_slot = a.cfg.dqk / 8 + (a.cfg.layout == SNAP_LAYOUT_GQA ? a.cfg.dv / 8 : 0);
    const long long total = (long long)a.cfg.C * per_slot;
    long long want = (total + 255) / 256;
    int bx = (int)(want < 1 ? 1 : want);
    const int cap = (num_sms * 8 + a.cfg.Hkv - 1) / a.cfg.Hkv;
    if (bx > cap) bx = cap;
    dim3 grid(bx, a.cfg.Hkv);
    cache_write_kernel<<<grid, 256, 0, st>>>(a);
    return cudaGetLastError();
}

}  // namespace snap
