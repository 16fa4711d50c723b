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
#include "tc.cuh"

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

// Prefill cache build ("Fixed-Size Cache Layout"): every slot of the sequence is
// written, with the row of the position it holds, or zeros when it holds nothing (so a
// reused cache slot never carries a previous request's rows).

// Prompt position held by slot s of KV head h's cache, or -1 for none.
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

// Each copying warp owns a ring of NBUF buffers of CB_BYTES in shared memory, one
// mbarrier each.  Per batch of rows, every lane moves one row segment (the K half or
// the V half of a GQA row, or a whole MLA row) with a bulk asynchronous copy global ->
// shared that completes on the buffer's mbarrier; the batch then leaves shared memory
// with bulk copies shared -> global.  The loads of the next NBUF - 1 batches are in
// flight while a batch is stored, and no data passes through registers.  Slots that
// hold no position are zero-filled with plain stores.
constexpr int CB_BYTES = 8192;
constexpr int CB_WARPS = 8;                          // copying warps per CTA
constexpr int CW_NBUF = 3;
constexpr int CW_SMEM = CB_WARPS * CW_NBUF * CB_BYTES;

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}
__device__ __forceinline__ void bulk_s2g(void* dst, uint32_t src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;\n" ::"l"(dst), "r"(src), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;\n" ::"n"(N) : "memory");
}
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;\n" ::: "memory"); }

// One lane's segment of a batch: its cache row (index within the sequence's
// [H_kv][C] rows), its source (null when the slot holds no position) and its size.
struct RowSeg {
    int64_t lin;
    const bf16* src;
    int bytes;
};

__device__ __forceinline__ RowSeg cache_row_seg(const CompressArgs& a, int64_t r, int sg, int kb, int vb) {
    const DevConfig& c = a.cfg;
    const int h = (int)(r / c.C);
    const int s = (int)(r - (int64_t)h * c.C);
    const int pos = cache_row_position(a, a.sel + ((size_t)a.slot * c.Hkv + h) * c.K, s);
    RowSeg g;
    g.lin = r;
    g.bytes = sg ? vb : kb;
    g.src = pos < 0 ? nullptr : (sg ? a.V : a.K) + (size_t)pos * a.tok_stride + (size_t)h * a.head_stride;
    return g;
}

// Called by a whole warp: warp w of n_warps copies batches w, w + n_warps, ... of the
// sequence's H_kv x C cache rows.  buf: this warp's NBUF x CB_BYTES of shared memory
// (a batch's K segments first, then its V segments); bars: its NBUF mbarriers, 8 bytes
// apart (initialised here).  A batch whose rows all hold positions leaves as one bulk
// store per K / V run (its rows are consecutive in the cache); any other batch row by
// row.  Returns false if a wait gave up (the status word then holds SNAP_ERR_TIMEOUT).
template <int NBUF>
__device__ bool cache_copy_rows_bulk(const CompressArgs& a, int64_t w, int64_t n_warps, uint32_t buf,
                                     uint32_t bars, volatile int* abort_flag) {
    const DevConfig& c = a.cfg;
    const int lane = threadIdx.x & 31;
    const int kb = c.dqk * 2, vb = c.layout == SNAP_LAYOUT_GQA ? c.dv * 2 : 0;
    const int segs = vb ? 2 : 1;
    const int rpb = min(32 / segs, CB_BYTES / (kb + vb));    // rows per batch
    const int64_t rows = (int64_t)c.Hkv * c.C;
    const size_t slot_rows = (size_t)a.slot * c.Hkv * (size_t)c.C;
    const int u = lane / segs, sg = lane % segs;
    const uint32_t seg_off = sg ? rpb * kb + u * vb : u * kb;   // this lane's segment in a buffer
    const int64_t step = n_warps * rpb;
    if (lane == 0) {
        for (int i = 0; i < NBUF; ++i) mbar_init(bars + 8 * i, 1);
        fence_barrier_init();
    }
    __syncwarp();
    const int64_t first = w * rpb;
    auto seg = [&](int j, bool* act) {
        const int64_t r = first + j * step + u;
        *act = u < rpb && r < rows;
        RowSeg g{0, nullptr, 0};
        if (*act) g = cache_row_seg(a, r, sg, kb, vb);
        return g;
    };
    // batch j covers rows first + j * step + [0, rpb); its buffer is j % NBUF
    auto load = [&](int j) {
        bool act;
        const RowSeg g = seg(j, &act);
        const uint32_t bar = bars + 8 * (j % NBUF);
        const uint32_t tx = __reduce_add_sync(0xffffffffu, (uint32_t)(g.src ? g.bytes : 0));
        if (lane == 0) mbar_expect_tx(bar, tx);
        __syncwarp();
        if (g.src) bulk_g2s(buf + (j % NBUF) * CB_BYTES + seg_off, g.src, g.bytes, bar);
    };
    const int n_b = first < rows ? (int)((rows - first + step - 1) / step) : 0;
    for (int j = 0; j < NBUF - 1 && j < n_b; ++j) load(j);
    for (int j = 0; j < n_b; ++j) {
        bool act;
        const RowSeg g = seg(j, &act);
        bf16* dst = act ? (sg ? a.vc + (slot_rows + g.lin) * c.dv : a.kc + (slot_rows + g.lin) * c.dqk) : nullptr;
        if (act && !g.src)
            for (int i = 0; i < g.bytes / 16; ++i) reinterpret_cast<uint4*>(dst)[i] = make_uint4(0u, 0u, 0u, 0u);
        // one run: every active row holds a position (the rows of a batch are consecutive)
        const int64_t lin0 = __shfl_sync(0xffffffffu, g.lin, 0);
        const bool run = __all_sync(0xffffffffu, !act || g.src != nullptr);
        const int n_act = __popc(__ballot_sync(0xffffffffu, act && sg == 0));
        if (!__all_sync(0xffffffffu, mbar_wait_bounded(bars + 8 * (j % NBUF), (j / NBUF) & 1, abort_flag))) {
            if (lane == 0) report_error(a.status, SNAP_ERR_TIMEOUT, 400, (int)w, (int)(first + j * step));
            // the later batches' loads already issued: wait for them too (bounded), so
            // none lands after the CTA's shared memory is gone
            for (int k = j + 1; k < j + NBUF && k < n_b; ++k)
                mbar_wait_bounded(bars + 8 * (k % NBUF), (k / NBUF) & 1, abort_flag);
            bulk_wait_all();
            return false;
        }
        const uint32_t sb = buf + (j % NBUF) * CB_BYTES;
        if (run) {
            if (lane < segs)    // lane 0: the K run, lane 1: the V run
                bulk_s2g(lane ? (void*)(a.vc + (slot_rows + lin0) * c.dv) : (void*)(a.kc + (slot_rows + lin0) * c.dqk),
                         sb + (lane ? rpb * kb : 0), n_act * (lane ? vb : kb));
        } else if (g.src) {
            bulk_s2g(dst, sb + seg_off, g.bytes);
        }
        bulk_commit();
        // refill the buffer of batch j - 1 (free at j = 0) with batch j + NBUF - 1, once
        // the stores of batch j - 1 (all but this lane's latest group) have read it
        if (j + NBUF - 1 < n_b) {
            bulk_wait_read<1>();
            __syncwarp();
            load(j + NBUF - 1);
        }
    }
    bulk_wait_all();     // every store done before the buffers go away with the CTA
    return true;
}

// The cache rows, the unscored selection list and the sequence meta.  Eight copying
// warps per CTA, each with a ring of CW_NBUF buffers; one CTA per SM.
__global__ void __launch_bounds__(CB_WARPS * 32) cache_write_kernel(CompressArgs a) {
    extern __shared__ __align__(128) uint8_t cw_smem[];
    __shared__ __align__(8) uint64_t bars[CB_WARPS * CW_NBUF];
    __shared__ int abort_flag;
    const DevConfig& c = a.cfg;
    if (threadIdx.x == 0) abort_flag = 0;
    pdl_wait();                 // the selection (and everything before it) is complete and visible
    __syncthreads();
    const int warp = threadIdx.x >> 5;
    const int64_t n_warps = (int64_t)gridDim.x * CB_WARPS, w = (int64_t)blockIdx.x * CB_WARPS + warp;
    cache_copy_rows_bulk<CW_NBUF>(a, w, n_warps, smem_u32(cw_smem) + warp * CW_NBUF * CB_BYTES,
                                  smem_u32(bars + CW_NBUF * warp), &abort_flag);
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
    // one CTA per SM, fewer when the cache has fewer batches; at least one per KV head
    // (the unscored selection list)
    static std::atomic<uint64_t> smem_set{0};
    if (cudaError_t e = opt_in_smem(cache_write_kernel, CW_SMEM, smem_set); e != cudaSuccess) return e;
    const int row_b = 2 * (a.cfg.dqk + (a.cfg.layout == SNAP_LAYOUT_GQA ? a.cfg.dv : 0));
    const int segs = a.cfg.layout == SNAP_LAYOUT_GQA ? 2 : 1;
    const int rpb = (32 / segs) < (CB_BYTES / row_b) ? 32 / segs : CB_BYTES / row_b;
    const long long batches = ((long long)a.cfg.Hkv * a.cfg.C + rpb - 1) / rpb;
    long long blocks = (batches + CB_WARPS - 1) / CB_WARPS;
    if (blocks > num_sms) blocks = num_sms;
    if (blocks < a.cfg.Hkv) blocks = a.cfg.Hkv;
    return launch_dependent(cache_write_kernel, dim3((unsigned)blocks), dim3(CB_WARPS * 32), CW_SMEM, st, a);
}

}  // namespace snap
