// common.cuh -- device-side helpers shared by the libsnap kernels (sm_103a).
//
// Inline PTX wrappers for the instructions the kernels are built from:
// cp.async (16-byte global->shared copies), ldmatrix, mma.sync m16n8k16 bf16 with
// fp32 accumulation, movmatrix (register transpose of an 8x8 b16 tile) and ex2.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "snap.h"

namespace snap {

// Kernel-side copy of the cache configuration.
struct DevConfig {
    int layout;
    int Hq, Hkv, G;
    int dqk, dv;
    int L_sink, K, L_recent;
    int W, P;
    int C;             // L_sink + K + L_recent
    int max_batch;
    float scale;       // sm_scale
    float scale_log2;  // sm_scale * log2(e): scores kept in the base-2 domain
};

// Records the first kernel-side error in the cache's status word.
__device__ __forceinline__ void report_error(int32_t* status, int code, int a, int b, int c) {
    if (atomicCAS(status, 0, code) == 0) {
        status[1] = a;
        status[2] = b;
        status[3] = c;
    }
}

// Slot validity of a sequence at its current length (see snap_decode_attn).
struct SlotValidity {
    int n_sink, L_sink, mid_end;   // middle slots [L_sink, mid_end) valid
    int ring0, L_recent, n_ring;   // ring slots: offset (r - lo mod L_recent) < n_ring
    int lo_mod;

    __device__ __forceinline__ void init(const snap_seq_meta& m, const DevConfig& c) {
        n_sink = m.n_sink;
        L_sink = c.L_sink;
        mid_end = c.L_sink + m.n_mid;
        ring0 = c.L_sink + c.K;
        L_recent = c.L_recent;
        int n = m.T - m.R0;
        n_ring = n < c.L_recent ? n : c.L_recent;
        int lo = m.T - n_ring;
        lo_mod = lo % c.L_recent;
    }
    __device__ __forceinline__ bool valid(int s) const {
        if (s < L_sink) return s < n_sink;
        if (s < ring0) return s < mid_end;
        int off = s - ring0 - lo_mod;
        if (off < 0) off += L_recent;
        return off < n_ring;
    }
    // true if any slot in [a, b) may be valid (conservative for the ring).
    __device__ __forceinline__ bool any_valid(int a, int b) const {
        if (a < L_sink && n_sink > a) return true;
        if (b > L_sink && a < ring0) {
            int lo = a > L_sink ? a : L_sink;
            if (lo < mid_end) return true;
        }
        if (b > ring0) {
            if (n_ring >= L_recent) return true;
            if (n_ring <= 0) return false;
            int r0 = (a > ring0 ? a : ring0) - ring0;
            int r1 = b - ring0;  // exclusive
            // valid ring offsets: [lo_mod, lo_mod + n_ring) modulo L_recent
            int e = lo_mod + n_ring;
            if (r1 > lo_mod && r0 < (e < L_recent ? e : L_recent)) return true;
            if (e > L_recent && r0 < e - L_recent) return true;
        }
        return false;
    }
};

// ------------------------------------------------------------------ PTX wrappers

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte async copy; src_bytes 0 zero-fills the destination.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes = 16) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;\n" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// D(16x8 fp32) += A(16x16 bf16, row) * B(16x8 bf16, col)
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Transpose of an 8x8 b16 matrix held one row-pair per thread.
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n" : "=r"(y) : "r"(x));
    return y;
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
    return y;
}

// Programmatic dependent launch.  A kernel launched with the programmatic stream
// serialization attribute may start while the previous kernel on its stream still
// runs: pdl_wait() returns once that kernel has completed and its writes are visible
// (at once after a normal launch), and pdl_launch_dependents() lets the next such
// kernel start (it launches once every CTA of this grid has called it or exited).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}

// L2 policy for data that the next kernel reads again: its lines are evicted after
// those of streaming traffic (evict_last, on the whole access).
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// Global store of one float with an L2 policy.
__device__ __forceinline__ void st_global_policy(float* ptr, float v, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.f32 [%0], %1, %2;" ::"l"(ptr), "f"(v), "l"(pol) : "memory");
}

// max of three floats in one instruction (-inf is the identity; a NaN operand is ignored
// unless all are NaN, as for fmaxf)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float m;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(m) : "f"(a), "f"(b), "f"(c));
    return m;
}
// acc (two fp32 lanes) += (lo, hi), one packed add
__device__ __forceinline__ void add_f32x2(uint64_t& acc, uint32_t lo, uint32_t hi) {
    asm("{\n .reg .b64 t;\n mov.b64 t, {%1, %2};\n add.rn.f32x2 %0, %0, t;\n}\n" : "+l"(acc) : "r"(lo), "r"(hi));
}
// (a0, a1) = (x0, x1) * m + b, lane by lane, one packed fma (m, b: packed pairs)
__device__ __forceinline__ void fma_f32x2(float& a0, float& a1, float x0, float x1, uint64_t m, uint64_t b) {
    asm("{\n .reg .b64 x, y;\n mov.b64 x, {%2, %3};\n fma.rn.f32x2 y, x, %4, %5;\n mov.b64 {%0, %1}, y;\n}\n"
        : "=f"(a0), "=f"(a1)
        : "f"(x0), "f"(x1), "l"(m), "l"(b));
}
// the packed pair (lo, hi)
__device__ __forceinline__ uint64_t f32x2_pack(float lo, float hi) {
    return (uint64_t)__float_as_uint(lo) | ((uint64_t)__float_as_uint(hi) << 32);
}
// both lanes of a packed pair set to x
__device__ __forceinline__ uint64_t f32x2_splat(float x) {
    const uint64_t u = __float_as_uint(x);
    return u | (u << 32);
}
// the sum of a packed pair's two fp32 lanes
__device__ __forceinline__ float f32x2_sum(uint64_t x) {
    return __uint_as_float((uint32_t)x) + __uint_as_float((uint32_t)(x >> 32));
}
__device__ __forceinline__ float bf16_round(float x) {
    return __bfloat162float(__float2bfloat16_rn(x));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// Byte offset of 16-byte chunk `c` of row `r` in a shared tile whose rows are
// `row_bytes` long (a multiple of 128): chunks are XOR-swizzled inside each
// 128-byte segment so that 8 rows read at the same column hit 8 distinct banks.
__device__ __forceinline__ uint32_t swz(int r, int c, int row_bytes) {
    return static_cast<uint32_t>(r * row_bytes + ((((c & ~7) | ((c & 7) ^ (r & 7)))) << 4));
}

}  // namespace snap
