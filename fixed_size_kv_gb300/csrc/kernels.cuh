// kernels.cuh -- launch interfaces between the C-ABI layer and the kernels.
#pragma once

#include <cuda.h>

#include <atomic>
#include <cstdint>

#include "common.cuh"

namespace snap {

using bf16 = __nv_bfloat16;

// ----------------------------------------------------------------- decode
struct DecodeArgs {
    const bf16* kc;              // cache keys   [max_batch][Hkv][C][dqk]
    const bf16* vc;              // cache values [max_batch][Hkv][C][dv] (GQA)
    const snap_seq_meta* meta;   // [max_batch]
    const int32_t* slots;        // [n]
    int n;
    const bf16* q;               // [n][Hq][dqk]
    float* out;                  // [n][Hq][dv] fp32
    float* part_o;               // [n][Hkv][splits][G][dv]
    float* part_ml;              // [n][Hkv][splits][G][2]  (max, sum) base-2 domain
    int splits;
    int tiles_per_split;         // in units of the kernel's key tile
    int32_t* status;
    DevConfig cfg;
    // fused ring append (snap_decode_step): the new token of sequence b is written into
    // ring slot L_sink + K + (T mod L_recent) by the CTA(s) whose key range holds it, the
    // attention sees T + 1 tokens, and the last CTA of the sequence to finish advances
    // meta.T (meta.pad[0] counts the CTAs of the sequence that have read the meta)
    const bf16* k_new;           // [n][Hkv][dqk] or null (no append)
    const bf16* v_new;           // [n][Hkv][dv] (GQA)
    snap_seq_meta* meta_rw;      // the same meta, writable (append only)
    int32_t* merge_cnt;          // [max_batch][Hkv] CTAs of (slot, head) done; zero between calls
    // GQA: the splits of one (sequence, KV head) run as one thread-block cluster and
    // merge through distributed shared memory (set by the launch when 2..8 splits)
    int cluster_merge;
};

constexpr int GQA_KEYS = 32;     // keys per warp step of the GQA decode kernel
constexpr int MLA_KEYS = 64;     // keys per tile of the MLA decode kernel
constexpr int MLA_HEADS = 128;   // query heads of the MLA layout (the M of its MMAs)

// Launches `kernel` with programmatic stream serialization: it may start while the
// previous kernel on `st` still runs, so its first statement must be pdl_wait().
template <typename... Exp, typename... Act>
cudaError_t launch_dependent(void (*kernel)(Exp...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                             Act&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Act&&>(args)...);
}

// As launch_dependent, with clusters of cluster_x CTAs along the grid's x.
template <typename... Exp, typename... Act>
cudaError_t launch_dependent_clustered(void (*kernel)(Exp...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                                       unsigned cluster_x, Act&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    at[1].id = cudaLaunchAttributeClusterDimension;
    at[1].val.clusterDim.x = cluster_x;
    at[1].val.clusterDim.y = 1;
    at[1].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Act&&>(args)...);
}

// Opts `kernel` into `bytes` of dynamic shared memory on the current device.  The
// attribute is per device, so `done` keeps one bit per device (devices 0..63; others
// set it on every call); concurrent first calls may both set it, which is harmless.
template <typename... Exp>
cudaError_t opt_in_smem(void (*kernel)(Exp...), int bytes, std::atomic<uint64_t>& done) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = (dev >= 0 && dev < 64) ? (uint64_t(1) << dev) : 0;
    if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_acq_rel);
    return e;
}

cudaError_t launch_decode_gqa(const DecodeArgs& a, cudaStream_t st);
// tkv: cache [max_batch][C][576], box {64, 64, 1}; tq: queries [n][128][576], box {64, 128, 1}
cudaError_t launch_decode_mla_tc(const DecodeArgs& a, const CUtensorMap& tkv, const CUtensorMap& tq,
                                 cudaStream_t st);
// CTAs of the MLA decode kernel that can be resident at once on the current device
// (one per SM at its shared-memory size; 0 if the occupancy query fails).
int mla_decode_wave_ctas();
cudaError_t launch_decode_merge(const DecodeArgs& a, cudaStream_t st);
// One kernel whose only (bounded) wait can never be satisfied: records SNAP_ERR_TIMEOUT.
cudaError_t launch_bounded_wait_selftest(int32_t* status, cudaStream_t st);

// ----------------------------------------------------------------- append
struct AppendArgs {
    bf16* kc;
    bf16* vc;
    snap_seq_meta* meta;
    const int32_t* slots;
    int n;
    const bf16* k_new;           // [n][Hkv][dqk]
    const bf16* v_new;           // [n][Hkv][dv]
    int32_t* status;
    DevConfig cfg;
};
cudaError_t launch_append(const AppendArgs& a, cudaStream_t st);

// --------------------------------------------------------------- compress
struct CompressArgs {
    const bf16* K;               // prompt keys (strided)
    const bf16* V;               // prompt values (GQA)
    int64_t tok_stride, head_stride;   // elements
    const bf16* Q;               // [W][Hq][dqk]
    int S;
    int R;                       // G * W observation rows per KV head
    int R0, n_sink, n_mid;
    int scored;                  // 1 when the SnapKV selection runs
    int slot;
    // workspace
    float* part_ml;              // [Hkv][R][row_splits][2]
    float* nlse2;                // [Hkv][R_pad]  -lse2 per observation row (-inf padding)
    float* col;                  // [SCORE_PARTS][Hkv][S_pad] column-sum parts (summed by select)
    uint32_t* pool;              // [Hkv][S_pad] pooled score bits
    int row_splits;              // partials per row (SCORE_PARTS per key split)
    int R_pad;
    int64_t S_pad;
    // cache
    bf16* kc;
    bf16* vc;
    snap_seq_meta* meta;
    int32_t* sel;                // [max_batch][Hkv][K]
    int32_t* status;
    DevConfig cfg;
};

cudaError_t launch_lse_merge(const CompressArgs& a, cudaStream_t st);
// -lse2 of every observation row from a caller-supplied natural-log LSE [W][Hq]
cudaError_t launch_lse_import(const CompressArgs& a, const float* lse_obs, cudaStream_t st);
cudaError_t launch_select(const CompressArgs& a, cudaStream_t st);

// ------------------------------------------------- score GEMM (tcgen05 + TMA)
struct ScoreParams {
    int S, W, R, G, Hkv;
    float sl2;                   // sm_scale * log2(e)
    int n_sc;                    // S - W scored prefix positions
    int n_units, splits, x_tiles;
    int Ny;                      // rows of the Y operand per MMA (N), multiple of 64, <= 256
    int R_pad;
    float* part_ml;              // ROWSTAT out: [Hkv][R][2*splits][2]
    const float* nlse2;          // COLSUM in:  [Hkv][R_pad]
    float* col;                  // COLSUM out: [SCORE_PARTS][Hkv][S_pad]
    int64_t S_pad;
    float* logits;               // LOGITS out: [Hkv][R][S]
    int32_t* status;
};
enum { SCORE_ROWSTAT = 0, SCORE_COLSUM = 1, SCORE_LOGITS = 2 };
// The score kernel's epilogue splits an accumulator's columns into this many parts (four
// warps each, one per TMEM lane quarter): the row pass leaves SCORE_PARTS partials per
// row and key split, the column pass SCORE_PARTS column-sum arrays.
constexpr int SCORE_PARTS = 4;
cudaError_t launch_score_tc(int mode, const CUtensorMap& tx, const CUtensorMap& ty, const ScoreParams& p,
                            int D, bool x_is_q, bool x_resident, int num_sms, bool pdl, cudaStream_t st);
cudaError_t launch_cache_write(const CompressArgs& a, int num_sms, cudaStream_t st);

// ------------------------------------------- causal prefill attention (tcgen05 + TMA)
struct PrefillArgs {
    int S, Hq, G, W;
    float sl2;                   // sm_scale * log2(e)
    bf16* O;                     // [S][Hq][128] output
    int64_t o_tok_stride;        // elements
    float* lse_obs;              // [W][Hq] natural-log LSE of the last W rows (nullable)
    int32_t* status;
};
// tq: Q {128, S, Hq}, tk / tv: K / V {128, S, Hkv}; boxes {64, 128, 1}, 128-byte swizzle
cudaError_t launch_prefill_tc(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                              const PrefillArgs& a, cudaStream_t st);

}  // namespace snap
