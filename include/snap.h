/*
 * snap.h -- C ABI of libsnap: the SnapStream fixed-size KV cache on GB300 (sm_103a).
 *
 * Method: SnapStream: Efficient Long Sequence Decoding on Dataflow Accelerators
 * (arXiv 2511.03092).  Its episode companion page, section "Fixed-Size Cache
 * Layout", fixes one static cache per sequence built once at prefill,
 *
 *        [ L_sink sink tokens | K SnapKV-selected middle tokens | L_recent recent ]
 *
 * with the three sizes as configurable hyperparameters; section "Ring Buffer vs.
 * Naive Slicing" fixes that decode only rotates the recent window, writing each
 * new token into a fixed index (scatter, no gather, no concat).  The SnapKV
 * step ("pooling-based top-K selection", section "Infinity-Bench KV Retrieval")
 * scores every prefix position by the softmax of the last W prompt queries
 * (the observation window), summed over the window and over the query heads
 * that share a KV head, max-pools the scores with an odd kernel P, and keeps the
 * K best middle positions (ties go to the lower position; kept in ascending
 * order).
 *
 * Conventions (every entry point):
 *  - All data pointers are DEVICE pointers unless a comment says host.  bf16 data
 *    is passed as void*; it must be 16-byte aligned, as must every row stride in
 *    bytes.
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).
 *    Every call is asynchronous on that stream, performs no host synchronisation
 *    and allocates no memory: buffers and workspaces are owned by the caller.
 *  - Argument and shape errors are detected on the host and returned synchronously;
 *    nothing is launched then.  Errors found by a kernel (a slot index out of range,
 *    a bounded wait that expired) are recorded in the cache's device status word and
 *    read back by snap_check_device().
 *  - Not thread-safe per cache handle: calls on one handle must be ordered by the
 *    caller (same stream, or events).
 */
#ifndef SNAP_H
#define SNAP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SNAP_OK = 0,
    SNAP_ERR_INVALID_ARG = 1,  /* null pointer, misaligned pointer/stride, bad slot count */
    SNAP_ERR_SHAPE = 2,        /* sizes violate the method's preconditions */
    SNAP_ERR_UNSUPPORTED = 3,  /* valid for the method, not implemented by these kernels */
    SNAP_ERR_CUDA = 4,         /* a CUDA runtime/driver call failed */
    SNAP_ERR_TIMEOUT = 5,      /* a kernel's bounded wait expired (device status word) */
    SNAP_ERR_DEVICE_CHECK = 6  /* a kernel rejected an index (device status word) */
} snap_status;

/* Layout of the attention the cache serves. */
enum { SNAP_LAYOUT_GQA = 0, SNAP_LAYOUT_MLA = 1 };

/*
 * Cache configuration.
 *  layout      SNAP_LAYOUT_GQA: separate K and V, n_q_heads / n_kv_heads query heads per
 *              KV head (query head i reads KV head i / G).  Supported: d_qk == d_v == 128,
 *              G = n_q_heads / n_kv_heads in {1, 2, 4, 8}.
 *              SNAP_LAYOUT_MLA: one latent KV head (n_kv_heads == 1); the key row is
 *              [latent (d_v) | rope (d_qk - d_v)] and the value is its first d_v columns
 *              (absorbed-query attention, DeepSeek-V2 style).  Supported: d_qk == 576,
 *              d_v == 512, n_q_heads == 128 (the M side of the decode MMAs).
 *  L_sink, K, L_recent   segment sizes; C = L_sink + K + L_recent slots per KV head.
 *  W           observation window (last W prompt queries); 1 <= W <= L_recent.
 *  P           max-pool kernel width, odd, >= 1.
 *  sm_scale    softmax scale applied to q.k (> 0).
 */
typedef struct {
    int layout;
    int n_q_heads;
    int n_kv_heads;
    int d_qk;
    int d_v;
    int L_sink;
    int K;
    int L_recent;
    int W;
    int P;
    float sm_scale;
} snap_config;

/* Per-sequence bookkeeping kept on the device (one entry per cache slot). */
typedef struct {
    int32_t S;       /* prompt length at compression */
    int32_t T;       /* current length: S + appended tokens */
    int32_t R0;      /* first prompt position that was written into the ring */
    int32_t n_sink;  /* valid sink slots = min(L_sink, S) */
    int32_t n_mid;   /* valid middle slots = min(K, R0 - n_sink) */
    int32_t pad[3];  /* library use: pad[0] counts the CTAs of a decode step in flight (zero
                        between calls) */
} snap_seq_meta;

/* Device addresses of the regions a cache occupies inside the caller's buffer. */
typedef struct {
    void* k;               /* bf16 [max_batch][n_kv_heads][C][d_qk] */
    void* v;               /* bf16 [max_batch][n_kv_heads][C][d_v]; NULL for MLA */
    snap_seq_meta* meta;   /* [max_batch] */
    int32_t* sel;          /* [max_batch][n_kv_heads][K] selected middle positions */
    int32_t* status;       /* device status word: [0] = snap_status, [1..3] = detail */
    int64_t C;             /* slots per KV head */
    int max_batch;
} snap_cache_view;

typedef struct snap_cache snap_cache; /* opaque host-side handle */

/* Human-readable text of a status code (static string, never NULL). */
const char* snap_status_string(int status);

/* Library ABI version (incremented on incompatible changes). */
int snap_abi_version(void);

/* Checks a configuration against the method's preconditions and these kernels. */
snap_status snap_config_check(const snap_config* cfg);

/*
 * Bytes of device memory a cache of `max_batch` sequences needs (host call, no
 * CUDA).  The cache is exactly C / T_full of a full KV cache of T_full tokens:
 * for C = 32768 against 131072 tokens that is 4x smaller (the page's "4.0x lower
 * KV memory").
 */
snap_status snap_cache_bytes(const snap_config* cfg, int max_batch, size_t* bytes);

/*
 * Binds a cache to a caller-owned device buffer of at least snap_cache_bytes()
 * bytes (256-byte aligned): max_batch static-shape caches of the "Fixed-Size Cache
 * Layout" section ([L_sink | K | L_recent] slots per KV head, fixed at creation, as the
 * "Why This Wasn't Already Standard" section asks of static-graph hardware), plus the
 * per-sequence meta, the selection lists, split-merge counters and the status word.
 * The handle owns host state only; the buffer stays the caller's and must outlive the
 * handle.  Zeroes the whole buffer on `stream` (every slot starts empty).  *out
 * receives the handle.  SNAP_ERR_INVALID_ARG for a null or misaligned buffer, a
 * buffer smaller than snap_cache_bytes(), or max_batch < 1; SNAP_ERR_CUDA if the
 * zeroing cannot be queued.
 */
snap_status snap_cache_create(const snap_config* cfg, int max_batch, void* dev_buf,
                              size_t bytes, void* stream, snap_cache** out);
void snap_cache_destroy(snap_cache* cache);

/* Fills *out with the device addresses of the cache regions (host call). */
snap_status snap_cache_view_get(const snap_cache* cache, snap_cache_view* out);

/* Workspace bytes snap_compress() needs for prompts of up to S_max tokens. */
snap_status snap_compress_ws_bytes(const snap_config* cfg, int64_t S_max, size_t* bytes);

/*
 * Prefill compression of one sequence into cache slot `slot` (0 <= slot < max_batch),
 * the SnapKV + StreamingLLM fusion of the "Fixed-Size Cache Layout" section.
 *  K       bf16 keys: element (token j, kv head h, e) at K + j*tok_stride + h*head_stride + e
 *          (strides in elements; post-RoPE keys; MLA: the [latent | rope] rows).
 *  V       bf16 values with the same strides (GQA); must be NULL for MLA.
 *  S       prompt length >= 1.  Scoring runs only when the middle [L_sink, S - L_recent)
 *          holds more than K positions.
 *  Q_obs   bf16 [W][n_q_heads][d_qk], the queries of prompt positions S-W .. S-1.
 *  ws      device workspace of at least snap_compress_ws_bytes(cfg, S) bytes.
 * Writes every slot of the sequence (unused ones zeroed), the selected positions and
 * the meta {S, T = S, R0, n_sink, n_mid}.  The softmax denominator of each window row
 * runs over all keys up to the query's own position (the prefill attention's row).
 */
snap_status snap_compress(snap_cache* cache, int slot, const void* K, const void* V, int64_t S,
                          int64_t tok_stride, int64_t head_stride, const void* Q_obs,
                          void* ws, size_t ws_bytes, void* stream);

/*
 * snap_compress() for a caller whose prefill attention already produced the
 * log-sum-exp of the observation rows (a flash-attention kernel returns it for every
 * query position).  lse_obs: device fp32 [W][n_q_heads], natural log of
 * sum_j exp(sm_scale * q.k_j) over the causal row of query head i at prompt position
 * S-W+w.  The row pass is skipped; everything else is snap_compress().  The result is
 * the same as snap_compress() up to the rounding of the supplied LSE.
 */
snap_status snap_compress_lse(snap_cache* cache, int slot, const void* K, const void* V, int64_t S,
                              int64_t tok_stride, int64_t head_stride, const void* Q_obs, const float* lse_obs,
                              void* ws, size_t ws_bytes, void* stream);

/* Stages of a compression, in the order they run (snap_compress_stages). */
enum {
    SNAP_STAGE_ROWS = 1,     /* row pass: log-sum-exp of every observation row (or import of lse_obs) */
    SNAP_STAGE_COLUMNS = 2,  /* column pass: per prompt position, the window softmax summed over rows */
    SNAP_STAGE_SELECT = 4,   /* max-pool of width P and top-K of the middle positions */
    SNAP_STAGE_WRITE = 8,    /* cache build: sinks, selected rows, ring; sequence meta */
    SNAP_STAGE_ALL = 15
};

/*
 * snap_compress() (lse_obs NULL) or snap_compress_lse() (lse_obs given), running only
 * the stages set in `stages`.  The stages hand their results to the next one through
 * the workspace `ws` and the cache's selection list, so running every stage in order,
 * in one call or in several calls on the same stream with the same arguments and
 * workspace, gives exactly the result of the one-call form.  For profiling the steps
 * of the "Fixed-Size Cache Layout" build (score passes, pooling + top-K, cache write)
 * one at a time, and for callers that interleave the stages of several sequences.
 * When the prompt needs no scoring (the middle holds <= K positions) only the write
 * stage does anything.  SNAP_ERR_INVALID_ARG for bits outside SNAP_STAGE_ALL.
 */
snap_status snap_compress_stages(snap_cache* cache, int slot, const void* K, const void* V, int64_t S,
                                 int64_t tok_stride, int64_t head_stride, const void* Q_obs,
                                 const float* lse_obs, void* ws, size_t ws_bytes, int stages, void* stream);

/*
 * Inspection of the compression's score GEMM: the base-2 logits
 * out[h][r][j] = log2(e) * sm_scale * q_r . k_j  (fp32 [n_kv_heads][G*W][S]) of every
 * observation row r = w*G + g (query head h*G+g at position S-W+w) against every
 * prompt key j, computed by the same tensor-core kernel that scores prompts in
 * snap_compress().  Arguments as for snap_compress(); S >= W.  Uses the cache handle
 * for its configuration and status word only.
 */
snap_status snap_window_logits(snap_cache* cache, const void* K, int64_t S, int64_t tok_stride,
                               int64_t head_stride, const void* Q_obs, float* out, void* stream);

/*
 * Causal prefill attention of one prompt, GQA layout (head_dim 128), on the tensor
 * cores: O[i][h] = softmax_j<=i(sm_scale * q_{i,h} . k_{j,h/G}) v_{j,h/G}, plus the
 * log-sum-exp of the last W rows in the layout snap_compress_lse() takes.  The episode
 * companion page's headline figure puts the compression at "2-5% extra prefill
 * latency": a prefill that already holds each query row's log-sum-exp hands it over,
 * and the compression skips its own row pass.
 *  Q        bf16 [S][n_q_heads][128], contiguous
 *  K, V     bf16 keys / values with element (j, h, e) at base + j*tok_stride +
 *           h*head_stride + e (the strides of snap_compress)
 *  O        bf16 [S][n_q_heads][128] output (contiguous)
 *  lse_obs  fp32 [W][n_q_heads] (nullable): natural-log LSE of rows S-W .. S-1
 * The cache handle supplies the configuration (heads, W, sm_scale) and the status word
 * only.  SNAP_ERR_UNSUPPORTED for the MLA layout; SNAP_ERR_SHAPE for S < 1 or, with
 * lse_obs, S < W; SNAP_ERR_INVALID_ARG for null or misaligned pointers or strides.
 */
snap_status snap_prefill_attn(snap_cache* cache, const void* Q, int64_t S, const void* K, const void* V,
                              int64_t tok_stride, int64_t head_stride, void* O, float* lse_obs, void* stream);

/*
 * Decode-step append for a continuous batch ("Ring Buffer vs. Naive Slicing"): for each
 * b < n, the new token of sequence slots[b] (position T) is written into ring slot
 * L_sink + K + (T mod L_recent), then T += 1.  No gather, no concat.
 *  slots   device int32 [n], distinct cache slots (a repeated slot is a caller error)
 *  k_new   bf16 [n][n_kv_heads][d_qk];  v_new bf16 [n][n_kv_heads][d_v] (NULL for MLA)
 */
snap_status snap_decode_append(snap_cache* cache, const int32_t* slots, int n, const void* k_new,
                               const void* v_new, void* stream);

/*
 * Workspace bytes snap_decode_attn() needs for batches of up to max_n sequences: the
 * split-KV partial results (max, sum, un-normalised output) of the "Prefill / Decode
 * Pipeline" section's memory-bound decode, split over key ranges to fill the GPU.
 * Host call, no CUDA.  SNAP_ERR_INVALID_ARG for max_n < 1 or a null pointer.
 */
snap_status snap_decode_attn_ws_bytes(const snap_config* cfg, int max_n, size_t* bytes);

/*
 * The launch plan snap_decode_attn() uses for a batch of n sequences on the current
 * device: *splits key ranges per sequence (merged at the end when > 1), each walking
 * *tiles_per_split key tiles (32 keys for GQA, 64 for MLA), and *ctas_per_wave CTAs of
 * the attention kernel resident at once.  The split count follows a cost model of the
 * kernels measured on GB300 (one wave of ~128 CTAs at 16 x 128k GQA, no merge).  Host-side only (no kernel runs); for profiling and
 * capacity planning.  SNAP_ERR_INVALID_ARG for a null pointer or n < 1,
 * SNAP_ERR_CUDA when no device is current.
 */
snap_status snap_decode_attn_plan(const snap_cache* cache, int n, int* splits, int* tiles_per_split,
                                  int* ctas_per_wave);

/*
 * Split-KV decode attention over the fixed-size cache for a continuous batch whose
 * sequences sit at different ring offsets ("Prefill / Decode Pipeline": decode is
 * memory-bound, each step streams the cache once; "Why This Wasn't Already Standard":
 * requests of one batch sit at different points of their lifecycle; "Fixed-Size Cache
 * Layout": the attention runs over sinks, selected middle and recent ring).  For each b < n and query head i, a plain
 * softmax over the VALID slots of sequence slots[b] (sinks < n_sink, middle < n_mid,
 * ring slots holding positions max(R0, T - L_recent) .. T-1) of sm_scale * q.k,
 * weighted sum of the values.  The query attends to what the cache holds now: call
 * snap_decode_append() first to include the current token.
 *  q     bf16 [n][n_q_heads][d_qk];  out fp32 [n][n_q_heads][d_v] (the fp32 accumulation,
 *        not rounded to bf16)
 *  ws    device workspace of snap_decode_attn_ws_bytes(cfg, n) bytes
 * A full (uncompressed) KV cache is the same call on a cache configured with
 * L_sink = 0, K = 0, L_recent = maximum length.
 */
snap_status snap_decode_attn(snap_cache* cache, const int32_t* slots, int n, const void* q,
                             void* out, void* ws, size_t ws_bytes, void* stream);

/*
 * One decode step ("Ring Buffer vs. Naive Slicing": each new token is scattered into
 * its fixed ring slot, then decode attends over the fixed-size cache; "Prefill / Decode
 * Pipeline": the step streams the cache once): the result of snap_decode_append() of
 * k_new/v_new followed by snap_decode_attn() of q, with the same arguments and
 * workspace.  GQA runs it as ONE kernel: the CTA whose key range holds the new token's
 * ring slot writes the row before reading, every CTA attends over T + 1 tokens, the
 * last CTA of each sequence advances T and the last CTA of each (sequence, KV head)
 * merges the key splits.  MLA runs the attention kernel (with the same fused append)
 * and, when the plan splits the keys, the merge kernel.  Static shapes and no host
 * synchronisation: the form a serving loop captures into a CUDA graph.
 * SNAP_ERR_INVALID_ARG for a null k_new (and, for GQA, a null v_new).
 */
snap_status snap_decode_step(snap_cache* cache, const int32_t* slots, int n, const void* q, const void* k_new,
                             const void* v_new, void* out, void* ws, size_t ws_bytes, void* stream);

/*
 * Synchronises `stream`, reads the device status word, clears it, and returns it
 * (SNAP_OK when no kernel reported an error since the last check).
 */
snap_status snap_check_device(snap_cache* cache, void* stream);

/*
 * Self-test of the error path that every kernel's bounded waits share: launches one
 * kernel whose single wait can never be satisfied (an mbarrier that nothing arrives
 * on).  The wait gives up after its bound (about 2 s of the device's global timer) and
 * the kernel records SNAP_ERR_TIMEOUT (detail 900) in the cache's status word, which
 * the next snap_check_device() returns.  Nothing faults or hangs; the device context
 * stays usable.  SNAP_ERR_INVALID_ARG for a null cache.
 */
snap_status snap_selftest_bounded_wait(snap_cache* cache, void* stream);

/*
 * Bytes of device scratch that snap_decode_attn_noalloc() draws on (32 MiB).  The
 * array is part of the library's device image: every GPU that loads libsnap holds
 * it until the process exits.
 */
#define SNAP_NOALLOC_SCRATCH_BYTES (32u << 20)

/*
 * snap_decode_attn() for callers that cannot allocate device memory.  The paper has
 * no counterpart: this is a packaging variant of the same decode attention.
 *
 * Who needs it: code that runs where cudaMalloc is unavailable or unwelcome, for
 * example a real-time thread that must not block in the allocator, a stream being
 * captured into a CUDA graph (after this entry point's first call on the device), or
 * an embedding runtime that owns every device allocation itself.  Such a caller cannot obtain the workspace snap_decode_attn()
 * needs for its split-KV partial results.  This entry point takes the same inputs
 * and output (q, out, slots; the cache it attends over) and keeps the partial results
 * in a fixed scratch array compiled into the library instead.  It never calls
 * cudaMalloc, cudaFree or any allocating routine.
 *
 *  - Limit: the partial results of one call (n * n_q_heads * splits * (d_v + 2) floats,
 *    splits chosen as in snap_decode_attn) must fit SNAP_NOALLOC_SCRATCH_BYTES; larger
 *    batches are rejected with SNAP_ERR_SHAPE (and a line on stderr) before anything is
 *    launched.  Whether a batch fits depends on its split count (snap_decode_attn_plan):
 *    a call with one split needs no scratch at all (16 sequences of 32 x 128 GQA heads
 *    with a 32768-slot cache); 64 such sequences with a 8192-slot cache fit; 8 sequences
 *    of the 128-head MLA shape with a 32768-slot cache fit, 13 do not.
 *  - Set-up: the first call on each device, whatever its batch, looks up the scratch
 *    array's device address (cudaGetSymbolAddress, with that device current).  That
 *    lookup may also load the library module holding the array, which is when the
 *    32 MiB are reserved on the device.  Make that first call before capturing a
 *    stream into a graph.
 *  - Sharing: every call on a device uses the same array, and it keeps the previous
 *    call's contents.  Each call overwrites every partial it reads, so nothing needs
 *    clearing, but calls that overlap on the GPU (different streams without ordering,
 *    or concurrent graphs) race on the scratch: order them.
 */
snap_status snap_decode_attn_noalloc(snap_cache* cache, const int32_t* slots, int n, const void* q,
                                     void* out, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* SNAP_H */
