/*
 * snap_oracle.h -- plain, slow CPU oracle of the SnapStream fixed-size KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link or
 * call this code; only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark do.  It shares no code with the CUDA library.
 *
 * What it computes (SnapStream: Efficient Long Sequence Decoding on Dataflow
 * Accelerators, episode companion page, sections "Fixed-Size Cache Layout" and
 * "Ring Buffer vs. Naive Slicing"; SnapKV and StreamingLLM as named there):
 *
 *   one static cache per sequence  [ L_sink sinks | K selected | L_recent ring ]
 *   built once at prefill, after which decode only rotates the recent window.
 *
 * The SnapKV-style selection: the last W prompt queries (the observation window)
 * attend causally over the prompt; each prefix position j < S-W gets the sum,
 * over the window rows and the query heads that share its KV head, of its softmax
 * probability; the scores are max-pooled with an odd kernel P ("pooling-based
 * top-K selection", Infinity-Bench section of the same page), and the K best
 * middle positions are kept (ties: lower position wins), stored ascending.
 *
 * It also holds plain causal prefill attention (with the per-row log-sum-exp that a
 * prefill flash-attention kernel hands to the compression).
 *
 * Arithmetic: every input is a bf16 bit pattern (uint16_t); all arithmetic is
 * IEEE double.  Readings of points the pages leave open are listed beside each
 * function.  Parity pins live in tests/test_oracle_pins.py.
 *
 * Parity unpinned: which keys the softmax denominator of a window row runs over
 * (reading: the whole causal row, window included).  No page prints a score, so no
 * pin fixes that choice; the arithmetic given the reading is pinned (closed forms,
 * brute force, a textbook softmax row, column mass G*W).
 */
#ifndef SNAP_ORACLE_H
#define SNAP_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same fields as the library's configuration, kept separate on purpose. */
typedef struct {
    int layout;      /* 0 = GQA (separate K and V), 1 = MLA latent (V = first d_v columns of K) */
    int n_q_heads;   /* H_q */
    int n_kv_heads;  /* H_kv; query head i reads KV head i / (H_q / H_kv) */
    int d_qk;        /* key/query width (GQA: head_dim; MLA: latent + rope) */
    int d_v;         /* value width (GQA: head_dim; MLA: latent width) */
    int L_sink;      /* attention sinks kept at the front */
    int K;           /* number of selected middle tokens */
    int L_recent;    /* ring of most recent tokens */
    int W;           /* observation window (last W prompt queries) */
    int P;           /* max-pool kernel, odd */
    double sm_scale; /* softmax scale applied to q.k */
} snap_oracle_config;

/* Per-sequence bookkeeping after compression / append. */
typedef struct {
    int64_t S;      /* prompt length */
    int64_t T;      /* current length (S + appended tokens) */
    int64_t n_sink; /* valid sink slots: min(L_sink, S) */
    int64_t R0;     /* first prompt position written to the ring at prefill */
    int64_t n_mid;  /* valid middle slots */
} snap_oracle_meta;

/* 0 on success, negative on a rejected configuration or shape. */
int snap_oracle_check_config(const snap_oracle_config* c);

/* Total slots C = L_sink + K + L_recent. */
int64_t snap_oracle_cache_slots(const snap_oracle_config* c);

/* Segment bookkeeping of a prompt of length S (no data touched). */
int snap_oracle_plan(const snap_oracle_config* c, int64_t S, snap_oracle_meta* m);

/*
 * Observation-window scores.
 *   Kp:   keys, element (j, h, e) at Kp[j*k_tok_stride + h*k_head_stride + e]
 *   Q:    window queries [W][H_q][d_qk]; row (w, g) of KV head h is query head h*G+g
 *         at absolute position S-W+w.
 *   lse:  out, [H_kv][W][G]  log-sum-exp of the causal row (reading: the softmax
 *         denominator runs over every key up to and including the query's own
 *         position, window included; parity unpinned for this reading).
 *   col:  out, [H_kv][S]     sum over (w, g) of the row probability at column j,
 *         for all j < S (window columns included, so each head sums to G*W).
 */
int snap_oracle_window_scores(const snap_oracle_config* c, int64_t S,
                              const uint16_t* Kp, int64_t k_tok_stride, int64_t k_head_stride,
                              const uint16_t* Q, double* lse, double* col);

/* y[j] = max of x[i] over |i-j| <= P/2, 0 <= i < n (edges clipped). */
void snap_oracle_maxpool(const double* x, int64_t n, int P, double* y);

/*
 * Top-K over candidate positions [lo, hi) by (score descending, position ascending).
 * Writes min(K, hi-lo) positions to sel in ascending order; returns that count.
 */
int64_t snap_oracle_select(const double* score, int64_t lo, int64_t hi, int64_t K, int32_t* sel);

/*
 * Whole prefill compression of one sequence.
 *   cache_k: out [H_kv][C][d_qk];  cache_v: out [H_kv][C][d_v] (GQA) or NULL (MLA)
 *   Vp:      values, same strides as Kp (GQA) or NULL (MLA)
 *   sel:     out [H_kv][K] selected middle positions (ascending, -1 past n_mid)
 *   pool:    optional out [H_kv][S-W] pooled scores (NULL to skip; unused when no
 *            selection is needed)
 * Slots that hold nothing are zero-filled and marked invalid by the meta.
 */
int snap_oracle_compress(const snap_oracle_config* c, int64_t S,
                         const uint16_t* Kp, const uint16_t* Vp,
                         int64_t k_tok_stride, int64_t k_head_stride,
                         const uint16_t* Q,
                         uint16_t* cache_k, uint16_t* cache_v,
                         int32_t* sel, double* pool, snap_oracle_meta* m);

/*
 * snap_oracle_compress() with the column scores supplied instead of the window
 * queries: col [H_kv][S] is what snap_oracle_window_scores() returns in `col`.  The
 * scores are additive over the observation rows, so a caller may compute them as
 * sums over disjoint groups of query heads (one window_scores call per group).
 * Everything after scoring (pool, select, cache layout) is snap_oracle_compress().
 */
int snap_oracle_compress_scored(const snap_oracle_config* c, int64_t S,
                                const uint16_t* Kp, const uint16_t* Vp,
                                int64_t k_tok_stride, int64_t k_head_stride,
                                const double* col,
                                uint16_t* cache_k, uint16_t* cache_v,
                                int32_t* sel, double* pool, snap_oracle_meta* m);

/*
 * Causal prefill attention of one prompt (the prefill that precedes compression; the
 * episode companion page's headline figure puts compression at 2-5% extra prefill
 * latency).  Plain definition, every query against every key up to its own position:
 *   Q:   [S][H_q][d_qk];  Kp/Vp: keys / values with the strides of snap_oracle_compress
 *   out: [S][H_q][d_v]  softmax(sm_scale * q.k) weighted sum of the values (double)
 *   lse: [S][H_q]       natural log of sum_j exp(sm_scale * q.k_j) over the causal row,
 *                       the quantity a flash-attention kernel keeps per query row
 * GQA only (query head i reads KV head i / G).  Either output may be NULL.
 */
int snap_oracle_prefill_attn(const snap_oracle_config* c, int64_t S, const uint16_t* Q,
                             const uint16_t* Kp, const uint16_t* Vp,
                             int64_t k_tok_stride, int64_t k_head_stride,
                             double* out, double* lse);

/* Ring slot (within the whole cache) that holds absolute position p. */
int64_t snap_oracle_ring_slot(const snap_oracle_config* c, int64_t p);

/* Position held by cache slot s, or -1 when the slot holds nothing valid. */
int64_t snap_oracle_slot_position(const snap_oracle_config* c, const snap_oracle_meta* m,
                                  const int32_t* sel_h, int64_t s);

/* Validity of cache slot s under meta m (1 valid, 0 not). */
int snap_oracle_slot_valid(const snap_oracle_config* c, const snap_oracle_meta* m, int64_t s);

/* Decode append of one token: k_new [H_kv][d_qk], v_new [H_kv][d_v] (NULL for MLA). */
int snap_oracle_append(const snap_oracle_config* c, uint16_t* cache_k, uint16_t* cache_v,
                       snap_oracle_meta* m, const uint16_t* k_new, const uint16_t* v_new);

/*
 * Decode attention of one sequence over its cache.
 *   q:   [H_q][d_qk];  out: [H_q][d_v] (double)
 */
int snap_oracle_decode_attn(const snap_oracle_config* c, const uint16_t* cache_k,
                            const uint16_t* cache_v, const snap_oracle_meta* m,
                            const uint16_t* q, double* out);

#ifdef __cplusplus
}
#endif
#endif
