/*
 * snap_oracle.c -- plain, slow CPU oracle of the SnapStream fixed-size KV cache.
 *
 * TEST INFRASTRUCTURE ONLY (see snap_oracle.h).  Single-threaded C99, IEEE
 * double arithmetic on bf16 inputs, no blocking, no fusion: each function does
 * one step of the method in the order the pages give it.
 *
 * Sources: SnapStream episode companion page, "Fixed-Size Cache Layout"
 * (sinks + SnapKV top-K middle + recent window, built once at prefill, sizes
 * are hyperparameters L-sink, K, L-recent) and "Ring Buffer vs. Naive Slicing"
 * (decode only rotates the recent window, writing into a fixed index);
 * "Infinity-Bench KV Retrieval" (pooling-based top-K).  The scoring rule (window
 * softmax summed over the window and the grouped query heads, 1-D max-pool of
 * width P, ties to the lower index, ring slot = position mod L_recent) is the
 * problem statement that accompanies those pages.
 */
#include "snap_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ORACLE_MUTANT selects one deliberately wrong variant (tests only: it shows that the
 * pins in tests/test_oracle_pins.py catch plausible mistakes).  0 = the oracle. */
#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

static double bf16_value(uint16_t b)
{
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

int snap_oracle_check_config(const snap_oracle_config* c)
{
    if (!c) return -1;
    if (c->layout != 0 && c->layout != 1) return -1;
    if (c->n_q_heads <= 0 || c->n_kv_heads <= 0) return -1;
    if (c->n_q_heads % c->n_kv_heads != 0) return -1;
    if (c->d_qk <= 0 || c->d_v <= 0) return -1;
    if (c->layout == 1 && (c->n_kv_heads != 1 || c->d_v > c->d_qk)) return -1;
    if (c->L_sink < 0 || c->K < 0 || c->L_recent < 1) return -1;
    if (c->W < 1 || c->W > c->L_recent) return -1;
    if (c->P < 1 || (c->P % 2) == 0) return -1;
    if (!(c->sm_scale > 0.0)) return -1;
    return 0;
}

int64_t snap_oracle_cache_slots(const snap_oracle_config* c)
{
    return (int64_t)c->L_sink + c->K + c->L_recent;
}

/*
 * Segment bookkeeping.  Sinks are the first min(L_sink, S) positions; the ring
 * receives the last L_recent prompt positions that are not sinks; what lies
 * between is the middle, from which at most K positions are kept.
 */
int snap_oracle_plan(const snap_oracle_config* c, int64_t S, snap_oracle_meta* m)
{
    if (snap_oracle_check_config(c) != 0 || S < 1 || !m) return -1;
    int64_t n_sink = S < c->L_sink ? S : c->L_sink;
    int64_t R0;
    if (S <= c->L_sink) {
        R0 = S;
    } else {
        R0 = S - c->L_recent;
        if (R0 < c->L_sink) R0 = c->L_sink;
    }
    int64_t M = R0 - n_sink;
    m->S = S;
    m->T = S;
    m->n_sink = n_sink;
    m->R0 = R0;
    m->n_mid = M < c->K ? M : c->K;
    return 0;
}

int snap_oracle_window_scores(const snap_oracle_config* c, int64_t S,
                              const uint16_t* Kp, int64_t k_tok_stride, int64_t k_head_stride,
                              const uint16_t* Q, double* lse, double* col)
{
    if (snap_oracle_check_config(c) != 0) return -1;
    if (S < c->W) return -2;
    const int G = c->n_q_heads / c->n_kv_heads;
    const int d = c->d_qk;
    double* s = (double*)malloc(sizeof(double) * (size_t)S);
    if (!s) return -3;
    for (int h = 0; h < c->n_kv_heads; ++h) {
        double* colh = col + (int64_t)h * S;
        for (int64_t j = 0; j < S; ++j) colh[j] = 0.0;
        for (int w = 0; w < c->W; ++w) {
            const int64_t pos = S - c->W + w; /* absolute position of this query */
            for (int g = 0; g < G; ++g) {
                const uint16_t* q = Q + ((int64_t)w * c->n_q_heads +
                                         (ORACLE_MUTANT == 3 ? (int64_t)g * c->n_kv_heads + h
                                                             : (int64_t)h * G + g)) * d;
                /* causal row: keys 0..pos */
                double mx = -INFINITY;
                for (int64_t j = 0; j <= pos - (ORACLE_MUTANT == 2); ++j) {
                    const uint16_t* k = Kp + j * k_tok_stride + (int64_t)h * k_head_stride;
                    double dot = 0.0;
                    for (int e = 0; e < d; ++e) dot += bf16_value(q[e]) * bf16_value(k[e]);
                    s[j] = (ORACLE_MUTANT == 1 ? 1.0 : c->sm_scale) * dot;
                    if (s[j] > mx) mx = s[j];
                }
                double l = 0.0;
                for (int64_t j = 0; j <= pos; ++j) l += exp(s[j] - mx);
                const double row_lse = mx + log(l);
                if (lse) lse[((int64_t)h * c->W + w) * G + g] = row_lse;
                for (int64_t j = 0; j <= pos; ++j) colh[j] += exp(s[j] - row_lse);
            }
        }
    }
    free(s);
    return 0;
}

void snap_oracle_maxpool(const double* x, int64_t n, int P, double* y)
{
    const int64_t r = P / 2 + (ORACLE_MUTANT == 4);
    for (int64_t j = 0; j < n; ++j) {
        int64_t a = j - r < 0 ? 0 : j - r;
        int64_t b = j + r > n - 1 ? n - 1 : j + r;
        double m = x[a];
        for (int64_t i = a + 1; i <= b; ++i)
            if (x[i] > m) m = x[i];
        y[j] = m;
    }
}

typedef struct {
    double score;
    int64_t pos;
} scored_pos;

static int by_score_then_pos(const void* a, const void* b)
{
    const scored_pos* x = (const scored_pos*)a;
    const scored_pos* y = (const scored_pos*)b;
    if (x->score > y->score) return -1;
    if (x->score < y->score) return 1;
    return ORACLE_MUTANT == 5 ? (x->pos < y->pos) - (x->pos > y->pos)
                              : (x->pos > y->pos) - (x->pos < y->pos);
}

static int ascending_i32(const void* a, const void* b)
{
    int32_t x = *(const int32_t*)a, y = *(const int32_t*)b;
    return (x > y) - (x < y);
}

int64_t snap_oracle_select(const double* score, int64_t lo, int64_t hi, int64_t K, int32_t* sel)
{
    int64_t n = hi - lo;
    if (n <= 0 || K <= 0) return 0;
    if (n <= K) {
        for (int64_t i = 0; i < n; ++i) sel[i] = (int32_t)(lo + i);
        return n;
    }
    scored_pos* v = (scored_pos*)malloc(sizeof(scored_pos) * (size_t)n);
    if (!v) return -1;
    for (int64_t i = 0; i < n; ++i) {
        v[i].score = score[lo + i];
        v[i].pos = lo + i;
    }
    qsort(v, (size_t)n, sizeof(scored_pos), by_score_then_pos);
    for (int64_t i = 0; i < K; ++i) sel[i] = (int32_t)v[i].pos;
    free(v);
    qsort(sel, (size_t)K, sizeof(int32_t), ascending_i32);
    return K;
}

int64_t snap_oracle_ring_slot(const snap_oracle_config* c, int64_t p)
{
    return (ORACLE_MUTANT == 6 ? 0 : (int64_t)c->L_sink + c->K) + (p % c->L_recent);
}

static void copy_row(uint16_t* dst, const uint16_t* src, int n)
{
    memcpy(dst, src, sizeof(uint16_t) * (size_t)n);
}

/* Compression; the column scores come from window_scores(Q) when col_in is NULL,
 * else from col_in ([H_kv][S], the same quantity computed by the caller). */
static int compress_core(const snap_oracle_config* c, int64_t S,
                         const uint16_t* Kp, const uint16_t* Vp,
                         int64_t k_tok_stride, int64_t k_head_stride,
                         const uint16_t* Q, const double* col_in,
                         uint16_t* cache_k, uint16_t* cache_v,
                         int32_t* sel, double* pool, snap_oracle_meta* m)
{
    if (snap_oracle_plan(c, S, m) != 0) return -1;
    if (c->layout == 0 && (!Vp || !cache_v)) return -1;
    const int64_t C = snap_oracle_cache_slots(c);
    const int Hkv = c->n_kv_heads;
    const int dk = c->d_qk, dv = c->d_v;
    const int64_t M = m->R0 - m->n_sink;

    memset(cache_k, 0, sizeof(uint16_t) * (size_t)(Hkv * C * dk));
    if (cache_v) memset(cache_v, 0, sizeof(uint16_t) * (size_t)(Hkv * C * dv));
    for (int64_t i = 0; i < (int64_t)Hkv * c->K; ++i) sel[i] = -1;

    /* 1. middle selection (SnapKV scoring only when the middle overflows K) */
    if (M > c->K && c->K > 0) {
        const int64_t n_scored = S - c->W;
        double* lse = (double*)malloc(sizeof(double) * (size_t)(Hkv * c->W * (c->n_q_heads / Hkv)));
        double* col = (double*)malloc(sizeof(double) * (size_t)(Hkv * S));
        double* pl = (double*)malloc(sizeof(double) * (size_t)n_scored);
        if (!lse || !col || !pl) { free(lse); free(col); free(pl); return -3; }
        if (col_in) {
            memcpy(col, col_in, sizeof(double) * (size_t)(Hkv * S));
        } else {
            if (!Q) { free(lse); free(col); free(pl); return -1; }
            int rc = snap_oracle_window_scores(c, S, Kp, k_tok_stride, k_head_stride, Q, lse, col);
            if (rc != 0) { free(lse); free(col); free(pl); return rc; }
        }
        for (int h = 0; h < Hkv; ++h) {
            /* pool over the scored prefix [0, S-W), then select in the middle */
            snap_oracle_maxpool(col + (int64_t)h * S, n_scored, c->P, pl);
            if (pool) memcpy(pool + (int64_t)h * n_scored, pl, sizeof(double) * (size_t)n_scored);
            snap_oracle_select(pl, m->n_sink, m->R0, c->K, sel + (int64_t)h * c->K);
        }
        free(lse); free(col); free(pl);
    } else {
        for (int h = 0; h < Hkv; ++h)
            for (int64_t i = 0; i < m->n_mid; ++i) sel[(int64_t)h * c->K + i] = (int32_t)(m->n_sink + i);
    }

    /* 2. write the static-shape cache: sinks | selected | ring */
    for (int h = 0; h < Hkv; ++h) {
        uint16_t* ck = cache_k + (int64_t)h * C * dk;
        uint16_t* cv = cache_v ? cache_v + (int64_t)h * C * dv : NULL;
        for (int64_t i = 0; i < m->n_sink; ++i) {
            copy_row(ck + i * dk, Kp + i * k_tok_stride + (int64_t)h * k_head_stride, dk);
            if (cv) copy_row(cv + i * dv, Vp + i * k_tok_stride + (int64_t)h * k_head_stride, dv);
        }
        for (int64_t i = 0; i < m->n_mid; ++i) {
            int64_t p = sel[(int64_t)h * c->K + i];
            int64_t s = (int64_t)c->L_sink + i;
            copy_row(ck + s * dk, Kp + p * k_tok_stride + (int64_t)h * k_head_stride, dk);
            if (cv) copy_row(cv + s * dv, Vp + p * k_tok_stride + (int64_t)h * k_head_stride, dv);
        }
        for (int64_t p = m->R0; p < S; ++p) {
            int64_t s = snap_oracle_ring_slot(c, p);
            copy_row(ck + s * dk, Kp + p * k_tok_stride + (int64_t)h * k_head_stride, dk);
            if (cv) copy_row(cv + s * dv, Vp + p * k_tok_stride + (int64_t)h * k_head_stride, dv);
        }
    }
    return 0;
}

int snap_oracle_compress(const snap_oracle_config* c, int64_t S,
                         const uint16_t* Kp, const uint16_t* Vp,
                         int64_t k_tok_stride, int64_t k_head_stride,
                         const uint16_t* Q,
                         uint16_t* cache_k, uint16_t* cache_v,
                         int32_t* sel, double* pool, snap_oracle_meta* m)
{
    return compress_core(c, S, Kp, Vp, k_tok_stride, k_head_stride, Q, NULL, cache_k, cache_v, sel,
                         pool, m);
}

int snap_oracle_compress_scored(const snap_oracle_config* c, int64_t S,
                                const uint16_t* Kp, const uint16_t* Vp,
                                int64_t k_tok_stride, int64_t k_head_stride,
                                const double* col,
                                uint16_t* cache_k, uint16_t* cache_v,
                                int32_t* sel, double* pool, snap_oracle_meta* m)
{
    if (!col) return -1;
    return compress_core(c, S, Kp, Vp, k_tok_stride, k_head_stride, NULL, col, cache_k, cache_v, sel,
                         pool, m);
}

/* Number of ring-held positions and the oldest one, at length T. */
static void ring_window(const snap_oracle_config* c, const snap_oracle_meta* m,
                        int64_t* n_ring, int64_t* lo)
{
    int64_t n = m->T - m->R0;
    if (n > c->L_recent) n = c->L_recent;
    *n_ring = n;
    *lo = m->T - n;
}

int snap_oracle_slot_valid(const snap_oracle_config* c, const snap_oracle_meta* m, int64_t s)
{
    if (s < 0) return 0;
    if (s < c->L_sink) return s < m->n_sink;
    if (s < (int64_t)c->L_sink + c->K) return ORACLE_MUTANT == 7 ? 1 : s - c->L_sink < m->n_mid;
    int64_t r = s - c->L_sink - c->K;
    if (r >= c->L_recent) return 0;
    int64_t n_ring, lo;
    ring_window(c, m, &n_ring, &lo);
    int64_t off = ((r - lo) % c->L_recent + c->L_recent) % c->L_recent;
    return off < n_ring;
}

int64_t snap_oracle_slot_position(const snap_oracle_config* c, const snap_oracle_meta* m,
                                  const int32_t* sel_h, int64_t s)
{
    if (!snap_oracle_slot_valid(c, m, s)) return -1;
    if (s < c->L_sink) return s;
    if (s < (int64_t)c->L_sink + c->K) return sel_h[s - c->L_sink];
    int64_t r = s - c->L_sink - c->K;
    int64_t n_ring, lo;
    ring_window(c, m, &n_ring, &lo);
    return lo + ((r - lo) % c->L_recent + c->L_recent) % c->L_recent;
}

int snap_oracle_append(const snap_oracle_config* c, uint16_t* cache_k, uint16_t* cache_v,
                       snap_oracle_meta* m, const uint16_t* k_new, const uint16_t* v_new)
{
    if (snap_oracle_check_config(c) != 0) return -1;
    const int64_t C = snap_oracle_cache_slots(c);
    const int64_t s = snap_oracle_ring_slot(c, m->T);
    for (int h = 0; h < c->n_kv_heads; ++h) {
        copy_row(cache_k + ((int64_t)h * C + s) * c->d_qk, k_new + (int64_t)h * c->d_qk, c->d_qk);
        if (c->layout == 0)
            copy_row(cache_v + ((int64_t)h * C + s) * c->d_v, v_new + (int64_t)h * c->d_v, c->d_v);
    }
    m->T += 1;
    return 0;
}

int snap_oracle_decode_attn(const snap_oracle_config* c, const uint16_t* cache_k,
                            const uint16_t* cache_v, const snap_oracle_meta* m,
                            const uint16_t* q, double* out)
{
    if (snap_oracle_check_config(c) != 0) return -1;
    const int64_t C = snap_oracle_cache_slots(c);
    const int G = c->n_q_heads / c->n_kv_heads;
    const int dk = c->d_qk, dv = c->d_v;
    double* s = (double*)malloc(sizeof(double) * (size_t)C);
    if (!s) return -3;
    for (int i = 0; i < c->n_q_heads; ++i) {
        const int h = i / G;
        const uint16_t* qi = q + (int64_t)i * dk;
        const uint16_t* kh = cache_k + (int64_t)h * C * dk;
        double mx = -INFINITY;
        for (int64_t t = 0; t < C; ++t) {
            if (!snap_oracle_slot_valid(c, m, t)) continue;
            double dot = 0.0;
            for (int e = 0; e < dk; ++e) dot += bf16_value(qi[e]) * bf16_value(kh[t * dk + e]);
            s[t] = c->sm_scale * dot;
            if (s[t] > mx) mx = s[t];
        }
        double* o = out + (int64_t)i * dv;
        for (int e = 0; e < dv; ++e) o[e] = 0.0;
        if (mx == -INFINITY) continue; /* nothing valid: zero output */
        double l = 0.0;
        for (int64_t t = 0; t < C; ++t) {
            if (!snap_oracle_slot_valid(c, m, t)) continue;
            const double p = exp(s[t] - mx);
            l += p;
            /* GQA reads the V cache; MLA's value is the first d_v columns of the key row */
            const uint16_t* v = c->layout == 0 ? cache_v + ((int64_t)h * C + t) * dv
                                               : kh + t * dk;
            for (int e = 0; e < dv; ++e) o[e] += p * bf16_value(v[ORACLE_MUTANT == 8 ? dv - 1 - e : e]);
        }
        for (int e = 0; e < dv; ++e) o[e] /= l;
    }
    free(s);
    return 0;
}

int snap_oracle_prefill_attn(const snap_oracle_config* c, int64_t S, const uint16_t* Q,
                             const uint16_t* Kp, const uint16_t* Vp,
                             int64_t k_tok_stride, int64_t k_head_stride,
                             double* out, double* lse)
{
    if (snap_oracle_check_config(c) != 0 || c->layout != 0 || S < 1 || !Q || !Kp || !Vp) return -1;
    const int G = c->n_q_heads / c->n_kv_heads;
    const int dk = c->d_qk, dv = c->d_v;
    double* s = (double*)malloc(sizeof(double) * (size_t)S);
    if (!s) return -3;
    for (int64_t i = 0; i < S; ++i) {
        for (int hq = 0; hq < c->n_q_heads; ++hq) {
            const int h = hq / G;
            const uint16_t* q = Q + (i * c->n_q_heads + hq) * (int64_t)dk;
            /* scores of the causal row: keys 0..i */
            const int64_t last = i - (ORACLE_MUTANT == 9 && i > 0);
            double mx = -INFINITY;
            for (int64_t j = 0; j <= last; ++j) {
                const uint16_t* k = Kp + j * k_tok_stride + (int64_t)h * k_head_stride;
                double dot = 0.0;
                for (int e = 0; e < dk; ++e) dot += bf16_value(q[e]) * bf16_value(k[e]);
                s[j] = c->sm_scale * dot;
                if (s[j] > mx) mx = s[j];
            }
            double l = 0.0;
            for (int64_t j = 0; j <= last; ++j) l += exp(s[j] - mx);
            if (lse) lse[i * c->n_q_heads + hq] = mx + log(l);
            if (out) {
                double* o = out + (i * c->n_q_heads + hq) * (int64_t)dv;
                for (int e = 0; e < dv; ++e) o[e] = 0.0;
                for (int64_t j = 0; j <= last; ++j) {
                    const double p = exp(s[j] - mx) / l;
                    const uint16_t* v = Vp + j * k_tok_stride + (int64_t)h * k_head_stride;
                    for (int e = 0; e < dv; ++e) o[e] += p * bf16_value(v[e]);
                }
            }
        }
    }
    free(s);
    return 0;
}
