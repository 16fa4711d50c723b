// snap_api.cu -- the C ABI of libsnap (see include/snap.h): argument checks,
// cache/workspace layout, and the launch sequence of each entry point.
#include <cudaTypedefs.h>

#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>

#include "kernels.cuh"

using namespace snap;

struct snap_cache {
    snap_config cfg;
    int max_batch;
    int64_t C;
    void* base;
    size_t bytes;
    bf16* k;
    bf16* v;
    snap_seq_meta* meta;
    int32_t* sel;
    int32_t* status;
    int32_t* merge_cnt;   // [max_batch][n_kv_heads] split-merge arrival counts (zero between calls)
};

namespace {

constexpr int ABI_VERSION = 1;
constexpr int MAX_KEY_SPLITS = 32;   // key splits of the row pass (SCORE_PARTS partials each)
constexpr int MAX_DECODE_SPLITS = 32;

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// SMs of the current device (cached per device); 0 if the query fails.  Every entry
// point that plans launches checks it first (SNAP_ERR_CUDA), so the helpers below
// only see a positive count.
int num_sms() {
    static std::atomic<int> cached[64];     // zero-initialised (static storage)
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    const bool cacheable = dev >= 0 && dev < 64;
    if (cacheable) {
        const int c = cached[dev].load(std::memory_order_relaxed);
        if (c > 0) return c;
    }
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 0;
    if (cacheable) cached[dev].store(n, std::memory_order_relaxed);
    return n;
}

DevConfig dev_config(const snap_config& c, int max_batch) {
    DevConfig d;
    d.layout = c.layout;
    d.Hq = c.n_q_heads;
    d.Hkv = c.n_kv_heads;
    d.G = c.n_q_heads / c.n_kv_heads;
    d.dqk = c.d_qk;
    d.dv = c.d_v;
    d.L_sink = c.L_sink;
    d.K = c.K;
    d.L_recent = c.L_recent;
    d.W = c.W;
    d.P = c.P;
    d.C = c.L_sink + c.K + c.L_recent;
    d.max_batch = max_batch;
    d.scale = c.sm_scale;
    d.scale_log2 = c.sm_scale * 1.4426950408889634f;
    return d;
}

struct CacheRegions {
    size_t meta, status, cnt, sel, k, v, total;
};

CacheRegions regions(const snap_config& c, int max_batch) {
    const size_t C = (size_t)c.L_sink + c.K + c.L_recent;
    CacheRegions r;
    size_t off = 0;
    r.meta = off;
    off = align_up(off + sizeof(snap_seq_meta) * max_batch, 256);
    r.status = off;
    off = align_up(off + 16, 256);
    r.cnt = off;
    off = align_up(off + sizeof(int32_t) * (size_t)max_batch * c.n_kv_heads, 256);
    r.sel = off;
    off = align_up(off + sizeof(int32_t) * (size_t)max_batch * c.n_kv_heads * c.K, 256);
    r.k = off;
    off = align_up(off + 2 * (size_t)max_batch * c.n_kv_heads * C * c.d_qk, 256);
    r.v = off;
    if (c.layout == SNAP_LAYOUT_GQA) off = align_up(off + 2 * (size_t)max_batch * c.n_kv_heads * C * c.d_v, 256);
    r.total = off;
    return r;
}

// Compress workspace regions for a prompt of S tokens.
struct CompressWs {
    size_t part_ml, nlse2, col, pool, total;
    int64_t S_pad;
    int R, R_pad;
};

CompressWs compress_ws(const snap_config& c, int64_t S) {
    const int G = c.n_q_heads / c.n_kv_heads;
    CompressWs w;
    w.R = G * c.W;
    w.R_pad = (w.R + 255) / 256 * 256;
    w.S_pad = (S + 127) / 128 * 128;
    size_t off = 0;
    w.part_ml = off;
    off = align_up(off + sizeof(float) * 2 * c.n_kv_heads * (size_t)w.R * SCORE_PARTS * MAX_KEY_SPLITS, 256);
    w.nlse2 = off;
    off = align_up(off + sizeof(float) * c.n_kv_heads * (size_t)w.R_pad, 256);
    w.col = off;
    off = align_up(off + sizeof(float) * SCORE_PARTS * c.n_kv_heads * (size_t)w.S_pad, 256);
    w.pool = off;
    off = align_up(off + sizeof(uint32_t) * c.n_kv_heads * (size_t)w.S_pad, 256);
    w.total = off;
    return w;
}

// ------------------------------------------------------------ TMA tensor maps
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

bool encode(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
            const cuuint32_t* box) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint32_t es[5] = {1, 1, 1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Observation queries [W][Hq][d] of KV head h as rows (w, g): dims {d, G, W, Hkv}.
bool q_map(CUtensorMap* m, const void* Q, const snap_config& c, int box_rows) {
    const int G = c.n_q_heads / c.n_kv_heads;
    const cuuint64_t dims[4] = {(cuuint64_t)c.d_qk, (cuuint64_t)G, (cuuint64_t)c.W, (cuuint64_t)c.n_kv_heads};
    const cuuint64_t strides[3] = {(cuuint64_t)c.d_qk * 2, (cuuint64_t)c.n_q_heads * c.d_qk * 2,
                                   (cuuint64_t)G * c.d_qk * 2};
    const cuuint32_t box[4] = {64, (cuuint32_t)G, (cuuint32_t)(box_rows / G), 1};
    return encode(m, Q, 4, dims, strides, box);
}

// Prompt keys (strided): dims {d, S, Hkv}.
bool k_map(CUtensorMap* m, const void* K, int64_t S, const snap_config& c, int64_t tok_stride,
           int64_t head_stride, int box_rows) {
    const cuuint64_t dims[3] = {(cuuint64_t)c.d_qk, (cuuint64_t)S, (cuuint64_t)c.n_kv_heads};
    const cuuint64_t strides[2] = {(cuuint64_t)tok_stride * 2,
                                   (cuuint64_t)(head_stride > 0 ? head_stride : c.d_qk) * 2};
    const cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
    return encode(m, K, 3, dims, strides, box);
}

ScoreParams score_params(const snap_config& c, int64_t S, const CompressWs& w, uint8_t* ws, int32_t* status) {
    ScoreParams sp;
    std::memset(&sp, 0, sizeof sp);
    sp.S = (int)S;
    sp.W = c.W;
    sp.R = w.R;
    sp.G = c.n_q_heads / c.n_kv_heads;
    sp.Hkv = c.n_kv_heads;
    sp.sl2 = c.sm_scale * 1.4426950408889634f;
    sp.n_sc = (int)S - c.W;
    sp.R_pad = w.R_pad;
    sp.S_pad = w.S_pad;
    if (ws) {
        sp.part_ml = reinterpret_cast<float*>(ws + w.part_ml);
        sp.nlse2 = reinterpret_cast<const float*>(ws + w.nlse2);
        sp.col = reinterpret_cast<float*>(ws + w.col);
    }
    sp.status = status;
    return sp;
}

// Key splits of the row pass.  The persistent CTAs take the (head, split, row tile)
// units in rounds of one per SM, so a split count s costs
//     ceil(units(s) / SMs) x (key tiles per split + 2)
// in key-tile times; the 2 covers a unit's start (the resident rows' load and the
// MMA pipeline's refill).  The smallest cost wins, ties going to fewer splits.
int row_key_splits(const snap_config& c, int R, int64_t S) {
    const int per = c.n_kv_heads * ((R + 127) / 128);
    const int ny = (int)((S + 255) / 256);
    const int sms = num_sms();
    const int top = ny < MAX_KEY_SPLITS ? ny : MAX_KEY_SPLITS;
    int best = 1;
    int64_t best_cost = -1;
    for (int s = 1; s <= top; ++s) {
        const int64_t rounds = ((int64_t)per * s + sms - 1) / sms;
        const int64_t cost = rounds * ((ny + s - 1) / s + 2);
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best = s;
        }
    }
    return best;
}

// Row pass: X = 128 observation rows, Y = 256-key tiles.
cudaError_t run_rowstat(int mode, const snap_config& c, ScoreParams sp, const void* K, int64_t S,
                        int64_t tok_stride, int64_t head_stride, const void* Q, cudaStream_t st) {
    CUtensorMap tx, ty;
    if (!q_map(&tx, Q, c, 128) || !k_map(&ty, K, S, c, tok_stride, head_stride, 256)) return cudaErrorInvalidValue;
    sp.Ny = 256;
    sp.x_tiles = (sp.R + 127) / 128;
    sp.splits = row_key_splits(c, sp.R, S);
    sp.n_units = c.n_kv_heads * sp.x_tiles * sp.splits;
    return launch_score_tc(mode, tx, ty, sp, c.d_qk, true, true, num_sms(), false, st);
}

// MLA decode tensor map of the cache rows [max_batch][C][576] (box 64 x 64).
bool mla_cache_map(CUtensorMap* tkv, const snap_cache* cache);

// Split count and launches of one decode-attention call (shared by the entry points).
cudaError_t run_decode(snap_cache* cache, DecodeArgs& a, cudaStream_t st);

size_t decode_ws_bytes(const snap_config& c, int max_n) {
    const size_t parts = (size_t)max_n * c.n_q_heads * MAX_DECODE_SPLITS;
    return align_up(parts * sizeof(float) * c.d_v, 256) + align_up(parts * sizeof(float) * 2, 256);
}

snap_status check_config(const snap_config* c) {
    if (!c) return SNAP_ERR_INVALID_ARG;
    if (c->layout != SNAP_LAYOUT_GQA && c->layout != SNAP_LAYOUT_MLA) return SNAP_ERR_SHAPE;
    if (c->n_q_heads <= 0 || c->n_kv_heads <= 0 || c->n_q_heads % c->n_kv_heads) return SNAP_ERR_SHAPE;
    if (c->d_qk <= 0 || c->d_v <= 0) return SNAP_ERR_SHAPE;
    if (c->L_sink < 0 || c->K < 0 || c->L_recent < 1) return SNAP_ERR_SHAPE;
    if (c->W < 1 || c->W > c->L_recent) return SNAP_ERR_SHAPE;
    if (c->P < 1 || c->P % 2 == 0) return SNAP_ERR_SHAPE;
    if (!(c->sm_scale > 0.f)) return SNAP_ERR_SHAPE;
    if ((int64_t)c->L_sink + c->K + c->L_recent > (1ll << 30)) return SNAP_ERR_SHAPE;
    if (c->layout == SNAP_LAYOUT_MLA) {
        if (c->n_kv_heads != 1 || c->d_v > c->d_qk) return SNAP_ERR_SHAPE;
        if (c->d_qk != 576 || c->d_v != 512 || c->n_q_heads != MLA_HEADS) return SNAP_ERR_UNSUPPORTED;
    } else {
        if (c->d_qk != 128 || c->d_v != 128) return SNAP_ERR_UNSUPPORTED;
        if (c->n_q_heads / c->n_kv_heads > 8) return SNAP_ERR_UNSUPPORTED;
    }
    // observation rows are loaded as whole query-head groups by the score GEMM
    if (128 % (c->n_q_heads / c->n_kv_heads)) return SNAP_ERR_UNSUPPORTED;
    return SNAP_OK;
}

snap_status cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return SNAP_OK;
    std::fprintf(stderr, "libsnap: CUDA error %s\n", cudaGetErrorString(e));
    return SNAP_ERR_CUDA;
}

// GQA decode split count.  A wave of resident CTAs streams as fast as HBM allows once
// about 84% of the SMs read (a partial wave below that takes as long as one that
// size), every CTA pays about one warp step of set-up and drain, and any split count
// above one adds the merge (~3%).  The count minimises
//   (warp steps per split + 1) x sum over waves of max(CTAs in the wave, 0.84 wave),
// which picks one wave of ~128 CTAs at 16 x 128k (one split, no merge) and two
// splits at 8 x 16-32k (measured on GB300 against every split count).
int decode_splits_gqa(int base, int tiles, int wave) {
    const int sat = (wave * 84 + 99) / 100;
    int best = 1;
    double best_cost = -1.0;
    for (int s = 1; s <= MAX_DECODE_SPLITS; ++s) {
        const int per_split = (tiles + s - 1) / s;
        if (s > 1 && (tiles + per_split - 1) / per_split < s) break;   // would leave a split empty
        const int steps = (per_split + 3) / 4;                         // 4 warps, one 32-key tile each per step
        const long long ctas = (long long)base * s;
        const long long full = ctas / wave, rem = ctas % wave;
        const long long units = full * wave + (rem ? (rem > sat ? rem : sat) : 0);
        double cost = (double)(steps + 1) * (double)units;
        if (s > 1) cost *= 1.03;
        if (best_cost < 0.0 || cost < best_cost) {
            best_cost = cost;
            best = s;
        }
    }
    return best;
}

// MLA decode: each CTA also pays a fixed cost (TMEM setup, the q load,
// writing its partial output) worth about this many 64-key tiles, so its split
// count minimises waves x (tiles per split + that cost) instead.
constexpr int MLA_FIXED_TILES = 8;

int decode_splits_fixed_cost(int base, int tiles, int wave, int fixed_tiles) {
    int best = 1;
    long long best_cost = -1;
    for (int s = 1; s <= MAX_DECODE_SPLITS; ++s) {
        const int per = (tiles + s - 1) / s;
        if (s > 1 && per < 4) break;
        const long long waves = ((long long)base * s + wave - 1) / wave;
        const long long cost = waves * (per + fixed_tiles);
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best = s;
        }
    }
    return best;
}

// CTAs of one decode-attention kernel resident at once: one per SM for GQA; for MLA
// as many as the occupancy query reports (one per SM).
int decode_wave_ctas(const snap_cache* cache) {
    if (cache->cfg.layout == SNAP_LAYOUT_GQA) return num_sms();
    const int w = mla_decode_wave_ctas();
    return w > 0 ? w : num_sms();
}

// Splits of one decode-attention call: enough CTAs for whole waves (GQA: 4 warps walk
// a split, one 32-key tile each per step; MLA: two CTAs per split, 64-key tiles).
int decode_split_count(const snap_cache* cache, int n) {
    const snap_config& c = cache->cfg;
    if (c.layout == SNAP_LAYOUT_GQA) {
        const int tiles = (int)((cache->C + GQA_KEYS - 1) / GQA_KEYS);
        return decode_splits_gqa(n * c.n_kv_heads, tiles, decode_wave_ctas(cache));
    }
    const int tiles = (int)((cache->C + MLA_KEYS - 1) / MLA_KEYS);
    return decode_splits_fixed_cost(2 * n, tiles, decode_wave_ctas(cache), MLA_FIXED_TILES);
}

// Splits and key tiles per split of one decode-attention call: the split count is
// recomputed from the rounded-up tiles per split, so that no split is empty.
void decode_plan(const snap_cache* cache, int n, int* splits, int* tiles_per_split) {
    const int key_tile = cache->cfg.layout == SNAP_LAYOUT_GQA ? GQA_KEYS : MLA_KEYS;
    const int tiles = (int)((cache->C + key_tile - 1) / key_tile);
    const int s = decode_split_count(cache, n);
    const int per = (tiles + s - 1) / s;
    *tiles_per_split = per;
    *splits = (tiles + per - 1) / per;
}

bool mla_cache_map(CUtensorMap* tkv, const snap_cache* cache) {
    const snap_config& c = cache->cfg;
    const cuuint64_t kd[3] = {(cuuint64_t)c.d_qk, (cuuint64_t)cache->C, (cuuint64_t)cache->max_batch};
    const cuuint64_t ks[2] = {(cuuint64_t)c.d_qk * 2, (cuuint64_t)cache->C * c.d_qk * 2};
    const cuuint32_t kb[3] = {64, (cuuint32_t)MLA_KEYS, 1};
    return encode(tkv, cache->k, 3, kd, ks, kb);
}

// GQA: one kernel (append, attention, split merge); MLA: the attention kernel (with the
// append) and, when the plan splits the keys, the merge kernel.
cudaError_t run_decode(snap_cache* cache, DecodeArgs& a, cudaStream_t st) {
    a.meta_rw = cache->meta;
    a.merge_cnt = cache->merge_cnt;
    if (cache->cfg.layout == SNAP_LAYOUT_GQA) return launch_decode_gqa(a, st);
    CUtensorMap tkv, tq;
    if (!mla_cache_map(&tkv, cache)) return cudaErrorInvalidValue;
    const snap_config& c = cache->cfg;
    const cuuint64_t qd[3] = {(cuuint64_t)c.d_qk, (cuuint64_t)c.n_q_heads, (cuuint64_t)a.n};
    const cuuint64_t qs[2] = {(cuuint64_t)c.d_qk * 2, (cuuint64_t)c.n_q_heads * c.d_qk * 2};
    const cuuint32_t qb[3] = {64, (cuuint32_t)c.n_q_heads, 1};
    if (!encode(&tq, a.q, 3, qd, qs, qb)) return cudaErrorInvalidValue;
    cudaError_t e = launch_decode_mla_tc(a, tkv, tq, st);
    if (e == cudaSuccess && a.splits > 1) e = launch_decode_merge(a, st);
    return e;
}

// Arguments shared by the decode-attention entry points (plan, workspace aside).
snap_status decode_args(snap_cache* cache, const int32_t* slots, int n, const void* q, void* out,
                        const void* k_new, const void* v_new, DecodeArgs* a) {
    if (!slots || !q || !out || !aligned16(q) || !aligned16(out)) return SNAP_ERR_INVALID_ARG;
    if (n > cache->max_batch) return SNAP_ERR_INVALID_ARG;
    if (num_sms() <= 0) return SNAP_ERR_CUDA;
    const snap_config& c = cache->cfg;
    if (k_new) {
        if (!aligned16(k_new)) return SNAP_ERR_INVALID_ARG;
        if (c.layout == SNAP_LAYOUT_GQA && (!v_new || !aligned16(v_new))) return SNAP_ERR_INVALID_ARG;
        if (c.layout == SNAP_LAYOUT_MLA && v_new) return SNAP_ERR_INVALID_ARG;
    }
    std::memset(a, 0, sizeof *a);
    a->kc = cache->k;
    a->vc = cache->v;
    a->meta = cache->meta;
    a->slots = slots;
    a->n = n;
    a->q = static_cast<const bf16*>(q);
    a->out = static_cast<float*>(out);
    a->status = cache->status;
    a->cfg = dev_config(c, cache->max_batch);
    a->k_new = static_cast<const bf16*>(k_new);
    a->v_new = static_cast<const bf16*>(v_new);
    int splits = 1;
    decode_plan(cache, n, &splits, &a->tiles_per_split);
    a->splits = splits;
    return SNAP_OK;
}

// Decode attention (with the fused append when k_new is given) using the caller's workspace.
snap_status decode_with_ws(snap_cache* cache, const int32_t* slots, int n, const void* q, const void* k_new,
                           const void* v_new, void* out, void* ws, size_t ws_bytes, void* stream) {
    if (!cache || n < 0) return SNAP_ERR_INVALID_ARG;
    if (n == 0) return SNAP_OK;
    DecodeArgs a;
    if (const snap_status s = decode_args(cache, slots, n, q, out, k_new, v_new, &a); s != SNAP_OK) return s;
    const snap_config& c = cache->cfg;
    if (a.splits > 1) {
        const size_t need = decode_ws_bytes(c, n);
        if (!ws || ws_bytes < need || (reinterpret_cast<uintptr_t>(ws) & 255u)) return SNAP_ERR_INVALID_ARG;
        const size_t parts = (size_t)n * c.n_q_heads * MAX_DECODE_SPLITS;
        a.part_o = static_cast<float*>(ws);
        a.part_ml = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + align_up(parts * sizeof(float) * c.d_v, 256));
    }
    return cuda_status(run_decode(cache, a, static_cast<cudaStream_t>(stream)));
}

}  // namespace

extern "C" {

const char* snap_status_string(int s) {
    switch (s) {
        case SNAP_OK: return "ok";
        case SNAP_ERR_INVALID_ARG: return "invalid argument (null or misaligned pointer, bad count)";
        case SNAP_ERR_SHAPE: return "shape violates the method's preconditions";
        case SNAP_ERR_UNSUPPORTED: return "configuration not supported by these kernels";
        case SNAP_ERR_CUDA: return "CUDA call failed";
        case SNAP_ERR_TIMEOUT: return "a kernel's bounded wait expired";
        case SNAP_ERR_DEVICE_CHECK: return "a kernel rejected an index (slot out of range)";
        default: return "unknown status";
    }
}

int snap_abi_version(void) { return ABI_VERSION; }

snap_status snap_config_check(const snap_config* cfg) { return check_config(cfg); }

snap_status snap_cache_bytes(const snap_config* cfg, int max_batch, size_t* bytes) {
    snap_status s = check_config(cfg);
    if (s != SNAP_OK) return s;
    if (max_batch < 1 || !bytes) return SNAP_ERR_INVALID_ARG;
    *bytes = regions(*cfg, max_batch).total;
    return SNAP_OK;
}

snap_status snap_cache_create(const snap_config* cfg, int max_batch, void* dev_buf, size_t bytes,
                              void* stream, snap_cache** out) {
    snap_status s = check_config(cfg);
    if (s != SNAP_OK) return s;
    if (max_batch < 1 || !dev_buf || !out) return SNAP_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(dev_buf) & 255u) return SNAP_ERR_INVALID_ARG;
    const CacheRegions r = regions(*cfg, max_batch);
    if (bytes < r.total) return SNAP_ERR_INVALID_ARG;
    snap_cache* c = new (std::nothrow) snap_cache;
    if (!c) return SNAP_ERR_INVALID_ARG;
    uint8_t* base = static_cast<uint8_t*>(dev_buf);
    c->cfg = *cfg;
    c->max_batch = max_batch;
    c->C = (int64_t)cfg->L_sink + cfg->K + cfg->L_recent;
    c->base = dev_buf;
    c->bytes = bytes;
    c->meta = reinterpret_cast<snap_seq_meta*>(base + r.meta);
    c->status = reinterpret_cast<int32_t*>(base + r.status);
    c->merge_cnt = reinterpret_cast<int32_t*>(base + r.cnt);
    c->sel = reinterpret_cast<int32_t*>(base + r.sel);
    c->k = reinterpret_cast<bf16*>(base + r.k);
    c->v = cfg->layout == SNAP_LAYOUT_GQA ? reinterpret_cast<bf16*>(base + r.v) : nullptr;
    cudaError_t e = cudaMemsetAsync(dev_buf, 0, r.total, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        delete c;
        return cuda_status(e);
    }
    *out = c;
    return SNAP_OK;
}

void snap_cache_destroy(snap_cache* cache) { delete cache; }

snap_status snap_cache_view_get(const snap_cache* cache, snap_cache_view* out) {
    if (!cache || !out) return SNAP_ERR_INVALID_ARG;
    out->k = cache->k;
    out->v = cache->v;
    out->meta = cache->meta;
    out->sel = cache->sel;
    out->status = cache->status;
    out->C = cache->C;
    out->max_batch = cache->max_batch;
    return SNAP_OK;
}

snap_status snap_compress_ws_bytes(const snap_config* cfg, int64_t S_max, size_t* bytes) {
    snap_status s = check_config(cfg);
    if (s != SNAP_OK) return s;
    if (S_max < 1 || !bytes) return SNAP_ERR_INVALID_ARG;
    *bytes = compress_ws(*cfg, S_max).total;
    return SNAP_OK;
}

}  // extern "C"

namespace {

// Compression of one sequence, the stages selected by `stages` (SNAP_STAGE_*);
// lse_obs (nullable) replaces the row pass.
snap_status compress_impl(snap_cache* cache, int slot, const void* K, const void* V, int64_t S,
                          int64_t tok_stride, int64_t head_stride, const void* Q_obs, const float* lse_obs,
                          void* ws, size_t ws_bytes, int stages, void* stream) {
    if (stages & ~SNAP_STAGE_ALL) return SNAP_ERR_INVALID_ARG;
    if (num_sms() <= 0) return SNAP_ERR_CUDA;
    if (!cache || !K || !Q_obs) return SNAP_ERR_INVALID_ARG;
    const snap_config& c = cache->cfg;
    if (slot < 0 || slot >= cache->max_batch) return SNAP_ERR_INVALID_ARG;
    if (S < 1 || S > (1ll << 30)) return SNAP_ERR_SHAPE;
    if (c.layout == SNAP_LAYOUT_GQA && !V) return SNAP_ERR_INVALID_ARG;
    if (c.layout == SNAP_LAYOUT_MLA && V) return SNAP_ERR_INVALID_ARG;
    if (!aligned16(K) || (V && !aligned16(V)) || !aligned16(Q_obs)) return SNAP_ERR_INVALID_ARG;
    if (tok_stride < 0 || head_stride < 0 || (tok_stride * 2) % 16 || (head_stride * 2) % 16)
        return SNAP_ERR_INVALID_ARG;
    if (c.n_kv_heads > 1 && head_stride < c.d_qk) return SNAP_ERR_INVALID_ARG;
    if (S > 1 && tok_stride < c.d_qk) return SNAP_ERR_INVALID_ARG;

    const int64_t n_sink = S < c.L_sink ? S : c.L_sink;
    int64_t R0 = S <= c.L_sink ? S : (S - c.L_recent > c.L_sink ? S - c.L_recent : c.L_sink);
    const int64_t M = R0 - n_sink;
    const int64_t n_mid = M < c.K ? M : c.K;
    const bool scored = M > c.K && c.K > 0;

    CompressArgs a;
    std::memset(&a, 0, sizeof a);
    a.K = static_cast<const bf16*>(K);
    a.V = static_cast<const bf16*>(V);
    a.tok_stride = tok_stride;
    a.head_stride = head_stride;
    a.Q = static_cast<const bf16*>(Q_obs);
    a.S = (int)S;
    a.R = (c.n_q_heads / c.n_kv_heads) * c.W;
    a.R0 = (int)R0;
    a.n_sink = (int)n_sink;
    a.n_mid = (int)n_mid;
    a.scored = scored ? 1 : 0;
    a.slot = slot;
    a.kc = cache->k;
    a.vc = cache->v;
    a.meta = cache->meta;
    a.sel = cache->sel;
    a.status = cache->status;
    a.cfg = dev_config(c, cache->max_batch);
    cudaStream_t st = static_cast<cudaStream_t>(stream);

    if (scored) {
        const CompressWs w = compress_ws(c, S);
        if (!ws || ws_bytes < w.total) return SNAP_ERR_INVALID_ARG;
        if (reinterpret_cast<uintptr_t>(ws) & 255u) return SNAP_ERR_INVALID_ARG;
        uint8_t* wb = static_cast<uint8_t*>(ws);
        a.part_ml = reinterpret_cast<float*>(wb + w.part_ml);
        a.nlse2 = reinterpret_cast<float*>(wb + w.nlse2);
        a.col = reinterpret_cast<float*>(wb + w.col);
        a.pool = reinterpret_cast<uint32_t*>(wb + w.pool);
        a.S_pad = w.S_pad;
        a.R_pad = w.R_pad;
        ScoreParams sp = score_params(c, S, w, wb, cache->status);
        cudaError_t e = cudaSuccess;
        if (!(stages & SNAP_STAGE_ROWS)) {
        } else if (lse_obs) {
            // 1-2. the caller's row log-sum-exp, in the base-2 domain the GEMM uses
            e = launch_lse_import(a, lse_obs, st);
        } else {
            // 1. row pass: partial log-sum-exp of every observation row
            e = run_rowstat(SCORE_ROWSTAT, c, sp, K, S, tok_stride, head_stride, Q_obs, st);
            // 2. merge into -lse2 per row
            if (e == cudaSuccess) {
                a.row_splits = SCORE_PARTS * row_key_splits(c, w.R, S);
                e = launch_lse_merge(a, st);
            }
        }
        // 3. column pass: X = 128-key tiles, Y = observation rows
        if (e == cudaSuccess && (stages & SNAP_STAGE_COLUMNS)) {
            CUtensorMap tx, ty;
            const int nx = (int)((S - c.W + 127) / 128);
            const int ny64 = (w.R + 63) / 64 * 64;
            const bool y_resident = c.d_qk == 128 && ny64 <= 256;
            sp.Ny = y_resident ? ny64 : 256;
            if (!k_map(&tx, K, S, c, tok_stride, head_stride, 128) || !q_map(&ty, Q_obs, c, sp.Ny))
                return SNAP_ERR_INVALID_ARG;
            if (y_resident) {
                int splits = (num_sms() + c.n_kv_heads - 1) / c.n_kv_heads;
                if (splits > nx) splits = nx;
                if (splits < 1) splits = 1;
                sp.splits = splits;
                sp.n_units = c.n_kv_heads * splits;
            } else {
                sp.splits = 1;
                sp.n_units = c.n_kv_heads * nx;
            }
            // behind this call's own row stage (a normal launch first) the pass may launch
            // early: it reads the caller's K and Q, complete before that stage started
            e = launch_score_tc(SCORE_COLSUM, tx, ty, sp, c.d_qk, false, !y_resident, num_sms(),
                                (stages & SNAP_STAGE_ROWS) != 0, st);
        }
        // 4. pool + top-K
        if (e == cudaSuccess && (stages & SNAP_STAGE_SELECT)) e = launch_select(a, st);
        if (e != cudaSuccess) return cuda_status(e);
    }
    if (!(stages & SNAP_STAGE_WRITE)) return SNAP_OK;
    // 5. cache write: every slot
    return cuda_status(launch_cache_write(a, num_sms(), st));
}

}  // namespace

extern "C" {

snap_status snap_compress(snap_cache* cache, int slot, const void* K, const void* V, int64_t S,
                          int64_t tok_stride, int64_t head_stride, const void* Q_obs, void* ws,
                          size_t ws_bytes, void* stream) {
    return compress_impl(cache, slot, K, V, S, tok_stride, head_stride, Q_obs, nullptr, ws, ws_bytes,
                         SNAP_STAGE_ALL, stream);
}

snap_status snap_compress_stages(snap_cache* cache, int slot, const void* K, const void* V, int64_t S,
                                 int64_t tok_stride, int64_t head_stride, const void* Q_obs, const float* lse_obs,
                                 void* ws, size_t ws_bytes, int stages, void* stream) {
    if (lse_obs && (reinterpret_cast<uintptr_t>(lse_obs) & 3u)) return SNAP_ERR_INVALID_ARG;
    return compress_impl(cache, slot, K, V, S, tok_stride, head_stride, Q_obs, lse_obs, ws, ws_bytes, stages,
                         stream);
}

snap_status snap_compress_lse(snap_cache* cache, int slot, const void* K, const void* V, int64_t S,
                              int64_t tok_stride, int64_t head_stride, const void* Q_obs, const float* lse_obs,
                              void* ws, size_t ws_bytes, void* stream) {
    if (!lse_obs || (reinterpret_cast<uintptr_t>(lse_obs) & 3u)) return SNAP_ERR_INVALID_ARG;
    return compress_impl(cache, slot, K, V, S, tok_stride, head_stride, Q_obs, lse_obs, ws, ws_bytes,
                         SNAP_STAGE_ALL, stream);
}

snap_status snap_window_logits(snap_cache* cache, const void* K, int64_t S, int64_t tok_stride,
                               int64_t head_stride, const void* Q_obs, float* out, void* stream) {
    if (!cache || !K || !Q_obs || !out) return SNAP_ERR_INVALID_ARG;
    const snap_config& c = cache->cfg;
    if (S < c.W || S > (1ll << 30)) return SNAP_ERR_SHAPE;
    if (!aligned16(K) || !aligned16(Q_obs) || !aligned16(out)) return SNAP_ERR_INVALID_ARG;
    if (tok_stride < c.d_qk || (tok_stride * 2) % 16 || head_stride < 0 || (head_stride * 2) % 16)
        return SNAP_ERR_INVALID_ARG;
    if (c.n_kv_heads > 1 && head_stride < c.d_qk) return SNAP_ERR_INVALID_ARG;
    if (num_sms() <= 0) return SNAP_ERR_CUDA;
    const CompressWs w = compress_ws(c, S);
    ScoreParams sp = score_params(c, S, w, nullptr, cache->status);
    sp.logits = out;
    return cuda_status(run_rowstat(SCORE_LOGITS, c, sp, K, S, tok_stride, head_stride, Q_obs,
                                   static_cast<cudaStream_t>(stream)));
}

snap_status snap_prefill_attn(snap_cache* cache, const void* Q, int64_t S, const void* K, const void* V,
                              int64_t tok_stride, int64_t head_stride, void* O, float* lse_obs, void* stream) {
    if (!cache || !Q || !K || !V || !O) return SNAP_ERR_INVALID_ARG;
    const snap_config& c = cache->cfg;
    if (c.layout != SNAP_LAYOUT_GQA) return SNAP_ERR_UNSUPPORTED;
    if (S < 1 || S > (1ll << 30)) return SNAP_ERR_SHAPE;
    if (lse_obs && S < c.W) return SNAP_ERR_SHAPE;
    if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O)) return SNAP_ERR_INVALID_ARG;
    if (lse_obs && (reinterpret_cast<uintptr_t>(lse_obs) & 3u)) return SNAP_ERR_INVALID_ARG;
    if (tok_stride < c.d_qk || (tok_stride * 2) % 16 || head_stride < 0 || (head_stride * 2) % 16)
        return SNAP_ERR_INVALID_ARG;
    if (c.n_kv_heads > 1 && head_stride < c.d_qk) return SNAP_ERR_INVALID_ARG;
    if (num_sms() <= 0) return SNAP_ERR_CUDA;
    CUtensorMap tq, tk, tv;
    const cuuint64_t qd[3] = {(cuuint64_t)c.d_qk, (cuuint64_t)S, (cuuint64_t)c.n_q_heads};
    const cuuint64_t qs[2] = {(cuuint64_t)c.n_q_heads * c.d_qk * 2, (cuuint64_t)c.d_qk * 2};
    const cuuint32_t qb[3] = {64, 128, 1};
    if (!encode(&tq, Q, 3, qd, qs, qb) || !k_map(&tk, K, S, c, tok_stride, head_stride, 128) ||
        !k_map(&tv, V, S, c, tok_stride, head_stride, 128))
        return SNAP_ERR_INVALID_ARG;
    PrefillArgs a;
    a.S = (int)S;
    a.Hq = c.n_q_heads;
    a.G = c.n_q_heads / c.n_kv_heads;
    a.W = c.W;
    a.sl2 = c.sm_scale * 1.4426950408889634f;
    a.O = static_cast<bf16*>(O);
    a.o_tok_stride = (int64_t)c.n_q_heads * c.d_qk;
    a.lse_obs = lse_obs;
    a.status = cache->status;
    return cuda_status(launch_prefill_tc(tq, tk, tv, a, static_cast<cudaStream_t>(stream)));
}

snap_status snap_decode_append(snap_cache* cache, const int32_t* slots, int n, const void* k_new,
                               const void* v_new, void* stream) {
    if (!cache || n < 0) return SNAP_ERR_INVALID_ARG;
    if (n == 0) return SNAP_OK;
    if (!slots || !k_new || !aligned16(k_new)) return SNAP_ERR_INVALID_ARG;
    const snap_config& c = cache->cfg;
    if (c.layout == SNAP_LAYOUT_GQA && (!v_new || !aligned16(v_new))) return SNAP_ERR_INVALID_ARG;
    if (c.layout == SNAP_LAYOUT_MLA && v_new) return SNAP_ERR_INVALID_ARG;
    if (n > cache->max_batch) return SNAP_ERR_INVALID_ARG;
    AppendArgs a;
    a.kc = cache->k;
    a.vc = cache->v;
    a.meta = cache->meta;
    a.slots = slots;
    a.n = n;
    a.k_new = static_cast<const bf16*>(k_new);
    a.v_new = static_cast<const bf16*>(v_new);
    a.status = cache->status;
    a.cfg = dev_config(c, cache->max_batch);
    return cuda_status(launch_append(a, static_cast<cudaStream_t>(stream)));
}

snap_status snap_decode_attn_ws_bytes(const snap_config* cfg, int max_n, size_t* bytes) {
    snap_status s = check_config(cfg);
    if (s != SNAP_OK) return s;
    if (max_n < 1 || !bytes) return SNAP_ERR_INVALID_ARG;
    *bytes = decode_ws_bytes(*cfg, max_n);
    return SNAP_OK;
}

snap_status snap_decode_attn_plan(const snap_cache* cache, int n, int* splits, int* tiles_per_split,
                                  int* ctas_per_wave) {
    if (!cache || n < 1 || !splits || !tiles_per_split || !ctas_per_wave) return SNAP_ERR_INVALID_ARG;
    if (num_sms() <= 0) return SNAP_ERR_CUDA;
    decode_plan(cache, n, splits, tiles_per_split);
    *ctas_per_wave = decode_wave_ctas(cache);
    return SNAP_OK;
}

snap_status snap_decode_attn(snap_cache* cache, const int32_t* slots, int n, const void* q,
                             void* out, void* ws, size_t ws_bytes, void* stream) {
    return decode_with_ws(cache, slots, n, q, nullptr, nullptr, out, ws, ws_bytes, stream);
}

snap_status snap_decode_step(snap_cache* cache, const int32_t* slots, int n, const void* q, const void* k_new,
                             const void* v_new, void* out, void* ws, size_t ws_bytes, void* stream) {
    if (!k_new) return SNAP_ERR_INVALID_ARG;
    return decode_with_ws(cache, slots, n, q, k_new, v_new, out, ws, ws_bytes, stream);
}

snap_status snap_selftest_bounded_wait(snap_cache* cache, void* stream) {
    if (!cache) return SNAP_ERR_INVALID_ARG;
    return cuda_status(launch_bounded_wait_selftest(cache->status, static_cast<cudaStream_t>(stream)));
}

snap_status snap_check_device(snap_cache* cache, void* stream) {
    if (!cache) return SNAP_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int32_t h[4] = {0, 0, 0, 0};
    cudaError_t e = cudaMemcpyAsync(h, cache->status, sizeof h, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_status(e);
    if (h[0] != 0) {
        std::fprintf(stderr, "libsnap: device status %d (%s) detail %d %d %d\n", h[0], snap_status_string(h[0]),
                     h[1], h[2], h[3]);
        e = cudaMemsetAsync(cache->status, 0, sizeof h, st);
        if (e == cudaSuccess) e = cudaStreamSynchronize(st);
        if (e != cudaSuccess) return cuda_status(e);
        return static_cast<snap_status>(h[0]);
    }
    return SNAP_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Decode attention without a caller workspace (snap_decode_attn_noalloc).
//
// The split-KV partial results live in this file-scope device array instead of a
// caller-allocated workspace.  Host code cannot use the array's name as a device
// address: the device address is looked up once per device with
// cudaGetSymbolAddress and then passed to the kernels as an ordinary pointer.

static __device__ __align__(256) unsigned char g_noalloc_scratch[SNAP_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int NOALLOC_MAX_DEVICES = 64;
std::mutex g_noalloc_mutex;
void* g_noalloc_addr[NOALLOC_MAX_DEVICES] = {};

// Device address of the scratch array on the current device (looked up on first use).
snap_status noalloc_scratch(void** out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_status(e);
    if (dev < 0 || dev >= NOALLOC_MAX_DEVICES) return SNAP_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (!g_noalloc_addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return cuda_status(e);
        g_noalloc_addr[dev] = p;
    }
    *out = g_noalloc_addr[dev];
    return SNAP_OK;
}

}  // namespace

extern "C" snap_status snap_decode_attn_noalloc(snap_cache* cache, const int32_t* slots, int n, const void* q,
                                                void* out, void* stream) {
    if (!cache || n < 0) return SNAP_ERR_INVALID_ARG;
    if (n == 0) return SNAP_OK;
    const snap_config& c = cache->cfg;
    DecodeArgs a;
    if (const snap_status s = decode_args(cache, slots, n, q, out, nullptr, nullptr, &a); s != SNAP_OK) return s;
    // The scratch address is looked up on every device's first call, whatever its
    // split plan, so that this first call (which may also load the module holding
    // the array) is the one the header tells callers to make before any capture.
    void* scratch = nullptr;
    if (const snap_status s = noalloc_scratch(&scratch); s != SNAP_OK) return s;
    const int splits = a.splits;
    if (splits > 1) {
        // compact partial layout for this call: O then (max, sum)
        const size_t parts = (size_t)n * c.n_q_heads * splits;
        const size_t o_bytes = align_up(parts * sizeof(float) * c.d_v, 256);
        const size_t need = o_bytes + parts * sizeof(float) * 2;
        if (need > SNAP_NOALLOC_SCRATCH_BYTES) {
            std::fprintf(stderr,
                         "libsnap: snap_decode_attn_noalloc needs %zu bytes of scratch for %d sequences; the "
                         "limit is %u (use snap_decode_attn with a workspace)\n",
                         need, n, SNAP_NOALLOC_SCRATCH_BYTES);
            return SNAP_ERR_SHAPE;
        }
        a.part_o = static_cast<float*>(scratch);
        a.part_ml = reinterpret_cast<float*>(static_cast<uint8_t*>(scratch) + o_bytes);
    }
    return cuda_status(run_decode(cache, a, static_cast<cudaStream_t>(stream)));
}
