// k_decode.cu -- split-KV decode attention over the fixed-size cache.
//
// SnapStream episode companion page, "Prefill / Decode Pipeline": decode is
// memory-bound, so the cache bytes streamed per step set the time per token.
// GQA: each CTA streams one contiguous range of cache slots of one (sequence, KV head)
// once from HBM and produces an un-normalised partial (max, sum, O) per query head;
// the splits are combined by flash-decoding's log-sum-exp merge inside the same launch:
// within a thread-block cluster (2-8 splits, through distributed shared memory) or by
// the last CTA of the (sequence, KV head) to finish (through global memory), so a decode
// step is one launch.  The ring append of the step ("Ring Buffer vs. Naive Slicing":
// scatter the new token into its fixed ring slot) is fused in: the warp whose tile holds
// the slot writes the new row to the cache and into its own copy of the tile.
// Invalid slots (unused middle slots, ring slots not holding a live position) are
// masked; whole tiles with no valid slot are not read.  The MLA layout's split merge
// runs as its own kernel (decode_merge_kernel): 128 heads x 512 values per sequence.
#include <cooperative_groups.h>

#include "kernels.cuh"

namespace snap {

namespace {

constexpr float NEG_INF = -__builtin_huge_valf();

// ===================================================================== GQA
// d = 128, G <= 8 query heads per KV head.  Keys sit on the MMA's M side
// (16 keys per m16 tile), the G heads on the N side (n8): S^T = K Q^T, then
// O^T += V^T P^T with P^T moved into B-fragment layout by movmatrix.
constexpr int GD = 128;
constexpr int G_ROWB = GD * 2;                              // 256 bytes per key row
constexpr int G_WARPS = 4;
constexpr int G_STAGES = 3;
constexpr int G_STAGE_BYTES = GQA_KEYS * G_ROWB * 2;        // K + V tile = 16 KB
constexpr int G_SMEM = G_WARPS * G_STAGES * G_STAGE_BYTES;  // 192 KB
static_assert(G_WARPS * 32 == GD, "the cross-warp fold gives each thread one of the GD output dimensions");

__global__ void __launch_bounds__(G_WARPS * 32, 1) gqa_decode_kernel(DecodeArgs a) {
    pdl_wait();                 // the previous kernel on the stream has completed
    pdl_launch_dependents();    // the next step's kernel may set up (it waits for this grid)
    extern __shared__ __align__(1024) uint8_t smem[];
    __shared__ int last_sh;
    const DevConfig& c = a.cfg;
    const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int slot = a.slots[b];

    // Loads that need neither the slot nor its meta go out first.
    // Q^T as B fragments: n = head (lane/4), k = d.
    uint32_t qf[8][2];
    {
        const int hq = lane >> 2;
        const bf16* qp = a.q + ((size_t)b * c.Hq + (size_t)h * c.G + (hq < c.G ? hq : 0)) * GD;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            if (hq < c.G) {
                qf[ks][0] = *reinterpret_cast<const uint32_t*>(qp + ks * 16 + 2 * (lane & 3));
                qf[ks][1] = *reinterpret_cast<const uint32_t*>(qp + ks * 16 + 8 + 2 * (lane & 3));
            } else {
                qf[ks][0] = qf[ks][1] = 0u;
            }
        }
    }
    // this lane's 16 bytes of the appended token: K row (lanes 0-15) or V row (16-31)
    uint4 new_row = make_uint4(0u, 0u, 0u, 0u);
    if (a.k_new)
        new_row = reinterpret_cast<const uint4*>((lane < 16 ? a.k_new : a.v_new) +
                                                 ((size_t)b * c.Hkv + h) * GD)[lane & 15];

    if (slot < 0 || slot >= c.max_batch) {
        if (threadIdx.x == 0 && split == 0 && h == 0)
            report_error(a.status, SNAP_ERR_DEVICE_CHECK, 1, b, slot);
        if (split == 0)  // no CTA of this sequence goes on: split 0 writes the zero output
            for (int i = threadIdx.x; i < c.G * GD; i += blockDim.x)
                a.out[((size_t)b * c.Hq + (size_t)h * c.G) * GD + i] = 0.f;
        return;
    }
    // the sequence's meta (S, T, R0, n_sink, n_mid, pad): two 16-byte loads, used below
    const int4* mp = reinterpret_cast<const int4*>(a.meta + slot);
    const int4 m0 = mp[0], m1 = mp[1];

    const size_t row0 = ((size_t)slot * c.Hkv + h) * (size_t)c.C;
    const bf16* kbase = a.kc + row0 * GD;
    const bf16* vbase = a.vc + row0 * GD;
    const int ntiles = (c.C + GQA_KEYS - 1) / GQA_KEYS;
    const int t_begin = split * a.tiles_per_split;
    const int t_end = min(ntiles, t_begin + a.tiles_per_split);
    const uint32_t wsm = smem_u32(smem) + warp * G_STAGES * G_STAGE_BYTES;

    auto load_tile = [&](int t, int st) {
        const uint32_t sk = wsm + st * G_STAGE_BYTES;
        const uint32_t svv = sk + GQA_KEYS * G_ROWB;
#pragma unroll 4
        for (int i = lane; i < GQA_KEYS * 16; i += 32) {
            const int r = i >> 4, ch = i & 15;
            const int key = t * GQA_KEYS + r;
            const bool ok = key < c.C;
            const size_t off = (size_t)(ok ? key : 0) * GD + ch * 8;
            cp_async16(sk + swz(r, ch, G_ROWB), kbase + off, ok ? 16 : 0);
            cp_async16(svv + swz(r, ch, G_ROWB), vbase + off, ok ? 16 : 0);
        }
    };
    // Speculative prologue: the warp's first G_STAGES - 1 tiles (every G_WARPS-th tile
    // of the range) are requested while the meta is in flight; the validity walk below
    // confirms them or reloads.
#pragma unroll
    for (int st = 0; st < G_STAGES - 1; ++st) {
        const int t = t_begin + warp + st * G_WARPS;
        if (t < t_end) load_tile(t, st);
        cp_async_commit();
    }

    snap_seq_meta m;
    m.S = m0.x;
    m.T = m0.y;
    m.R0 = m0.z;
    m.n_sink = m0.w;
    m.n_mid = m1.x;
    // Fused ring append: the new token's ring slot s_app.  The warp that computes the
    // tile holding it writes the row to the cache and patches it into its stage (its
    // load may have read the old row); the attention sees T + 1 tokens.
    int t_app = -1, s_app = 0;
    if (a.k_new) {
        s_app = c.L_sink + c.K + m.T % c.L_recent;
        m.T += 1;
        const int t = s_app / GQA_KEYS;
        if (t >= t_begin && t < t_end && (t - t_begin) % G_WARPS == warp) {
            t_app = t;
            bf16* dst = const_cast<bf16*>(lane < 16 ? kbase : vbase) + (size_t)s_app * GD;
            reinterpret_cast<uint4*>(dst)[lane & 15] = new_row;
        }
    }
    SlotValidity sv;
    sv.init(m, c);

    auto next_tile = [&](int t) {
        while (t < t_end && !sv.any_valid(t * GQA_KEYS, min(c.C, (t + 1) * GQA_KEYS))) t += G_WARPS;
        return t;
    };
    // the tiles the warp computes: every G_WARPS-th tile with a valid slot
    const int t_first = next_tile(t_begin + warp);
    int t_load = t_first;
    bool spec_ok = true;
    int chain[G_STAGES - 1];
#pragma unroll
    for (int st = 0; st < G_STAGES - 1; ++st) {
        chain[st] = t_load;
        if (t_load < t_end) {
            if (t_load != t_begin + warp + st * G_WARPS) spec_ok = false;
            t_load = next_tile(t_load + G_WARPS);
        }
    }
    if (!spec_ok) {             // a skipped tile: drop the speculative stages, load the walk's
        cp_async_wait<0>();
        __syncwarp();
#pragma unroll
        for (int st = 0; st < G_STAGES - 1; ++st) {
            if (chain[st] < t_end) load_tile(chain[st], st);
            cp_async_commit();
        }
    }

    float m_run[2] = {NEG_INF, NEG_INF};
    float l_run[2] = {0.f, 0.f};
    float o[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;

    int t_comp = t_first;
    int st_comp = 0, st_load = G_STAGES - 1;
    const float sl2 = c.scale_log2;
    while (t_comp < t_end) {
        if (t_load < t_end) {
            load_tile(t_load, st_load);
            t_load = next_tile(t_load + G_WARPS);
        }
        cp_async_commit();
        cp_async_wait<G_STAGES - 1>();
        __syncwarp();

        const uint32_t sk = wsm + st_comp * G_STAGE_BYTES;
        const uint32_t svv = sk + GQA_KEYS * G_ROWB;
        if (t_comp == t_app) {  // the appended row replaces whatever the load read there
            const uint32_t dst = (lane < 16 ? sk : svv) + swz(s_app - t_comp * GQA_KEYS, lane & 15, G_ROWB);
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};\n" ::"r"(dst), "r"(new_row.x),
                         "r"(new_row.y), "r"(new_row.z), "r"(new_row.w)
                         : "memory");
            __syncwarp();
        }
        float s[2][4];
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
            s[mt][0] = s[mt][1] = s[mt][2] = s[mt][3] = 0.f;
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const int r = mt * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
                const int ch = ks * 2 + (lane >> 4);
                uint32_t af[4];
                ldsm_x4(sk + swz(r, ch, G_ROWB), af[0], af[1], af[2], af[3]);
                mma_bf16(s[mt], af, qf[ks][0], qf[ks][1]);
            }
        }
        // mask + scale into the base-2 domain; per-head tile max
        float mx0 = NEG_INF, mx1 = NEG_INF;
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const int key = t_comp * GQA_KEYS + mt * 16 + (lane >> 2) + 8 * half;
                const bool ok = key < c.C && sv.valid(key);
                s[mt][2 * half + 0] = ok ? s[mt][2 * half + 0] * sl2 : NEG_INF;
                s[mt][2 * half + 1] = ok ? s[mt][2 * half + 1] * sl2 : NEG_INF;
                mx0 = fmaxf(mx0, s[mt][2 * half + 0]);
                mx1 = fmaxf(mx1, s[mt][2 * half + 1]);
            }
#pragma unroll
        for (int x = 4; x < 32; x <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, x));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, x));
        }
        const float mn0 = fmaxf(m_run[0], mx0), mn1 = fmaxf(m_run[1], mx1);
        const float al0 = mn0 == NEG_INF ? 1.f : ex2(m_run[0] - mn0);
        const float al1 = mn1 == NEG_INF ? 1.f : ex2(m_run[1] - mn1);
        m_run[0] = mn0;
        m_run[1] = mn1;
        float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                // weights rounded to bf16 here, so that the normaliser sums exactly
                // the weights the P V product uses
                float p0 = mn0 == NEG_INF ? 0.f : bf16_round(ex2(s[mt][2 * half + 0] - mn0));
                float p1 = mn1 == NEG_INF ? 0.f : bf16_round(ex2(s[mt][2 * half + 1] - mn1));
                s[mt][2 * half + 0] = p0;
                s[mt][2 * half + 1] = p1;
                ps0 += p0;
                ps1 += p1;
            }
        l_run[0] = l_run[0] * al0 + ps0;
        l_run[1] = l_run[1] * al1 + ps1;
#pragma unroll
        for (int dt = 0; dt < 8; ++dt) {
            o[dt][0] *= al0;
            o[dt][1] *= al1;
            o[dt][2] *= al0;
            o[dt][3] *= al1;
        }
        // O^T[d][head] += V^T[d][key] * P^T[key][head]
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
            const uint32_t b0 = movmatrix_t(pack_bf16(s[mt][0], s[mt][1]));
            const uint32_t b1 = movmatrix_t(pack_bf16(s[mt][2], s[mt][3]));
#pragma unroll
            for (int dt = 0; dt < 8; ++dt) {
                const int r = mt * 16 + (lane & 7) + ((lane >> 4) << 3);
                const int ch = dt * 2 + ((lane >> 3) & 1);
                uint32_t af[4];
                ldsm_x4_t(svv + swz(r, ch, G_ROWB), af[0], af[1], af[2], af[3]);
                mma_bf16(o[dt], af, b0, b1);
            }
        }
        __syncwarp();
        t_comp = next_tile(t_comp + G_WARPS);
        st_comp = (st_comp + 1) % G_STAGES;
        st_load = (st_load + 1) % G_STAGES;
    }
    cp_async_wait<0>();

    // per-head sums over the lanes holding the same head columns
#pragma unroll
    for (int x = 4; x < 32; x <<= 1) {
        l_run[0] += __shfl_xor_sync(0xffffffffu, l_run[0], x);
        l_run[1] += __shfl_xor_sync(0xffffffffu, l_run[1], x);
    }
    __syncthreads();
    // cross-warp merge through shared memory (pipeline buffers are free now)
    float* ob = reinterpret_cast<float*>(smem);                 // [warps][8 heads][128]
    float* mlb = ob + G_WARPS * 8 * GD;                         // [warps][8][2]
    {
        const int g = lane >> 2, t = lane & 3;
#pragma unroll
        for (int dt = 0; dt < 8; ++dt)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int d = dt * 16 + g + 8 * (i >> 1);
                const int hh = 2 * t + (i & 1);
                ob[(warp * 8 + hh) * GD + d] = o[dt][i];
            }
        if (lane < 4) {
            mlb[(warp * 8 + 2 * t) * 2 + 0] = m_run[0];
            mlb[(warp * 8 + 2 * t) * 2 + 1] = l_run[0];
            mlb[(warp * 8 + 2 * t + 1) * 2 + 0] = m_run[1];
            mlb[(warp * 8 + 2 * t + 1) * 2 + 1] = l_run[1];
        }
    }
    __syncthreads();
    const int d = threadIdx.x;  // 128 threads == 128 dims
    // this CTA's (max, sum, O[d]) per query head, kept for the split merge: every warp's
    // values of every head are loaded first, then combined
    float Mh[8], Lh[8], Oh[8];
    {
        float wm[G_WARPS][8], wl[G_WARPS][8], wo[G_WARPS][8];
#pragma unroll
        for (int w = 0; w < G_WARPS; ++w)
#pragma unroll
            for (int hh = 0; hh < 8; ++hh) {
                wm[w][hh] = mlb[(w * 8 + hh) * 2];
                wl[w][hh] = mlb[(w * 8 + hh) * 2 + 1];
                wo[w][hh] = ob[(w * 8 + hh) * GD + d];
            }
#pragma unroll
        for (int hh = 0; hh < 8; ++hh) {
            Mh[hh] = NEG_INF;
#pragma unroll
            for (int w = 0; w < G_WARPS; ++w) Mh[hh] = fmaxf(Mh[hh], wm[w][hh]);
            Lh[hh] = Oh[hh] = 0.f;
#pragma unroll
            for (int w = 0; w < G_WARPS; ++w) {
                const float f = Mh[hh] == NEG_INF ? 0.f : ex2(wm[w][hh] - Mh[hh]);
                Lh[hh] += f * wl[w][hh];
                Oh[hh] += f * wo[w][hh];
            }
        }
    }
    if (a.splits > 1 && !a.cluster_merge) {
#pragma unroll
        for (int hh = 0; hh < 8; ++hh) {
            if (hh >= c.G) continue;
            const size_t pi = (((size_t)b * c.Hkv + h) * a.splits + split) * c.G + hh;
            a.part_o[pi * GD + d] = Oh[hh];
            if (d == 0) {
                a.part_ml[pi * 2 + 0] = Mh[hh];
                a.part_ml[pi * 2 + 1] = Lh[hh];
            }
        }
    }
    if (a.splits > 1 && a.cluster_merge) {
        // the splits of this (sequence, KV head) are one cluster (rank = split).  Once
        // every rank's loop is done, each writes its (max, sum, O) into rank 0's pipeline
        // buffers (free by then) through distributed shared memory; after the second
        // barrier rank 0 folds them in rank order from its own shared memory.
        namespace cg = cooperative_groups;
        cg::cluster_group cl = cg::this_cluster();
        constexpr int ML_OFF = 8 * 8 * GD;        // [rank][8 heads][GD] O, then [rank][8][2]
        static_assert((ML_OFF + 8 * 8 * 2) * 4 <= G_SMEM, "landing area inside the pipeline buffers");
        cl.sync();
        float* land = cl.map_shared_rank(reinterpret_cast<float*>(smem), 0);
#pragma unroll
        for (int hh = 0; hh < 8; ++hh)
            if (hh < c.G) {
                land[(split * 8 + hh) * GD + d] = Oh[hh];
                if (d == 0) {
                    land[ML_OFF + (split * 8 + hh) * 2 + 0] = Mh[hh];
                    land[ML_OFF + (split * 8 + hh) * 2 + 1] = Lh[hh];
                }
            }
        cl.sync();
        if (split != 0) return;
        const float* xo = reinterpret_cast<const float*>(smem);
        float Mr[8], Lr[8], Or[8];
#pragma unroll
        for (int hh = 0; hh < 8; ++hh) {
            Mr[hh] = NEG_INF;
            Lr[hh] = Or[hh] = 0.f;
        }
        for (int s2 = 0; s2 < a.splits; ++s2) {
            // a rank's values of every head loaded first (slots of heads >= G are unused)
            float ms[8], ls[8], os[8];
#pragma unroll
            for (int hh = 0; hh < 8; ++hh) {
                ms[hh] = xo[ML_OFF + (s2 * 8 + hh) * 2];
                ls[hh] = xo[ML_OFF + (s2 * 8 + hh) * 2 + 1];
                os[hh] = xo[(s2 * 8 + hh) * GD + d];
            }
#pragma unroll
            for (int hh = 0; hh < 8; ++hh) {
                if (hh >= c.G || ms[hh] == NEG_INF) continue;
                const float Mn = fmaxf(Mr[hh], ms[hh]);
                const float fa = ex2(Mr[hh] - Mn), fb = ex2(ms[hh] - Mn);
                Lr[hh] = Lr[hh] * fa + ls[hh] * fb;
                Or[hh] = Or[hh] * fa + os[hh] * fb;
                Mr[hh] = Mn;
            }
        }
#pragma unroll
        for (int hh = 0; hh < 8; ++hh) {
            Lh[hh] = Lr[hh];
            Oh[hh] = Or[hh];
        }
    } else if (a.splits > 1) {
        // split merge in the last CTA of (sequence, KV head) to finish: flash-decoding's
        // log-sum-exp merge of every split's (max, sum, O) of the G query heads
        __threadfence();
        __syncthreads();
        if (threadIdx.x == 0) {
            int* cnt = a.merge_cnt + (size_t)slot * c.Hkv + h;
            const int last = atomicAdd(cnt, 1) == a.splits - 1;
            if (last) *cnt = 0;      // every other CTA has counted: ready for the next call
            last_sh = last;
        }
        __syncthreads();
        if (!last_sh) return;
        __threadfence();
        // splits folded in index order (this CTA's own from registers), so that the
        // result does not depend on which CTA finished last
        const size_t p0 = ((size_t)b * c.Hkv + h) * a.splits;
        float Mr[8], Lr[8], Or[8];
#pragma unroll
        for (int hh = 0; hh < 8; ++hh) {
            Mr[hh] = NEG_INF;
            Lr[hh] = Or[hh] = 0.f;
        }
        for (int s2 = 0; s2 < a.splits; ++s2) {
            // one split's partials of every head, all loads in flight together
            float ms[8], ls[8], os[8];
#pragma unroll
            for (int hh = 0; hh < 8; ++hh) {
                ms[hh] = Mh[hh];
                ls[hh] = Lh[hh];
                os[hh] = Oh[hh];
                if (hh < c.G && s2 != split) {
                    const size_t pi = (p0 + s2) * c.G + hh;
                    ms[hh] = __ldcg(a.part_ml + pi * 2);
                    ls[hh] = __ldcg(a.part_ml + pi * 2 + 1);
                    os[hh] = __ldcg(a.part_o + pi * GD + d);
                }
            }
#pragma unroll
            for (int hh = 0; hh < 8; ++hh) {
                if (ms[hh] == NEG_INF) continue;
                const float Mn = fmaxf(Mr[hh], ms[hh]);
                const float fa = ex2(Mr[hh] - Mn), fb = ex2(ms[hh] - Mn);
                Lr[hh] = Lr[hh] * fa + ls[hh] * fb;
                Or[hh] = Or[hh] * fa + os[hh] * fb;
                Mr[hh] = Mn;
            }
        }
#pragma unroll
        for (int hh = 0; hh < 8; ++hh) {
            Lh[hh] = Lr[hh];
            Oh[hh] = Or[hh];
        }
    }
#pragma unroll
    for (int hh = 0; hh < 8; ++hh)
        if (hh < c.G)
            a.out[((size_t)b * c.Hq + (size_t)h * c.G + hh) * GD + d] = Lh[hh] > 0.f ? Oh[hh] / Lh[hh] : 0.f;
    // T advances once per step: counted by the CTA that finishes each (sequence, KV head)
    // (the merging CTA, or the only split), every CTA of the sequence having read the meta
    if (a.k_new && threadIdx.x == 0) {
        if (atomicAdd(&a.meta_rw[slot].pad[0], 1) == (int)gridDim.y - 1) {
            a.meta_rw[slot].T = m.T;
            a.meta_rw[slot].pad[0] = 0;
        }
    }
}

// =================================================================== merge
// out[b][i][:] = sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s  (zero if empty).
// Partial index: ((b * Hkv + h) * splits + s) * G + hh  for query head i = h*G + hh.
// Every thread first requests its columns of the first MERGE_PRE splits (they do not
// depend on the weights), then one warp turns the (max, sum) pairs into weights in
// shared memory; the splits are added in index order.
constexpr int MERGE_PRE = 8;
__global__ void decode_merge_kernel(DecodeArgs a) {
    pdl_wait();                 // the attention's partials are complete and visible
    __shared__ float w_s[32];
    __shared__ float inv_l;
    const DevConfig& c = a.cfg;
    const int i = blockIdx.x, b = blockIdx.y;
    const int h = i / c.G, hh = i % c.G;
    const int slot = a.slots[b];
    const bool ok = slot >= 0 && slot < c.max_batch;
    const size_t p0 = ((size_t)b * c.Hkv + h) * a.splits;
    const int dv4 = c.dv / 4;
    auto part = [&](int s, int d4) {
        return reinterpret_cast<const float4*>(a.part_o + ((p0 + s) * c.G + hh) * c.dv)[d4];
    };
    // this thread's first column group: its loads overlap the weights below
    float4 pre[MERGE_PRE];
#pragma unroll
    for (int s = 0; s < MERGE_PRE; ++s)
        pre[s] = (ok && s < a.splits && (int)threadIdx.x < dv4) ? part(s, threadIdx.x) : make_float4(0.f, 0.f, 0.f, 0.f);
    if (threadIdx.x < 32) {
        const int s = threadIdx.x;
        const bool in = ok && s < a.splits;
        const float m = in ? a.part_ml[((p0 + s) * c.G + hh) * 2] : NEG_INF;
        const float l = in ? a.part_ml[((p0 + s) * c.G + hh) * 2 + 1] : 0.f;
        float M = m;
#pragma unroll
        for (int x = 16; x > 0; x >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, x));
        const float w = (M == NEG_INF || m == NEG_INF) ? 0.f : ex2(m - M);
        float L = w * l;
#pragma unroll
        for (int x = 16; x > 0; x >>= 1) L += __shfl_xor_sync(0xffffffffu, L, x);
        w_s[s] = w;
        if (s == 0) inv_l = L > 0.f ? 1.f / L : 0.f;
    }
    __syncthreads();
    const float il = inv_l;
    // four output columns per thread (d_v is 128 or 512)
    for (int d4 = threadIdx.x; d4 < dv4; d4 += blockDim.x) {
        float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
        if (il != 0.f) {
            int s0 = 0;
            if (d4 == (int)threadIdx.x) {     // the prefetched splits
#pragma unroll
                for (int s = 0; s < MERGE_PRE; ++s) {
                    if (s < a.splits) {
                        const float w = w_s[s];
                        O.x += w * pre[s].x;
                        O.y += w * pre[s].y;
                        O.z += w * pre[s].z;
                        O.w += w * pre[s].w;
                    }
                }
                s0 = a.splits < MERGE_PRE ? a.splits : MERGE_PRE;
            }
#pragma unroll 8
            for (int s = s0; s < a.splits; ++s) {
                const float4 v = part(s, d4);
                const float w = w_s[s];
                O.x += w * v.x;
                O.y += w * v.y;
                O.z += w * v.z;
                O.w += w * v.w;
            }
        }
        reinterpret_cast<float4*>(a.out + ((size_t)b * c.Hq + i) * c.dv)[d4] =
            make_float4(O.x * il, O.y * il, O.z * il, O.w * il);
    }
}

}  // namespace

// Clusters of `csize` decode CTAs that can be resident at once on this device (0 if
// the query fails); cached per device and cluster size.
int gqa_active_clusters(int csize) {
    static std::atomic<int> cached[64][9];     // zero-initialised (static storage)
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    const bool cacheable = dev >= 0 && dev < 64 && csize >= 0 && csize <= 8;
    if (cacheable) {
        const int v = cached[dev][csize].load(std::memory_order_relaxed);
        if (v > 0) return v;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(csize, 1, 1);
    cfg.blockDim = dim3(G_WARPS * 32);
    cfg.dynamicSmemBytes = G_SMEM;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = csize;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, gqa_decode_kernel, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    if (cacheable && n > 0) cached[dev][csize].store(n, std::memory_order_relaxed);
    return n;
}

cudaError_t launch_decode_gqa(const DecodeArgs& a0, cudaStream_t st) {
    static std::atomic<uint64_t> smem_set{0};
    if (cudaError_t e = opt_in_smem(gqa_decode_kernel, G_SMEM, smem_set); e != cudaSuccess) return e;
    dim3 grid(a0.splits, a0.cfg.Hkv, a0.n);
    // the splits of a (sequence, KV head) as one cluster when a portable cluster holds
    // them and every cluster of the launch is resident at once (else the global merge)
    if (a0.splits >= 2 && a0.splits <= 8) {
        const long long ctas = (long long)a0.splits * a0.cfg.Hkv * a0.n;
        if (ctas <= (long long)gqa_active_clusters(a0.splits) * a0.splits) {
            DecodeArgs a = a0;
            a.cluster_merge = 1;
            return launch_dependent_clustered(gqa_decode_kernel, grid, dim3(G_WARPS * 32), G_SMEM, st,
                                              (unsigned)a.splits, a);
        }
    }
    return launch_dependent(gqa_decode_kernel, grid, dim3(G_WARPS * 32), G_SMEM, st, a0);
}

cudaError_t launch_decode_merge(const DecodeArgs& a, cudaStream_t st) {
    dim3 grid(a.cfg.Hq, a.n);
    const int threads = a.cfg.dv / 4 < 32 ? 32 : (a.cfg.dv / 4 > 128 ? 128 : a.cfg.dv / 4);   // one float4 each
    return launch_dependent(decode_merge_kernel, grid, dim3(threads), 0, st, a);
}

}  // namespace snap
