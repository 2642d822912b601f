// Unordered-tree row kernels (TR_ORDER_UNORDERED_TREE).
//
// Mapping ("TIRx Metal reduction lowering" §4 "Execution mapping algebra"):
// a row is served by W workers. Worker w owns the 16-byte slots
// e = W*chunk + w of the row's aligned body (§4.4 "Coverage and ancestry",
// blocked-cyclic ownership with V = 4: one float4 per slot), so a warp's loads
// of one chunk are 512 contiguous bytes. The unaligned head (< 4 floats before
// the first 16-byte boundary) and tail (< 4 floats) are owned by workers
// 0..head-1 and 0..tail-1. Missing slots hold the reducer's identity.
//
// Reuse (§5 "Logical Tile materialization to physical worker storage"): in
// the cached plans each worker keeps its stripe in registers (K float4 slots,
// at most 64 floats: the §5.1 stripe budget), so every input element is read
// from memory exactly once and the epilogue runs on the cached values. The
// stream plans keep nothing and read the row again after the statistics.
#pragma once

#include <type_traits>

#include "tr_device.cuh"
#include "tr_internal.h"

namespace tr {

// Largest CTA a K-slot cached kernel is compiled for: 64 cached floats need
// about 90 registers (at most 512 threads per CTA); a LayerNorm stripe of 16
// or more floats, with its prefetched weights and biases, needs more than the
// 64 registers a 1024-thread CTA allows.
// K == 6 is the one-wave shape for rows of up to 6144 columns: 256 threads a
// row and six rows on every SM (1536 threads, so at most 40 registers a
// thread), which keeps 912 rows resident on 152 SMs; a CTA holds one, two or
// three rows (256, 512 or 768 threads).
template <int OP, int K>
constexpr int max_threads_for() {
    return K == 6 ? 768 : K >= 16 ? 512 : (K >= 4 && OP == OP_LAYERNORM) ? 768 : 1024;
}
template <int K>
constexpr int min_blocks_for() {
    return K == 6 ? 2 : 1;
}
// Fused residual variants hold the residual's stripe in flight beside x's
// (2K float4 at the peak): half the threads of a plain kernel for K >= 4.
template <int OP, int K, bool RES>
constexpr int max_threads_res() {
    return !RES ? max_threads_for<OP, K>() : K >= 16 ? 256 : K >= 4 ? 512 : 1024;
}
template <int K, bool RES>
constexpr int min_blocks_res() {
    return RES ? 1 : min_blocks_for<K>();
}

// Staged kernels that also hold K float4 of weights (and of biases) per worker.
template <int OP, int K, bool PRE>
constexpr int staged_max_threads() {
    if (!PRE) return (K >= 8 || (K >= 4 && OP == OP_LAYERNORM)) ? 768 : 1024;
    return K <= 2 ? 1024 : K == 4 ? 768 : (OP == OP_LAYERNORM ? 384 : 512);
}

template <int OP>
__device__ __forceinline__ float first_identity() {
    return OP == OP_SOFTMAX ? MaxOp::id() : 0.0f;
}

__device__ __forceinline__ float4 ld_param(const float* p, bool vec) {
    if (vec) return ld_param4(p);
    return make_float4(__ldg(p), __ldg(p + 1), __ldg(p + 2), __ldg(p + 3));
}

__device__ __forceinline__ void st_out(float* p, float4 o, bool vec) {
    if (vec) {
        st4(p, o);
    } else {
        p[0] = o.x;
        p[1] = o.y;
        p[2] = o.z;
        p[3] = o.w;
    }
}

__device__ __forceinline__ float4 f4(float v) { return make_float4(v, v, v, v); }

// Which body slot a cached register slot j holds.
struct SlotMapRows {  // a row per W workers: slot j <-> vector j*W + w
    int W, w, nvec;
    __device__ __forceinline__ int idx(int j) const { return j * W + w; }
    __device__ __forceinline__ bool ok(int j) const { return idx(j) < nvec; }
};
struct SlotMapSeg {  // a CTA's segment [v0, v1) of the row: slot j <-> v0 + j*T + t
    int T, t, v0, v1;
    __device__ __forceinline__ int idx(int j) const { return v0 + j * T + t; }
    __device__ __forceinline__ bool ok(int j) const { return idx(j) < v1; }
};

// Merge a worker statistic over the workers of one row (inside one CTA).
template <int G>
struct RowsReducer {
    RowPos p;
    float4 (*part)[32];
    int buf;
    template <class T>
    __device__ __forceinline__ T operator()(T v) {
        return cta_row_merge<T, G>(v, p, part, buf);
    }
};
// ... over the CTA, then over the C CTAs of the cluster (distributed shared memory).
struct ClusterReducer {
    RowPos p;
    float4 (*part)[32];
    int buf;
    float4* cpart;
    int cbuf;
    int C;
    template <class T>
    __device__ __forceinline__ T operator()(T v) {
        v = cta_row_merge<T, 32>(v, p, part, buf);
        return cluster_merge<T>(v, cpart, cbuf, C);
    }
};

__device__ __forceinline__ float max4(float4 v) { return fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w)); }
__device__ __forceinline__ float sum4(float4 v) { return (v.x + v.y) + (v.z + v.w); }

// Load a worker's stripe: K float4 slots plus its head/tail scalar.
template <int OP, int K, class Map>
__device__ __forceinline__ void load_stripe(const float* xr, const RowGeom& g, const Map& map, bool active,
                                            int wi, bool own_h, bool own_t, float4 (&v)[K], float& hv,
                                            float& tv) {
    const float id = first_identity<OP>();
    const float* xb = xr + g.head;
#pragma unroll
    for (int j = 0; j < K; ++j) {
        v[j] = f4(id);
        if (active && map.ok(j)) v[j] = ld_stream4(xb + 4 * map.idx(j));
    }
    hv = id;
    tv = id;
    if (active && own_h) hv = ld_stream1(xr + wi);
    if (active && own_t) tv = ld_stream1(xb + 4 * g.nvec + wi);
}

// Fused residual norms: add the residual's stripe to the loaded x stripe
// (h = x + r, one rounded add per element, the residual read with 16-byte
// loads when its rows have x's 16-byte phase) and, when h is requested, write
// h at once: it does not depend on the row statistics, so the stores overlap
// the merges. Padding slots keep the identity.
template <int K, class Map>
__device__ __forceinline__ void add_residual(const RowArgs& a, int64_t row, const RowGeom& g, const Map& map,
                                             bool active, int wi, bool own_h, bool own_t, float4 (&v)[K],
                                             float& hv, float& tv) {
    const float* rr = a.r + row * a.cols;
    const float* rb = rr + g.head;
    float4 rq[K];
#pragma unroll
    for (int j = 0; j < K; ++j) {
        rq[j] = f4(0.0f);
        if (active && map.ok(j)) {
            const float* p = rb + 4 * map.idx(j);
            rq[j] = a.r_vec ? ld_stream4(p) : make_float4(ld_stream1(p), ld_stream1(p + 1), ld_stream1(p + 2),
                                                          ld_stream1(p + 3));
        }
    }
    float rh = 0.0f, rt = 0.0f;
    if (active && own_h) rh = ld_stream1(rr + wi);
    if (active && own_t) rt = ld_stream1(rb + 4 * g.nvec + wi);
#pragma unroll
    for (int j = 0; j < K; ++j)
        if (active && map.ok(j)) {
            v[j].x += rq[j].x;
            v[j].y += rq[j].y;
            v[j].z += rq[j].z;
            v[j].w += rq[j].w;
        }
    if (active && own_h) hv += rh;
    if (active && own_t) tv += rt;
    if (a.h && active) {
        float* hr = a.h + row * a.cols;
        float* hb = hr + g.head;
#pragma unroll
        for (int j = 0; j < K; ++j)
            if (map.ok(j)) st_out(hb + 4 * map.idx(j), v[j], a.h_vec);
        if (own_h) hr[wi] = hv;
        if (own_t) hb[4 * g.nvec + wi] = tv;
    }
}

// Norm weights and biases staged in shared memory (rows plans with
// TR_PLAN_FLAG_PARAMS_IN_SHARED): one thread issues bulk asynchronous copies
// of the whole weight (and bias) vector when the kernel starts, while the rows
// load, and the epilogue reads them once `bar` completes instead of making a
// dependent trip to L2 after the merges. All rows of the CTA share the copy.
struct SharedParams {
    const float* w;  // cols floats (16-byte aligned rows: column = body index)
    const float* b;
    uint64_t* bar;
};
__device__ __forceinline__ float4 ld_shared4(const float* p) { return *reinterpret_cast<const float4*>(p); }

// The three cached epilogues. Every worker of the row calls this uniformly
// (merges may contain a barrier); only the stores are predicated on `active`.
//   softmax:   m = max (merge 1); e = 2^(x log2e - mb(m)) with one FMA per
//              element; s = sum e (merge 2); y = e * (1/s)
//   RMSNorm:   sum of squares (one merge); y = x * rsqrt(ss/N + eps) * w
//   LayerNorm: mean = sum / N (merge 1, one rounded division); var = sum of
//              (x - mean)^2 over the cached stripe / N (merge 2: the second pass
//              runs on registers, no cancellation); y = (x - mean) * rsqrt(var + eps)
//              * gamma + beta
// Two cheap float butterflies are shorter on the critical path than one merge
// of compound statistics, which matters when a CTA reduces rows back to back.
// PRE: the weight/bias float4s of this worker's slots are already in wr/br
// (persistent CTAs whose workers see the same columns in every row).
template <int OP, int K, bool PRE = false, bool SP = false, class Map, class Red>
__device__ __forceinline__ void cached_epilogue(const RowArgs& a, float* yr, const RowGeom& g, float4 (&v)[K],
                                                float hv, float tv, bool own_h, bool own_t, bool active, int wi,
                                                const Map& map, Red& red, const float4 (&wr)[K],
                                                const float4 (&br)[K], const SharedParams& sp = SharedParams{}) {
    float* yb = yr + g.head;
    const int ti = g.head + 4 * g.nvec + wi;  // column of this worker's tail scalar
    if constexpr (OP == OP_SOFTMAX) {
        // missing slots hold -inf: they give e = 0
        float m = fmaxf(hv, tv);
#pragma unroll
        for (int j = 0; j < K; ++j) m = fmaxf(m, max4(v[j]));
        m = red(MaxF{m}).v;
        const float mb = mb_of(m);
        float s = 0.0f;
#pragma unroll
        for (int j = 0; j < K; ++j) {
            v[j].x = ex2(fmaf(v[j].x, kL2E, -mb));
            v[j].y = ex2(fmaf(v[j].y, kL2E, -mb));
            v[j].z = ex2(fmaf(v[j].z, kL2E, -mb));
            v[j].w = ex2(fmaf(v[j].w, kL2E, -mb));
            s += sum4(v[j]);
        }
        hv = ex2(fmaf(hv, kL2E, -mb));
        tv = ex2(fmaf(tv, kL2E, -mb));
        s += hv + tv;
        s = red(s);
        const float inv = 1.0f / s;
        if (!active) return;
#pragma unroll
        for (int j = 0; j < K; ++j)
            if (map.ok(j))
                st_out(yb + 4 * map.idx(j), make_float4(v[j].x * inv, v[j].y * inv, v[j].z * inv, v[j].w * inv),
                       a.y_vec);
        if (own_h) yr[wi] = hv * inv;
        if (own_t) yr[ti] = tv * inv;
    } else if constexpr (OP == OP_RMSNORM) {
        // short stripes fetch their weights now, so the load overlaps the merge
        constexpr bool kFetchEarly = !PRE && !SP && K <= 4;
        const bool wv = a.has_w && aligned16(a.w + g.head);
        float4 wq[K];
        if constexpr (kFetchEarly) {
#pragma unroll
            for (int j = 0; j < K; ++j)
                wq[j] = (a.has_w && active && map.ok(j)) ? ld_param(a.w + g.head + 4 * map.idx(j), wv) : f4(1.0f);
        }
        // missing slots hold 0
        float ss = fmaf(hv, hv, tv * tv);
#pragma unroll
        for (int j = 0; j < K; ++j)
            ss = fmaf(v[j].x, v[j].x, fmaf(v[j].y, v[j].y, fmaf(v[j].z, v[j].z, fmaf(v[j].w, v[j].w, ss))));
        ss = red(ss);
        const float rstd = rsqrtf(fmaf(ss, a.inv_cols, a.eps));
        if constexpr (SP) mbar_wait_bounded(sp.bar, 0, a.wait_ns, a.err);  // uniform: before any return
        if (!active) return;
#pragma unroll
        for (int j = 0; j < K; ++j)
            if (map.ok(j)) {
                const int e = 4 * map.idx(j);
                float4 o = make_float4(v[j].x * rstd, v[j].y * rstd, v[j].z * rstd, v[j].w * rstd);
                if (a.has_w) {
                    const float4 wj = SP ? ld_shared4(sp.w + e)
                                      : PRE ? wr[j] : kFetchEarly ? wq[j] : ld_param(a.w + g.head + e, wv);
                    o.x *= wj.x; o.y *= wj.y; o.z *= wj.z; o.w *= wj.w;
                }
                st_out(yb + e, o, a.y_vec);
            }
        if (own_h) yr[wi] = hv * rstd * (a.has_w ? __ldg(a.w + wi) : 1.0f);
        if (own_t) yr[ti] = tv * rstd * (a.has_w ? __ldg(a.w + ti) : 1.0f);
    } else if constexpr (OP == OP_LAYERNORM) {
        // short stripes fetch their weights and biases now, overlapping the merges
        constexpr bool kFetchEarly = !PRE && !SP && K <= 4;
        const bool wv = a.has_w && aligned16(a.w + g.head);
        const bool bv = a.has_b && aligned16(a.b + g.head);
        float4 wq[K], bq[K];
        if constexpr (kFetchEarly) {
#pragma unroll
            for (int j = 0; j < K; ++j) {
                const bool here = active && map.ok(j);
                const int e = 4 * map.idx(j);
                wq[j] = (a.has_w && here) ? ld_param(a.w + g.head + e, wv) : f4(1.0f);
                bq[j] = (a.has_b && here) ? ld_param(a.b + g.head + e, bv) : f4(0.0f);
            }
        }
        // missing slots hold 0 for the sum; they are excluded from the second pass
        float sm = hv + tv;
#pragma unroll
        for (int j = 0; j < K; ++j) sm += sum4(v[j]);
        sm = red(sm);
        // one rounded division: a product sm * (1/N) could be contracted into
        // fma(-sm, 1/N, x) below, leaving the mean unrounded (a constant row
        // would then not centre to exactly 0)
        const float mean = __fdiv_rn(sm, a.cols_f);
        float sq = 0.0f;
#pragma unroll
        for (int j = 0; j < K; ++j)
            if (map.ok(j)) {
                const float dx = v[j].x - mean, dy = v[j].y - mean, dz = v[j].z - mean, dw = v[j].w - mean;
                sq = fmaf(dx, dx, fmaf(dy, dy, fmaf(dz, dz, fmaf(dw, dw, sq))));
            }
        if (own_h) sq = fmaf(hv - mean, hv - mean, sq);
        if (own_t) sq = fmaf(tv - mean, tv - mean, sq);
        sq = red(sq);
        const float rstd = rsqrtf(fmaf(sq, a.inv_cols, a.eps));
        if constexpr (SP) mbar_wait_bounded(sp.bar, 0, a.wait_ns, a.err);  // uniform: before any return
        if (!active) return;
#pragma unroll
        for (int j = 0; j < K; ++j)
            if (map.ok(j)) {
                const int e = 4 * map.idx(j);
                float4 o = make_float4((v[j].x - mean) * rstd, (v[j].y - mean) * rstd, (v[j].z - mean) * rstd,
                                       (v[j].w - mean) * rstd);
                if (a.has_w) {
                    const float4 wj = SP ? ld_shared4(sp.w + e)
                                      : PRE ? wr[j] : kFetchEarly ? wq[j] : ld_param(a.w + g.head + e, wv);
                    o.x *= wj.x; o.y *= wj.y; o.z *= wj.z; o.w *= wj.w;
                }
                if (a.has_b) {
                    const float4 bj = SP ? ld_shared4(sp.b + e)
                                      : PRE ? br[j] : kFetchEarly ? bq[j] : ld_param(a.b + g.head + e, bv);
                    o.x += bj.x; o.y += bj.y; o.z += bj.z; o.w += bj.w;
                }
                st_out(yb + e, o, a.y_vec);
            }
        if (own_h) {
            float o = (hv - mean) * rstd;
            if (a.has_w) o *= __ldg(a.w + wi);
            if (a.has_b) o += __ldg(a.b + wi);
            yr[wi] = o;
        }
        if (own_t) {
            float o = (tv - mean) * rstd;
            if (a.has_w) o *= __ldg(a.w + ti);
            if (a.has_b) o += __ldg(a.b + ti);
            yr[ti] = o;
        }
    }
}

// ---------------------------------------------------------------------------
// TR_PLAN_ROWS: G lanes per row inside a warp (G = 4, 8, 16), or S warps per
// row (G = 32); Q rows per CTA; K float4 slots per worker.
// ---------------------------------------------------------------------------
template <int OP, int G, int K, bool SP = false, bool RES = false>
__global__ void __launch_bounds__(max_threads_res<OP, K, RES>(), min_blocks_res<K, RES>())
    rows_cached_kernel(const RowArgs a) {
    __shared__ float4 part[2][32];
    extern __shared__ __align__(16) float sparams[];  // SP: weight (cols floats), then bias
    __shared__ __align__(8) uint64_t pbar;
    const SharedParams sp{sparams, sparams + (a.has_w ? a.cols : 0), &pbar};
    if constexpr (SP) {
        if (threadIdx.x == 0) {
            mbar_init(&pbar, 1);
            fence_barrier_init();
        }
        __syncthreads();
    }
    RowPos p;
    p.lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    int64_t row;
    if constexpr (G < 32) {
        p.W = G;
        p.w = p.lane & (G - 1);
        p.S = 1;
        p.s = 0;
        p.q = warp * (32 / G) + p.lane / G;
        row = static_cast<int64_t>(blockIdx.x) * ((blockDim.x >> 5) * (32 / G)) + p.q;
    } else {
        p.S = a.S;
        p.W = 32 * a.S;
        p.s = warp % a.S;
        p.q = warp / a.S;
        p.w = p.s * 32 + p.lane;
        row = static_cast<int64_t>(blockIdx.x) * (blockDim.x / p.W) + p.q;
    }
    const bool active = row < a.rows;
    const int64_t rr = active ? row : a.rows - 1;
    const float* xr = a.x + rr * a.cols;
    const RowGeom g = row_geom(xr, a.cols);
    const SlotMapRows map{p.W, p.w, g.nvec};
    const bool own_h = p.w < g.head, own_t = p.w < g.tail;
    float4 v[K];
    float hv, tv;
    pdl_enter();
    if constexpr (SP) {
        // the whole weight (and bias) vector, once per CTA, while the rows load
        if (threadIdx.x == 0) {
            const uint32_t bytes = static_cast<uint32_t>(a.cols) * 4u;
            mbar_arrive_expect_tx(&pbar, bytes * ((a.has_w ? 1u : 0u) + (a.has_b ? 1u : 0u)));
            if (a.has_w) bulk_g2s(sparams, a.w, bytes, &pbar);
            if (a.has_b) bulk_g2s(sparams + (a.has_w ? a.cols : 0), a.b, bytes, &pbar);
        }
    }
    // Packed rows of short stripes (G < 32 lanes, K <= 4): the norms' weight
    // (and bias) quads are requested before the row. Requested after it, they
    // would return behind the row loads that the SM's other CTAs still have
    // in flight, even as L1 hits, and hold up the epilogue.
    constexpr bool kParamsFirst = G < 32 && K <= 4 && !SP && !RES && OP != OP_SOFTMAX;
    float4 wr[K], br[K];
    if constexpr (kParamsFirst) {
        const bool wv = a.has_w && aligned16(a.w + g.head);
        const bool bv = a.has_b && aligned16(a.b + g.head);
#pragma unroll
        for (int j = 0; j < K; ++j) {
            const bool here = active && map.ok(j);
            const int e = 4 * map.idx(j);
            wr[j] = (a.has_w && here) ? ld_param(a.w + g.head + e, wv) : f4(1.0f);
            br[j] = (OP == OP_LAYERNORM && a.has_b && here) ? ld_param(a.b + g.head + e, bv) : f4(0.0f);
        }
    }
    load_stripe<OP, K>(xr, g, map, active, p.w, own_h, own_t, v, hv, tv);
    if constexpr (RES) add_residual<K>(a, rr, g, map, active, p.w, own_h, own_t, v, hv, tv);
    RowsReducer<G> red{p, part, 0};
    if constexpr (kParamsFirst) {
        cached_epilogue<OP, K, true, false>(a, a.y + rr * a.cols, g, v, hv, tv, own_h, own_t, active, p.w, map, red,
                                            wr, br, sp);
    } else {
        float4 none[K];
        cached_epilogue<OP, K, false, SP>(a, a.y + rr * a.cols, g, v, hv, tv, own_h, own_t, active, p.w, map, red,
                                          none, none, sp);
    }
    // the weight copy has landed unless the epilogue's wait gave up: then wait
    // for it once more before the CTA's shared memory goes away
    if constexpr (SP)
        if (threadIdx.x == 0) mbar_wait_bounded(&pbar, 0, a.wait_ns, nullptr);
}

// Two rows per worker group, in sequence (TR_PLAN_FLAG_TWO_ROWS): the stripes of
// both rows are loaded first, so the second row's loads are still landing while
// the first row is reduced and written. Across the device, the writes of first
// rows overlap the reads of second rows, instead of every CTA reading, then
// merging, then writing in lockstep. Group q of the CTA owns rows 2g and 2g + 1,
// g = blockIdx.x * (groups per CTA) + q. Warp rows only (G == 32).
// K = 6 (rows of up to 6144 columns at 256 threads): three CTAs, six rows per SM.
template <int K>
constexpr int pair_max_threads() {
    return K == 6 ? 256 : 512;
}
template <int K>
constexpr int pair_min_blocks() {
    return K == 6 ? 3 : 2;
}

template <int OP, int K, bool SP = false>
__global__ void __launch_bounds__(pair_max_threads<K>(), pair_min_blocks<K>()) rows_pair_kernel(const RowArgs a) {
    __shared__ float4 part[2][32];
    extern __shared__ __align__(16) float sparams[];  // SP: weight (cols floats), then bias
    __shared__ __align__(8) uint64_t pbar;
    const SharedParams sp{sparams, sparams + (a.has_w ? a.cols : 0), &pbar};
    if constexpr (SP) {
        if (threadIdx.x == 0) {
            mbar_init(&pbar, 1);
            fence_barrier_init();
        }
        __syncthreads();
    }
    RowPos p;
    p.lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    p.S = a.S;
    p.W = 32 * a.S;
    p.s = warp % a.S;
    p.q = warp / a.S;
    p.w = p.s * 32 + p.lane;
    const int64_t row0 = (static_cast<int64_t>(blockIdx.x) * (blockDim.x / p.W) + p.q) * 2;
    const bool act0 = row0 < a.rows, act1 = row0 + 1 < a.rows;
    const int64_t r0 = act0 ? row0 : a.rows - 1, r1 = act1 ? row0 + 1 : a.rows - 1;
    const float* x0 = a.x + r0 * a.cols;
    const float* x1 = a.x + r1 * a.cols;
    const RowGeom g0 = row_geom(x0, a.cols), g1 = row_geom(x1, a.cols);
    const SlotMapRows m0{p.W, p.w, g0.nvec}, m1{p.W, p.w, g1.nvec};
    const bool h0 = p.w < g0.head, t0 = p.w < g0.tail, h1 = p.w < g1.head, t1 = p.w < g1.tail;
    float4 v0[K], v1[K];
    float hv0, tv0, hv1, tv1;
    pdl_enter();
    if constexpr (SP) {
        if (threadIdx.x == 0) {
            const uint32_t bytes = static_cast<uint32_t>(a.cols) * 4u;
            mbar_arrive_expect_tx(&pbar, bytes * ((a.has_w ? 1u : 0u) + (a.has_b ? 1u : 0u)));
            if (a.has_w) bulk_g2s(sparams, a.w, bytes, &pbar);
            if (a.has_b) bulk_g2s(sparams + (a.has_w ? a.cols : 0), a.b, bytes, &pbar);
        }
    }
    load_stripe<OP, K>(x0, g0, m0, act0, p.w, h0, t0, v0, hv0, tv0);
    load_stripe<OP, K>(x1, g1, m1, act1, p.w, h1, t1, v1, hv1, tv1);
    RowsReducer<32> red{p, part, 0};
    float4 none[K];
    cached_epilogue<OP, K, false, SP>(a, a.y + r0 * a.cols, g0, v0, hv0, tv0, h0, t0, act0, p.w, m0, red, none,
                                      none, sp);
    cached_epilogue<OP, K, false, SP>(a, a.y + r1 * a.cols, g1, v1, hv1, tv1, h1, t1, act1, p.w, m1, red, none,
                                      none, sp);
    if constexpr (SP)
        if (threadIdx.x == 0) mbar_wait_bounded(&pbar, 0, a.wait_ns, nullptr);  // as in rows_cached_kernel
}

// ---------------------------------------------------------------------------
// TR_PLAN_CLUSTER: a row per cluster of C CTAs (launched with a cluster
// dimension of C). CTA rank c owns the body slots [c*seg, (c+1)*seg).
// ---------------------------------------------------------------------------
template <int OP, int K, bool RES = false>
__global__ void __launch_bounds__(max_threads_res<OP, K, RES>()) cluster_cached_kernel(const RowArgs a) {
    __shared__ float4 part[2][32];
    __shared__ float4 cpart[2];
    cg::cluster_group cl = cg::this_cluster();
    const int C = a.C;
    const int rank = static_cast<int>(cl.block_rank());
    const int64_t row = static_cast<int64_t>(blockIdx.x) / C;  // every CTA of a cluster has the same row
    const float* xr = a.x + row * a.cols;
    const RowGeom g = row_geom(xr, a.cols);
    const int seg = (g.nvec + C - 1) / C;
    const int v0 = min(g.nvec, rank * seg), v1 = min(g.nvec, v0 + seg);
    const int t = threadIdx.x;
    const SlotMapSeg map{static_cast<int>(blockDim.x), t, v0, v1};
    const bool own_h = rank == 0 && t < g.head;
    const bool own_t = rank == C - 1 && t < g.tail;
    RowPos p;
    p.w = t;
    p.W = blockDim.x;
    p.q = 0;
    p.s = t >> 5;
    p.S = blockDim.x >> 5;
    p.lane = t & 31;
    float4 v[K];
    float hv, tv;
    pdl_enter();
    load_stripe<OP, K>(xr, g, map, true, t, own_h, own_t, v, hv, tv);
    if constexpr (RES) add_residual<K>(a, row, g, map, true, t, own_h, own_t, v, hv, tv);
    ClusterReducer red{p, part, 0, cpart, 0, C};
    float4 none[K];
    cached_epilogue<OP, K>(a, a.y + row * a.cols, g, v, hv, tv, own_h, own_t, true, t, map, red, none, none);
    cl.sync();  // peers may still be reading this CTA's cpart
}

// ---------------------------------------------------------------------------
// TR_PLAN_STAGED: persistent CTAs over rows blockIdx.x, blockIdx.x + gridDim.x,
// ...; a ring of nbuf shared-memory slots, each filled by one bulk
// asynchronous copy (TMA) of a row, so every row of a CTA is requested as soon
// as a slot is free and reads overlap the writes of earlier rows. One thread
// issues the copies; the whole CTA reduces each row from registers.
// ---------------------------------------------------------------------------

// The global window copied for a row: its 16-byte-aligned body plus the
// partial 16-byte chunks holding the head and the tail, when those chunks lie
// inside the tensor (they may hold neighbouring rows' elements: x is read-only).
struct StagedWindow {
    const float* lo;  // first float copied
    int dst;          // slot float index receiving lo
    int bytes;        // multiple of 16
    int off;          // slot float index of body float4 0
    bool head_global, tail_global;  // head / tail scalars not in the slot
};
__device__ __forceinline__ StagedWindow staged_window(const float* xr, const RowGeom& g, const float* x0,
                                                      const float* x1) {
    StagedWindow w;
    const float* body = xr + g.head;
    w.off = g.head > 0 ? 4 : 0;
    const float* lo = body - w.off;
    const float* hi = body + 4 * g.nvec + (g.tail > 0 ? 4 : 0);
    w.head_global = lo < x0;
    w.tail_global = hi > x1;
    if (w.head_global) lo = body;
    if (w.tail_global) hi = body + 4 * g.nvec;
    w.lo = lo;
    w.dst = lo == body ? w.off : 0;
    w.bytes = static_cast<int>(hi - lo) * 4;
    return w;
}

// PRE (norms only): every row starts 16-byte aligned and cols % 4 == 0, so a
// worker owns the same columns in every row and keeps their weights (and
// biases) in registers for the whole kernel instead of re-reading them per row.
template <int OP, int K, bool PRE>
__global__ void __launch_bounds__(staged_max_threads<OP, K, PRE>()) staged_kernel(const RowArgs a) {
    extern __shared__ __align__(16) float ring[];
    __shared__ __align__(8) uint64_t full[kMaxRing];
    __shared__ __align__(8) uint64_t never;  // testing: a barrier nothing completes
    __shared__ float4 part[2][32];
    __shared__ volatile int s_abort;
    const int T = blockDim.x, t = threadIdx.x;
    const int nbuf = a.nbuf;
    const int64_t G = gridDim.x;
    const int64_t mine = (a.rows - blockIdx.x + G - 1) / G;  // rows blockIdx.x + i*G, i < mine
    const float* x0 = a.x;
    const float* x1 = a.x + a.rows * a.cols;
    if (t == 0) {
        for (int b = 0; b < nbuf; ++b) mbar_init(&full[b], 1);
        mbar_init(&never, 1);
        s_abort = 0;
        fence_barrier_init();
    }
    __syncthreads();
    pdl_enter();
    if ((a.debug_flags & kDebugForceTimeout) && t == 0) mbar_wait_bounded(&never, 0, 1000000LL, a.err);

    auto issue = [&](int64_t i) {  // thread 0: copy the CTA's i-th row into slot i % nbuf
        const int64_t row = blockIdx.x + i * G;
        const float* xr = a.x + row * a.cols;
        const RowGeom g = row_geom(xr, a.cols);
        const StagedWindow w = staged_window(xr, g, x0, x1);
        const int b = static_cast<int>(i % nbuf);
        float* slot = ring + static_cast<int64_t>(b) * a.slot_floats;
        if (w.bytes > 0) {
            mbar_arrive_expect_tx(&full[b], static_cast<uint32_t>(w.bytes));
            bulk_g2s(slot + w.dst, w.lo, static_cast<uint32_t>(w.bytes), &full[b]);
        } else {
            mbar_arrive(&full[b]);
        }
    };
    if (t == 0)
        for (int64_t i = 0; i < mine && i < nbuf; ++i) issue(i);

    RowPos p;
    p.w = t;
    p.W = T;
    p.q = 0;
    p.s = t >> 5;
    p.S = T >> 5;
    p.lane = t & 31;
    const float id = first_identity<OP>();
    float4 wr[K], br[K];
    if constexpr (PRE) {
        const int nvec = a.cols >> 2;
#pragma unroll
        for (int j = 0; j < K; ++j) {
            const int e = 4 * (j * T + t);
            wr[j] = f4(1.0f);
            br[j] = f4(0.0f);
            if (j * T + t < nvec) {
                if (a.has_w) wr[j] = ld_param4(a.w + e);
                if (OP == OP_LAYERNORM && a.has_b) br[j] = ld_param4(a.b + e);
            }
        }
    }
    // one reducer for all rows: its two shared buffers alternate, so a row's
    // merge never overwrites a slot the previous row's merge may still read
    RowsReducer<32> red{p, part, 0};
    for (int64_t i = 0; i < mine; ++i) {
        const int b = static_cast<int>(i % nbuf);
        const uint32_t parity = static_cast<uint32_t>((i / nbuf) & 1);
        const int64_t row = blockIdx.x + i * G;
        const float* xr = a.x + row * a.cols;
        const RowGeom g = row_geom(xr, a.cols);
        const StagedWindow w = staged_window(xr, g, x0, x1);
        const float* slot = ring + static_cast<int64_t>(b) * a.slot_floats;
        if (!mbar_wait_bounded(&full[b], parity, a.wait_ns, a.err, a.debug_flags & kDebugExpireCopies)) s_abort = 1;
        const SlotMapRows map{T, t, g.nvec};
        float4 v[K];
#pragma unroll
        for (int j = 0; j < K; ++j) {
            v[j] = f4(id);
            if (map.ok(j)) v[j] = *reinterpret_cast<const float4*>(slot + w.off + 4 * map.idx(j));
        }
        const bool own_h = t < g.head, own_t = t < g.tail;
        float hv = id, tv = id;
        if (own_h) hv = w.head_global ? ld_stream1(xr + t) : slot[w.off - g.head + t];
        if (own_t) tv = w.tail_global ? ld_stream1(xr + g.head + 4 * g.nvec + t) : slot[w.off + 4 * g.nvec + t];
        cached_epilogue<OP, K, PRE>(a, a.y + row * a.cols, g, v, hv, tv, own_h, own_t, true, t, map, red, wr, br);
        // the merge's barrier (or, for one warp, this __syncwarp) orders every
        // thread's reads of the slot, and the abort flag, before what follows
        if (p.S == 1) __syncwarp();
        if (s_abort) {
            // give up without trapping: wait for the copies still in flight, then leave
            if (t == 0)
                for (int64_t j = i; j < mine && j < i + nbuf; ++j)
                    mbar_wait_bounded(&full[j % nbuf], static_cast<uint32_t>((j / nbuf) & 1), a.wait_ns, a.err);
            return;
        }
        if (t == 0 && i + nbuf < mine) {
            fence_proxy_async_smem();
            issue(i + nbuf);
        }
    }
}

// Merge over the CTA's threads and then over the C CTAs of the cluster.
// `part` holds 2 x 32 values of T and `cpart` 2 values of T (shared memory).
template <class T>
__device__ __forceinline__ T block_cluster_merge(T v, T (*part)[32], T* cpart, int& buf, int C) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    v = warp_merge<T, 32>(v);
    if (nw > 1) {
        T* slot = part[buf];
        if (lane == 0) slot[warp] = v;
        __syncthreads();
        v = warp_merge<T, 32>(lane < nw ? slot[lane] : identity_of<T>());
    }
    if (C > 1) {
        cg::cluster_group cl = cg::this_cluster();
        T* cs = cpart + buf;
        if (threadIdx.x == 0) *cs = v;
        cl.sync();
        v = warp_merge<T, 32>(lane < C ? *cl.map_shared_rank(cs, lane) : identity_of<T>());
    }
    buf ^= 1;
    return v;
}

// ---------------------------------------------------------------------------
// TR_PLAN_STREAM: a row per C CTAs (a cluster when C > 1). Statistics are
// streamed in chunks of U float4 per thread; then the row slice is read again
// (from L2 when the working set fits) and the epilogue is written.
// ---------------------------------------------------------------------------
constexpr int kStreamU = 8;

template <int OP>
__global__ void __launch_bounds__(1024) stream_kernel(const RowArgs a) {
    using Stat = typename std::conditional<OP == OP_SOFTMAX, MaxSum,
                 typename std::conditional<OP == OP_LAYERNORM, Moments, float>::type>::type;
    __shared__ Stat part[2][32];
    __shared__ Stat cpart[2];
    int buf = 0;
    const int C = a.C;
    int rank = 0;
    if (C > 1) rank = static_cast<int>(cg::this_cluster().block_rank());
    const int64_t row = static_cast<int64_t>(blockIdx.x) / C;
    const float* xr = a.x + row * a.cols;
    float* yr = a.y + row * a.cols;
    const RowGeom g = row_geom(xr, a.cols);
    const int seg = (g.nvec + C - 1) / C;
    const int v0 = min(g.nvec, rank * seg), v1 = min(g.nvec, v0 + seg);
    const int T = blockDim.x, t = threadIdx.x;
    const bool own_h = rank == 0 && t < g.head;
    const bool own_t = rank == C - 1 && t < g.tail;
    const float* xb = xr + g.head;
    const int ti = g.head + 4 * g.nvec + t;

    pdl_enter();
    // ---- pass 1: statistics ----
    Stat st = identity_of<Stat>();
    for (int base = v0; base < v1; base += kStreamU * T) {
        float4 c[kStreamU];
#pragma unroll
        for (int u = 0; u < kStreamU; ++u) {
            const int i = base + u * T + t;
            c[u] = f4(first_identity<OP>());
            if (i < v1) c[u] = ld_stream4(xb + 4 * i);
        }
        if constexpr (OP == OP_SOFTMAX) {
            float cm = MaxOp::id();
#pragma unroll
            for (int u = 0; u < kStreamU; ++u) cm = fmaxf(cm, fmaxf(fmaxf(c[u].x, c[u].y), fmaxf(c[u].z, c[u].w)));
            const float m = fmaxf(st.m, cm);
            if (m != MaxOp::id()) {
                const float mb = mb_of(m);
                float s = st.s * ex2(mb_of(st.m) - mb);
#pragma unroll
                for (int u = 0; u < kStreamU; ++u)
                    s += (ex2(fmaf(c[u].x, kL2E, -mb)) + ex2(fmaf(c[u].y, kL2E, -mb))) +
                         (ex2(fmaf(c[u].z, kL2E, -mb)) + ex2(fmaf(c[u].w, kL2E, -mb)));
                st = MaxSum{m, s};
            }
        } else if constexpr (OP == OP_RMSNORM) {
#pragma unroll
            for (int u = 0; u < kStreamU; ++u)
                st = fmaf(c[u].x, c[u].x, fmaf(c[u].y, c[u].y, fmaf(c[u].z, c[u].z, fmaf(c[u].w, c[u].w, st))));
        } else {
            // chunk moments by two passes over the registers, then a Chan merge
            int cnt = 0;
            float sm = 0.0f;
#pragma unroll
            for (int u = 0; u < kStreamU; ++u)
                if (base + u * T + t < v1) {
                    cnt += 4;
                    sm += (c[u].x + c[u].y) + (c[u].z + c[u].w);
                }
            if (cnt > 0) {
                const float n = static_cast<float>(cnt);
                const float mu = sm / n;
                float m2 = 0.0f;
#pragma unroll
                for (int u = 0; u < kStreamU; ++u)
                    if (base + u * T + t < v1) {
                        const float dx = c[u].x - mu, dy = c[u].y - mu, dz = c[u].z - mu, dw = c[u].w - mu;
                        m2 = fmaf(dx, dx, fmaf(dy, dy, fmaf(dz, dz, fmaf(dw, dw, m2))));
                    }
                st = mo_merge(st, Moments{n, mu, m2});
            }
        }
    }
    float hv = 0.0f, tv = 0.0f;
    if (own_h) hv = ld_stream1(xr + t);
    if (own_t) tv = ld_stream1(xb + 4 * g.nvec + t);
    if constexpr (OP == OP_SOFTMAX) {
        if (own_h) st = ms_merge(st, ms_single(hv));
        if (own_t) st = ms_merge(st, ms_single(tv));
    } else if constexpr (OP == OP_RMSNORM) {
        st = fmaf(hv, hv, fmaf(tv, tv, st));
    } else {
        if (own_h) st = mo_merge(st, Moments{1.0f, hv, 0.0f});
        if (own_t) st = mo_merge(st, Moments{1.0f, tv, 0.0f});
    }
    st = block_cluster_merge<Stat>(st, part, cpart, buf, C);

    // ---- pass 2: epilogue over the re-read slice ----
    float scale, shift;  // norms: y = (x - shift) * scale [* w + b]; softmax: y = 2^(x*log2e - mb) * scale
    float mb = 0.0f;
    if constexpr (OP == OP_SOFTMAX) {
        mb = mb_of(st.m);
        scale = 1.0f / st.s;
        shift = 0.0f;
    } else if constexpr (OP == OP_RMSNORM) {
        scale = rsqrtf(fmaf(st, a.inv_cols, a.eps));
        shift = 0.0f;
    } else {
        scale = rsqrtf(fmaf(st.m2, a.inv_cols, a.eps));
        shift = st.mean;
    }
    const bool wv = a.has_w && aligned16(a.w + g.head);
    const bool bv = a.has_b && aligned16(a.b + g.head);
    auto apply = [&](float x, int col) -> float {
        if constexpr (OP == OP_SOFTMAX) {
            return ex2(fmaf(x, kL2E, -mb)) * scale;
        } else {
            float o = (x - shift) * scale;
            if (a.has_w) o *= __ldg(a.w + col);
            if (OP == OP_LAYERNORM && a.has_b) o += __ldg(a.b + col);
            return o;
        }
    };
    for (int base = v0; base < v1; base += kStreamU * T) {
        float4 c[kStreamU];
#pragma unroll
        for (int u = 0; u < kStreamU; ++u) {
            const int i = base + u * T + t;
            if (i < v1) c[u] = ld_stream4(xb + 4 * i);
        }
#pragma unroll
        for (int u = 0; u < kStreamU; ++u) {
            const int i = base + u * T + t;
            if (i < v1) {
                float4 o;
                if constexpr (OP == OP_SOFTMAX) {
                    o = make_float4(ex2(fmaf(c[u].x, kL2E, -mb)) * scale, ex2(fmaf(c[u].y, kL2E, -mb)) * scale,
                                    ex2(fmaf(c[u].z, kL2E, -mb)) * scale, ex2(fmaf(c[u].w, kL2E, -mb)) * scale);
                } else {
                    o = make_float4((c[u].x - shift) * scale, (c[u].y - shift) * scale,
                                    (c[u].z - shift) * scale, (c[u].w - shift) * scale);
                    if (a.has_w) {
                        const float4 wq = ld_param(a.w + g.head + 4 * i, wv);
                        o.x *= wq.x; o.y *= wq.y; o.z *= wq.z; o.w *= wq.w;
                    }
                    if constexpr (OP == OP_LAYERNORM) {
                        if (a.has_b) {
                            const float4 bq = ld_param(a.b + g.head + 4 * i, bv);
                            o.x += bq.x; o.y += bq.y; o.z += bq.z; o.w += bq.w;
                        }
                    }
                }
                st_out(yr + g.head + 4 * i, o, a.y_vec);
            }
        }
    }
    if (own_h) yr[t] = apply(hv, t);
    if (own_t) yr[ti] = apply(tv, ti);
    if (C > 1) cg::this_cluster().sync();  // peers may still read this CTA's cpart
}

// ---------------------------------------------------------------------------
// TR_PLAN_XENT: cross-entropy, one streaming pass per row (the row is read
// once; nothing is written but the loss). G lanes per row (G < 32) or S warps
// per row (G == 32); Q rows per CTA; chunks of K float4 per worker.
// ---------------------------------------------------------------------------
template <int G, int K>
__global__ void __launch_bounds__(1024) xent_kernel(const RowArgs a) {
    __shared__ MaxSum part[2][32];
    RowPos p;
    p.lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    int64_t row;
    if constexpr (G < 32) {
        p.W = G;
        p.w = p.lane & (G - 1);
        p.S = 1;
        p.s = 0;
        p.q = warp * (32 / G) + p.lane / G;
        row = static_cast<int64_t>(blockIdx.x) * ((blockDim.x >> 5) * (32 / G)) + p.q;
    } else {
        p.S = a.S;
        p.W = 32 * a.S;
        p.s = warp % a.S;
        p.q = warp / a.S;
        p.w = p.s * 32 + p.lane;
        row = static_cast<int64_t>(blockIdx.x) * (blockDim.x / p.W) + p.q;
    }
    const bool active = row < a.rows;
    const int64_t rr = active ? row : a.rows - 1;
    const float* xr = a.x + rr * a.cols;
    const RowGeom g = row_geom(xr, a.cols);
    const float* xb = xr + g.head;
    MaxSum st{MaxOp::id(), 0.0f};
    pdl_enter();
    if (active) {
        for (int base = 0; base < g.nvec; base += K * p.W) {
            float4 c[K];
#pragma unroll
            for (int j = 0; j < K; ++j) {
                const int i = base + j * p.W + p.w;
                c[j] = f4(MaxOp::id());
                if (i < g.nvec) c[j] = ld_stream4(xb + 4 * i);
            }
            float cm = MaxOp::id();
#pragma unroll
            for (int j = 0; j < K; ++j) cm = fmaxf(cm, fmaxf(fmaxf(c[j].x, c[j].y), fmaxf(c[j].z, c[j].w)));
            const float m = fmaxf(st.m, cm);
            if (m != MaxOp::id()) {
                const float mb = mb_of(m);
                float s = st.s * ex2(mb_of(st.m) - mb);
#pragma unroll
                for (int j = 0; j < K; ++j)
                    s += (ex2(fmaf(c[j].x, kL2E, -mb)) + ex2(fmaf(c[j].y, kL2E, -mb))) +
                         (ex2(fmaf(c[j].z, kL2E, -mb)) + ex2(fmaf(c[j].w, kL2E, -mb)));
                st = MaxSum{m, s};
            }
        }
        if (p.w < g.head) st = ms_merge(st, ms_single(ld_stream1(xr + p.w)));
        if (p.w < g.tail) st = ms_merge(st, ms_single(ld_stream1(xb + 4 * g.nvec + p.w)));
    }
    // merge over the row's workers
    if constexpr (G < 32) {
        st = warp_merge<MaxSum, G>(st);
    } else {
        st = warp_merge<MaxSum, 32>(st);
        if (p.S > 1) {
            if (p.lane == 0) part[0][p.q * p.S + p.s] = st;
            __syncthreads();
            st = warp_merge<MaxSum, 32>(p.lane < p.S ? part[0][p.q * p.S + p.lane] : identity_of<MaxSum>());
        }
    }
    if (active && p.w == 0) {
        // log(sum e^(x-m)) + m = ln2 * (log2(s) + m*log2e), s scaled by 2^(-m*log2e)
        const float lse = (log2f(st.s) + mb_of(st.m)) * kLN2;
        const int64_t label = a.labels[rr];
        const float sel = (label >= 0 && label < a.cols) ? __ldg(xr + label) : 0.0f;
        a.loss[rr] = lse - sel;
    }
}

// ---------------------------------------------------------------------------
// Standalone row reductions (sum, max, min, min and max together): one
// streaming pass per row like the cross-entropy kernel (TR_PLAN_XENT shapes: G
// lanes per row or S warps per row, Q rows per CTA, chunks of K float4 per
// worker); one value per row (two for min/max). Max and min are the hardware
// maxNum/minNum (NaN operands skipped); the sum is a tree in worker order.
// ---------------------------------------------------------------------------
// The identity of these folds is NaN: maxNum/minNum skip it, so a row (or a
// padding lane) contributes nothing, and the result is NaN only when every
// element of the row is NaN.
struct MinMax {
    float lo, hi;
};
__device__ __forceinline__ MinMax merge(MinMax a, MinMax b) { return MinMax{fminf(a.lo, b.lo), fmaxf(a.hi, b.hi)}; }
__device__ __forceinline__ MinMax shfl_xor(MinMax v, int o) {
    return MinMax{__shfl_xor_sync(kFull, v.lo, o), __shfl_xor_sync(kFull, v.hi, o)};
}
struct RMax {
    float v;
};
__device__ __forceinline__ RMax merge(RMax a, RMax b) { return RMax{fmaxf(a.v, b.v)}; }
__device__ __forceinline__ RMax shfl_xor(RMax v, int o) { return RMax{__shfl_xor_sync(kFull, v.v, o)}; }
struct RMin {
    float v;
};
__device__ __forceinline__ RMin merge(RMin a, RMin b) { return RMin{fminf(a.v, b.v)}; }
__device__ __forceinline__ RMin shfl_xor(RMin v, int o) { return RMin{__shfl_xor_sync(kFull, v.v, o)}; }
template <>
__device__ __forceinline__ MinMax identity_of<MinMax>() {
    return MinMax{__int_as_float(0x7fc00000), __int_as_float(0x7fc00000)};
}
template <>
__device__ __forceinline__ RMax identity_of<RMax>() { return RMax{__int_as_float(0x7fc00000)}; }
template <>
__device__ __forceinline__ RMin identity_of<RMin>() { return RMin{__int_as_float(0x7fc00000)}; }

template <int OP>
using ReduceStat = typename std::conditional<
    OP == OP_RSUM, float,
    typename std::conditional<OP == OP_RMAX, RMax,
                              typename std::conditional<OP == OP_RMIN, RMin, MinMax>::type>::type>::type;

template <int OP>
__device__ __forceinline__ ReduceStat<OP> reduce_elem(ReduceStat<OP> s, float v) {
    if constexpr (OP == OP_RSUM) {
        return s + v;
    } else if constexpr (OP == OP_RMAX) {
        return RMax{fmaxf(s.v, v)};
    } else if constexpr (OP == OP_RMIN) {
        return RMin{fminf(s.v, v)};
    } else {
        return MinMax{fminf(s.lo, v), fmaxf(s.hi, v)};
    }
}

template <int OP, int G, int K>
__global__ void __launch_bounds__(1024) reduce_kernel(const RowArgs a) {
    using Stat = ReduceStat<OP>;
    __shared__ float4 part[2][32];
    RowPos p;
    p.lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    int64_t row;
    if constexpr (G < 32) {
        p.W = G;
        p.w = p.lane & (G - 1);
        p.S = 1;
        p.s = 0;
        p.q = warp * (32 / G) + p.lane / G;
        row = static_cast<int64_t>(blockIdx.x) * ((blockDim.x >> 5) * (32 / G)) + p.q;
    } else {
        p.S = a.S;
        p.W = 32 * a.S;
        p.s = warp % a.S;
        p.q = warp / a.S;
        p.w = p.s * 32 + p.lane;
        row = static_cast<int64_t>(blockIdx.x) * (blockDim.x / p.W) + p.q;
    }
    const bool active = row < a.rows;
    const int64_t rr = active ? row : a.rows - 1;
    const float* xr = a.x + rr * a.cols;
    const RowGeom g = row_geom(xr, a.cols);
    const float* xb = xr + g.head;
    Stat st = identity_of<Stat>();
    pdl_enter();
    if (active) {
        for (int base = 0; base < g.nvec; base += K * p.W) {
            float4 c[K];
            bool ok[K];
#pragma unroll
            for (int j = 0; j < K; ++j) {
                const int i = base + j * p.W + p.w;
                ok[j] = i < g.nvec;
                if (ok[j]) c[j] = ld_stream4(xb + 4 * i);
            }
#pragma unroll
            for (int j = 0; j < K; ++j)
                if (ok[j]) {
                    if constexpr (OP == OP_RSUM) {
                        st += (c[j].x + c[j].y) + (c[j].z + c[j].w);
                    } else {
                        st = reduce_elem<OP>(reduce_elem<OP>(st, c[j].x), c[j].y);
                        st = reduce_elem<OP>(reduce_elem<OP>(st, c[j].z), c[j].w);
                    }
                }
        }
        if (p.w < g.head) st = reduce_elem<OP>(st, ld_stream1(xr + p.w));
        if (p.w < g.tail) st = reduce_elem<OP>(st, ld_stream1(xb + 4 * g.nvec + p.w));
    }
    int buf = 0;
    st = cta_row_merge<Stat, G>(st, p, part, buf);
    if (active && p.w == 0) {
        if constexpr (OP == OP_RSUM) {
            a.loss[rr] = st;
        } else if constexpr (OP == OP_RMINMAX) {
            a.loss[rr] = st.lo;
            a.out2[rr] = st.hi;
        } else {
            a.loss[rr] = st.v;
        }
    }
}

}  // namespace tr
