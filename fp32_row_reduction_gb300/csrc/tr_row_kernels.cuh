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
// about 90 registers (at most 512 threads per CTA); LayerNorm's 32-float
// stripe needs more than the 64 registers a 1024-thread CTA allows.
template <int OP, int K>
constexpr int max_threads_for() {
    return K >= 16 ? 512 : (K >= 8 && OP == OP_LAYERNORM) ? 768 : 1024;
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

// Reduce over the workers of one row.
template <int G>
struct RowsReducer {
    RowPos p;
    float (*part)[32];
    int buf;
    template <class R>
    __device__ __forceinline__ float operator()(float v, R) {
        return cta_row_allreduce<R, G>(v, p, part, buf);
    }
};
struct ClusterReducer {
    float (*part)[32];
    int buf;
    float* cpart;
    int cbuf;
    int C;
    template <class R>
    __device__ __forceinline__ float operator()(float v, R) {
        v = cta_allreduce<R>(v, part, buf);
        return cluster_allreduce<R>(v, cpart, cbuf, C);
    }
};

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

// The three cached epilogues. Every worker of the row calls this uniformly
// (reductions may contain barriers); only stores are predicated on `active`.
template <int OP, int K, class Map, class Red>
__device__ __forceinline__ void cached_epilogue(const RowArgs& a, float* yr, const RowGeom& g, float4 (&v)[K],
                                                float hv, float tv, bool own_h, bool own_t, bool active, int wi,
                                                const Map& map, Red& red) {
    float* yb = yr + g.head;
    const int ti = g.head + 4 * g.nvec + wi;  // column of this worker's tail scalar
    if constexpr (OP == OP_SOFTMAX) {
        // m = max; e = exp(x - m) computed as 2^(x*log2e - m*log2e) with one FMA;
        // y = e * (1/sum e). Missing slots hold -inf, so they contribute e = 0.
        float m = fmaxf(hv, tv);
#pragma unroll
        for (int j = 0; j < K; ++j) m = fmaxf(m, fmaxf(fmaxf(v[j].x, v[j].y), fmaxf(v[j].z, v[j].w)));
        m = red(m, MaxOp{});
        const float mb = mb_of(m);
        float s = 0.0f;
#pragma unroll
        for (int j = 0; j < K; ++j) {
            v[j].x = ex2(fmaf(v[j].x, kL2E, -mb));
            v[j].y = ex2(fmaf(v[j].y, kL2E, -mb));
            v[j].z = ex2(fmaf(v[j].z, kL2E, -mb));
            v[j].w = ex2(fmaf(v[j].w, kL2E, -mb));
            s += (v[j].x + v[j].y) + (v[j].z + v[j].w);
        }
        hv = ex2(fmaf(hv, kL2E, -mb));
        tv = ex2(fmaf(tv, kL2E, -mb));
        s += hv + tv;
        s = red(s, SumOp{});
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
        // r = sqrt(sum x^2 / N + eps); y = x * (1/r) * w. Missing slots hold 0.
        float ss = fmaf(hv, hv, tv * tv);
#pragma unroll
        for (int j = 0; j < K; ++j)
            ss = fmaf(v[j].x, v[j].x, fmaf(v[j].y, v[j].y, fmaf(v[j].z, v[j].z, fmaf(v[j].w, v[j].w, ss))));
        ss = red(ss, SumOp{});
        const float rstd = rsqrtf(fmaf(ss, a.inv_cols, a.eps));
        if (!active) return;
        const bool wv = a.has_w && aligned16(a.w + g.head);
#pragma unroll
        for (int j = 0; j < K; ++j)
            if (map.ok(j)) {
                const int e = 4 * map.idx(j);
                float4 o = make_float4(v[j].x * rstd, v[j].y * rstd, v[j].z * rstd, v[j].w * rstd);
                if (a.has_w) {
                    const float4 wq = ld_param(a.w + g.head + e, wv);
                    o.x *= wq.x; o.y *= wq.y; o.z *= wq.z; o.w *= wq.w;
                }
                st_out(yb + e, o, a.y_vec);
            }
        if (own_h) yr[wi] = hv * rstd * (a.has_w ? __ldg(a.w + wi) : 1.0f);
        if (own_t) yr[ti] = tv * rstd * (a.has_w ? __ldg(a.w + ti) : 1.0f);
    } else if constexpr (OP == OP_LAYERNORM) {
        // mean = sum x / N; c = x - mean; var = sum c^2 / N (second pass over the
        // cached stripe, no cancellation); y = c * rsqrt(var + eps) * gamma + beta.
        float sm = hv + tv;
#pragma unroll
        for (int j = 0; j < K; ++j) sm += (v[j].x + v[j].y) + (v[j].z + v[j].w);
        sm = red(sm, SumOp{});
        const float mean = sm * a.inv_cols;
        float sq = 0.0f;
#pragma unroll
        for (int j = 0; j < K; ++j) {
            if (map.ok(j)) {
                v[j].x -= mean; v[j].y -= mean; v[j].z -= mean; v[j].w -= mean;
            } else {
                v[j] = f4(0.0f);
            }
            sq = fmaf(v[j].x, v[j].x, fmaf(v[j].y, v[j].y, fmaf(v[j].z, v[j].z, fmaf(v[j].w, v[j].w, sq))));
        }
        hv = own_h ? hv - mean : 0.0f;
        tv = own_t ? tv - mean : 0.0f;
        sq = fmaf(hv, hv, fmaf(tv, tv, sq));
        sq = red(sq, SumOp{});
        const float rstd = rsqrtf(fmaf(sq, a.inv_cols, a.eps));
        if (!active) return;
        const bool wv = a.has_w && aligned16(a.w + g.head);
        const bool bv = a.has_b && aligned16(a.b + g.head);
#pragma unroll
        for (int j = 0; j < K; ++j)
            if (map.ok(j)) {
                const int e = 4 * map.idx(j);
                float4 o = make_float4(v[j].x * rstd, v[j].y * rstd, v[j].z * rstd, v[j].w * rstd);
                if (a.has_w) {
                    const float4 wq = ld_param(a.w + g.head + e, wv);
                    o.x *= wq.x; o.y *= wq.y; o.z *= wq.z; o.w *= wq.w;
                }
                if (a.has_b) {
                    const float4 bq = ld_param(a.b + g.head + e, bv);
                    o.x += bq.x; o.y += bq.y; o.z += bq.z; o.w += bq.w;
                }
                st_out(yb + e, o, a.y_vec);
            }
        if (own_h) {
            float o = hv * rstd;
            if (a.has_w) o *= __ldg(a.w + wi);
            if (a.has_b) o += __ldg(a.b + wi);
            yr[wi] = o;
        }
        if (own_t) {
            float o = tv * rstd;
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
template <int OP, int G, int K>
__global__ void __launch_bounds__(max_threads_for<OP, K>()) rows_cached_kernel(const RowArgs a) {
    __shared__ float part[2][32];
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
    load_stripe<OP, K>(xr, g, map, active, p.w, own_h, own_t, v, hv, tv);
    RowsReducer<G> red{p, part, 0};
    cached_epilogue<OP, K>(a, a.y + rr * a.cols, g, v, hv, tv, own_h, own_t, active, p.w, map, red);
}

// ---------------------------------------------------------------------------
// TR_PLAN_CLUSTER: a row per cluster of C CTAs (launched with a cluster
// dimension of C). CTA rank c owns the body slots [c*seg, (c+1)*seg).
// ---------------------------------------------------------------------------
template <int OP, int K>
__global__ void __launch_bounds__(max_threads_for<OP, K>()) cluster_cached_kernel(const RowArgs a) {
    __shared__ float part[2][32];
    __shared__ float cpart[2];
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
    float4 v[K];
    float hv, tv;
    load_stripe<OP, K>(xr, g, map, true, t, own_h, own_t, v, hv, tv);
    ClusterReducer red{part, 0, cpart, 0, C};
    cached_epilogue<OP, K>(a, a.y + row * a.cols, g, v, hv, tv, own_h, own_t, true, t, map, red);
    cl.sync();  // peers may still be reading this CTA's cpart
}

// ---------------------------------------------------------------------------
// Merges of partial statistics for the streaming plans.
// ---------------------------------------------------------------------------

// (m, s): m is the max of the elements seen and s = sum of 2^(x*log2e - mb(m))
// with mb(m) = RN(m * log2e). Rescaling by 2^(mb(m_old) - mb(m_new)) keeps every
// partial sum relative to the same rounded offset its terms were computed with.
struct MaxSum {
    float m, s;
};
__device__ __forceinline__ MaxSum ms_merge(MaxSum a, MaxSum b) {
    const float m = fmaxf(a.m, b.m);
    if (m == MaxOp::id()) return MaxSum{m, 0.0f};
    const float mb = mb_of(m);
    return MaxSum{m, a.s * ex2(mb_of(a.m) - mb) + b.s * ex2(mb_of(b.m) - mb)};
}
// one element x as a (m, s) pair
__device__ __forceinline__ MaxSum ms_single(float x) { return MaxSum{x, ex2(fmaf(x, kL2E, -mb_of(x)))}; }
// (n, mean, M2) merged as in Chan, Golub and LeVeque, "Updating formulae and a
// pairwise algorithm for computing sample variances" (1979).
struct Moments {
    float n, mean, m2;
};
__device__ __forceinline__ Moments mo_merge(Moments a, Moments b) {
    const float n = a.n + b.n;
    if (n == 0.0f) return Moments{0.0f, 0.0f, 0.0f};
    const float d = b.mean - a.mean;
    const float fb = b.n / n;
    return Moments{n, fmaf(d, fb, a.mean), a.m2 + b.m2 + d * d * a.n * fb};
}

__device__ __forceinline__ MaxSum shfl_xor(MaxSum v, int o) {
    return MaxSum{__shfl_xor_sync(kFull, v.m, o), __shfl_xor_sync(kFull, v.s, o)};
}
__device__ __forceinline__ Moments shfl_xor(Moments v, int o) {
    return Moments{__shfl_xor_sync(kFull, v.n, o), __shfl_xor_sync(kFull, v.mean, o),
                   __shfl_xor_sync(kFull, v.m2, o)};
}
__device__ __forceinline__ MaxSum merge(MaxSum a, MaxSum b) { return ms_merge(a, b); }
__device__ __forceinline__ Moments merge(Moments a, Moments b) { return mo_merge(a, b); }
__device__ __forceinline__ float merge(float a, float b) { return a + b; }
__device__ __forceinline__ float shfl_xor(float v, int o) { return __shfl_xor_sync(kFull, v, o); }

template <class T>
__device__ __forceinline__ T identity_of();
template <>
__device__ __forceinline__ float identity_of<float>() { return 0.0f; }
template <>
__device__ __forceinline__ MaxSum identity_of<MaxSum>() { return MaxSum{MaxOp::id(), 0.0f}; }
template <>
__device__ __forceinline__ Moments identity_of<Moments>() { return Moments{0.0f, 0.0f, 0.0f}; }

template <class T, int WIDTH>
__device__ __forceinline__ T warp_merge(T v) {
#pragma unroll
    for (int o = WIDTH / 2; o > 0; o >>= 1) v = merge(v, shfl_xor(v, o));
    return v;
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

}  // namespace tr
