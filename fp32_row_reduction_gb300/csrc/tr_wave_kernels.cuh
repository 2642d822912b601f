// TR_PLAN_WAVE: rows whose 16-byte-aligned body fits 256 threads x K slots,
// all resident in one wave, both reduction policies.
//
// Mapping ("TIRx Metal reduction lowering" §4.4, blocked-cyclic ownership with
// V = 4): a 256-thread CTA serves R consecutive rows; thread t owns the
// 16-byte slots t, t + 256, ..., t + 256 (K - 1) of EVERY one of its rows, so
// the same thread sees the same columns R times. That is what the norms need:
// a weight (and bias) quad is loaded once per thread and applied to R rows,
// which divides the epilogue's L1 parameter traffic by R, the cost that keeps
// one-row-per-thread norm kernels below the copy bandwidth at 768 x 6144.
//
// The layout is also the OT-1024 leaf layout: the slots t + 256 j, j = 0..K-1,
// are the columns 1024 j + 4 t .. 1024 j + 4 t + 3, i.e. the leaves 4t .. 4t+3,
// each folded over j in increasing column order. The ordered policy therefore
// runs in the same kernel with IEEE round-to-nearest steps, the fixed tree
// above the leaves (quad pairing, xor butterfly 16..1, the fixed top over the
// eight warps) and the library's own exp, and gives the bits of every other
// OT-1024 realisation. The unordered policy uses the same tree shape with
// contracted arithmetic and the hardware exp2.
//
// Requirements (checked by the plan selector): cols % 4 == 0, x 16-byte
// aligned, cols <= 1024 K (y at another 16-byte phase takes scalar stores). All loads of a CTA are issued before any
// reduction; every CTA of the grid is resident at once when the plan is chosen
// for a single wave.
#pragma once

#include <type_traits>

#include "tr_device.cuh"
#include "tr_internal.h"
#include "tr_ot.cuh"

namespace tr {
namespace wave {

constexpr int kThreads = 256;

// Resident CTAs per SM each instantiation is compiled for (register budget of
// 4 K R cached floats plus addresses and statistics): K = 6 gives 6, 3 and 2
// CTAs for R = 1, 2, 3, i.e. 912 rows resident on 152 SMs in every case.
template <int K, int R>
constexpr int min_blocks() {
    return K * R <= 4 ? 8 : K * R <= 6 ? 6 : K * R <= 8 ? 4 : K * R <= 12 ? 3 : K * R <= 18 ? 2 : 1;
}

// Reducers. The ordered ones round every step; max is the hardware maxNum in
// both policies (see the ordered kernels: it changes no output bit).
struct AddU {
    static __device__ __forceinline__ float f(float a, float b) { return a + b; }
};
struct AddO {
    static __device__ __forceinline__ float f(float a, float b) { return __fadd_rn(a, b); }
};
struct MaxR {
    static __device__ __forceinline__ float f(float a, float b) { return fmaxf(a, b); }
};

// The tree above each thread's value for R rows at once: xor butterfly with
// offsets 16, 8, 4, 2, 1, one shared-memory exchange of the 8 warp values
// (one barrier for all R rows), then ((p0+p1)+(p2+p3)) + ((p4+p5)+(p6+p7)),
// evaluated identically by every thread. `part` is this tree's own [R][8]
// slot block, so consecutive trees never share a slot.
template <class Rd, int R>
__device__ __forceinline__ void tree_rows(float (&v)[R], float (*part)[8]) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1)
#pragma unroll
        for (int r = 0; r < R; ++r) v[r] = Rd::f(v[r], __shfl_xor_sync(kFull, v[r], o));
    if ((threadIdx.x & 31) == 0)
#pragma unroll
        for (int r = 0; r < R; ++r) part[r][threadIdx.x >> 5] = v[r];
    __syncthreads();
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const float4 lo = *reinterpret_cast<const float4*>(&part[r][0]);
        const float4 hi = *reinterpret_cast<const float4*>(&part[r][4]);
        v[r] = Rd::f(Rd::f(Rd::f(lo.x, lo.y), Rd::f(lo.z, lo.w)), Rd::f(Rd::f(hi.x, hi.y), Rd::f(hi.z, hi.w)));
    }
}

// A thread's value from its four leaves of one row: (l0 + l1) + (l2 + l3).
template <class Rd>
__device__ __forceinline__ float quad_top(float4 l) {
    return Rd::f(Rd::f(l.x, l.y), Rd::f(l.z, l.w));
}

__device__ __forceinline__ float4 param4(const float* p, bool vec) {
    if (vec) return ld_param4(p);
    return make_float4(__ldg(p), __ldg(p + 1), __ldg(p + 2), __ldg(p + 3));
}

// y rows may sit at another 16-byte phase than x rows: then scalar stores.
__device__ __forceinline__ void store4(float* p, float4 o, bool vec) {
    if (vec) {
        st4(p, o);
    } else {
        p[0] = o.x;
        p[1] = o.y;
        p[2] = o.z;
        p[3] = o.w;
    }
}

// One group of R rows starting at row0. `part` holds two [R][8] slot blocks;
// the group's trees use part[tb], part[tb ^ 1], ... alternately, continuing
// from the previous group (the caller passes the next block index in tb).
template <int OP, bool ORD, int K, int R>
__device__ __forceinline__ void wave_group(const RowArgs& a, int64_t row0, float (*part)[R][8], int& tb) {
    using Add = typename std::conditional<ORD, AddO, AddU>::type;
    const int t = threadIdx.x;
    const int nvec = a.cols >> 2;
    // slots past the end of the row hold the reducer's identity (folded last,
    // where they change no bit of an ordered leaf)
    bool okj[K];
#pragma unroll
    for (int j = 0; j < K; ++j) okj[j] = t + kThreads * j < nvec;
    const float kId = OP == OP_SOFTMAX ? -__int_as_float(0x7f800000) : 0.0f;
    float4 v[R][K];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int64_t row = min(row0 + r, a.rows - 1);  // rows past the end repeat the last (not stored)
        const float* xr = a.x + row * a.cols + 4 * t;
#pragma unroll
        for (int j = 0; j < K; ++j) v[r][j] = okj[j] ? ld_stream4(xr + 4 * kThreads * j) : make_float4(kId, kId, kId, kId);
    }
    const float n = a.cols_f;

    if constexpr (OP == OP_SOFTMAX) {
        float m[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            float4 l = v[r][0];
#pragma unroll
            for (int j = 1; j < K; ++j) {
                l.x = fmaxf(l.x, v[r][j].x);
                l.y = fmaxf(l.y, v[r][j].y);
                l.z = fmaxf(l.z, v[r][j].z);
                l.w = fmaxf(l.w, v[r][j].w);
            }
            m[r] = quad_top<MaxR>(l);
        }
        tree_rows<MaxR, R>(m, part[tb]);
        tb ^= 1;
        float s[R];
        if constexpr (ORD) {
            // e = exp_ot(x - m) in place. The differences of a finite row lie in
            // (-86, 0] almost always: then the whole thread takes the branch-free
            // form; otherwise (a huge spread, infinities, NaN) every element
            // takes the general form. Padding slots stay 0.
            bool fast = true;
#pragma unroll
            for (int r = 0; r < R; ++r)
#pragma unroll
                for (int j = 0; j < K; ++j)
                    if (okj[j]) {
                        v[r][j].x = __fsub_rn(v[r][j].x, m[r]);
                        v[r][j].y = __fsub_rn(v[r][j].y, m[r]);
                        v[r][j].z = __fsub_rn(v[r][j].z, m[r]);
                        v[r][j].w = __fsub_rn(v[r][j].w, m[r]);
                        fast &= ordered::exp_ot_in_fast_range(v[r][j].x) & ordered::exp_ot_in_fast_range(v[r][j].y) &
                                ordered::exp_ot_in_fast_range(v[r][j].z) & ordered::exp_ot_in_fast_range(v[r][j].w);
                    }
            if (fast) {
#pragma unroll
                for (int r = 0; r < R; ++r)
#pragma unroll
                    for (int j = 0; j < K; ++j)
                        if (okj[j]) {
                            v[r][j].x = ordered::exp_ot_fast(v[r][j].x);
                            v[r][j].y = ordered::exp_ot_fast(v[r][j].y);
                            v[r][j].z = ordered::exp_ot_fast(v[r][j].z);
                            v[r][j].w = ordered::exp_ot_fast(v[r][j].w);
                        }
            } else {
#pragma unroll
                for (int r = 0; r < R; ++r)
#pragma unroll
                    for (int j = 0; j < K; ++j)
                        if (okj[j]) {
                            v[r][j].x = ordered::exp_ot(v[r][j].x);
                            v[r][j].y = ordered::exp_ot(v[r][j].y);
                            v[r][j].z = ordered::exp_ot(v[r][j].z);
                            v[r][j].w = ordered::exp_ot(v[r][j].w);
                        }
            }
#pragma unroll
            for (int j = 0; j < K; ++j)
                if (!okj[j])
#pragma unroll
                    for (int r = 0; r < R; ++r) v[r][j] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        } else {
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const float mb = mb_of(m[r]);
#pragma unroll
                for (int j = 0; j < K; ++j) {  // padding: ex2(-inf) = 0
                    v[r][j].x = ex2(fmaf(v[r][j].x, kL2E, -mb));
                    v[r][j].y = ex2(fmaf(v[r][j].y, kL2E, -mb));
                    v[r][j].z = ex2(fmaf(v[r][j].z, kL2E, -mb));
                    v[r][j].w = ex2(fmaf(v[r][j].w, kL2E, -mb));
                }
            }
        }
#pragma unroll
        for (int r = 0; r < R; ++r) {
            float4 l = v[r][0];
#pragma unroll
            for (int j = 1; j < K; ++j) {
                l.x = Add::f(l.x, v[r][j].x);
                l.y = Add::f(l.y, v[r][j].y);
                l.z = Add::f(l.z, v[r][j].z);
                l.w = Add::f(l.w, v[r][j].w);
            }
            s[r] = quad_top<Add>(l);
        }
        tree_rows<Add, R>(s, part[tb]);
        tb ^= 1;
#pragma unroll
        for (int r = 0; r < R; ++r) {
            if (row0 + r >= a.rows) break;
            const float inv = ORD ? __fdiv_rn(1.0f, s[r]) : 1.0f / s[r];
            float* yr = a.y + (row0 + r) * a.cols + 4 * t;
#pragma unroll
            for (int j = 0; j < K; ++j)
                if (okj[j])
                    store4(yr + 4 * kThreads * j,
                        ORD ? make_float4(__fmul_rn(v[r][j].x, inv), __fmul_rn(v[r][j].y, inv),
                                          __fmul_rn(v[r][j].z, inv), __fmul_rn(v[r][j].w, inv))
                            : make_float4(v[r][j].x * inv, v[r][j].y * inv, v[r][j].z * inv, v[r][j].w * inv),
                        a.y_vec);
        }
    } else if constexpr (OP == OP_RMSNORM) {
        float ss[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            if constexpr (ORD) {
                float4 l = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
                for (int j = 0; j < K; ++j) {
                    l.x = __fadd_rn(l.x, __fmul_rn(v[r][j].x, v[r][j].x));
                    l.y = __fadd_rn(l.y, __fmul_rn(v[r][j].y, v[r][j].y));
                    l.z = __fadd_rn(l.z, __fmul_rn(v[r][j].z, v[r][j].z));
                    l.w = __fadd_rn(l.w, __fmul_rn(v[r][j].w, v[r][j].w));
                }
                ss[r] = quad_top<AddO>(l);
            } else {
                float acc = 0.0f;
#pragma unroll
                for (int j = 0; j < K; ++j)
                    acc = fmaf(v[r][j].x, v[r][j].x,
                               fmaf(v[r][j].y, v[r][j].y, fmaf(v[r][j].z, v[r][j].z, fmaf(v[r][j].w, v[r][j].w, acc))));
                ss[r] = acc;
            }
        }
        tree_rows<Add, R>(ss, part[tb]);
        tb ^= 1;
        float sc[R];
#pragma unroll
        for (int r = 0; r < R; ++r)
            sc[r] = ORD ? __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ss[r], n), a.eps)))
                        : rsqrtf(fmaf(ss[r], a.inv_cols, a.eps));
        const bool wv = a.has_w && aligned16(a.w);
#pragma unroll
        for (int j = 0; j < K; ++j) {
            if (!okj[j]) continue;
            const int c = 4 * (t + kThreads * j);
            const float4 w = a.has_w ? param4(a.w + c, wv) : make_float4(1.0f, 1.0f, 1.0f, 1.0f);
#pragma unroll
            for (int r = 0; r < R; ++r) {
                if (row0 + r >= a.rows) break;
                const float4 x = v[r][j];
                float4 o;
                if constexpr (ORD) {
                    o = make_float4(__fmul_rn(x.x, sc[r]), __fmul_rn(x.y, sc[r]), __fmul_rn(x.z, sc[r]),
                                    __fmul_rn(x.w, sc[r]));
                    if (a.has_w)
                        o = make_float4(__fmul_rn(o.x, w.x), __fmul_rn(o.y, w.y), __fmul_rn(o.z, w.z),
                                        __fmul_rn(o.w, w.w));
                } else {
                    o = make_float4(x.x * sc[r] * w.x, x.y * sc[r] * w.y, x.z * sc[r] * w.z, x.w * sc[r] * w.w);
                }
                store4(a.y + (row0 + r) * a.cols + c, o, a.y_vec);
            }
        }
    } else {  // OP_LAYERNORM: mean, then the centred sum of squares on the cached row
        float mu[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            float4 l = v[r][0];
#pragma unroll
            for (int j = 1; j < K; ++j) {
                l.x = Add::f(l.x, v[r][j].x);
                l.y = Add::f(l.y, v[r][j].y);
                l.z = Add::f(l.z, v[r][j].z);
                l.w = Add::f(l.w, v[r][j].w);
            }
            mu[r] = quad_top<Add>(l);
        }
        tree_rows<Add, R>(mu, part[tb]);
        tb ^= 1;
        float q[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            // one rounded division (a contracted x - sum * (1/N) would leave a
            // constant row at ~1e-7 instead of 0)
            mu[r] = __fdiv_rn(mu[r], n);
            if constexpr (ORD) {
                float4 l = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
                for (int j = 0; j < K; ++j) {
                    if (!okj[j]) continue;  // padding is no column of the row
                    const float cx = __fsub_rn(v[r][j].x, mu[r]), cy = __fsub_rn(v[r][j].y, mu[r]);
                    const float cz = __fsub_rn(v[r][j].z, mu[r]), cw = __fsub_rn(v[r][j].w, mu[r]);
                    l.x = __fadd_rn(l.x, __fmul_rn(cx, cx));
                    l.y = __fadd_rn(l.y, __fmul_rn(cy, cy));
                    l.z = __fadd_rn(l.z, __fmul_rn(cz, cz));
                    l.w = __fadd_rn(l.w, __fmul_rn(cw, cw));
                }
                q[r] = quad_top<AddO>(l);
            } else {
                float acc = 0.0f;
#pragma unroll
                for (int j = 0; j < K; ++j) {
                    if (!okj[j]) continue;
                    const float cx = v[r][j].x - mu[r], cy = v[r][j].y - mu[r];
                    const float cz = v[r][j].z - mu[r], cw = v[r][j].w - mu[r];
                    acc = fmaf(cx, cx, fmaf(cy, cy, fmaf(cz, cz, fmaf(cw, cw, acc))));
                }
                q[r] = acc;
            }
        }
        tree_rows<Add, R>(q, part[tb]);
        tb ^= 1;
        float sc[R];
#pragma unroll
        for (int r = 0; r < R; ++r)
            sc[r] = ORD ? __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(q[r], n), a.eps)))
                        : rsqrtf(fmaf(q[r], a.inv_cols, a.eps));
        const bool wv = a.has_w && aligned16(a.w), bv = a.has_b && aligned16(a.b);
#pragma unroll
        for (int j = 0; j < K; ++j) {
            if (!okj[j]) continue;
            const int c = 4 * (t + kThreads * j);
            const float4 w = a.has_w ? param4(a.w + c, wv) : make_float4(1.0f, 1.0f, 1.0f, 1.0f);
            const float4 b = a.has_b ? param4(a.b + c, bv) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
            for (int r = 0; r < R; ++r) {
                if (row0 + r >= a.rows) break;
                const float4 x = v[r][j];
                float4 o;
                if constexpr (ORD) {
                    o = make_float4(__fmul_rn(__fsub_rn(x.x, mu[r]), sc[r]), __fmul_rn(__fsub_rn(x.y, mu[r]), sc[r]),
                                    __fmul_rn(__fsub_rn(x.z, mu[r]), sc[r]), __fmul_rn(__fsub_rn(x.w, mu[r]), sc[r]));
                    if (a.has_w)
                        o = make_float4(__fmul_rn(o.x, w.x), __fmul_rn(o.y, w.y), __fmul_rn(o.z, w.z),
                                        __fmul_rn(o.w, w.w));
                    if (a.has_b)
                        o = make_float4(__fadd_rn(o.x, b.x), __fadd_rn(o.y, b.y), __fadd_rn(o.z, b.z),
                                        __fadd_rn(o.w, b.w));
                } else {
                    o = make_float4(fmaf((x.x - mu[r]) * sc[r], w.x, b.x), fmaf((x.y - mu[r]) * sc[r], w.y, b.y),
                                    fmaf((x.z - mu[r]) * sc[r], w.z, b.z), fmaf((x.w - mu[r]) * sc[r], w.w, b.w));
                }
                store4(a.y + (row0 + r) * a.cols + c, o, a.y_vec);
            }
        }
    }
}

// Groups blockIdx.x, blockIdx.x + gridDim.x, ... (one group per CTA when the
// grid covers the rows). A block index alternates over consecutive trees, so a
// tree never writes a slot block that a thread may still be reading: between
// two uses of one block lies the other tree's barrier.
template <int OP, bool ORD, int K, int R>
__global__ void __launch_bounds__(kThreads, min_blocks<K, R>()) wave_kernel(const RowArgs a) {
    __shared__ __align__(16) float part[2][R][8];
    int tb = 0;
    pdl_enter();
    if constexpr (OP != OP_SOFTMAX) {
        // The norms read their weight (and bias) quads only in the epilogue, and
        // in a stream of launches those vectors have usually left L2, so the
        // first read per SM would wait on DRAM after the merges. CTA 0 asks L2
        // for both vectors now (one prefetch per 128-byte line, two per
        // thread at 6144 columns): they land while the rows load, and each
        // SM's epilogue finds them in L2 or, after its first CTA, in L1.
        // Prefetching from every CTA measured slower: the redundant requests
        // compete with the row loads.
        if (blockIdx.x == 0) {
            // 128-byte steps over one vector, plus its last element (a vector
            // need not start on a line); every address lies inside the vector
            const int lines = (a.cols + 31) / 32 + 1;
            const int nvecs = (a.has_w ? 1 : 0) + (OP == OP_LAYERNORM && a.has_b ? 1 : 0);
            for (int i = threadIdx.x; i < nvecs * lines; i += kThreads) {
                const float* base = (a.has_w && i < lines) ? a.w : a.b;
                prefetch_l2(base + min(32 * (i < lines ? i : i - lines), a.cols - 1));
            }
        }
    }
    for (int64_t g = blockIdx.x; g * R < a.rows; g += gridDim.x) wave_group<OP, ORD, K, R>(a, g * R, part, tb);
}

}  // namespace wave
}  // namespace tr
