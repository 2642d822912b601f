// Ordered-tree kernels (TR_ORDER_ORDERED_TREE): the canonical OT-1024 tree.
//
// "TIRx Metal reduction lowering" §1: a reduction's ReductionPolicy may be an
// ordered tree, which "stays ordered", and a kernel with an ordered reduction
// must not be compiled with fast math. The page fixes no tree shape; this
// library's ordered policy is the fixed tree OT-1024, defined on columns and
// independent of the launch configuration:
//   leaf k (k < 1024)   fold_left, in increasing column e, of the columns
//                       e = k (mod 1024), starting from the identity;
//   partial t (t < 256) (leaf 4t (+) leaf 4t+1) (+) (leaf 4t+2 (+) leaf 4t+3);
//   group g (g < 8)     partials 32g..32g+31 combined by an xor butterfly with
//                       offsets 16, 8, 4, 2, 1 (every lane ends with the same bits,
//                       since IEEE add and the canonical max are commutative);
//   result              ((g0 (+) g1) (+) (g2 (+) g3)) (+) ((g4 (+) g5) (+) (g6 (+) g7)).
// Realisation: one CTA of 256 threads per row; thread t owns leaves 4t..4t+3,
// i.e. the float4 at columns 1024j + 4t (a single 128-bit load when the row
// start is 16-byte aligned). Rows of at most 1024*K columns are cached in
// registers; longer rows are read again for each pass (K = 0).
//
// Every floating-point step is an explicit round-to-nearest intrinsic
// (__fadd_rn, __fmul_rn, __fdiv_rn, __fsqrt_rn, __fmaf_rn): nothing can be
// contracted, approximated or flushed, so the bits equal the CPU emulation.
#include <cuda_runtime.h>
#include <stdint.h>

#include "tr_device.cuh"
#include "tr_internal.h"

namespace tr {
namespace ordered {

// exp on binary32 by Cody & Waite argument reduction (W. J. Cody and W. Waite,
// "Software Manual for the Elementary Functions", 1980): k = rint(x * RN(1/ln2)),
// r = x - k*ln2 with ln2 = RN(ln2) + RN(ln2 - RN(ln2)) applied by two FMAs,
// e^r by its Taylor series through r^7/7! (coefficients RN(1/i!)) in Horner
// form, and the result scaled by 2^floor(k/2) and then by 2^(k - floor(k/2)).
__device__ __forceinline__ float pow2i(int n) { return __int_as_float((n + 127) << 23); }

__device__ __forceinline__ float exp_ot(float x) {
    if (x != x) return __fadd_rn(x, x);
    if (x > 100.0f) return __int_as_float(0x7f800000);
    if (x < -110.0f) return 0.0f;
    const float kf = rintf(__fmul_rn(x, 0x1.715476p+0f));
    const int k = static_cast<int>(kf);
    float r = __fmaf_rn(-kf, 0x1.62e430p-1f, x);
    r = __fmaf_rn(-kf, -0x1.05c610p-29f, r);
    float p = 0x1.a01a02p-13f;           // 1/7!
    p = __fmaf_rn(p, r, 0x1.6c16c2p-10f);  // 1/6!
    p = __fmaf_rn(p, r, 0x1.111112p-7f);   // 1/5!
    p = __fmaf_rn(p, r, 0x1.555556p-5f);   // 1/4!
    p = __fmaf_rn(p, r, 0x1.555556p-3f);   // 1/3!
    p = __fmaf_rn(p, r, 0x1.000000p-1f);   // 1/2!
    p = __fmaf_rn(p, r, 1.0f);
    p = __fmaf_rn(p, r, 1.0f);
    const int k1 = k >> 1;
    return __fmul_rn(__fmul_rn(p, pow2i(k1)), pow2i(k - k1));
}

// log on binary32: x = 2^e m, m in (sqrt(1/2), sqrt(2)], f = m - 1,
// s = f / (2 + f), log m = f - s (f - R(s^2)) with
// R(z) = z (2/3 + z (2/5 + z (2/7 + z 2/9))) (the atanh series written so that
// the leading term f is exact), log x = e RN(ln2) + (e RN(ln2 - RN(ln2)) + log m).
__device__ __forceinline__ float log_ot(float x) {
    if (x != x) return __fadd_rn(x, x);
    if (x < 0.0f) return __int_as_float(0x7fc00000);
    if (x == 0.0f) return __int_as_float(0xff800000);
    if (x == __int_as_float(0x7f800000)) return x;
    int e = 0;
    if (x < 0x1p-126f) {
        x = __fmul_rn(x, 0x1p23f);
        e = -23;
    }
    const unsigned u = __float_as_uint(x);
    e += static_cast<int>((u >> 23) & 0xffu) - 127;
    float m = __uint_as_float((u & 0x007fffffu) | 0x3f800000u);
    if (m > 0x1.6a09e6p+0f) {
        m = __fmul_rn(m, 0.5f);
        e += 1;
    }
    const float f = __fsub_rn(m, 1.0f);
    const float s = __fdiv_rn(f, __fadd_rn(2.0f, f));
    const float z = __fmul_rn(s, s);
    float q = 0x1.c71c72p-3f;           // 2/9
    q = __fmaf_rn(q, z, 0x1.24924ap-2f);  // 2/7
    q = __fmaf_rn(q, z, 0x1.99999ap-2f);  // 2/5
    q = __fmaf_rn(q, z, 0x1.555556p-1f);  // 2/3
    const float rr = __fmul_rn(z, q);
    const float lm = __fmaf_rn(-s, __fsub_rn(f, rr), f);
    const float ef = static_cast<float>(e);
    return __fmaf_rn(ef, 0x1.62e430p-1f, __fmaf_rn(ef, -0x1.05c610p-29f, lm));
}

// Canonical max: NaN in the first operand wins, +0 beats -0; commutative for
// every non-NaN pair, so the butterfly leaves identical bits in all lanes.
__device__ __forceinline__ float max2(float a, float b) {
    if (a != a) return a;
    if (b != b) return b;
    if (a > b) return a;
    if (b > a) return b;
    return (__float_as_uint(a) >> 31) ? b : a;
}
struct Add {
    static __device__ __forceinline__ float f(float a, float b) { return __fadd_rn(a, b); }
};
struct Max {
    static __device__ __forceinline__ float f(float a, float b) { return max2(a, b); }
};

// The tree above this thread's four leaves. `gpart` is 2 x 8 shared floats;
// `buf` alternates so consecutive trees never share a slot.
template <class R>
__device__ __forceinline__ float tree(const float (&leaf)[4], float (*gpart)[8], int& buf) {
    float v = R::f(R::f(leaf[0], leaf[1]), R::f(leaf[2], leaf[3]));
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v = R::f(v, __shfl_xor_sync(kFull, v, o));
    float* g = gpart[buf];
    buf ^= 1;
    if ((threadIdx.x & 31) == 0) g[threadIdx.x >> 5] = v;
    __syncthreads();
    return R::f(R::f(R::f(g[0], g[1]), R::f(g[2], g[3])), R::f(R::f(g[4], g[5]), R::f(g[6], g[7])));
}

// Columns 1024j + 4t .. +3 of a row; `ok[v]` marks the columns inside the row.
__device__ __forceinline__ void load_quad(const float* xr, int cols, int j, bool aligned, float (&q)[4],
                                          bool (&ok)[4]) {
    const int c0 = 1024 * j + 4 * static_cast<int>(threadIdx.x);
    if (aligned && c0 + 3 < cols) {
        const float4 v = ld_stream4(xr + c0);
        q[0] = v.x; q[1] = v.y; q[2] = v.z; q[3] = v.w;
        ok[0] = ok[1] = ok[2] = ok[3] = true;
    } else {
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            ok[v] = c0 + v < cols;
            q[v] = ok[v] ? ld_stream1(xr + c0 + v) : 0.0f;
        }
    }
}

__device__ __forceinline__ void store_quad(float* yr, int cols, int j, bool vec, const float (&o)[4],
                                           const bool (&ok)[4]) {
    const int c0 = 1024 * j + 4 * static_cast<int>(threadIdx.x);
    if (vec && ok[3]) {
        st4(yr + c0, make_float4(o[0], o[1], o[2], o[3]));
    } else {
#pragma unroll
        for (int v = 0; v < 4; ++v)
            if (ok[v]) yr[c0 + v] = o[v];
    }
}

__device__ __forceinline__ float param(const float* p, int col, bool has, float dflt) {
    return has ? __ldg(p + col) : dflt;
}

// K > 0: the row (cols <= 1024*K) is cached in registers. K == 0: re-read.
template <int OP, int K>
__global__ void __launch_bounds__(kOrderedThreads) ot_kernel(const RowArgs a) {
    __shared__ float gpart[2][8];
    int buf = 0;
    const int64_t row = blockIdx.x;
    const int cols = a.cols;
    const float* xr = a.x + row * cols;
    const bool aligned = aligned16(xr);
    const int nj = (cols + 1023) / 1024;  // column blocks of 1024
    constexpr bool kCached = K > 0;
    constexpr int KC = kCached ? K : 1;
    float q[KC][4];
    bool ok[KC][4];
    pdl_enter();
    if constexpr (kCached) {
#pragma unroll
        for (int j = 0; j < K; ++j) {
            if (j < nj) {
                load_quad(xr, cols, j, aligned, q[j], ok[j]);
            } else {
                q[j][0] = q[j][1] = q[j][2] = q[j][3] = 0.0f;
                ok[j][0] = ok[j][1] = ok[j][2] = ok[j][3] = false;
            }
        }
    }
    // fold f(x) into the four leaves, column blocks in increasing order
    auto fold = [&](auto elem, auto comb, float init, float (&leaf)[4]) {
        leaf[0] = leaf[1] = leaf[2] = leaf[3] = init;
        if constexpr (kCached) {
#pragma unroll
            for (int j = 0; j < K; ++j)
#pragma unroll
                for (int v = 0; v < 4; ++v)
                    if (ok[j][v]) leaf[v] = comb(leaf[v], elem(q[j][v], j * 1024 + 4 * static_cast<int>(threadIdx.x) + v));
        } else {
            for (int j = 0; j < nj; ++j) {
                float qq[4];
                bool oo[4];
                load_quad(xr, cols, j, aligned, qq, oo);
#pragma unroll
                for (int v = 0; v < 4; ++v)
                    if (oo[v]) leaf[v] = comb(leaf[v], elem(qq[v], j * 1024 + 4 * static_cast<int>(threadIdx.x) + v));
            }
        }
    };
    // apply out(x, col) to every element and store it
    auto emit = [&](auto out) {
        float* yr = a.y + row * cols;
        const bool vec = aligned && a.y_vec;
        if constexpr (kCached) {
#pragma unroll
            for (int j = 0; j < K; ++j) {
                if (j < nj) {
                    float o[4];
#pragma unroll
                    for (int v = 0; v < 4; ++v) o[v] = out(q[j][v], j * 1024 + 4 * static_cast<int>(threadIdx.x) + v);
                    store_quad(yr, cols, j, vec, o, ok[j]);
                }
            }
        } else {
            for (int j = 0; j < nj; ++j) {
                float qq[4], o[4];
                bool oo[4];
                load_quad(xr, cols, j, aligned, qq, oo);
#pragma unroll
                for (int v = 0; v < 4; ++v) o[v] = oo[v] ? out(qq[v], j * 1024 + 4 * static_cast<int>(threadIdx.x) + v) : 0.0f;
                store_quad(yr, cols, j, vec, o, oo);
            }
        }
    };
    auto add = [](float p, float v) { return __fadd_rn(p, v); };
    auto mx = [](float p, float v) { return max2(p, v); };
    auto ident = [](float v, int) { return v; };
    float leaf[4];
    const float n = static_cast<float>(cols);

    if constexpr (OP == OP_SOFTMAX || OP == OP_XENT) {
        fold(ident, mx, __int_as_float(0xff800000), leaf);
        const float m = tree<Max>(leaf, gpart, buf);
        float s;
        if constexpr (kCached) {
            // exp once per element, kept in place: the sum below folds the same
            // values in the same leaf order as exp_ot(x - m) would
#pragma unroll
            for (int j = 0; j < K; ++j)
#pragma unroll
                for (int v = 0; v < 4; ++v)
                    if (ok[j][v]) q[j][v] = exp_ot(__fsub_rn(q[j][v], m));
            fold(ident, add, 0.0f, leaf);
            s = tree<Add>(leaf, gpart, buf);
        } else {
            fold([m](float v, int) { return exp_ot(__fsub_rn(v, m)); }, add, 0.0f, leaf);
            s = tree<Add>(leaf, gpart, buf);
        }
        if constexpr (OP == OP_SOFTMAX) {
            if constexpr (kCached)
                emit([s](float e, int) { return __fdiv_rn(e, s); });
            else
                emit([m, s](float v, int) { return __fdiv_rn(exp_ot(__fsub_rn(v, m)), s); });
        } else {
            if (threadIdx.x == 0) {
                const int64_t label = a.labels[row];
                const float sel = (label >= 0 && label < cols) ? __ldg(xr + label) : 0.0f;
                a.loss[row] = __fsub_rn(__fadd_rn(log_ot(s), m), sel);
            }
        }
    } else if constexpr (OP == OP_RMSNORM) {
        fold([](float v, int) { return __fmul_rn(v, v); }, add, 0.0f, leaf);
        const float ss = tree<Add>(leaf, gpart, buf);
        const float r = __fsqrt_rn(__fadd_rn(__fdiv_rn(ss, n), a.eps));
        const bool hw = a.has_w;
        const float* w = a.w;
        emit([r, hw, w](float v, int c) {
            const float t = __fdiv_rn(v, r);
            return hw ? __fmul_rn(t, __ldg(w + c)) : t;
        });
    } else {  // OP_LAYERNORM
        fold(ident, add, 0.0f, leaf);
        const float mean = __fdiv_rn(tree<Add>(leaf, gpart, buf), n);
        fold([mean](float v, int) {
            const float c = __fsub_rn(v, mean);
            return __fmul_rn(c, c);
        }, add, 0.0f, leaf);
        const float var = __fdiv_rn(tree<Add>(leaf, gpart, buf), n);
        const float d = __fsqrt_rn(__fadd_rn(var, a.eps));
        const bool hw = a.has_w, hb = a.has_b;
        const float *w = a.w, *b = a.b;
        emit([mean, d, hw, hb, w, b](float v, int c) {
            float t = __fdiv_rn(__fsub_rn(v, mean), d);
            if (hw) t = __fmul_rn(t, __ldg(w + c));
            if (hb) t = __fadd_rn(t, __ldg(b + c));
            return t;
        });
    }
}

}  // namespace ordered

const void* kernel_ordered(int op, int slots) {
#define TR_OT_CASES(OPV)                                                    \
    switch (slots) {                                                        \
        case 0: return reinterpret_cast<const void*>(ordered::ot_kernel<OPV, 0>);   \
        case 1: return reinterpret_cast<const void*>(ordered::ot_kernel<OPV, 1>);   \
        case 2: return reinterpret_cast<const void*>(ordered::ot_kernel<OPV, 2>);   \
        case 4: return reinterpret_cast<const void*>(ordered::ot_kernel<OPV, 4>);   \
        case 8: return reinterpret_cast<const void*>(ordered::ot_kernel<OPV, 8>);   \
        case 16: return reinterpret_cast<const void*>(ordered::ot_kernel<OPV, 16>); \
    }                                                                       \
    return nullptr;
    switch (op) {
        case TR_OP_SOFTMAX: { TR_OT_CASES(OP_SOFTMAX) }
        case TR_OP_RMSNORM: { TR_OT_CASES(OP_RMSNORM) }
        case TR_OP_LAYERNORM: { TR_OT_CASES(OP_LAYERNORM) }
        case TR_OP_CROSS_ENTROPY: { TR_OT_CASES(OP_XENT) }
    }
#undef TR_OT_CASES
    return nullptr;
}

}  // namespace tr
