// OT-1024 building blocks shared by the ordered row kernels and the ordered
// backward kernels: the library's own binary32 exp and log, the reducers, the
// fixed tree above a thread's four leaves, and the quad loads and stores of
// the layout (thread t of 256 owns columns 1024j + 4t .. 1024j + 4t + 3).
#pragma once

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

// The clamped, two-step form for any x: clamping to [-110, 100] changes
// nothing inside the range and reproduces the out-of-range results by
// overflow to +inf (x > 100) and underflow to +0 (x < -110).
static __device__ __noinline__ float exp_ot_wide(float x) {
    const float xc = fminf(fmaxf(x, -110.0f), 100.0f);
    const float kf = rintf(__fmul_rn(xc, 0x1.715476p+0f));
    const int k = static_cast<int>(kf);
    float r = __fmaf_rn(-kf, 0x1.62e430p-1f, xc);
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

// Fast form for |x| < 86 (so |k| <= 124), the same bits with full-rate
// instructions only:
//  - rint(t) for |t| < 2^22 is (t + M) - M with M = 1.5 * 2^23: the sum lands
//    in [2^23, 2^24), where the float spacing is 1, so adding M rounds t to an
//    integer with ties to even (M is even), and the difference is exact; k is
//    the sum's bit pattern minus M's.
//  - p lies in [2^-0.5, 2^0.5], so p * 2^k is normal: adding k to p's exponent
//    field is exact and equals the two-step product.
// Other x (|x| >= 86, infinities, NaN) take the clamped form.
__device__ __forceinline__ bool exp_ot_in_fast_range(float x) { return fabsf(x) < 86.0f; }
__device__ __forceinline__ float exp_ot_fast(float x) {
    constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23
    const float u = __fadd_rn(__fmul_rn(x, 0x1.715476p+0f), kMagic);
    const float kf = __fsub_rn(u, kMagic);
    const int k = __float_as_int(u) - 0x4b400000;
    float r = __fmaf_rn(-kf, 0x1.62e430p-1f, x);
    r = __fmaf_rn(-kf, -0x1.05c610p-29f, r);
    float p = 0x1.a01a02p-13f;
    p = __fmaf_rn(p, r, 0x1.6c16c2p-10f);
    p = __fmaf_rn(p, r, 0x1.111112p-7f);
    p = __fmaf_rn(p, r, 0x1.555556p-5f);
    p = __fmaf_rn(p, r, 0x1.555556p-3f);
    p = __fmaf_rn(p, r, 0x1.000000p-1f);
    p = __fmaf_rn(p, r, 1.0f);
    p = __fmaf_rn(p, r, 1.0f);
    return __int_as_float(__float_as_int(p) + static_cast<int>(static_cast<unsigned>(k) << 23));
}
__device__ __forceinline__ float exp_ot(float x) {
    if (!exp_ot_in_fast_range(x)) return x != x ? __fadd_rn(x, x) : exp_ot_wide(x);
    return exp_ot_fast(x);
}

// exp_ot_fast on two values at once with the packed binary32 FMA
// (__ffma2_rn: each lane rounds exactly as __fmaf_rn), so every lane gives
// exp_ot_fast's bits:
//  - u = RN(RN(x * RN(1/ln2)) + M) stays two scalar steps per lane: the
//    scalar _rn forms are never fused, and a fused u (one rounding) would
//    pick another k for rare x; such a difference was seen in a kernel that
//    formed u with the packed multiply and add;
//  - -kf = M - u exactly (u - M is an integer of at most 2^22 in magnitude), as
//    one packed FMA u * -1 + M;
//  - the scaling adds k << 23 to p's bits, and k << 23 equals u's bits << 23
//    modulo 2^32 (M's bits, 0x4b400000, vanish under the shift).
__device__ __forceinline__ float2 exp_ot_fast2(float2 x) {
    const float2 magic = make_float2(12582912.0f, 12582912.0f);
    const float2 u = make_float2(__fadd_rn(__fmul_rn(x.x, 0x1.715476p+0f), 12582912.0f),
                                 __fadd_rn(__fmul_rn(x.y, 0x1.715476p+0f), 12582912.0f));
    const float2 nkf = __ffma2_rn(u, make_float2(-1.0f, -1.0f), magic);
    float2 r = __ffma2_rn(nkf, make_float2(0x1.62e430p-1f, 0x1.62e430p-1f), x);
    r = __ffma2_rn(nkf, make_float2(-0x1.05c610p-29f, -0x1.05c610p-29f), r);
    float2 p = make_float2(0x1.a01a02p-13f, 0x1.a01a02p-13f);
    p = __ffma2_rn(p, r, make_float2(0x1.6c16c2p-10f, 0x1.6c16c2p-10f));
    p = __ffma2_rn(p, r, make_float2(0x1.111112p-7f, 0x1.111112p-7f));
    p = __ffma2_rn(p, r, make_float2(0x1.555556p-5f, 0x1.555556p-5f));
    p = __ffma2_rn(p, r, make_float2(0x1.555556p-3f, 0x1.555556p-3f));
    p = __ffma2_rn(p, r, make_float2(0x1.000000p-1f, 0x1.000000p-1f));
    p = __ffma2_rn(p, r, make_float2(1.0f, 1.0f));
    p = __ffma2_rn(p, r, make_float2(1.0f, 1.0f));
    return make_float2(__uint_as_float(__float_as_uint(p.x) + (__float_as_uint(u.x) << 23)),
                       __uint_as_float(__float_as_uint(p.y) + (__float_as_uint(u.y) << 23)));
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

// Row maximum of the softmax and cross-entropy trees: the hardware maxNum
// (NaN operands skipped). It can differ from the canonical max of the tree's
// definition (NaN wins, +0 over -0) only in rows that hold a NaN or whose
// maximum is a signed zero, and neither changes an output bit: a NaN element
// still reaches the sum as exp(NaN - m) = NaN, so every output of the row is
// NaN either way, and x - (+0) and x - (-0) give exponentials of equal value.
// maxNum of two non-NaN values is exact and commutative up to the sign of a
// zero, so the butterfly's lanes agree on the value.
__device__ __forceinline__ float max2(float a, float b) { return fmaxf(a, b); }
struct Add {
    static __device__ __forceinline__ float f(float a, float b) { return __fadd_rn(a, b); }
};
struct CMax {
    static __device__ __forceinline__ float f(float a, float b) { return cmax2(a, b); }
};
struct CMin {
    static __device__ __forceinline__ float f(float a, float b) { return cmin2(a, b); }
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

}  // namespace ordered
}  // namespace tr
