// Device building blocks shared by the unordered row kernels.
//
// The reduction protocol follows "TIRx Metal reduction lowering" §2 ("Warp and
// SIMD-group intrinsics in the generated code") and §4.2 ("cooperative
// striping"): each worker folds its own stripe, a 32-lane collective combines
// a warp, lane 0 of each warp publishes one partial to shared memory, one
// barrier, and every warp re-reduces the partials (padding with the reducer's
// identity) so that every worker holds the result without a broadcast
// barrier. On sm_103a the 32-lane collective is a __shfl_xor_sync butterfly
// and, for rows split across the CTAs of a cluster, the third level reads the
// peers' partials through distributed shared memory.
#pragma once

#include <cooperative_groups.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace tr {

namespace cg = cooperative_groups;

constexpr float kL2E = 1.44269504088896340736f;  // log2(e)
constexpr float kLN2 = 0.69314718055994530942f;  // ln(2)
constexpr unsigned kFull = 0xffffffffu;

enum Op : int { OP_SOFTMAX = 0, OP_RMSNORM = 1, OP_LAYERNORM = 2, OP_XENT = 3 };

// 2^t with the SFU (ex2.approx): max relative error ~2^-22 on [-126, 128];
// results below 2^-126 flush to zero, which the unordered tolerance absorbs.
__device__ __forceinline__ float ex2(float t) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(t));
    return r;
}

// m * log2(e) rounded on its own. __fmul_rn is never fused into a following
// add, so mb_of(a) - mb_of(b) is exactly 0 when a == b; a plain a*L2E - mb
// may be contracted into fma(a, L2E, -mb), which leaves the rounding residual
// of mb and lets every rescale of a running sum drift by 2^residual.
__device__ __forceinline__ float mb_of(float m) { return __fmul_rn(m, kL2E); }

// Read-only 128-bit load of data that is read exactly once (no L1 allocation).
__device__ __forceinline__ float4 ld_stream4(const float* p) {
    float4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(p));
    return v;
}
__device__ __forceinline__ float ld_stream1(const float* p) {
    float v;
    asm volatile("ld.global.nc.L1::no_allocate.f32 %0, [%1];" : "=f"(v) : "l"(p));
    return v;
}
// Parameter vectors (weights, biases) are re-read by every row: keep them cached.
__device__ __forceinline__ float4 ld_param4(const float* p) {
    return __ldg(reinterpret_cast<const float4*>(p));
}

__device__ __forceinline__ bool aligned16(const void* p) {
    return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

__device__ __forceinline__ void st4(float* p, float4 v) {
    *reinterpret_cast<float4*>(p) = v;
}

struct SumOp {
    static __device__ __forceinline__ float id() { return 0.0f; }
    static __device__ __forceinline__ float op(float a, float b) { return a + b; }
};
struct MaxOp {
    static __device__ __forceinline__ float id() { return -__int_as_float(0x7f800000); }
    static __device__ __forceinline__ float op(float a, float b) { return fmaxf(a, b); }
};

// Butterfly over aligned groups of WIDTH lanes (all 32 lanes participate).
template <class R, int WIDTH>
__device__ __forceinline__ float warp_allreduce(float v) {
#pragma unroll
    for (int o = WIDTH / 2; o > 0; o >>= 1) v = R::op(v, __shfl_xor_sync(kFull, v, o));
    return v;
}

// The place of one thread inside the row it works on.
struct RowPos {
    int w;      // worker index within the row's workers (0 .. W-1)
    int W;      // workers per row inside this CTA
    int q;      // row slot inside the CTA
    int s;      // warp index within the row (G == 32)
    int S;      // warps per row (G == 32)
    int lane;
};

// Reduce one value over the W workers of a row inside one CTA.
// G < 32: a sub-warp butterfly. G == 32: warp butterfly, then (S > 1) one
// shared-memory exchange through `part` (2 x 32 floats; `buf` alternates so
// that consecutive reductions never race on a slot).
template <class R, int G>
__device__ __forceinline__ float cta_row_allreduce(float v, const RowPos& p, float (*part)[32], int& buf) {
    if constexpr (G < 32) {
        return warp_allreduce<R, G>(v);
    } else {
        v = warp_allreduce<R, 32>(v);
        if (p.S == 1) return v;
        float* slot = part[buf];
        buf ^= 1;
        if (p.lane == 0) slot[p.q * p.S + p.s] = v;
        __syncthreads();
        float t = (p.lane < p.S) ? slot[p.q * p.S + p.lane] : R::id();
        return warp_allreduce<R, 32>(t);
    }
}

// Reduce over all threads of a CTA (one row slice per CTA), result in every thread.
template <class R>
__device__ __forceinline__ float cta_allreduce(float v, float (*part)[32], int& buf) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    v = warp_allreduce<R, 32>(v);
    if (nw == 1) return v;
    float* slot = part[buf];
    buf ^= 1;
    if (lane == 0) slot[warp] = v;
    __syncthreads();
    float t = (lane < nw) ? slot[lane] : R::id();
    return warp_allreduce<R, 32>(t);
}

// Combine one per-CTA value across the C CTAs of a cluster. `cpart` is a
// 2-slot shared array; slots alternate between consecutive reductions, and
// the cluster barrier inside each reduction orders a slot's reads before its
// next write. The caller ends with cluster.sync() before exiting so that no
// CTA leaves while a peer may still read its shared memory.
template <class R>
__device__ __forceinline__ float cluster_allreduce(float v_cta, float* cpart, int& cbuf, int C) {
    cg::cluster_group cl = cg::this_cluster();
    float* slot = cpart + cbuf;
    cbuf ^= 1;
    if (threadIdx.x == 0) *slot = v_cta;
    cl.sync();
    const int lane = threadIdx.x & 31;
    float t = R::id();
    if (lane < C) t = *cl.map_shared_rank(slot, lane);
    return warp_allreduce<R, 32>(t);
}

// Geometry of one row's 16-byte body: `head` scalars up to the first 16-byte
// boundary, `nvec` float4 slots, `tail` trailing scalars.
struct RowGeom {
    int head, nvec, tail;
};
__device__ __forceinline__ RowGeom row_geom(const float* xr, int cols) {
    const int mis = static_cast<int>((reinterpret_cast<uintptr_t>(xr) >> 2) & 3u);
    int head = (4 - mis) & 3;
    if (head > cols) head = cols;
    const int body = cols - head;
    return RowGeom{head, body >> 2, body & 3};
}

}  // namespace tr
