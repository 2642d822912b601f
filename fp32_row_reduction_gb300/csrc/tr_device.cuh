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

enum Op : int {
    OP_SOFTMAX = 0,
    OP_RMSNORM = 1,
    OP_LAYERNORM = 2,
    OP_XENT = 3,
    // standalone row reductions: one value per row (two for min/max)
    OP_RSUM = 4,
    OP_RMAX = 5,
    OP_RMIN = 6,
    OP_RMINMAX = 7
};

// Canonical max / min of the ordered standalone reductions, whose result is
// the output itself: NaN in the first operand wins, then NaN in the second,
// then the larger (smaller) value, +0 over -0 for the max and -0 over +0 for
// the min. Selects only, so a NaN keeps its payload; the predicates combine
// with bitwise operators, so no branch is taken per element.
__device__ __forceinline__ float cmax2(float a, float b) {
    const bool a_wins = (a != a) | (!(b != b) & ((a > b) | ((a == b) & (__float_as_int(a) >= 0))));
    return a_wins ? a : b;
}
__device__ __forceinline__ float cmin2(float a, float b) {
    const bool a_wins = (a != a) | (!(b != b) & ((a < b) | ((a == b) & (__float_as_int(a) < 0))));
    return a_wins ? a : b;
}
// Integer key of a float whose signed order is the total order of the floats
// with -0 below +0 (negative values have their magnitude bits flipped); NaNs
// map above key(+inf) or below key(-inf). The map is its own inverse.
__device__ __forceinline__ int order_key(float x) {
    const int b = __float_as_int(x);
    return b ^ ((b >> 31) & 0x7fffffff);
}
__device__ __forceinline__ float from_order_key(int k) { return __int_as_float(k ^ ((k >> 31) & 0x7fffffff)); }

// 2^t with the SFU (ex2.approx): max relative error ~2^-22 on [-126, 128];
// results below 2^-126 flush to zero, which the unordered tolerance absorbs.
__device__ __forceinline__ float ex2(float t) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(t));
    return r;
}

// Programmatic dependent launch. Every kernel waits for the grids it depends
// on (their memory operations complete and visible) before its first global
// read or write; without a programmatic predecessor the wait returns at once.
// No kernel signals its dependents early: the next launch on the stream is
// released as this grid's CTAs exit. An early signal lets the next grid's CTAs
// take free slots and sit in their own wait while this grid still streams,
// and in back-to-back launches at 768 x 6144 that cost about 1 us a launch.
__device__ __forceinline__ void pdl_enter() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

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

// Bring the line holding p into L1 (no register, no wait).
__device__ __forceinline__ void prefetch_l1(const void* p) { asm volatile("prefetch.global.L1 [%0];" ::"l"(p)); }
// Bring the line holding p into L2.
__device__ __forceinline__ void prefetch_l2(const void* p) { asm volatile("prefetch.global.L2 [%0];" ::"l"(p)); }

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

// ---------------------------------------------------------------------------
// Statistics merged across workers (one shuffle butterfly / shared exchange each).
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
// A float merged by max (a float alone merges by addition).
struct MaxF {
    float v;
};
__device__ __forceinline__ MaxF merge(MaxF a, MaxF b) { return MaxF{fmaxf(a.v, b.v)}; }
__device__ __forceinline__ MaxF shfl_xor(MaxF a, int o) { return MaxF{__shfl_xor_sync(kFull, a.v, o)}; }
__device__ __forceinline__ MaxSum merge(MaxSum a, MaxSum b) { return ms_merge(a, b); }
__device__ __forceinline__ Moments merge(Moments a, Moments b) { return mo_merge(a, b); }
__device__ __forceinline__ float merge(float a, float b) { return a + b; }
__device__ __forceinline__ float shfl_xor(float v, int o) { return __shfl_xor_sync(kFull, v, o); }

template <class T>
__device__ __forceinline__ T identity_of();
template <>
__device__ __forceinline__ float identity_of<float>() { return 0.0f; }
template <>
__device__ __forceinline__ MaxF identity_of<MaxF>() { return MaxF{MaxOp::id()}; }
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

// The place of one thread inside the row it works on.
struct RowPos {
    int w;      // worker index within the row's workers (0 .. W-1)
    int W;      // workers per row inside this CTA
    int q;      // row slot inside the CTA
    int s;      // warp index within the row (G == 32)
    int S;      // warps per row (G == 32)
    int lane;
};

// Merge one statistic over the W workers of a row inside one CTA.
// G < 32: a sub-warp butterfly. G == 32: warp butterfly, then (S > 1) lane 0
// of each warp publishes its value in `part` (2 x 32 slots of 16 bytes; `buf`
// alternates so consecutive merges never race on a slot), one barrier, and
// every warp merges the S published values (identity-padded).
template <class T, int G>
__device__ __forceinline__ T cta_row_merge(T v, const RowPos& p, float4 (*part)[32], int& buf) {
    if constexpr (G < 32) {
        return warp_merge<T, G>(v);
    } else {
        v = warp_merge<T, 32>(v);
        if (p.S == 1) return v;
        T* slot = reinterpret_cast<T*>(part[buf]);
        buf ^= 1;
        if (p.lane == 0) slot[p.q * p.S + p.s] = v;
        __syncthreads();
        return warp_merge<T, 32>(p.lane < p.S ? slot[p.q * p.S + p.lane] : identity_of<T>());
    }
}

// Merge a per-CTA statistic over the C CTAs of a cluster through distributed
// shared memory. `cpart` has 2 slots of 16 bytes that alternate between merges;
// the cluster barrier orders a slot's remote reads before its next write. The
// kernel ends with a cluster barrier so that no CTA exits while a peer may
// still read its slot.
template <class T>
__device__ __forceinline__ T cluster_merge(T v_cta, float4* cpart, int& cbuf, int C) {
    cg::cluster_group cl = cg::this_cluster();
    T* slot = reinterpret_cast<T*>(cpart + cbuf);
    cbuf ^= 1;
    if (threadIdx.x == 0) *slot = v_cta;
    cl.sync();
    const int lane = threadIdx.x & 31;
    return warp_merge<T, 32>(lane < C ? *cl.map_shared_rank(slot, lane) : identity_of<T>());
}

// ---------------------------------------------------------------------------
// Bulk asynchronous copies (TMA, non-tensor form) and mbarriers.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
// make initialised barriers visible to the async (TMA) proxy
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
// order this thread's earlier generic-proxy shared accesses before later async-proxy ones
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
// global -> shared bulk copy of `bytes` (multiple of 16, both addresses 16-byte
// aligned), completing `bytes` transactions on `bar`
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Error codes recorded in the device error word.
constexpr unsigned kErrWaitTimeout = 1u;

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for phase `parity` of `bar` for at most `limit_ns` nanoseconds. On
// timeout the error word gets kErrWaitTimeout and false is returned; the
// caller then finishes without trapping. `expire` (a testing mode) makes the
// wait give up at once without looking, as if its limit had passed, so that
// the caller's give-up path runs; waits that drain copies before a CTA exits
// never pass it.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, long long limit_ns,
                                                  unsigned* err, bool expire = false) {
    if (expire) {
        if (err) atomicOr(err, kErrWaitTimeout);
        return false;
    }
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (static_cast<long long>(global_ns() - t0) > limit_ns) break;
    }
    if (err) atomicOr(err, kErrWaitTimeout);
    return false;
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
