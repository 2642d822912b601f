// Cross-entropy backward, unordered policy, long rows (more than 8192 columns):
// dx_c = dloss (p_c - [c == label]), p = softmax(logits), as the 256-thread
// backward kernel computes it, realised for rows that do not fit registers.
//
// A row is read twice: once for its (max, sum of exponentials) pair, folded
// online per thread, and once to write dx. What decides the speed is where
// the second read is served from. Every CTA that is resident holds one row
// between its two passes, so the rows in flight are the resident CTAs, and
// their bytes must stay well inside L2 for the second read to hit there: at
// 4096 x 50257 the 256-thread kernel keeps ~1200 rows (240 MB) in flight and
// reads the row from DRAM twice. Here a CTA of 1024 threads takes a row, two
// CTAs per SM, so ~300 rows (60 MB) are in flight, and each thread keeps four
// 16-byte loads in flight per pass, enough to cover DRAM latency. The first
// pass loads with an L2 evict-last policy, the second pass and the dx stores
// with evict-first, so the rows waiting for their second pass are the lines L2
// keeps (without the hints ncu counts 1.62 GB of DRAM reads for 0.82 GB of
// logits at 4096 x 50257).
//
// Every global access is checked against its buffer and, for 16-byte
// accesses, its alignment before it is made; a failed check skips the access
// and sets kErrAccessCheck in the device error word. (This kernel's first form,
// without the checks, stopped with a misaligned-address error on rows whose
// logits and dlogits sat at different 16-byte phases; its checked form
// records no bad access on the same inputs.)
#include <cuda_runtime.h>
#include <stdint.h>

#include "tr_internal.h"
#include "tr_split_kernels.cuh"

namespace tr {

constexpr int kXbThreads = 1024;
constexpr int kXbU = 4;  // float4 per thread per chunk
static_assert(kXbU == kSplitU, "the chunk fold takes kSplitU quads");

// The buffers of one launch and the checked accesses to them.
struct XbIo {
    const float* x0;
    const float* x1;  // logits [x0, x1)
    float* y0;
    float* y1;        // dlogits [y0, y1)
    unsigned* err;
    __device__ __forceinline__ void bad() const { atomicOr(err, kErrAccessCheck); }
    // a 16-byte load under the L2 eviction policy `pol` (createpolicy)
    __device__ __forceinline__ float4 ld4(const float* p, uint64_t pol) const {
        if ((reinterpret_cast<uintptr_t>(p) & 15u) || p < x0 || p + 4 > x1) {
            bad();
            return make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        }
        float4 v;
        asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.f32 {%0, %1, %2, %3}, [%4], %5;"
                     : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                     : "l"(p), "l"(pol));
        return v;
    }
    __device__ __forceinline__ float ld1(const float* p) const {
        if (p < x0 || p + 1 > x1) {
            bad();
            return 0.0f;
        }
        return ld_stream1(p);
    }
    // four consecutive outputs: one 16-byte store (under the L2 policy `pol`)
    // when p is on the 16-byte grid
    __device__ __forceinline__ void st(float* p, float4 o, bool vec, uint64_t pol) const {
        if (p < y0 || p + 4 > y1) {
            bad();
            return;
        }
        if (vec) {
            if (reinterpret_cast<uintptr_t>(p) & 15u) {
                bad();
                return;
            }
            asm volatile("st.global.L2::cache_hint.v4.f32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(p), "f"(o.x), "f"(o.y),
                         "f"(o.z), "f"(o.w), "l"(pol)
                         : "memory");
        } else {
            p[0] = o.x;
            p[1] = o.y;
            p[2] = o.z;
            p[3] = o.w;
        }
    }
    __device__ __forceinline__ void st1(float* p, float v) const {
        if (p < y0 || p + 1 > y1) {
            bad();
            return;
        }
        *p = v;
    }
};

__global__ void __launch_bounds__(kXbThreads, 2) xent_bwd_stream_kernel(const BwArgs a, const XbIo io) {
    __shared__ float4 part[2][32];
    uint64_t keep, drop;  // L2 policies: rows between their passes stay, rows on their last pass go first
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(keep));
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(drop));
    const int cols = a.cols, T = blockDim.x, t = threadIdx.x;
    RowPos p;
    p.w = t;
    p.W = T;
    p.q = 0;
    p.s = t >> 5;
    p.S = T >> 5;
    p.lane = t & 31;
    int buf = 0;
    for (int64_t row = blockIdx.x; row < a.rows; row += gridDim.x) {
        const float* xr = a.x + row * cols;
        float* yr = a.dx + row * cols;
        const RowGeom g = row_geom(xr, cols);
        const float* xb = xr + g.head;
        float* yb = yr + g.head;
        const bool yv = ((reinterpret_cast<uintptr_t>(xr) ^ reinterpret_cast<uintptr_t>(yr)) & 15u) == 0;

        // ---- pass 1: the row's (max, sum of exponentials), online per thread
        MaxSum st = identity_of<MaxSum>();
        int i = t;
        for (; i + (kXbU - 1) * T < g.nvec; i += kXbU * T) {
            float4 c[kXbU];
            for (int u = 0; u < kXbU; ++u) c[u] = io.ld4(xb + 4 * (i + u * T), keep);
            st = fold_chunk<OP_SOFTMAX, kXbU>(st, c);
        }
        for (; i < g.nvec; i += T) {
            float4 c[kXbU];
            c[0] = io.ld4(xb + 4 * i, keep);
            st = fold_chunk<OP_SOFTMAX, 1>(st, c);
        }
        if (t < g.head) st = fold_one<OP_SOFTMAX>(st, io.ld1(xr + t));
        if (t < g.tail) st = fold_one<OP_SOFTMAX>(st, io.ld1(xb + 4 * g.nvec + t));
        st = cta_row_merge<MaxSum, 32>(st, p, part, buf);  // every thread holds the row's pair

        // ---- pass 2: dx, the row read again (from L2)
        const float mb = mb_of(st.m);
        const float inv = __fdividef(1.0f, st.s);
        const int64_t label = a.labels[row];
        const bool scaled = a.dloss != nullptr;
        const float dl = scaled ? a.dloss[row] : 1.0f;
        // every element as if it were not the label's; the label's element (one per
        // row, when in range) is written again after the barrier below
        auto grad = [&](float x) {
            const float d = ex2(fmaf(x, kL2E, -mb)) * inv;
            return scaled ? d * dl : d;
        };
        auto grad4 = [&](float4 c) { return make_float4(grad(c.x), grad(c.y), grad(c.z), grad(c.w)); };
        i = t;
        for (; i + (kXbU - 1) * T < g.nvec; i += kXbU * T) {
            float4 c[kXbU];
            for (int u = 0; u < kXbU; ++u) c[u] = io.ld4(xb + 4 * (i + u * T), drop);
            for (int u = 0; u < kXbU; ++u) io.st(yb + 4 * (i + u * T), grad4(c[u]), yv, drop);
        }
        for (; i < g.nvec; i += T) io.st(yb + 4 * i, grad4(io.ld4(xb + 4 * i, drop)), yv, drop);
        if (t < g.head) io.st1(yr + t, grad(io.ld1(xr + t)));
        if (t < g.tail) {
            const int c = g.head + 4 * g.nvec + t;
            io.st1(yr + c, grad(io.ld1(xr + c)));
        }
        // the barrier orders the CTA's stores of this row before the label's rewrite
        __syncthreads();
        if (t == 0 && label >= 0 && label < cols) {
            const float d = ex2(fmaf(io.ld1(xr + label), kL2E, -mb)) * inv - 1.0f;
            io.st1(yr + label, scaled ? d * dl : d);
        }
    }
}

cudaError_t launch_xent_backward_stream(const BwArgs& a, cudaStream_t stream) {
    const int64_t n = a.rows * static_cast<int64_t>(a.cols);
    const XbIo io{a.x, a.x + n, a.dx, a.dx + n, a.err};
    const int64_t ctas = a.rows < (1LL << 20) ? a.rows : (1LL << 20);
    xent_bwd_stream_kernel<<<dim3(static_cast<unsigned>(ctas)), kXbThreads, 0, stream>>>(a, io);
    return cudaGetLastError();
}

}  // namespace tr
