// OT-1024 for few long rows: a cluster of 8 CTAs per row, one per group of the
// tree.
//
// The fixed tree's top level combines 8 group values, ((g0 + g1) + (g2 + g3)) +
// ((g4 + g5) + (g6 + g7)), and group W is the subtree over quads 32W .. 32W + 31,
// that is over the leaves whose columns are 128W .. 128W + 127 modulo 1024. Each
// group is therefore independent up to the top: CTA W of a row's cluster copies
// the row's columns of its group into shared memory (asynchronous 16-byte copies,
// all in flight at once), warp 0 folds the group exactly as the one-CTA kernel's
// warp W does (lane L owns quad 32W + L, leaves folded in increasing column order,
// then the lane butterfly), and the 8 group values meet in distributed shared
// memory, where every CTA evaluates the top level in the same order. The result
// is the OT-1024 value bit for bit, with a row spread over 8 SMs instead of one.
#include <cooperative_groups.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "tr_device.cuh"
#include "tr_internal.h"
#include "tr_ot.cuh"

namespace tr {
namespace ordered {

namespace cg = cooperative_groups;

constexpr int kGroups = 8;

__device__ __forceinline__ void cp_async16_ot(void* dst, const float* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}

template <int OP>
__global__ void __launch_bounds__(kOrderedThreads) ot_cluster_kernel(const RowArgs a) {
    extern __shared__ float4 slab[];  // [nm][32]: quad L of this group at column 1024m + 128W + 4L
    __shared__ float gv[4];           // this CTA's group value of each pass, read by the whole cluster
    cg::cluster_group cl = cg::this_cluster();
    pdl_enter();
    const int W = static_cast<int>(cl.block_rank());
    const int64_t row = blockIdx.x / kGroups;
    const int cols = a.cols;
    const int nm = (cols + 1023) / 1024;
    const float* xr = a.x + row * cols;
    const bool al = aligned16(xr);
    const int lane = threadIdx.x & 31;

    // stage the group's columns
    for (int i = threadIdx.x; i < nm * 32; i += kOrderedThreads) {
        const int c0 = 1024 * (i >> 5) + 128 * W + 4 * (i & 31);
        if (al && c0 + 3 < cols) {
            cp_async16_ot(slab + i, xr + c0);
        } else {
            float q[4];
#pragma unroll
            for (int v = 0; v < 4; ++v) q[v] = c0 + v < cols ? ld_stream1(xr + c0 + v) : 0.0f;
            slab[i] = make_float4(q[0], q[1], q[2], q[3]);
        }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    __syncthreads();

    // warp 0: the group's subtree of elem(x, column) under the reducer R (lane 0 holds it)
    auto fold_group = [&](auto elem, auto R, float init) -> float {
        using F = decltype(R);
        float leaf[4] = {init, init, init, init};
        auto take = [&](const float4& q4, int m) {
            const float q[4] = {q4.x, q4.y, q4.z, q4.w};
            const int c0 = 1024 * m + 128 * W + 4 * lane;
#pragma unroll
            for (int v = 0; v < 4; ++v)
                if (c0 + v < cols) leaf[v] = F::f(leaf[v], elem(q[v], c0 + v));
        };
        int m = 0;
        for (; m + 7 < nm; m += 8) {  // eight shared-memory loads ahead of their folds
            float4 q[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) q[u] = slab[(m + u) * 32 + lane];
#pragma unroll
            for (int u = 0; u < 8; ++u) take(q[u], m + u);
        }
        for (; m < nm; ++m) take(slab[m * 32 + lane], m);
        float val = F::f(F::f(leaf[0], leaf[1]), F::f(leaf[2], leaf[3]));
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) val = F::f(val, __shfl_xor_sync(kFull, val, o));
        return val;
    };
    // the top level over the 8 group values of pass `slot`, identical in every CTA
    auto top = [&](float mine, auto R, int slot) -> float {
        using F = decltype(R);
        if (threadIdx.x == 0) gv[slot] = mine;
        cl.sync();
        float g[kGroups];
#pragma unroll
        for (int r = 0; r < kGroups; ++r) g[r] = *cl.map_shared_rank(&gv[slot], r);
        return F::f(F::f(F::f(g[0], g[1]), F::f(g[2], g[3])), F::f(F::f(g[4], g[5]), F::f(g[6], g[7])));
    };
    auto ident = [](float v, int) { return v; };
    // out(value, column) for every column of the group (all threads), written to y
    auto emit = [&](auto out) {
        float* yr = a.y + row * cols;
        for (int i = threadIdx.x; i < nm * 32; i += kOrderedThreads) {
            const int c0 = 1024 * (i >> 5) + 128 * W + 4 * (i & 31);
            const float4 q4 = slab[i];
            const float q[4] = {q4.x, q4.y, q4.z, q4.w};
            if (c0 + 3 < cols && aligned16(yr + c0)) {
                st4(yr + c0, make_float4(out(q[0], c0), out(q[1], c0 + 1), out(q[2], c0 + 2), out(q[3], c0 + 3)));
            } else {
#pragma unroll
                for (int v = 0; v < 4; ++v)
                    if (c0 + v < cols) yr[c0 + v] = out(q[v], c0 + v);
            }
        }
    };
    const float n = static_cast<float>(cols);
    float mine = 0.0f;

    if constexpr (OP == OP_SOFTMAX || OP == OP_XENT) {
        if (threadIdx.x < 32) mine = fold_group(ident, Max{}, __int_as_float(0xff800000));
        const float m = top(mine, Max{}, 0);
        // the exponentials once per element, in place (every thread), then their sum
        for (int i = threadIdx.x; i < nm * 32; i += kOrderedThreads) {
            const float4 q = slab[i];
            slab[i] = make_float4(exp_ot(__fsub_rn(q.x, m)), exp_ot(__fsub_rn(q.y, m)), exp_ot(__fsub_rn(q.z, m)),
                                  exp_ot(__fsub_rn(q.w, m)));
        }
        __syncthreads();
        if (threadIdx.x < 32) mine = fold_group(ident, Add{}, 0.0f);
        const float s = top(mine, Add{}, 1);
        if constexpr (OP == OP_SOFTMAX) {
            const float inv = __fdiv_rn(1.0f, s);
            emit([inv](float e, int) { return __fmul_rn(e, inv); });
        } else {
            if (W == 0 && threadIdx.x == 0) {
                const int64_t label = a.labels[row];
                const float sel = (label >= 0 && label < cols) ? __ldg(xr + label) : 0.0f;
                a.loss[row] = __fsub_rn(__fadd_rn(log_ot(s), m), sel);
            }
        }
    } else if constexpr (OP == OP_RMSNORM) {
        if (threadIdx.x < 32) mine = fold_group([](float v, int) { return __fmul_rn(v, v); }, Add{}, 0.0f);
        const float ss = top(mine, Add{}, 0);
        const float inv = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ss, n), a.eps)));
        const bool hw = a.has_w;
        const float* w = a.w;
        emit([inv, hw, w](float v, int c) {
            const float u = __fmul_rn(v, inv);
            return hw ? __fmul_rn(u, __ldg(w + c)) : u;
        });
    } else {  // OP_LAYERNORM
        if (threadIdx.x < 32) mine = fold_group(ident, Add{}, 0.0f);
        const float mean = __fdiv_rn(top(mine, Add{}, 0), n);
        if (threadIdx.x < 32)
            mine = fold_group([mean](float v, int) {
                const float c = __fsub_rn(v, mean);
                return __fmul_rn(c, c);
            }, Add{}, 0.0f);
        const float var = __fdiv_rn(top(mine, Add{}, 1), n);
        const float inv = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(var, a.eps)));
        const bool hw = a.has_w, hb = a.has_b;
        const float *w = a.w, *b = a.b;
        emit([mean, inv, hw, hb, w, b](float v, int c) {
            float u = __fmul_rn(__fsub_rn(v, mean), inv);
            if (hw) u = __fmul_rn(u, __ldg(w + c));
            if (hb) u = __fadd_rn(u, __ldg(b + c));
            return u;
        });
    }
    cl.sync();  // no CTA leaves while another may still read its group values
}

}  // namespace ordered

const void* kernel_ordered_cluster(int op) {
    switch (op) {
        case TR_OP_SOFTMAX: return reinterpret_cast<const void*>(ordered::ot_cluster_kernel<OP_SOFTMAX>);
        case TR_OP_RMSNORM: return reinterpret_cast<const void*>(ordered::ot_cluster_kernel<OP_RMSNORM>);
        case TR_OP_LAYERNORM: return reinterpret_cast<const void*>(ordered::ot_cluster_kernel<OP_LAYERNORM>);
        case TR_OP_CROSS_ENTROPY: return reinterpret_cast<const void*>(ordered::ot_cluster_kernel<OP_XENT>);
    }
    return nullptr;
}

}  // namespace tr
