// Reductions over a non-last axis: x viewed as [outer, extent, inner] (row
// major, contiguous), out[o * inner + i] = reduce over r of x[o, r, i].
//
// "TIRx Metal reduction lowering" (Reductions inside composed groups): the
// reduced axis need not be the last memory dimension; each output is one
// independent collective, missing elements contribute the identity, and the
// canonical FP32 add / max / min are the reducers. On GB300 the 32 lanes of a
// warp take 32 consecutive output columns, so every load of a warp reads
// consecutive floats of one x row (coalesced whenever inner >= 32), and the
// reduced axis is spread over the 8 warps of a CTA and, when the columns alone
// cannot fill the GPU, over `splits` CTAs whose partials the last CTA to
// arrive combines (a ticket, no waiting).
//
// Ordered policy: the result is the fixed tree OT-1024 applied to the column
// (leaf k folds the elements r = k mod 1024 in increasing r, then the fixed
// tree above the 1024 leaves), bit for bit the value the row reductions give
// for the same vector. That tree is a perfect binary tree over the leaf slots
// in the order (group w, bit-reversed lane, slot v) of the row kernels'
// thread layout, so any power-of-two block of consecutive slots is a subtree:
// every warp folds its block of quads with a stack of pending subtrees, the
// CTA combines its 8 blocks in order, and the last CTA combines the splits'
// blocks in order.
#include <cuda_runtime.h>
#include <stdint.h>

#include "tr_device.cuh"
#include "tr_internal.h"

namespace tr {
namespace axis {

constexpr int kWarps = kAxisThreads / 32;
constexpr int kQuads = 256;  // OT-1024: 1024 leaves, four per quad

template <int OP>
constexpr int nvals() { return OP == OP_RMINMAX ? 2 : 1; }

// Value k of the reduction (min and max together: 0 = min, 1 = max).
template <int OP, bool ORD>
__device__ __forceinline__ float comb(int k, float a, float b) {
    if constexpr (OP == OP_RSUM) {
        return __fadd_rn(a, b);
    } else {
        const bool mx = OP == OP_RMAX || (OP == OP_RMINMAX && k == 1);
        if constexpr (ORD) return mx ? cmax2(a, b) : cmin2(a, b);
        else return mx ? fmaxf(a, b) : fminf(a, b);
    }
}

// Identities: +0 for the sum; the ordered max / min start from -inf / +inf as
// the tree's leaves do; the unordered ones start from NaN, which maxNum and
// minNum skip, so a column gives NaN only when every element is NaN.
template <int OP, bool ORD>
__device__ __forceinline__ float ident(int k) {
    if constexpr (OP == OP_RSUM) {
        return 0.0f;
    } else if constexpr (!ORD) {
        return __int_as_float(0x7fffffff);
    } else {
        const bool mx = OP == OP_RMAX || (OP == OP_RMINMAX && k == 1);
        return __int_as_float(mx ? 0xff800000u : 0x7f800000u);
    }
}

__device__ __forceinline__ float ld_col(const float* p) { return ld_stream1(p); }

// Push the subtree value `cur` (the n-th of its block, n counting from 0) onto
// a stack of pending left siblings. After the last push of a block of 2^d
// values, `cur` holds the block's tree.
template <int OP, bool ORD, int N>
__device__ __forceinline__ void push(float (&stk)[6][N], float (&cur)[N], int n) {
    bool carry = true;  // no break: every level index stays a constant, the stack stays in registers
#pragma unroll
    for (int lv = 0; lv < 6; ++lv) {
        const bool bit = (n >> lv) & 1;
#pragma unroll
        for (int k = 0; k < N; ++k) {
            const float t = comb<OP, ORD>(k, stk[lv][k], cur[k]);
            if (carry && !bit) stk[lv][k] = cur[k];
            if (carry && bit) cur[k] = t;
        }
        carry = carry && bit;
    }
}

template <int OP, bool ORD>
__global__ void __launch_bounds__(kAxisThreads, 2) axis_kernel(AxisArgs a) {
    constexpr int N = nvals<OP>();
    __shared__ float g[N][kWarps][32];
    __shared__ unsigned s_ticket;
    const int lane = threadIdx.x & 31;
    const int w = threadIdx.x >> 5;
    const int64_t tile = blockIdx.x;
    const int s = blockIdx.y;
    const int S = gridDim.y;
    const int64_t R = a.extent;
    const int64_t inner = a.inner;
    const int64_t j = tile * 32 + lane;
    const bool jok = j < a.ncols;
    const int64_t o = jok ? j / inner : 0;
    const float* col = a.x + (o * R) * inner + (j - o * inner);

    float res[N];
    if constexpr (ORD) {
        // this warp's block of P consecutive quads in tree order
        const int P = kQuads / (S * kWarps);
        const int p0 = s * (kQuads / S) + w * P;
        float stk[6][N];
        float cur[N];
#pragma unroll
        for (int k = 0; k < N; ++k) {
            cur[k] = ident<OP, ORD>(k);
#pragma unroll
            for (int lv = 0; lv < 6; ++lv) stk[lv][k] = cur[k];
        }
        // the first leaf row of quad position p: 4t, t = 32 * group + bit-reversed lane
        auto first_row = [](int p) { return 4 * (32 * (p >> 5) + static_cast<int>(__brev(p & 31) >> 27)); };
        constexpr int B = 4;  // quads loaded together
        for (int n0 = 0; n0 < P; n0 += B) {
            const int nb = P - n0 < B ? P - n0 : B;
            float lf[B][4][N];
            int e0[B];
#pragma unroll
            for (int b = 0; b < B; ++b) {
                e0[b] = first_row(p0 + n0 + b);
#pragma unroll
                for (int v = 0; v < 4; ++v)
#pragma unroll
                    for (int k = 0; k < N; ++k) lf[b][v][k] = ident<OP, ORD>(k);
            }
            // leaf e folds rows e, e + 1024, ... in increasing order
            const float* qp[B];
            int64_t left[B];  // rows of quad b's first leaf at or after this round
#pragma unroll
            for (int b = 0; b < B; ++b) {
                qp[b] = col + e0[b] * inner;
                left[b] = (jok && b < nb) ? R - e0[b] : 0;
            }
            const int64_t step = 1024 * inner;
            for (int64_t m = 0; m < R; m += 1024) {
                float val[B][4];
#pragma unroll
                for (int b = 0; b < B; ++b)
#pragma unroll
                    for (int v = 0; v < 4; ++v) val[b][v] = v < left[b] ? ld_col(qp[b] + v * inner) : 0.0f;
#pragma unroll
                for (int b = 0; b < B; ++b) {
#pragma unroll
                    for (int v = 0; v < 4; ++v)
                        if (v < left[b]) {
#pragma unroll
                            for (int k = 0; k < N; ++k) lf[b][v][k] = comb<OP, ORD>(k, lf[b][v][k], val[b][v]);
                        }
                    qp[b] += step;
                    left[b] -= 1024;
                }
            }
#pragma unroll
            for (int b = 0; b < B; ++b) {
                if (b < nb) {
                    float q[N];
#pragma unroll
                    for (int k = 0; k < N; ++k)
                        q[k] = comb<OP, ORD>(k, comb<OP, ORD>(k, lf[b][0][k], lf[b][1][k]),
                                             comb<OP, ORD>(k, lf[b][2][k], lf[b][3][k]));
                    push<OP, ORD, N>(stk, q, n0 + b);
#pragma unroll
                    for (int k = 0; k < N; ++k) cur[k] = q[k];
                }
            }
        }
#pragma unroll
        for (int k = 0; k < N; ++k) res[k] = cur[k];
    } else {
        // rows [r0, r1) of this split, interleaved over the warps, eight loads in flight
        const int64_t base = R / S, extra = R % S;
        const int64_t r0 = s * base + (s < extra ? s : extra);
        const int64_t r1 = r0 + base + (s < extra ? 1 : 0);
        float acc[4][N];
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
            for (int k = 0; k < N; ++k) acc[u][k] = ident<OP, ORD>(k);
        if (jok) {
            int64_t r = r0 + w;
            for (; r + 7 * kWarps < r1; r += 8 * kWarps) {
                float v[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) v[u] = ld_col(col + (r + u * kWarps) * inner);
#pragma unroll
                for (int u = 0; u < 8; ++u)
#pragma unroll
                    for (int k = 0; k < N; ++k) acc[u & 3][k] = comb<OP, ORD>(k, acc[u & 3][k], v[u]);
            }
            for (; r < r1; r += kWarps) {
                const float v = ld_col(col + r * inner);
#pragma unroll
                for (int k = 0; k < N; ++k) acc[0][k] = comb<OP, ORD>(k, acc[0][k], v);
            }
        }
#pragma unroll
        for (int k = 0; k < N; ++k)
            res[k] = comb<OP, ORD>(k, comb<OP, ORD>(k, acc[0][k], acc[1][k]), comb<OP, ORD>(k, acc[2][k], acc[3][k]));
    }

    // the CTA's 8 blocks, combined in order by warp 0
#pragma unroll
    for (int k = 0; k < N; ++k) g[k][w][lane] = res[k];
    __syncthreads();
    if (w != 0) return;
    float v[N];
#pragma unroll
    for (int k = 0; k < N; ++k) {
        const float a01 = comb<OP, ORD>(k, g[k][0][lane], g[k][1][lane]);
        const float a23 = comb<OP, ORD>(k, g[k][2][lane], g[k][3][lane]);
        const float a45 = comb<OP, ORD>(k, g[k][4][lane], g[k][5][lane]);
        const float a67 = comb<OP, ORD>(k, g[k][6][lane], g[k][7][lane]);
        v[k] = comb<OP, ORD>(k, comb<OP, ORD>(k, a01, a23), comb<OP, ORD>(k, a45, a67));
    }
    if (S > 1) {
        // publish this split's partial; the last CTA of the tile combines all of them
        float* mine = a.part + ((tile * S + s) * N) * 32;
#pragma unroll
        for (int k = 0; k < N; ++k) mine[k * 32 + lane] = v[k];
        __threadfence();
        __syncwarp();
        if (lane == 0) s_ticket = atomicAdd(a.ticket + tile, 1u);
        __syncwarp();
        if (s_ticket != static_cast<unsigned>(S - 1)) return;
        __threadfence();
        float stk[6][N];
        for (int q = 0; q < S; ++q) {
            const float* pq = a.part + ((tile * S + q) * N) * 32;
#pragma unroll
            for (int k = 0; k < N; ++k) v[k] = __ldcg(pq + k * 32 + lane);
            push<OP, ORD, N>(stk, v, q);
        }
        if (lane == 0) a.ticket[tile] = 0u;
    }
    if (jok) {
        a.out[j] = v[0];
        if constexpr (N == 2) a.out2[j] = v[1];
    }
}

template <int OP>
cudaError_t launch(bool ordered, const AxisArgs& a, int64_t tiles, int splits, cudaStream_t stream) {
    const dim3 grid(static_cast<unsigned>(tiles), static_cast<unsigned>(splits));
    if (ordered)
        axis_kernel<OP, true><<<grid, kAxisThreads, 0, stream>>>(a);
    else
        axis_kernel<OP, false><<<grid, kAxisThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace axis

cudaError_t launch_axis(int op, bool ordered, const AxisArgs& a, int64_t tiles, int splits, cudaStream_t stream) {
    switch (op) {
        case TR_OP_ROW_SUM: return axis::launch<OP_RSUM>(ordered, a, tiles, splits, stream);
        case TR_OP_ROW_MAX: return axis::launch<OP_RMAX>(ordered, a, tiles, splits, stream);
        case TR_OP_ROW_MIN: return axis::launch<OP_RMIN>(ordered, a, tiles, splits, stream);
        case TR_OP_ROW_MINMAX: return axis::launch<OP_RMINMAX>(ordered, a, tiles, splits, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace tr
