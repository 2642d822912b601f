// The fold policies (TR_ORDER_FOLD_LEFT / TR_ORDER_FOLD_RIGHT).
//
// "TIRx Metal reduction lowering" §1 (ReductionPolicy): a reduction may be
// restricted to fold_left or fold_right, and an ordered reduction stays
// ordered. fold_left visits the columns in increasing order with the
// accumulator as the left operand (acc = acc + t_c), fold_right in decreasing
// order with the accumulator as the right operand (acc = t_c + acc), both
// from the identity. The operators keep the op sequences of the ordered tree
// with each tree reduction replaced by the fold, and the same exp and log.
//
// A fold is one chain of dependent additions per row: the chain is the floor
// of the run time (4 cycles an add), so each row gets one warp. The 32 lanes
// load 128 columns at a time (coalesced float4) and compute their terms (the
// exponentials of softmax and cross-entropy, the squares of the norms) in
// parallel; the warp then runs the chain on terms broadcast by shuffles while
// the loads of the next 128 columns are in flight. Max and min need no
// chain: without a NaN in the row the canonical fold's result is the largest
// (smallest) element in the total order with -0 below +0, whatever the
// order, so the lanes fold integer keys in any order; a row with a NaN is
// folded canonically by lane 0.
#include <climits>
#include <cuda_runtime.h>
#include <stdint.h>

#include "tr_device.cuh"
#include "tr_internal.h"
#include "tr_ot.cuh"

namespace tr {
namespace fold {

using ordered::exp_ot;
using ordered::log_ot;

constexpr int kWarps = 2;    // rows per CTA: few, so the rows spread over every SM (the chains share an SM's shuffle throughput)
constexpr int kChunk = 128;  // columns per step: 32 lanes x 4

// Columns c0 .. c0 + 3 of a row (0 outside it).
__device__ __forceinline__ void load4(const float* r, int cols, int64_t c0, bool aligned, float (&q)[4]) {
    if (aligned && c0 + 3 < cols) {
        const float4 v = ld_stream4(r + c0);
        q[0] = v.x; q[1] = v.y; q[2] = v.z; q[3] = v.w;
    } else {
#pragma unroll
        for (int v = 0; v < 4; ++v) q[v] = c0 + v < cols ? ld_stream1(r + c0 + v) : 0.0f;
    }
}

__device__ __forceinline__ void param4(const float* p, int cols, int64_t c0, float (&q)[4]) {
    if (aligned16(p + c0) && c0 + 3 < cols) {
        const float4 v = ld_param4(p + c0);
        q[0] = v.x; q[1] = v.y; q[2] = v.z; q[3] = v.w;
    } else {
#pragma unroll
        for (int v = 0; v < 4; ++v) q[v] = c0 + v < cols ? __ldg(p + c0 + v) : 0.0f;
    }
}

__device__ __forceinline__ void store4(float* r, int cols, int64_t c0, const float (&o)[4]) {
    if (aligned16(r + c0) && c0 + 3 < cols) {
        st4(r + c0, make_float4(o[0], o[1], o[2], o[3]));
    } else {
#pragma unroll
        for (int v = 0; v < 4; ++v)
            if (c0 + v < cols) r[c0 + v] = o[v];
    }
}

struct AddC {
    static __device__ __forceinline__ float f(float a, float b) { return __fadd_rn(a, b); }
};
struct MaxC {
    static __device__ __forceinline__ float f(float a, float b) { return cmax2(a, b); }
};
struct MinC {
    static __device__ __forceinline__ float f(float a, float b) { return cmin2(a, b); }
};

template <int OP, bool RIGHT>
__global__ void __launch_bounds__(kWarps * 32) fold_kernel(const RowArgs a) {
    const int lane = threadIdx.x & 31;
    const int w = threadIdx.x >> 5;
    const int64_t row = static_cast<int64_t>(blockIdx.x) * kWarps + w;
    if (row >= a.rows) return;  // whole warps leave; nothing below synchronises the CTA
    const int cols = a.cols;
    const float* xr = a.x + row * cols;
    const bool al = aligned16(xr);
    const int nch = (cols + kChunk - 1) / kChunk;
    const int64_t lc = 4 * lane;  // this lane's first column within a chunk

    // The fold of term(x_c) over the row in the policy's order, starting from
    // init. Every lane computes the terms of its 4 columns, then the whole
    // warp runs the chain, each term broadcast by a shuffle (independent of the
    // chain, so the shuffles issue ahead of the dependent adds) while the next
    // 128 columns load. Every lane ends with the result.
    auto fold_seq = [&](auto term, auto comb, float init) -> float {
        using C = decltype(comb);
        float acc = init;
        // the i-th chunk visited and the loads of four of them at a time
        auto chunk_of = [&](int i) { return RIGHT ? nch - 1 - i : i; };
        auto load_group = [&](int i0, float (&g)[4][4]) {
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                if (i0 + u < nch) {
                    load4(xr, cols, static_cast<int64_t>(chunk_of(i0 + u)) * kChunk + lc, al, g[u]);
                } else {
#pragma unroll
                    for (int v = 0; v < 4; ++v) g[u][v] = 0.0f;
                }
            }
        };
        float cur[4][4], nxt[4][4];
        load_group(0, cur);
        for (int i0 = 0; i0 < nch; i0 += 4) {
            if (i0 + 4 < nch) load_group(i0 + 4, nxt);  // four chunks of chain time to arrive
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int i = i0 + u;
                if (i < nch) {
                    const int ch = chunk_of(i);
                    float t[4];
#pragma unroll
                    for (int v = 0; v < 4; ++v) t[v] = term(cur[u][v]);
                    const int n = cols - ch * kChunk < kChunk ? cols - ch * kChunk : kChunk;
                    if (n == kChunk) {
                        // the shuffle of element q + 16 issues right after the combine
                        // of element q, in the shadow of the combine's latency (a warp
                        // issues in order); visit position q is column RIGHT ? 127 - q : q
                        float sh[16];
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            const int k = RIGHT ? kChunk - 1 - e : e;
                            sh[e] = __shfl_sync(kFull, t[k & 3], k >> 2);
                        }
#pragma unroll
                        for (int q = 0; q < kChunk; ++q) {
                            acc = RIGHT ? C::f(sh[q & 15], acc) : C::f(acc, sh[q & 15]);
                            if (q + 16 < kChunk) {
                                const int k = RIGHT ? kChunk - 1 - (q + 16) : q + 16;
                                sh[q & 15] = __shfl_sync(kFull, t[k & 3], k >> 2);
                            }
                        }
                    } else {
                        for (int q = 0; q < n; ++q) {
                            const int k = RIGHT ? n - 1 - q : q;
                            const int v = k & 3;
                            const float tk = __shfl_sync(kFull, v == 0 ? t[0] : v == 1 ? t[1] : v == 2 ? t[2] : t[3], k >> 2);
                            acc = RIGHT ? C::f(tk, acc) : C::f(acc, tk);
                        }
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
                for (int v = 0; v < 4; ++v) cur[u][v] = nxt[u][v];
        }
        return acc;
    };
    auto ident = [](float v) { return v; };

    // canonical max (want_max) or min of the row: integer keys in any order,
    // the canonical fold only for a row that holds a NaN
    auto extreme = [&](bool want_max, float& lo, float& hi) {
        int kmax = INT_MIN, kmin = INT_MAX;
        for (int ch0 = 0; ch0 < nch; ch0 += 4) {  // four chunks' loads in flight
            float q[4][4];
#pragma unroll
            for (int u = 0; u < 4; ++u) load4(xr, cols, static_cast<int64_t>(ch0 + u) * kChunk + lc, al, q[u]);
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
                for (int v = 0; v < 4; ++v)
                    if (static_cast<int64_t>(ch0 + u) * kChunk + lc + v < cols) {
                        const int k = order_key(q[u][v]);
                        kmax = max(kmax, k);
                        kmin = min(kmin, k);
                    }
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
            kmax = max(kmax, __shfl_xor_sync(kFull, kmax, o));
            kmin = min(kmin, __shfl_xor_sync(kFull, kmin, o));
        }
        const bool nan = kmax > 0x7f800000 || kmin < order_key(__int_as_float(0xff800000u));
        if (!nan) {
            lo = from_order_key(kmin);
            hi = from_order_key(kmax);
            return;
        }
        hi = want_max ? fold_seq(ident, MaxC{}, __int_as_float(0xff800000u)) : 0.0f;
        lo = fold_seq(ident, MinC{}, __int_as_float(0x7f800000u));
    };

    // y_c = out(x_c, c) for every column (any order)
    auto emit = [&](auto out) {
        float* yr = a.y + row * cols;
        for (int ch0 = 0; ch0 < nch; ch0 += 4) {  // four chunks' loads in flight
            float q[4][4];
#pragma unroll
            for (int u = 0; u < 4; ++u) load4(xr, cols, static_cast<int64_t>(ch0 + u) * kChunk + lc, al, q[u]);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int64_t c0 = static_cast<int64_t>(ch0 + u) * kChunk + lc;
                if (c0 < cols) {
                    float o[4];
                    out(q[u], c0, o);
                    store4(yr, cols, c0, o);
                }
            }
        }
    };
    const float n = static_cast<float>(cols);

    if constexpr (OP == OP_SOFTMAX || OP == OP_XENT) {
        float lo, m;
        extreme(true, lo, m);
        const float s = fold_seq([m](float v) { return exp_ot(__fsub_rn(v, m)); }, AddC{}, 0.0f);
        if constexpr (OP == OP_SOFTMAX) {
            const float inv = __fdiv_rn(1.0f, s);
            emit([m, inv](const float (&q)[4], int64_t, float (&o)[4]) {
#pragma unroll
                for (int v = 0; v < 4; ++v) o[v] = __fmul_rn(exp_ot(__fsub_rn(q[v], m)), inv);
            });
        } else if (lane == 0) {
            const int64_t label = a.labels[row];
            const float sel = (label >= 0 && label < cols) ? __ldg(xr + label) : 0.0f;
            a.loss[row] = __fsub_rn(__fadd_rn(log_ot(s), m), sel);
        }
    } else if constexpr (OP == OP_RMSNORM) {
        const float ss = fold_seq([](float v) { return __fmul_rn(v, v); }, AddC{}, 0.0f);
        const float inv = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ss, n), a.eps)));
        emit([&](const float (&q)[4], int64_t c0, float (&o)[4]) {
            float wq[4] = {1.0f, 1.0f, 1.0f, 1.0f};
            if (a.has_w) param4(a.w, cols, c0, wq);
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                const float u = __fmul_rn(q[v], inv);
                o[v] = a.has_w ? __fmul_rn(u, wq[v]) : u;
            }
        });
    } else if constexpr (OP == OP_LAYERNORM) {
        const float mean = __fdiv_rn(fold_seq(ident, AddC{}, 0.0f), n);
        const float var = __fdiv_rn(fold_seq([mean](float v) {
            const float c = __fsub_rn(v, mean);
            return __fmul_rn(c, c);
        }, AddC{}, 0.0f), n);
        const float inv = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(var, a.eps)));
        emit([&](const float (&q)[4], int64_t c0, float (&o)[4]) {
            float gq[4] = {1.0f, 1.0f, 1.0f, 1.0f}, bq[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            if (a.has_w) param4(a.w, cols, c0, gq);
            if (a.has_b) param4(a.b, cols, c0, bq);
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                float u = __fmul_rn(__fsub_rn(q[v], mean), inv);
                if (a.has_w) u = __fmul_rn(u, gq[v]);
                if (a.has_b) u = __fadd_rn(u, bq[v]);
                o[v] = u;
            }
        });
    } else if constexpr (OP == OP_RSUM) {
        const float s = fold_seq(ident, AddC{}, 0.0f);
        if (lane == 0) a.loss[row] = s;
    } else {
        float lo, hi;
        extreme(OP != OP_RMIN, lo, hi);
        if (lane == 0) {
            if constexpr (OP == OP_RMAX) a.loss[row] = hi;
            if constexpr (OP == OP_RMIN) a.loss[row] = lo;
            if constexpr (OP == OP_RMINMAX) {
                a.loss[row] = lo;
                a.out2[row] = hi;
            }
        }
    }
}

template <int OP>
cudaError_t launch_op(bool right, const RowArgs& a, cudaStream_t stream) {
    const dim3 grid(static_cast<unsigned>((a.rows + kWarps - 1) / kWarps));
    if (right)
        fold_kernel<OP, true><<<grid, kWarps * 32, 0, stream>>>(a);
    else
        fold_kernel<OP, false><<<grid, kWarps * 32, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace fold

cudaError_t launch_fold(int op, bool right, const RowArgs& a, cudaStream_t stream) {
    switch (op) {
        case TR_OP_SOFTMAX: return fold::launch_op<OP_SOFTMAX>(right, a, stream);
        case TR_OP_RMSNORM: return fold::launch_op<OP_RMSNORM>(right, a, stream);
        case TR_OP_LAYERNORM: return fold::launch_op<OP_LAYERNORM>(right, a, stream);
        case TR_OP_CROSS_ENTROPY: return fold::launch_op<OP_XENT>(right, a, stream);
        case TR_OP_ROW_SUM: return fold::launch_op<OP_RSUM>(right, a, stream);
        case TR_OP_ROW_MAX: return fold::launch_op<OP_RMAX>(right, a, stream);
        case TR_OP_ROW_MIN: return fold::launch_op<OP_RMIN>(right, a, stream);
        case TR_OP_ROW_MINMAX: return fold::launch_op<OP_RMINMAX>(right, a, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace tr
