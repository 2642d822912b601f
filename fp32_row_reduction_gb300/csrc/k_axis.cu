// Reductions over a non-last axis: x viewed as [outer, extent, inner] (row
// major, contiguous), out[o * inner + i] = reduce over r of x[o, r, i].
//
// "TIRx Metal reduction lowering" (Reductions inside composed groups): the
// reduced axis need not be the last memory dimension; each output is one
// independent collective, missing elements contribute the identity, and the
// canonical FP32 add / max / min are the reducers. On GB300 the 32 lanes of a
// warp take 32 consecutive output columns (32 float4 column quads when inner
// is a multiple of 4 and x is 16-byte aligned), so every load of a warp reads
// 128 (512) consecutive bytes of one x row. The reduced axis is spread over
// the 8 warps of a CTA and, when the columns alone cannot fill the GPU, over
// `splits` CTAs whose partials the last CTA to arrive combines (a ticket, no
// waiting).
//
// Three ways to fold a column:
// * free (unordered policy): rows split evenly, four accumulators per column,
//   any combine order;
// * tree (ordered sum): the fixed tree OT-1024 on the column (leaf k folds the
//   elements r = k mod 1024 in increasing r, then the fixed tree above the
//   1024 leaves), bit for bit the value of the row reductions for the same
//   vector. That tree is a perfect binary tree over the leaf slots in the
//   order (group w, bit-reversed lane, slot v) of the row kernels' thread
//   layout, so any power-of-two block of consecutive slots is a subtree: every
//   warp folds its block of quads with a stack of pending subtrees, the CTA
//   combines its 8 blocks in order, the last CTA the splits' blocks in order;
// * key (ordered max / min): without a NaN the canonical max (min) of the tree
//   is the largest (smallest) element in the total order with -0 below +0, in
//   any grouping, which is the signed order of the integer keys; the rows are
//   folded freely in key space, and a tile with a NaN in any column is
//   recomputed by its last CTA with the canonical tree.
#include <climits>
#include <type_traits>
#include <cuda_runtime.h>
#include <stdint.h>

#include "tr_device.cuh"
#include "tr_internal.h"

namespace tr {
namespace axis {

constexpr int kWarps = kAxisThreads / 32;
constexpr int kQuads = 256;  // OT-1024: 1024 leaves, four per quad
// STAGED: the tree mode for a reduced axis of at most 1024 rows (one element
// per leaf), with the split's rows staged in shared memory first, so that
// every load of the CTA is in flight at once before the tree is folded.
enum Mode : int { FREE = 0, TREE = 1, KEY = 2, STAGED = 3 };

template <int OP, int MODE, int TERM = AXIS_PLAIN>
constexpr int nvals() { return MODE == KEY ? 2 : (OP == OP_RMINMAX || TERM == AXIS_LN_BOTH ? 2 : 1); }

// Value k of the free / tree reductions (min and max together: 0 = min, 1 = max).
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

// Accumulators of each mode, as 32-bit patterns in floats. Free max / min
// start from NaN, which maxNum / minNum skip (a column gives NaN only when all
// of it is NaN); key mode keeps (min key, max key).
template <int OP, int MODE>
__device__ __forceinline__ float acc_init(int k) {
    if constexpr (MODE == KEY) return __int_as_float(k == 0 ? INT_MAX : INT_MIN);
    else if constexpr (OP == OP_RSUM) return 0.0f;
    else return __int_as_float(0x7fffffff);
}
template <int OP, int MODE>
__device__ __forceinline__ float acc_fold(int k, float acc, float x) {
    if constexpr (MODE == KEY) {
        const int a = __float_as_int(acc), e = order_key(x);
        return __int_as_float(k == 0 ? min(a, e) : max(a, e));
    } else {
        return comb<OP, MODE == TREE>(k, acc, x);
    }
}
template <int OP, int MODE>
__device__ __forceinline__ float acc_comb(int k, float a, float b) {
    if constexpr (MODE == KEY) {
        const int x = __float_as_int(a), y = __float_as_int(b);
        return __int_as_float(k == 0 ? min(x, y) : max(x, y));
    } else {
        return comb<OP, MODE == TREE>(k, a, b);
    }
}

// The canonical reducers of the tree, one value at a time.
struct AddF {
    static __device__ __forceinline__ float id() { return 0.0f; }
    static __device__ __forceinline__ float f(float a, float b) { return __fadd_rn(a, b); }
};
struct CMaxF {
    static __device__ __forceinline__ float id() { return __int_as_float(0xff800000u); }
    static __device__ __forceinline__ float f(float a, float b) { return cmax2(a, b); }
};
struct CMinF {
    static __device__ __forceinline__ float id() { return __int_as_float(0x7f800000u); }
    static __device__ __forceinline__ float f(float a, float b) { return cmin2(a, b); }
};

template <int V>
__device__ __forceinline__ void ld_cols(const float* p, float (&v)[V]) {
    if constexpr (V == 4) {
        const float4 q = ld_stream4(p);
        v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
    } else {
        v[0] = ld_stream1(p);
    }
}

// Element (row r) of this thread's V columns: x itself, or a backward term.
// Ordered (O): each binary32 step rounded in the written order.
template <int TERM, bool O, int V>
__device__ __forceinline__ void ld_elem(const AxisArgs& a, const float* p, int64_t r, float (&v)[V]) {
    if constexpr (TERM == AXIS_PLAIN) {
        ld_cols<V>(p, v);
    } else {
        float d[V];
        ld_cols<V>(a.dy + (p - a.x), d);
        if constexpr (TERM == AXIS_LN_BETA) {
#pragma unroll
            for (int c = 0; c < V; ++c) v[c] = d[c];
        } else {
            float x[V];
            ld_cols<V>(p, x);
            const float s0 = __ldg(a.sa + r);
            if constexpr (TERM == AXIS_RMS_W) {
#pragma unroll
                for (int c = 0; c < V; ++c) v[c] = O ? __fmul_rn(__fmul_rn(d[c], x[c]), s0) : d[c] * x[c] * s0;
            } else {
                const float s1 = __ldg(a.sb + r);
#pragma unroll
                for (int c = 0; c < V; ++c)
                    v[c] = O ? __fmul_rn(d[c], __fmul_rn(__fsub_rn(x[c], s0), s1)) : d[c] * ((x[c] - s0) * s1);
            }
        }
    }
}

// 4-byte asynchronous copy global -> shared.
__device__ __forceinline__ void cp_async4(float* dst, const float* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// The N values an element contributes: the LayerNorm's (dy xh, dy) for
// AXIS_LN_BOTH, otherwise the element (or term) itself for every value.
template <int TERM, bool O, int V, int N>
__device__ __forceinline__ void ld_terms(const AxisArgs& a, const float* p, int64_t r, float (&e)[N][V]) {
    if constexpr (TERM == AXIS_LN_BOTH) {
        static_assert(N == 2, "two gradients");
        float d[V], x[V];
        ld_cols<V>(a.dy + (p - a.x), d);
        ld_cols<V>(p, x);
        const float s0 = __ldg(a.sa + r), s1 = __ldg(a.sb + r);
#pragma unroll
        for (int c = 0; c < V; ++c) {
            e[0][c] = O ? __fmul_rn(d[c], __fmul_rn(__fsub_rn(x[c], s0), s1)) : d[c] * ((x[c] - s0) * s1);
            e[1][c] = d[c];
        }
    } else {
        ld_elem<TERM, O, V>(a, p, r, e[0]);
#pragma unroll
        for (int k = 1; k < N; ++k)
#pragma unroll
            for (int c = 0; c < V; ++c) e[k][c] = e[0][c];
    }
}

// Push the subtree value `cur` (the n-th of its block, n from 0) onto a stack
// of pending left siblings; after the last push of a block of 2^d values,
// `cur` holds the block's tree. No break: every level index stays a constant,
// so the stack lives in registers.
template <class F, int V>
__device__ __forceinline__ void push(float (&stk)[5][V], float (&cur)[V], int n) {
    bool carry = true;
#pragma unroll
    for (int lv = 0; lv < 5; ++lv) {
        const bool bit = (n >> lv) & 1;
#pragma unroll
        for (int c = 0; c < V; ++c) {
            const float t = F::f(stk[lv][c], cur[c]);
            if (carry && !bit) stk[lv][c] = cur[c];
            if (carry && bit) cur[c] = t;
        }
        carry = carry && bit;
    }
}

// The OT-1024 subtree over quad positions p0 .. p0 + P - 1 (P a power of two,
// at most 32) of this thread's columns; `col` points at row 0 of them.
template <class F, int V, int B, int TERM = AXIS_PLAIN>  // B quads loaded together
__device__ __forceinline__ void tree_block(const AxisArgs& a, const float* col, bool jok, int64_t R, int64_t inner,
                                           int p0, int P, float (&out)[V]) {
    float stk[5][V];
    float cur[V];
#pragma unroll
    for (int c = 0; c < V; ++c) {
        cur[c] = F::id();
#pragma unroll
        for (int lv = 0; lv < 5; ++lv) stk[lv][c] = cur[c];
    }
    const int64_t step = 1024 * inner;
    for (int n0 = 0; n0 < P; n0 += B) {
        const int nb = P - n0 < B ? P - n0 : B;
        float lf[B][4][V];
        const float* qp[B];
        int64_t left[B];  // rows of the quad's first leaf from this round on
        int64_t rowb[B];  // the row of the quad's first leaf in this round
#pragma unroll
        for (int b = 0; b < B; ++b) {
            // first leaf row of position p: 4t, t = 32 * group + bit-reversed lane
            const int p = p0 + n0 + b;
            const int e0 = 4 * (32 * (p >> 5) + static_cast<int>(__brev(p & 31) >> 27));
            qp[b] = col + e0 * inner;
            rowb[b] = e0;
            left[b] = (jok && b < nb) ? R - e0 : 0;
#pragma unroll
            for (int v = 0; v < 4; ++v)
#pragma unroll
                for (int c = 0; c < V; ++c) lf[b][v][c] = F::id();
        }
        // leaf e folds rows e, e + 1024, ... in increasing order
        for (int64_t m = 0; m < R; m += 1024) {
            float val[B][4][V];
#pragma unroll
            for (int b = 0; b < B; ++b)
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    if (v < left[b]) {
                        ld_elem<TERM, true, V>(a, qp[b] + v * inner, rowb[b] + v, val[b][v]);
                    } else {
#pragma unroll
                        for (int c = 0; c < V; ++c) val[b][v][c] = 0.0f;
                    }
                }
#pragma unroll
            for (int b = 0; b < B; ++b) {
#pragma unroll
                for (int v = 0; v < 4; ++v)
                    if (v < left[b]) {
#pragma unroll
                        for (int c = 0; c < V; ++c) lf[b][v][c] = F::f(lf[b][v][c], val[b][v][c]);
                    }
                qp[b] += step;
                left[b] -= 1024;
                rowb[b] += 1024;
            }
        }
#pragma unroll
        for (int b = 0; b < B; ++b) {
            if (b < nb) {
                float q[V];
#pragma unroll
                for (int c = 0; c < V; ++c)
                    q[c] = F::f(F::f(lf[b][0][c], lf[b][1][c]), F::f(lf[b][2][c], lf[b][3][c]));
                push<F, V>(stk, q, n0 + b);
#pragma unroll
                for (int c = 0; c < V; ++c) cur[c] = q[c];
            }
        }
    }
#pragma unroll
    for (int c = 0; c < V; ++c) out[c] = cur[c];
}

// In-order tree over the 8 warps' values g[w][i].
template <class F>
__device__ __forceinline__ float cta_tree(const float (*g)[kAxisCols * 4], int i) {
    return F::f(F::f(F::f(g[0][i], g[1][i]), F::f(g[2][i], g[3][i])),
                F::f(F::f(g[4][i], g[5][i]), F::f(g[6][i], g[7][i])));
}

// Resident CTAs per SM each mode is built for (the host sizes its splits to fit one wave).
template <int MODE>
constexpr int min_ctas() { return MODE == TREE || MODE == STAGED ? kAxisCtasTree : kAxisCtasFree; }

template <int OP, int MODE, int V, int TERM = AXIS_PLAIN>
__global__ void __launch_bounds__(kAxisThreads, min_ctas<MODE>()) axis_kernel(AxisArgs a) {
    constexpr int N = nvals<OP, MODE, TERM>();
    constexpr int W = kAxisCols * V;  // columns of the tile
    __shared__ float g[N][kWarps][kAxisCols * 4];
    __shared__ unsigned s_last;
    const int lane = threadIdx.x & 31;
    const int w = threadIdx.x >> 5;
    const int64_t tile = blockIdx.x;
    const int s = blockIdx.y;
    const int S = gridDim.y;
    const int64_t R = a.extent;
    const int64_t inner = a.inner;
    const int64_t j = tile * W + lane * V;  // first column of this thread (its V columns share o)
    const bool jok = j < a.ncols;
    const int64_t o = jok ? j / inner : 0;
    const float* col = a.x + (o * R) * inner + (j - o * inner);

    float res[N][V];
    if constexpr (MODE == STAGED) {
        static_assert(OP == OP_RSUM && V == 1, "the staged tree folds sums of single columns");
        // rows [rs, re) hold the leaves of this split's quad positions (S <= 8);
        // their x (and dy) are copied to shared memory asynchronously, all at once
        constexpr bool two = TERM == AXIS_RMS_W || TERM == AXIS_LN_GAMMA || TERM == AXIS_LN_BOTH;
        extern __shared__ float stage[];
        const int64_t per = 1024 / S;
        const int64_t rows_cta = R < per ? R : per;
        float* sx = stage;                 // x, or dy for the dbeta term
        float* sd = stage + rows_cta * 32;  // dy of the two-input terms
        const int64_t rs = static_cast<int64_t>(s) * per;
        const int64_t re = rs + per < R ? rs + per : R;
        if (jok) {
            // pointers advance by a stride: no 64-bit product per copy
            const float* gcol = TERM == AXIS_PLAIN ? col : a.dy + (col - a.x);
            const int64_t step = kWarps * inner;
            const float* src = (TERM == AXIS_LN_BETA ? gcol : col) + (rs + w) * inner;
            const float* srd = gcol + (rs + w) * inner;
            float* dx = sx + w * 32 + lane;
            float* dd = sd + w * 32 + lane;
            for (int64_t r = rs + w; r < re; r += kWarps) {
                cp_async4(dx, src);
                if constexpr (two) cp_async4(dd, srd);
                src += step;
                srd += step;
                dx += kWarps * 32;
                dd += kWarps * 32;
            }
        }
        cp_async_wait_all();
        __syncthreads();
        // value k of the element of row rs + i
        auto elem = [&](int i, int64_t r, int k) {
            const int at = i * 32 + lane;
            if constexpr (TERM == AXIS_PLAIN || TERM == AXIS_LN_BETA) {
                return sx[at];
            } else if constexpr (TERM == AXIS_RMS_W) {
                return __fmul_rn(__fmul_rn(sd[at], sx[at]), __ldg(a.sa + r));
            } else {
                if (TERM == AXIS_LN_BOTH && k == 1) return sd[at];
                return __fmul_rn(sd[at], __fmul_rn(__fsub_rn(sx[at], __ldg(a.sa + r)), __ldg(a.sb + r)));
            }
        };
        // this warp's P (a power of two, at most 32) quad positions, then the
        // perfect tree over them, adjacent pairs level by level; unrolled for at
        // most 8 positions (the usual splits) or for 32, so only one short path runs
        const int P = kQuads / (S * kWarps);
        const int p0 = s * (kQuads / S) + w * P;
        auto fold_positions = [&](auto pmax) {
            constexpr int PM = decltype(pmax)::value;
            float q[N][PM];
#pragma unroll
            for (int n = 0; n < PM; ++n) {
                if (n < P) {
                    const int p = p0 + n;
                    const int e0 = 4 * (32 * (p >> 5) + static_cast<int>(__brev(p & 31) >> 27));
#pragma unroll
                    for (int k = 0; k < N; ++k) {
                        float l[4];
#pragma unroll
                        for (int v = 0; v < 4; ++v)
                            l[v] = e0 + v < R ? __fadd_rn(0.0f, elem(static_cast<int>(e0 + v - rs), e0 + v, k)) : 0.0f;
                        q[k][n] = __fadd_rn(__fadd_rn(l[0], l[1]), __fadd_rn(l[2], l[3]));
                    }
                }
            }
#pragma unroll
            for (int wd = 1; wd < PM; wd *= 2)
#pragma unroll
                for (int n = 0; n + wd < PM; n += 2 * wd)
                    if (n + wd < P)
#pragma unroll
                        for (int k = 0; k < N; ++k) q[k][n] = __fadd_rn(q[k][n], q[k][n + wd]);
#pragma unroll
            for (int k = 0; k < N; ++k) res[k][0] = q[k][0];
        };
        if (P <= 8)
            fold_positions(std::integral_constant<int, 8>{});
        else
            fold_positions(std::integral_constant<int, 32>{});
    } else if constexpr (MODE == TREE) {
        static_assert(OP == OP_RSUM, "the tree mode folds sums");
        const int P = kQuads / (S * kWarps);
        // quads loaded together: fewer when each element is a term of two loads
        constexpr int B = V == 4 ? 1 : (TERM == AXIS_PLAIN ? 4 : 2);
        tree_block<AddF, V, B, TERM>(a, col, jok, R, inner, s * (kQuads / S) + w * P, P, res[0]);
    } else {
        // rows [r0, r1) of this split, interleaved over the warps
        const int64_t base = R / S, extra = R % S;
        const int64_t r0 = s * base + (s < extra ? s : extra);
        const int64_t r1 = r0 + base + (s < extra ? 1 : 0);
        // loads in flight per thread (a term loads two elements)
        constexpr int U = (V == 4 ? 4 : 8) / (TERM == AXIS_PLAIN || TERM == AXIS_LN_BETA ? 1 : 2);
        static_assert(MODE != TREE || TERM != AXIS_LN_BOTH, "the register tree takes one term");
        float acc[4][N][V];
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
            for (int k = 0; k < N; ++k)
#pragma unroll
                for (int c = 0; c < V; ++c) acc[u][k][c] = acc_init<OP, MODE>(k);
        if (jok) {
            for (int64_t r = r0 + w; r < r1; r += U * kWarps) {
                float v[U][N][V];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    if (r + u * kWarps < r1) {
                        ld_terms<TERM, false, V, N>(a, col + (r + u * kWarps) * inner, r + u * kWarps, v[u]);
                    } else {
#pragma unroll
                        for (int k = 0; k < N; ++k)
#pragma unroll
                            for (int c = 0; c < V; ++c) v[u][k][c] = 0.0f;
                    }
                }
#pragma unroll
                for (int u = 0; u < U; ++u)
                    if (r + u * kWarps < r1) {
#pragma unroll
                        for (int k = 0; k < N; ++k)
#pragma unroll
                            for (int c = 0; c < V; ++c)
                                acc[u & 3][k][c] = acc_fold<OP, MODE>(k, acc[u & 3][k][c], v[u][k][c]);
                    }
            }
        }
#pragma unroll
        for (int k = 0; k < N; ++k)
#pragma unroll
            for (int c = 0; c < V; ++c)
                res[k][c] = acc_comb<OP, MODE>(k, acc_comb<OP, MODE>(k, acc[0][k][c], acc[1][k][c]),
                                               acc_comb<OP, MODE>(k, acc[2][k][c], acc[3][k][c]));
    }

    // the CTA's 8 blocks, combined in order by warp 0
#pragma unroll
    for (int k = 0; k < N; ++k)
#pragma unroll
        for (int c = 0; c < V; ++c) g[k][w][lane * V + c] = res[k][c];
    __syncthreads();
    float v[N][V];
    if (w == 0) {
#pragma unroll
        for (int k = 0; k < N; ++k)
#pragma unroll
            for (int c = 0; c < V; ++c) {
                const int i = lane * V + c;
                auto f = [k](float x, float y) { return acc_comb<OP, MODE>(k, x, y); };
                v[k][c] = f(f(f(g[k][0][i], g[k][1][i]), f(g[k][2][i], g[k][3][i])),
                            f(f(g[k][4][i], g[k][5][i]), f(g[k][6][i], g[k][7][i])));
            }
    }
    if (S > 1) {
        // publish this split's partial; the last CTA of the tile combines all of them
        if (w == 0) {
#pragma unroll
            for (int k = 0; k < N; ++k)
#pragma unroll
                for (int c = 0; c < V; ++c) a.part[((tile * S + s) * N + k) * W + lane * V + c] = v[k][c];
            __threadfence();
            __syncwarp();
            if (lane == 0) s_last = atomicAdd(a.ticket + tile, 1u) == static_cast<unsigned>(S - 1) ? 1u : 0u;
        }
        __syncthreads();
        if (!s_last) return;
        // the splits' blocks in order: warp w folds blocks [w S/8, (w+1) S/8) (S >= 8)
        // or block w (S < 8, identities elsewhere), then the in-order tree over
        // the 8 warps; S is a power of two, so this is the perfect tree over S
        // blocks (a +0 beside a sum changes nothing: these sums are never -0)
        __threadfence();
        const int per = S >= kWarps ? S / kWarps : 1;
        const int q0 = S >= kWarps ? w * per : w;
        float t[N][V];
#pragma unroll
        for (int k = 0; k < N; ++k)
#pragma unroll
            for (int c = 0; c < V; ++c) t[k][c] = acc_init<OP, MODE>(k);
        if (q0 < S) {
            float pv[4][N][V];
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
                for (int k = 0; k < N; ++k)
#pragma unroll
                    for (int c = 0; c < V; ++c)
                        pv[u][k][c] = u < per ? __ldcg(a.part + ((tile * S + q0 + u) * N + k) * W + lane * V + c)
                                              : acc_init<OP, MODE>(k);
#pragma unroll
            for (int k = 0; k < N; ++k)
#pragma unroll
                for (int c = 0; c < V; ++c) {
                    auto f = [k](float x, float y) { return acc_comb<OP, MODE>(k, x, y); };
                    t[k][c] = per == 1 ? pv[0][k][c]
                            : per == 2 ? f(pv[0][k][c], pv[1][k][c])
                                       : f(f(pv[0][k][c], pv[1][k][c]), f(pv[2][k][c], pv[3][k][c]));
                }
        }
#pragma unroll
        for (int k = 0; k < N; ++k)
#pragma unroll
            for (int c = 0; c < V; ++c) g[k][w][lane * V + c] = t[k][c];
        __syncthreads();
        if (w == 0) {
#pragma unroll
            for (int k = 0; k < N; ++k)
#pragma unroll
                for (int c = 0; c < V; ++c) {
                    const int i = lane * V + c;
                    auto f = [k](float x, float y) { return acc_comb<OP, MODE>(k, x, y); };
                    v[k][c] = f(f(f(g[k][0][i], g[k][1][i]), f(g[k][2][i], g[k][3][i])),
                                f(f(g[k][4][i], g[k][5][i]), f(g[k][6][i], g[k][7][i])));
                }
            if (lane == 0) a.ticket[tile] = 0u;
        }
    }
    if constexpr (MODE == KEY) {
        // a NaN anywhere in the tile: every warp recomputes the tile with the canonical tree
        bool nan = false;
        if (w == 0) {
            const int hi_ok = 0x7f800000;                                  // key(+inf)
            const int lo_ok = order_key(__int_as_float(0xff800000u));     // key(-inf)
#pragma unroll
            for (int c = 0; c < V; ++c)
                nan |= jok && (__float_as_int(v[0][c]) < lo_ok || __float_as_int(v[1][c]) > hi_ok);
        }
        if (__syncthreads_or(nan)) {
            constexpr bool want_min = OP == OP_RMIN || OP == OP_RMINMAX;
            constexpr bool want_max = OP == OP_RMAX || OP == OP_RMINMAX;
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                if ((k == 0 && !want_min) || (k == 1 && !want_max)) continue;
                __syncthreads();  // warp 0 may still read g[0] from the previous pass
#pragma unroll 1
                for (int c = 0; c < V; ++c) {  // one column at a time keeps the registers low
                    float tc[1];
                    if (k == 0) tree_block<CMinF, 1, 1>(a, col + c, jok, R, inner, 32 * w, 32, tc);
                    else tree_block<CMaxF, 1, 1>(a, col + c, jok, R, inner, 32 * w, 32, tc);
                    g[0][w][lane * V + c] = tc[0];
                }
                __syncthreads();
                if (w == 0) {
#pragma unroll
                    for (int c = 0; c < V; ++c) {
                        const float r = k == 0 ? cta_tree<CMinF>(g[0], lane * V + c)
                                               : cta_tree<CMaxF>(g[0], lane * V + c);
                        v[k][c] = __int_as_float(order_key(r));  // the key map is undone below
                    }
                }
            }
        }
        if (w == 0 && jok) {
#pragma unroll
            for (int c = 0; c < V; ++c) {
                const float lo = from_order_key(__float_as_int(v[0][c]));
                const float hi = from_order_key(__float_as_int(v[1][c]));
                if constexpr (OP == OP_RMIN) a.out[j + c] = lo;
                if constexpr (OP == OP_RMAX) a.out[j + c] = hi;
                if constexpr (OP == OP_RMINMAX) {
                    a.out[j + c] = lo;
                    a.out2[j + c] = hi;
                }
            }
        }
    } else {
        if (w == 0 && jok) {
#pragma unroll
            for (int c = 0; c < V; ++c) {
                a.out[j + c] = v[0][c];
                if constexpr (N == 2) a.out2[j + c] = v[1][c];
            }
        }
    }
}

template <int OP, int MODE>
cudaError_t launch_mode(const AxisArgs& a, int vec, int64_t tiles, int splits, cudaStream_t stream) {
    const dim3 grid(static_cast<unsigned>(tiles), static_cast<unsigned>(splits));
    if (vec == 4)
        axis_kernel<OP, MODE, 4><<<grid, kAxisThreads, 0, stream>>>(a);
    else
        axis_kernel<OP, MODE, 1><<<grid, kAxisThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

template <int OP>
cudaError_t launch(bool ordered, const AxisArgs& a, int vec, int64_t tiles, int splits, cudaStream_t stream) {
    if (!ordered) return launch_mode<OP, FREE>(a, vec, tiles, splits, stream);
    // the ordered sum folds one column per thread (the host passes vec 1)
    if constexpr (OP == OP_RSUM) return launch_mode<OP, TREE>(a, 1, tiles, splits, stream);
    else return launch_mode<OP, KEY>(a, vec, tiles, splits, stream);
}

}  // namespace axis

cudaError_t launch_axis_staged(int term, const AxisArgs& a, int64_t tiles, int splits, size_t smem,
                               cudaStream_t stream) {
    const dim3 grid(static_cast<unsigned>(tiles), static_cast<unsigned>(splits));
    switch (term) {
        case AXIS_PLAIN:
            axis::axis_kernel<OP_RSUM, axis::STAGED, 1, AXIS_PLAIN><<<grid, kAxisThreads, smem, stream>>>(a);
            break;
        case AXIS_RMS_W:
            axis::axis_kernel<OP_RSUM, axis::STAGED, 1, AXIS_RMS_W><<<grid, kAxisThreads, smem, stream>>>(a);
            break;
        case AXIS_LN_GAMMA:
            axis::axis_kernel<OP_RSUM, axis::STAGED, 1, AXIS_LN_GAMMA><<<grid, kAxisThreads, smem, stream>>>(a);
            break;
        case AXIS_LN_BETA:
            axis::axis_kernel<OP_RSUM, axis::STAGED, 1, AXIS_LN_BETA><<<grid, kAxisThreads, smem, stream>>>(a);
            break;
        case AXIS_LN_BOTH:
            axis::axis_kernel<OP_RSUM, axis::STAGED, 1, AXIS_LN_BOTH><<<grid, kAxisThreads, smem, stream>>>(a);
            break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

template <int TERM>
cudaError_t launch_term(bool ordered, const AxisArgs& a, int vec, int64_t tiles, int splits, cudaStream_t stream) {
    const dim3 grid(static_cast<unsigned>(tiles), static_cast<unsigned>(splits));
    if (ordered) {
        if constexpr (TERM == AXIS_LN_BOTH) return cudaErrorInvalidValue;  // the ordered pair is staged only
        else axis::axis_kernel<OP_RSUM, axis::TREE, 1, TERM><<<grid, kAxisThreads, 0, stream>>>(a);
    } else if (vec == 4)
        axis::axis_kernel<OP_RSUM, axis::FREE, 4, TERM><<<grid, kAxisThreads, 0, stream>>>(a);
    else
        axis::axis_kernel<OP_RSUM, axis::FREE, 1, TERM><<<grid, kAxisThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_axis_term(int term, bool ordered, const AxisArgs& a, int vec, int64_t tiles, int splits,
                             cudaStream_t stream) {
    switch (term) {
        case AXIS_RMS_W: return launch_term<AXIS_RMS_W>(ordered, a, vec, tiles, splits, stream);
        case AXIS_LN_GAMMA: return launch_term<AXIS_LN_GAMMA>(ordered, a, vec, tiles, splits, stream);
        case AXIS_LN_BETA: return launch_term<AXIS_LN_BETA>(ordered, a, vec, tiles, splits, stream);
        case AXIS_LN_BOTH: return launch_term<AXIS_LN_BOTH>(ordered, a, vec, tiles, splits, stream);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_axis(int op, bool ordered, const AxisArgs& a, int vec, int64_t tiles, int splits,
                        cudaStream_t stream) {
    switch (op) {
        case TR_OP_ROW_SUM: return axis::launch<OP_RSUM>(ordered, a, vec, tiles, splits, stream);
        case TR_OP_ROW_MAX: return axis::launch<OP_RMAX>(ordered, a, vec, tiles, splits, stream);
        case TR_OP_ROW_MIN: return axis::launch<OP_RMIN>(ordered, a, vec, tiles, splits, stream);
        case TR_OP_ROW_MINMAX: return axis::launch<OP_RMINMAX>(ordered, a, vec, tiles, splits, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace tr
