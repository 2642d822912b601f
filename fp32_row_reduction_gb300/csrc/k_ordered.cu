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
// A row is divided by its normaliser (softmax sum, RMS, sigma) as a product with
// the correctly rounded reciprocal: one IEEE division per row, one rounded
// product per element.
#include <cuda_runtime.h>
#include <climits>
#include <stdint.h>

#include "tr_device.cuh"
#include "tr_internal.h"
#include "tr_ot.cuh"
#include "tr_row_kernels.cuh"

namespace tr {
namespace ordered {

// The OT-1024 epilogue of one row whose quads are cached in q: q[j][v] holds
// column 1024j + 4t + v of the row (t = threadIdx.x), valid when that column is
// < cols. `vec_out`: the row's output may be written with 16-byte stores.
template <int OP, int K>
__device__ __forceinline__ void ot_cached_row(const RowArgs& a, int64_t row, float (&q)[K][4], bool vec_out,
                                              float (*gpart)[8], int& buf) {
    const int cols = a.cols;
    const int t = static_cast<int>(threadIdx.x);
    const int nj = (cols + 1023) / 1024;
    auto col = [t](int j, int v) { return 1024 * j + 4 * t + v; };
    // validity, tested once per quad: `full` quads need no per-element test
    auto full = [&](int j) { return j < nj && col(j, 3) < cols; };
    auto okc = [&](int j, int v) { return j < nj && col(j, v) < cols; };
    // the norms' weight and bias quads: into L1 now, so that the epilogue after
    // the trees finds them there (every CTA on the SM reads the same vectors)
    if constexpr (OP == OP_RMSNORM || OP == OP_LAYERNORM) {
#pragma unroll
        for (int j = 0; j < K; ++j) {
            if (j < nj && col(j, 0) < cols) {
                if (a.has_w) prefetch_l1(a.w + col(j, 0));
                if (OP == OP_LAYERNORM && a.has_b) prefetch_l1(a.b + col(j, 0));
            }
        }
    }
    float leaf[4];
    // fold f(value, column) into the leaves in increasing column order
    auto fold = [&](auto elem, auto comb, float init) {
        leaf[0] = leaf[1] = leaf[2] = leaf[3] = init;
#pragma unroll
        for (int j = 0; j < K; ++j) {
            if (full(j)) {
#pragma unroll
                for (int v = 0; v < 4; ++v) leaf[v] = comb(leaf[v], elem(q[j][v], col(j, v)));
            } else {
#pragma unroll
                for (int v = 0; v < 4; ++v)
                    if (okc(j, v)) leaf[v] = comb(leaf[v], elem(q[j][v], col(j, v)));
            }
        }
    };
    float* yr = a.y + row * cols;
    auto emit = [&](auto out) {
#pragma unroll
        for (int j = 0; j < K; ++j) {
            if (j >= nj) continue;
            // `out` may read the column's weight: evaluate it for columns inside the row only
            if (full(j)) {
                float o[4];
#pragma unroll
                for (int v = 0; v < 4; ++v) o[v] = out(q[j][v], col(j, v));
                if (vec_out) {
                    st4(yr + col(j, 0), make_float4(o[0], o[1], o[2], o[3]));
                } else {
#pragma unroll
                    for (int v = 0; v < 4; ++v) yr[col(j, v)] = o[v];
                }
            } else {
#pragma unroll
                for (int v = 0; v < 4; ++v)
                    if (okc(j, v)) yr[col(j, v)] = out(q[j][v], col(j, v));
            }
        }
    };
    // emit with a whole-quad form for full quads (quad(v[4], first column, o[4]))
    // and the per-element form for the partial last quad
    auto emit_quads = [&](auto quad, auto elem) {
#pragma unroll
        for (int j = 0; j < K; ++j) {
            if (j >= nj) continue;
            if (full(j)) {
                float o[4];
                quad(q[j], col(j, 0), o);
                if (vec_out) {
                    st4(yr + col(j, 0), make_float4(o[0], o[1], o[2], o[3]));
                } else {
#pragma unroll
                    for (int v = 0; v < 4; ++v) yr[col(j, v)] = o[v];
                }
            } else {
#pragma unroll
                for (int v = 0; v < 4; ++v)
                    if (okc(j, v)) yr[col(j, v)] = elem(q[j][v], col(j, v));
            }
        }
    };
    auto add = [](float p, float v) { return __fadd_rn(p, v); };
    auto mx = [](float p, float v) { return max2(p, v); };
    auto ident = [](float v, int) { return v; };
    const float n = static_cast<float>(cols);

    if constexpr (OP == OP_SOFTMAX || OP == OP_XENT) {
        fold(ident, mx, __int_as_float(0xff800000));
        const float m = tree<Max>(leaf, gpart, buf);
        // exp once per element, kept in place: the sum folds the same values in
        // the same leaf order as exp_ot(x - m) would
#pragma unroll
        for (int j = 0; j < K; ++j) {
            if (full(j)) {
#pragma unroll
                for (int v = 0; v < 4; ++v) q[j][v] = exp_ot(__fsub_rn(q[j][v], m));
            } else {
#pragma unroll
                for (int v = 0; v < 4; ++v)
                    if (okc(j, v)) q[j][v] = exp_ot(__fsub_rn(q[j][v], m));
            }
        }
        fold(ident, add, 0.0f);
        const float s = tree<Add>(leaf, gpart, buf);
        if constexpr (OP == OP_SOFTMAX) {
            const float inv = __fdiv_rn(1.0f, s);
            emit([inv](float e, int) { return __fmul_rn(e, inv); });
        } else {
            if (t == 0) {
                const float* xr = a.x + row * cols;
                const int64_t label = a.labels[row];
                const float sel = (label >= 0 && label < cols) ? __ldg(xr + label) : 0.0f;
                a.loss[row] = __fsub_rn(__fadd_rn(log_ot(s), m), sel);
            }
        }
    } else if constexpr (OP == OP_RMSNORM) {
        fold([](float v, int) { return __fmul_rn(v, v); }, add, 0.0f);
        const float ss = tree<Add>(leaf, gpart, buf);
        const float r = __fsqrt_rn(__fadd_rn(__fdiv_rn(ss, n), a.eps));
        const float inv = __fdiv_rn(1.0f, r);
        const bool hw = a.has_w;
        const float* w = a.w;
        if (hw && aligned16(w)) {
            // whole quads: one 16-byte weight load per quad
            emit_quads([inv, w](const float (&v)[4], int c0, float (&o)[4]) {
                const float4 wq = ld_param4(w + c0);
                const float wv[4] = {wq.x, wq.y, wq.z, wq.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) o[e] = __fmul_rn(__fmul_rn(v[e], inv), wv[e]);
            }, [inv, w](float v, int c) { return __fmul_rn(__fmul_rn(v, inv), __ldg(w + c)); });
        } else {
            emit([inv, hw, w](float v, int c) {
                const float u = __fmul_rn(v, inv);
                return hw ? __fmul_rn(u, __ldg(w + c)) : u;
            });
        }
    } else {  // OP_LAYERNORM
        fold(ident, add, 0.0f);
        const float mean = __fdiv_rn(tree<Add>(leaf, gpart, buf), n);
        fold([mean](float v, int) {
            const float c = __fsub_rn(v, mean);
            return __fmul_rn(c, c);
        }, add, 0.0f);
        const float var = __fdiv_rn(tree<Add>(leaf, gpart, buf), n);
        const float d = __fsqrt_rn(__fadd_rn(var, a.eps));
        const float inv = __fdiv_rn(1.0f, d);
        const bool hw = a.has_w, hb = a.has_b;
        const float *w = a.w, *b = a.b;
        auto scalar = [mean, inv, hw, hb, w, b](float v, int c) {
            float u = __fmul_rn(__fsub_rn(v, mean), inv);
            if (hw) u = __fmul_rn(u, __ldg(w + c));
            if (hb) u = __fadd_rn(u, __ldg(b + c));
            return u;
        };
        if (hw && hb && aligned16(w) && aligned16(b)) {
            emit_quads([mean, inv, w, b](const float (&v)[4], int c0, float (&o)[4]) {
                const float4 wq = ld_param4(w + c0), bq = ld_param4(b + c0);
                const float wv[4] = {wq.x, wq.y, wq.z, wq.w}, bv[4] = {bq.x, bq.y, bq.z, bq.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) o[e] = __fadd_rn(__fmul_rn(__fmul_rn(__fsub_rn(v[e], mean), inv), wv[e]), bv[e]);
            }, scalar);
        } else {
            emit(scalar);
        }
    }
}

// One-shot realisation: a CTA per row. K > 0: the row (cols <= 1024*K) is
// cached in registers. K == 0: the row is read again for each pass.
// Rows of up to 6144 columns (K <= 6) fit six 256-thread CTAs per SM, so that
// 768 such rows are resident in one wave on 152 SMs.
template <int K>
constexpr int ot_min_blocks() {
    return K >= 1 && K <= 6 ? 6 : (K == 8 ? 5 : 1);
}

// RES (fused residual norms, K > 0): h = x + r by one IEEE add per element
// before the tree; h is written at once when requested.
template <int OP, int K, bool RES = false>
__global__ void __launch_bounds__(kOrderedThreads, ot_min_blocks<K>()) ot_kernel(const RowArgs a) {
    __shared__ float gpart[2][8];
    int buf = 0;
    const int64_t row = blockIdx.x;
    const int cols = a.cols;
    const float* xr = a.x + row * cols;
    const bool aligned = aligned16(xr);
    pdl_enter();
    if constexpr (K > 0) {
        const int nj = (cols + 1023) / 1024;
        float q[K][4];
#pragma unroll
        for (int j = 0; j < K; ++j) {
            bool ok[4];
            if (j < nj) {
                load_quad(xr, cols, j, aligned, q[j], ok);
            } else {
                q[j][0] = q[j][1] = q[j][2] = q[j][3] = 0.0f;
            }
        }
        if constexpr (RES) {
            const float* rr = a.r + row * cols;
            const bool raligned = aligned16(rr);
            float* hr = a.h ? a.h + row * cols : nullptr;
#pragma unroll
            for (int j = 0; j < K; ++j) {
                if (j >= nj) continue;
                float rq[4];
                bool ok[4];
                load_quad(rr, cols, j, raligned, rq, ok);
#pragma unroll
                for (int v = 0; v < 4; ++v) q[j][v] = __fadd_rn(q[j][v], rq[v]);
                if (hr) store_quad(hr, cols, j, aligned && a.h_vec, q[j], ok);
            }
        }
        ot_cached_row<OP, K>(a, row, q, aligned && a.y_vec, gpart, buf);
    } else {
        const int nj = (cols + 1023) / 1024;
        // four quads in flight at a time; the leaves still fold in increasing column order
        auto fold = [&](auto elem, auto comb, float init, float (&leaf)[4]) {
            leaf[0] = leaf[1] = leaf[2] = leaf[3] = init;
            int j = 0;
            for (; j + 3 < nj; j += 4) {
                float qq[4][4];
                bool oo[4][4];
#pragma unroll
                for (int u = 0; u < 4; ++u) load_quad(xr, cols, j + u, aligned, qq[u], oo[u]);
#pragma unroll
                for (int u = 0; u < 4; ++u)
#pragma unroll
                    for (int v = 0; v < 4; ++v)
                        if (oo[u][v])
                            leaf[v] = comb(leaf[v], elem(qq[u][v], (j + u) * 1024 + 4 * static_cast<int>(threadIdx.x) + v));
            }
            for (; j < nj; ++j) {
                float qq[4];
                bool oo[4];
                load_quad(xr, cols, j, aligned, qq, oo);
#pragma unroll
                for (int v = 0; v < 4; ++v)
                    if (oo[v]) leaf[v] = comb(leaf[v], elem(qq[v], j * 1024 + 4 * static_cast<int>(threadIdx.x) + v));
            }
        };
        auto emit = [&](auto out) {
            float* yr = a.y + row * cols;
            const bool vec = aligned && a.y_vec;
            auto one = [&](int jj, const float (&qq)[4], const bool (&oo)[4]) {
                float o[4];
#pragma unroll
                for (int v = 0; v < 4; ++v)
                    o[v] = oo[v] ? out(qq[v], jj * 1024 + 4 * static_cast<int>(threadIdx.x) + v) : 0.0f;
                store_quad(yr, cols, jj, vec, o, oo);
            };
            int j = 0;
            // softmax: four quads' loads in flight (the norms' per-element weight loads
            // measured slower batched)
            for (; OP == OP_SOFTMAX && j + 3 < nj; j += 4) {
                float qq[4][4];
                bool oo[4][4];
#pragma unroll
                for (int u = 0; u < 4; ++u) load_quad(xr, cols, j + u, aligned, qq[u], oo[u]);
#pragma unroll
                for (int u = 0; u < 4; ++u) one(j + u, qq[u], oo[u]);
            }
            for (; j < nj; ++j) {
                float qq[4];
                bool oo[4];
                load_quad(xr, cols, j, aligned, qq, oo);
                one(j, qq, oo);
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
            fold([m](float v, int) { return exp_ot(__fsub_rn(v, m)); }, add, 0.0f, leaf);
            const float s = tree<Add>(leaf, gpart, buf);
            if constexpr (OP == OP_SOFTMAX) {
                const float inv = __fdiv_rn(1.0f, s);
                emit([m, inv](float v, int) { return __fmul_rn(exp_ot(__fsub_rn(v, m)), inv); });
            } else {
                if (threadIdx.x == 0) {
                    const int64_t label = a.labels[row];
                    const float sel = (label >= 0 && label < cols) ? __ldg(xr + label) : 0.0f;
                    a.loss[row] = __fsub_rn(__fadd_rn(log_ot(s), m), sel);
                }
            }
        } else if constexpr (OP == OP_RSUM) {
            fold(ident, add, 0.0f, leaf);
            const float r = tree<Add>(leaf, gpart, buf);
            if (threadIdx.x == 0) a.loss[row] = r;
        } else if constexpr (OP == OP_RMAX || OP == OP_RMIN || OP == OP_RMINMAX) {
            // Without a NaN in the row the canonical max (min) of the tree is the
            // largest (smallest) element in the total order with -0 below +0, in
            // any grouping. That order is the signed order of the integer keys, so
            // one pass folds both key extremes with integer max / min; the keys of
            // NaNs fall outside [key(-inf), key(+inf)], which flags the rare row
            // that needs the canonical fold itself.
            int kmax[4], kmin[4];
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                kmax[v] = INT_MIN;
                kmin[v] = INT_MAX;
            }
            auto take = [&](const float (&qq)[4], const bool (&oo)[4]) {
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    const int k = order_key(qq[v]);
                    kmax[v] = oo[v] ? max(kmax[v], k) : kmax[v];
                    kmin[v] = oo[v] ? min(kmin[v], k) : kmin[v];
                }
            };
            int j = 0;
            for (; j + 3 < nj; j += 4) {
                float qq[4][4];
                bool oo[4][4];
#pragma unroll
                for (int u = 0; u < 4; ++u) load_quad(xr, cols, j + u, aligned, qq[u], oo[u]);
#pragma unroll
                for (int u = 0; u < 4; ++u) take(qq[u], oo[u]);
            }
            for (; j < nj; ++j) {
                float qq[4];
                bool oo[4];
                load_quad(xr, cols, j, aligned, qq, oo);
                take(qq, oo);
            }
            int hi = max(max(kmax[0], kmax[1]), max(kmax[2], kmax[3]));
            int lo = min(min(kmin[0], kmin[1]), min(kmin[2], kmin[3]));
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) {
                hi = max(hi, __shfl_xor_sync(kFull, hi, o));
                lo = min(lo, __shfl_xor_sync(kFull, lo, o));
            }
            if ((threadIdx.x & 31) == 0) {
                gpart[0][threadIdx.x >> 5] = __int_as_float(hi);
                gpart[1][threadIdx.x >> 5] = __int_as_float(lo);
            }
            __syncthreads();
#pragma unroll
            for (int w = 0; w < 8; ++w) {
                hi = max(hi, __float_as_int(gpart[0][w]));
                lo = min(lo, __float_as_int(gpart[1][w]));
            }
            __syncthreads();   // the canonical trees below reuse both slots
            if (hi <= order_key(__int_as_float(0x7f800000)) && lo >= order_key(__int_as_float(0xff800000))) {
                if (threadIdx.x == 0) {
                    if constexpr (OP == OP_RMAX) a.loss[row] = from_order_key(hi);
                    if constexpr (OP == OP_RMIN) a.loss[row] = from_order_key(lo);
                    if constexpr (OP == OP_RMINMAX) {
                        a.loss[row] = from_order_key(lo);
                        a.out2[row] = from_order_key(hi);
                    }
                }
            } else {
                // a NaN in the row: the canonical selects decide which one survives
                if constexpr (OP == OP_RMAX || OP == OP_RMINMAX) {
                    fold(ident, [](float p, float v) { return cmax2(p, v); }, __int_as_float(0xff800000), leaf);
                    const float r = tree<CMax>(leaf, gpart, buf);
                    if (threadIdx.x == 0) (OP == OP_RMAX ? a.loss : a.out2)[row] = r;
                }
                if constexpr (OP == OP_RMIN || OP == OP_RMINMAX) {
                    fold(ident, [](float p, float v) { return cmin2(p, v); }, __int_as_float(0x7f800000), leaf);
                    const float r = tree<CMin>(leaf, gpart, buf);
                    if (threadIdx.x == 0) a.loss[row] = r;
                }
            }
        } else if constexpr (OP == OP_RMSNORM) {
            fold([](float v, int) { return __fmul_rn(v, v); }, add, 0.0f, leaf);
            const float ss = tree<Add>(leaf, gpart, buf);
            const float r = __fsqrt_rn(__fadd_rn(__fdiv_rn(ss, n), a.eps));
            const float inv = __fdiv_rn(1.0f, r);
            const bool hw = a.has_w;
            const float* w = a.w;
            emit([inv, hw, w](float v, int c) {
                const float u = __fmul_rn(v, inv);
                return hw ? __fmul_rn(u, __ldg(w + c)) : u;
            });
        } else {
            fold(ident, add, 0.0f, leaf);
            const float mean = __fdiv_rn(tree<Add>(leaf, gpart, buf), n);
            fold([mean](float v, int) {
                const float c = __fsub_rn(v, mean);
                return __fmul_rn(c, c);
            }, add, 0.0f, leaf);
            const float var = __fdiv_rn(tree<Add>(leaf, gpart, buf), n);
            const float d = __fsqrt_rn(__fadd_rn(var, a.eps));
            const float inv = __fdiv_rn(1.0f, d);
            const bool hw = a.has_w, hb = a.has_b;
            const float *w = a.w, *b = a.b;
            emit([mean, inv, hw, hb, w, b](float v, int c) {
                float u = __fmul_rn(__fsub_rn(v, mean), inv);
                if (hw) u = __fmul_rn(u, __ldg(w + c));
                if (hb) u = __fadd_rn(u, __ldg(b + c));
                return u;
            });
        }
    }
}

// Staged realisation: persistent CTAs of 256 threads over rows blockIdx.x,
// blockIdx.x + gridDim.x, ...; each row arrives in a ring slot by one bulk
// asynchronous copy (the window of the unordered staged plans), so one row's
// arithmetic overlaps the loads of the next rows and the stores of the
// previous ones. The tree and every rounding are those of ot_cached_row.
template <int OP, int K>
__global__ void __launch_bounds__(kOrderedThreads) ot_staged_kernel(const RowArgs a) {
    extern __shared__ __align__(16) float ring[];
    __shared__ __align__(8) uint64_t full[kMaxRing];
    __shared__ __align__(8) uint64_t never;
    __shared__ float gpart[2][8];
    __shared__ volatile int s_abort;
    int buf = 0;
    const int t = threadIdx.x;
    const int nbuf = a.nbuf;
    const int64_t G = gridDim.x;
    const int64_t mine = (a.rows - blockIdx.x + G - 1) / G;
    const float* x0 = a.x;
    const float* x1 = a.x + a.rows * a.cols;
    const int cols = a.cols;
    const int nj = (cols + 1023) / 1024;
    if (t == 0) {
        for (int b = 0; b < nbuf; ++b) mbar_init(&full[b], 1);
        mbar_init(&never, 1);
        s_abort = 0;
        fence_barrier_init();
    }
    __syncthreads();
    pdl_enter();
    if ((a.debug_flags & kDebugForceTimeout) && t == 0) mbar_wait_bounded(&never, 0, 1000000LL, a.err);
    auto issue = [&](int64_t i) {
        const int64_t row = blockIdx.x + i * G;
        const float* xr = a.x + row * cols;
        const RowGeom g = row_geom(xr, cols);
        const StagedWindow w = staged_window(xr, g, x0, x1);
        const int b = static_cast<int>(i % nbuf);
        float* slot = ring + static_cast<int64_t>(b) * a.slot_floats;
        if (w.bytes > 0) {
            mbar_arrive_expect_tx(&full[b], static_cast<uint32_t>(w.bytes));
            bulk_g2s(slot + w.dst, w.lo, static_cast<uint32_t>(w.bytes), &full[b]);
        } else {
            mbar_arrive(&full[b]);
        }
    };
    if (t == 0)
        for (int64_t i = 0; i < mine && i < nbuf; ++i) issue(i);
    for (int64_t i = 0; i < mine; ++i) {
        const int b = static_cast<int>(i % nbuf);
        const uint32_t parity = static_cast<uint32_t>((i / nbuf) & 1);
        const int64_t row = blockIdx.x + i * G;
        const float* xr = a.x + row * cols;
        const RowGeom g = row_geom(xr, cols);
        const StagedWindow w = staged_window(xr, g, x0, x1);
        const float* slot = ring + static_cast<int64_t>(b) * a.slot_floats;
        if (!mbar_wait_bounded(&full[b], parity, a.wait_ns, a.err, a.debug_flags & kDebugExpireCopies)) s_abort = 1;
        // column c sits at slot[pre + c]; pre = 0 exactly when the row is aligned
        const int pre = w.off - g.head;
        const int body_end = g.head + 4 * g.nvec;
        float q[K][4];
#pragma unroll
        for (int j = 0; j < K; ++j) {
            const int c0 = 1024 * j + 4 * t;
            if (j < nj && pre == 0 && c0 + 3 < body_end && !(w.head_global && c0 < g.head)) {
                const float4 v4 = *reinterpret_cast<const float4*>(slot + c0);
                q[j][0] = v4.x; q[j][1] = v4.y; q[j][2] = v4.z; q[j][3] = v4.w;
            } else {
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    const int c = c0 + v;
                    float x = 0.0f;
                    if (j < nj && c < cols) {
                        const bool global = (w.head_global && c < g.head) || (w.tail_global && c >= body_end);
                        x = global ? ld_stream1(xr + c) : slot[pre + c];
                    }
                    q[j][v] = x;
                }
            }
        }
        ot_cached_row<OP, K>(a, row, q, pre == 0 && a.y_vec, gpart, buf);
        // each tree ends in a barrier after every thread loaded its quads, so
        // the slot is free and the abort flag is visible here
        if (s_abort) {
            if (t == 0)
                for (int64_t j = i; j < mine && j < i + nbuf; ++j)
                    mbar_wait_bounded(&full[j % nbuf], static_cast<uint32_t>((j / nbuf) & 1), a.wait_ns, a.err);
            return;
        }
        if (t == 0 && i + nbuf < mine) {
            fence_proxy_async_smem();
            issue(i + nbuf);
        }
    }
}

}  // namespace ordered

const void* kernel_ordered_staged(int op, int slots) {
#define TR_OTS_CASES(OPV)                                                          \
    switch (slots) {                                                               \
        case 1: return reinterpret_cast<const void*>(ordered::ot_staged_kernel<OPV, 1>); \
        case 2: return reinterpret_cast<const void*>(ordered::ot_staged_kernel<OPV, 2>); \
        case 4: return reinterpret_cast<const void*>(ordered::ot_staged_kernel<OPV, 4>); \
        case 8: return reinterpret_cast<const void*>(ordered::ot_staged_kernel<OPV, 8>); \
    }                                                                              \
    return nullptr;
    switch (op) {
        case TR_OP_SOFTMAX: { TR_OTS_CASES(OP_SOFTMAX) }
        case TR_OP_RMSNORM: { TR_OTS_CASES(OP_RMSNORM) }
        case TR_OP_LAYERNORM: { TR_OTS_CASES(OP_LAYERNORM) }
        case TR_OP_CROSS_ENTROPY: { TR_OTS_CASES(OP_XENT) }
    }
#undef TR_OTS_CASES
    return nullptr;
}

// Fused residual norms (op TR_OP_ADD_RMSNORM / TR_OP_ADD_LAYERNORM): cached plans only.
const void* kernel_ordered_residual(int op, int slots) {
#define TR_OTR_CASES(OPV)                                                            \
    switch (slots) {                                                                 \
        case 1: return reinterpret_cast<const void*>(ordered::ot_kernel<OPV, 1, true>);   \
        case 2: return reinterpret_cast<const void*>(ordered::ot_kernel<OPV, 2, true>);   \
        case 4: return reinterpret_cast<const void*>(ordered::ot_kernel<OPV, 4, true>);   \
        case 6: return reinterpret_cast<const void*>(ordered::ot_kernel<OPV, 6, true>);   \
        case 8: return reinterpret_cast<const void*>(ordered::ot_kernel<OPV, 8, true>);   \
        case 12: return reinterpret_cast<const void*>(ordered::ot_kernel<OPV, 12, true>); \
        case 16: return reinterpret_cast<const void*>(ordered::ot_kernel<OPV, 16, true>); \
    }                                                                                \
    return nullptr;
    switch (op) {
        case TR_OP_ADD_RMSNORM: { TR_OTR_CASES(OP_RMSNORM) }
        case TR_OP_ADD_LAYERNORM: { TR_OTR_CASES(OP_LAYERNORM) }
    }
#undef TR_OTR_CASES
    return nullptr;
}

const void* kernel_ordered(int op, int slots) {
    if (op >= TR_OP_ROW_SUM && op <= TR_OP_ROW_MINMAX) {
        // standalone reductions read each element once: the streaming realisation only
        if (slots != 0) return nullptr;
        switch (op) {
            case TR_OP_ROW_SUM: return reinterpret_cast<const void*>(ordered::ot_kernel<OP_RSUM, 0>);
            case TR_OP_ROW_MAX: return reinterpret_cast<const void*>(ordered::ot_kernel<OP_RMAX, 0>);
            case TR_OP_ROW_MIN: return reinterpret_cast<const void*>(ordered::ot_kernel<OP_RMIN, 0>);
            case TR_OP_ROW_MINMAX: return reinterpret_cast<const void*>(ordered::ot_kernel<OP_RMINMAX, 0>);
        }
        return nullptr;
    }
#define TR_OT_CASES(OPV)                                                    \
    switch (slots) {                                                        \
        case 0: return reinterpret_cast<const void*>(ordered::ot_kernel<OPV, 0>);   \
        case 1: return reinterpret_cast<const void*>(ordered::ot_kernel<OPV, 1>);   \
        case 2: return reinterpret_cast<const void*>(ordered::ot_kernel<OPV, 2>);   \
        case 4: return reinterpret_cast<const void*>(ordered::ot_kernel<OPV, 4>);   \
        case 6: return reinterpret_cast<const void*>(ordered::ot_kernel<OPV, 6>);   \
        case 8: return reinterpret_cast<const void*>(ordered::ot_kernel<OPV, 8>);   \
        case 12: return reinterpret_cast<const void*>(ordered::ot_kernel<OPV, 12>); \
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
