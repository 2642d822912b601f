// Backward passes of the four row operators: the gradients of softmax,
// cross-entropy, RMSNorm and LayerNorm, the next rows of the same row-reduction
// family (the pages define the forward operators only).
//
//   softmax        dx_c = y_c (dy_c - s),            s = sum_j dy_j y_j
//   cross-entropy  dx_c = dloss (p_c - [c == label]), p = softmax(logits)
//   RMSNorm        dx_c = r (g_c - x_c k),           g = dy w, k = (sum g x / N) r r,
//                  r = 1 / sqrt(sum x^2 / N + eps);  dw_c = sum_rows (dy_c x_c) r
//   LayerNorm      dx_c = r ((g_c - a) - xh_c b),    xh = (x - mean) r, g = dy gamma,
//                  a = sum g / N, b = sum g xh / N;  dgamma_c = sum_rows dy_c xh_c,
//                  dbeta_c = sum_rows dy_c
//
// Layout: one CTA of 256 threads per row, thread t owning columns 1024j + 4t
// .. +3, the OT-1024 layout of the ordered forward kernels, so every row sum is
// the fixed tree in both policies (the unordered policy uses the same tree
// with contracted arithmetic and the hardware exp2). Rows of at most 1024 K
// columns stay in registers; longer rows are read again for each pass.
//
// Column gradients (dw, dgamma, dbeta): the row kernel writes each row's
// statistics (1/rms; mean and 1/sigma), and a column sum over the rows of the
// per-element terms, recomputed from x, dy and those statistics, finishes them
// (ordered: OT-1024 over each column's terms, as every ordered column sum).
#include <cuda_runtime.h>
#include <algorithm>
#include <stdint.h>

#include "tr_device.cuh"
#include "tr_internal.h"
#include "tr_ot.cuh"

namespace tr {
namespace backward {

using ordered::Add;
using ordered::Max;
using ordered::exp_ot;
using ordered::load_quad;
using ordered::store_quad;
using ordered::tree;

// Binary32 steps: rounded one by one under the ordered policy, free to
// contract under the unordered one.
template <bool O>
__device__ __forceinline__ float add(float a, float b) { return O ? __fadd_rn(a, b) : a + b; }
template <bool O>
__device__ __forceinline__ float sub(float a, float b) { return O ? __fsub_rn(a, b) : a - b; }
template <bool O>
__device__ __forceinline__ float mul(float a, float b) { return O ? __fmul_rn(a, b) : a * b; }
template <bool O>
__device__ __forceinline__ float divide(float a, float b) { return O ? __fdiv_rn(a, b) : __fdividef(a, b); }
template <bool O>
__device__ __forceinline__ float root(float a) { return O ? __fsqrt_rn(a) : sqrtf(a); }
// exp(x - m): the library's exp under the ordered policy, the hardware exp2 otherwise
template <bool O>
__device__ __forceinline__ float exp_shift(float x, float m) {
    if constexpr (O) return exp_ot(__fsub_rn(x, m));
    else return ex2(x * kL2E - m * kL2E);
}

// Columns 1024j + 4t .. +3 of a parameter vector (cached loads; 0 outside the row).
__device__ __forceinline__ void load_param_quad(const float* w, int cols, int j, bool aligned, float (&q)[4]) {
    const int c0 = 1024 * j + 4 * static_cast<int>(threadIdx.x);
    if (aligned && c0 + 3 < cols) {
        const float4 v = ld_param4(w + c0);
        q[0] = v.x; q[1] = v.y; q[2] = v.z; q[3] = v.w;
    } else {
#pragma unroll
        for (int v = 0; v < 4; ++v) q[v] = c0 + v < cols ? __ldg(w + c0 + v) : 0.0f;
    }
}

// 16-byte asynchronous copy global -> shared (no registers held while in flight).
__device__ __forceinline__ void cp_async16(void* dst, const float* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Stage quad j of a row into this thread's shared-memory slot: an async copy
// when the quad is a whole aligned float4, plain loads otherwise (0 outside).
__device__ __forceinline__ void stage_quad(float4* slot, const float* r, int cols, int j, bool aligned) {
    const int c0 = 1024 * j + 4 * static_cast<int>(threadIdx.x);
    if (aligned && c0 + 3 < cols) {
        cp_async16(slot, r + c0);
    } else {
        float q[4];
#pragma unroll
        for (int v = 0; v < 4; ++v) q[v] = c0 + v < cols ? ld_stream1(r + c0 + v) : 0.0f;
        *slot = make_float4(q[0], q[1], q[2], q[3]);
    }
}

// Shared memory of a launch: x and (but for cross-entropy) dy, K quads per thread.
template <int OP>
constexpr size_t bw_smem_per_slot() { return (OP == BW_XENT ? 1 : 2) * kOrderedThreads * sizeof(float4); }

template <int OP, int K, bool O>
__global__ void __launch_bounds__(kOrderedThreads) bw_kernel(const BwArgs a) {
    extern __shared__ float4 smem_raw[];
    __shared__ float gpart[2][8];
    int buf = 0;
    const int cols = a.cols;
    const int nj = (cols + 1023) / 1024;
    const float n = static_cast<float>(cols);
    const int t4 = 4 * static_cast<int>(threadIdx.x);
    const bool w_al = a.w && aligned16(a.w);
    for (int64_t row = blockIdx.x; row < a.rows; row += gridDim.x) {
        const bool first = row == static_cast<int64_t>(blockIdx.x);
        const float* xr = a.x + row * cols;
        const float* dr = OP == BW_XENT ? nullptr : a.dy + row * cols;
        float* yr = a.dx + row * cols;
        const bool x_al = aligned16(xr);
        const bool d_al = dr && aligned16(dr);
        const bool y_al = aligned16(yr);
        // the row's quads in shared memory, each thread's own slots (no barrier):
        // x at cache[j][t], dy at cache[K + j][t]; staged by async copies, the
        // next row's quad j as soon as the last pass has used this row's
        float4* cache = reinterpret_cast<float4*>(smem_raw);
        auto slot_x = [&](int j) { return cache + j * kOrderedThreads + threadIdx.x; };
        auto slot_d = [&](int j) { return cache + (K + j) * kOrderedThreads + threadIdx.x; };
        const int64_t next = row + gridDim.x;
        auto stage_next = [&](int j) {
            if constexpr (K > 0) {
                if (next < a.rows) {
                    const float* nx = a.x + next * cols;
                    stage_quad(slot_x(j), nx, cols, j, aligned16(nx));
                    if constexpr (OP != BW_XENT) {
                        const float* nd = a.dy + next * cols;
                        stage_quad(slot_d(j), nd, cols, j, aligned16(nd));
                    }
                }
            }
        };
        if constexpr (K > 0) {
            if (first) {
#pragma unroll
                for (int j = 0; j < K; ++j) {
                    if (j < nj) {
                        stage_quad(slot_x(j), xr, cols, j, x_al);
                        if constexpr (OP != BW_XENT) stage_quad(slot_d(j), dr, cols, j, d_al);
                        // the norms' weight quads into L1 while the row lands
                        if ((OP == BW_RMSNORM || OP == BW_LAYERNORM) && a.w && 1024 * j + t4 < cols)
                            prefetch_l1(a.w + 1024 * j + t4);
                    }
                }
            }
            cp_async_wait_all();
        }
        // fn(j, x quad, dy quad, valid columns) for every quad of the row, in increasing j
        auto for_quads = [&](auto&& fn) {
            if constexpr (K > 0) {
#pragma unroll
                for (int j = 0; j < K; ++j) {
                    if (j < nj) {
                        bool ok[4];
#pragma unroll
                        for (int v = 0; v < 4; ++v) ok[v] = 1024 * j + t4 + v < cols;
                        const float4 vx = *slot_x(j);
                        float qx[4] = {vx.x, vx.y, vx.z, vx.w};
                        float qd[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                        if constexpr (OP != BW_XENT) {
                            const float4 vd = *slot_d(j);
                            qd[0] = vd.x; qd[1] = vd.y; qd[2] = vd.z; qd[3] = vd.w;
                        }
                        fn(j, qx, qd, ok);
                    }
                }
            } else {
                // four quads' loads in flight, then their folds in increasing j
                int j = 0;
                for (; j + 3 < nj; j += 4) {
                    float qx[4][4], qd[4][4] = {};
                    bool ok[4][4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        load_quad(xr, cols, j + u, x_al, qx[u], ok[u]);
                        if constexpr (OP != BW_XENT) load_quad(dr, cols, j + u, d_al, qd[u], ok[u]);
                    }
#pragma unroll
                    for (int u = 0; u < 4; ++u) fn(j + u, qx[u], qd[u], ok[u]);
                }
                for (; j < nj; ++j) {
                    float qx[4], qd[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                    bool ok[4];
                    load_quad(xr, cols, j, x_al, qx, ok);
                    if constexpr (OP != BW_XENT) load_quad(dr, cols, j, d_al, qd, ok);
                    fn(j, qx, qd, ok);
                }
            }
        };
        float leaf[4];
        auto clear = [&](float v0) { leaf[0] = leaf[1] = leaf[2] = leaf[3] = v0; };
        if constexpr (OP == BW_SOFTMAX) {
            clear(0.0f);
            for_quads([&](int, const float (&y)[4], const float (&d)[4], const bool (&ok)[4]) {
#pragma unroll
                for (int v = 0; v < 4; ++v)
                    if (ok[v]) leaf[v] = add<O>(leaf[v], mul<O>(d[v], y[v]));
            });
            const float s = tree<Add>(leaf, gpart, buf);
            for_quads([&](int j, const float (&y)[4], const float (&d)[4], const bool (&ok)[4]) {
                float o[4];
#pragma unroll
                for (int v = 0; v < 4; ++v) o[v] = mul<O>(y[v], sub<O>(d[v], s));
                store_quad(yr, cols, j, y_al, o, ok);
                stage_next(j);
            });
        } else if constexpr (OP == BW_XENT) {
            float m, inv;
            if constexpr (!O && K == 0) {
                // a row read from memory per pass: the maximum and the sum of
                // exponentials in one online pass (a running pair per leaf, the sum
                // rescaled when the maximum grows), so the row is read twice, not three times
                float lm[4], ls[4];
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    lm[v] = __int_as_float(0xff800000);
                    ls[v] = 0.0f;
                }
                for_quads([&](int, const float (&x)[4], const float (&)[4], const bool (&ok)[4]) {
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        if (!ok[v]) continue;
                        if (x[v] > lm[v]) {
                            ls[v] = ls[v] * ex2((lm[v] - x[v]) * kL2E) + 1.0f;
                            lm[v] = x[v];
                        } else {
                            ls[v] += ex2((x[v] - lm[v]) * kL2E);
                        }
                    }
                });
                auto merge = [](float& ma, float& sa, float mb, float sb) {
                    const float mm = fmaxf(ma, mb);
                    if (mm == __int_as_float(0xff800000)) return;  // both empty
                    sa = sa * ex2((ma - mm) * kL2E) + sb * ex2((mb - mm) * kL2E);
                    ma = mm;
                };
                float pm = lm[0], ps = ls[0];
#pragma unroll
                for (int v = 1; v < 4; ++v) merge(pm, ps, lm[v], ls[v]);
#pragma unroll
                for (int o = 16; o >= 1; o >>= 1) {
                    const float om = __shfl_xor_sync(kFull, pm, o), os = __shfl_xor_sync(kFull, ps, o);
                    merge(pm, ps, om, os);
                }
                if ((threadIdx.x & 31) == 0) {
                    gpart[0][threadIdx.x >> 5] = pm;
                    gpart[1][threadIdx.x >> 5] = ps;
                }
                __syncthreads();
                float gm = gpart[0][0], gs = gpart[1][0];
#pragma unroll
                for (int q = 1; q < 8; ++q) merge(gm, gs, gpart[0][q], gpart[1][q]);
                __syncthreads();  // the next row writes both slots again
                m = gm;
                inv = divide<O>(1.0f, gs);
            } else {
                clear(__int_as_float(0xff800000));
                for_quads([&](int, const float (&x)[4], const float (&)[4], const bool (&ok)[4]) {
#pragma unroll
                    for (int v = 0; v < 4; ++v)
                        if (ok[v]) leaf[v] = fmaxf(leaf[v], x[v]);
                });
                m = tree<Max>(leaf, gpart, buf);
                clear(0.0f);
                for_quads([&](int, const float (&x)[4], const float (&)[4], const bool (&ok)[4]) {
#pragma unroll
                    for (int v = 0; v < 4; ++v)
                        if (ok[v]) leaf[v] = add<O>(leaf[v], exp_shift<O>(x[v], m));
                });
                inv = divide<O>(1.0f, tree<Add>(leaf, gpart, buf));
            }
            const int64_t label = a.labels[row];
            const bool scaled = a.dloss != nullptr;
            const float dl = scaled ? a.dloss[row] : 1.0f;
            for_quads([&](int j, const float (&x)[4], const float (&)[4], const bool (&ok)[4]) {
                float o[4];
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    const float p = mul<O>(exp_shift<O>(x[v], m), inv);
                    const float d = (1024 * j + t4 + v == label) ? sub<O>(p, 1.0f) : p;
                    o[v] = scaled ? mul<O>(d, dl) : d;
                }
                store_quad(yr, cols, j, y_al, o, ok);
                stage_next(j);
            });
        } else if constexpr (OP == BW_RMSNORM) {
            clear(0.0f);
            for_quads([&](int, const float (&x)[4], const float (&)[4], const bool (&ok)[4]) {
#pragma unroll
                for (int v = 0; v < 4; ++v)
                    if (ok[v]) leaf[v] = add<O>(leaf[v], mul<O>(x[v], x[v]));
            });
            const float ss = tree<Add>(leaf, gpart, buf);
            const float inv = divide<O>(1.0f, root<O>(add<O>(divide<O>(ss, n), a.eps)));
            // g = dy w, column by column
            auto grad_in = [&](int j, const float (&d)[4], float (&g)[4]) {
                if (a.w) {
                    float wq[4];
                    load_param_quad(a.w, cols, j, w_al, wq);
#pragma unroll
                    for (int v = 0; v < 4; ++v) g[v] = mul<O>(d[v], wq[v]);
                } else {
#pragma unroll
                    for (int v = 0; v < 4; ++v) g[v] = d[v];
                }
            };
            clear(0.0f);
            for_quads([&](int j, const float (&x)[4], const float (&d)[4], const bool (&ok)[4]) {
                float g[4];
                grad_in(j, d, g);
#pragma unroll
                for (int v = 0; v < 4; ++v)
                    if (ok[v]) leaf[v] = add<O>(leaf[v], mul<O>(g[v], x[v]));
            });
            const float cs = tree<Add>(leaf, gpart, buf);
            const float k = mul<O>(mul<O>(divide<O>(cs, n), inv), inv);
            if (a.stat_a && threadIdx.x == 0) a.stat_a[row] = inv;
            for_quads([&](int j, const float (&x)[4], const float (&d)[4], const bool (&ok)[4]) {
                float g[4], o[4];
                grad_in(j, d, g);
#pragma unroll
                for (int v = 0; v < 4; ++v) o[v] = mul<O>(inv, sub<O>(g[v], mul<O>(x[v], k)));
                store_quad(yr, cols, j, y_al, o, ok);
                stage_next(j);
            });
        } else {
            clear(0.0f);
            for_quads([&](int, const float (&x)[4], const float (&)[4], const bool (&ok)[4]) {
#pragma unroll
                for (int v = 0; v < 4; ++v)
                    if (ok[v]) leaf[v] = add<O>(leaf[v], x[v]);
            });
            const float mean = divide<O>(tree<Add>(leaf, gpart, buf), n);
            clear(0.0f);
            for_quads([&](int, const float (&x)[4], const float (&)[4], const bool (&ok)[4]) {
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    const float c = sub<O>(x[v], mean);
                    if (ok[v]) leaf[v] = add<O>(leaf[v], mul<O>(c, c));
                }
            });
            const float var = divide<O>(tree<Add>(leaf, gpart, buf), n);
            const float inv = divide<O>(1.0f, root<O>(add<O>(var, a.eps)));
            auto grad_in = [&](int j, const float (&d)[4], float (&g)[4]) {
                if (a.w) {
                    float wq[4];
                    load_param_quad(a.w, cols, j, w_al, wq);
#pragma unroll
                    for (int v = 0; v < 4; ++v) g[v] = mul<O>(d[v], wq[v]);
                } else {
#pragma unroll
                    for (int v = 0; v < 4; ++v) g[v] = d[v];
                }
            };
            float lb[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            clear(0.0f);
            for_quads([&](int j, const float (&x)[4], const float (&d)[4], const bool (&ok)[4]) {
                float g[4];
                grad_in(j, d, g);
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    const float xh = mul<O>(sub<O>(x[v], mean), inv);
                    if (ok[v]) {
                        leaf[v] = add<O>(leaf[v], g[v]);
                        lb[v] = add<O>(lb[v], mul<O>(g[v], xh));
                    }
                }
            });
            const float ga = divide<O>(tree<Add>(leaf, gpart, buf), n);
            const float gb = divide<O>(tree<Add>(lb, gpart, buf), n);
            if (a.stat_a && threadIdx.x == 0) {
                a.stat_a[row] = mean;
                a.stat_b[row] = inv;
            }
            for_quads([&](int j, const float (&x)[4], const float (&d)[4], const bool (&ok)[4]) {
                float g[4], o[4];
                grad_in(j, d, g);
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    const float xh = mul<O>(sub<O>(x[v], mean), inv);
                    o[v] = mul<O>(inv, sub<O>(sub<O>(g[v], ga), mul<O>(xh, gb)));
                }
                store_quad(yr, cols, j, y_al, o, ok);
                stage_next(j);
            });
        }
    }
}

template <int OP, int K, bool O>
cudaError_t launch_k(const BwArgs& a, int ctas, cudaStream_t stream) {
    const size_t smem = K * bw_smem_per_slot<OP>();
    // (once per instantiation) the shared-memory opt-in and the CTAs the device
    // holds at once: a grid of more rows than that would run a partial second
    // wave, while resident CTAs that loop over their rows stage each next row
    // during the current one's passes
    static int resident = 0;
    if (resident == 0) {
        if (smem > 40 * 1024) {  // beyond the default 48 KB once the static shared memory is added
            const cudaError_t e = cudaFuncSetAttribute(bw_kernel<OP, K, O>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                       static_cast<int>(smem));
            if (e != cudaSuccess) return e;
        }
        int dev = 0, sms = 0, per_sm = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e == cudaSuccess)
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, bw_kernel<OP, K, O>, kOrderedThreads, smem);
        if (e != cudaSuccess) return e;
        resident = std::max(1, per_sm * sms);
    }
    if (K > 0) ctas = std::min(ctas, resident);
    bw_kernel<OP, K, O><<<dim3(static_cast<unsigned>(ctas)), kOrderedThreads, smem, stream>>>(a);
    return cudaGetLastError();
}

template <int OP, bool O>
cudaError_t launch_op(int slots, const BwArgs& a, int ctas, cudaStream_t stream) {
    switch (slots) {
        case 0: return launch_k<OP, 0, O>(a, ctas, stream);
        case 1: return launch_k<OP, 1, O>(a, ctas, stream);
        case 2: return launch_k<OP, 2, O>(a, ctas, stream);
        case 4: return launch_k<OP, 4, O>(a, ctas, stream);
        case 6: return launch_k<OP, 6, O>(a, ctas, stream);
        case 8: return launch_k<OP, 8, O>(a, ctas, stream);
    }
    return cudaErrorInvalidValue;
}

template <int OP>
cudaError_t launch_policy(bool ordered, int slots, const BwArgs& a, int ctas, cudaStream_t stream) {
    return ordered ? launch_op<OP, true>(slots, a, ctas, stream) : launch_op<OP, false>(slots, a, ctas, stream);
}

}  // namespace backward

cudaError_t launch_backward(int op, bool ordered, int slots, const BwArgs& a, int ctas, cudaStream_t stream) {
    switch (op) {
        case BW_SOFTMAX: return backward::launch_policy<BW_SOFTMAX>(ordered, slots, a, ctas, stream);
        case BW_XENT: return backward::launch_policy<BW_XENT>(ordered, slots, a, ctas, stream);
        case BW_RMSNORM: return backward::launch_policy<BW_RMSNORM>(ordered, slots, a, ctas, stream);
        case BW_LAYERNORM: return backward::launch_policy<BW_LAYERNORM>(ordered, slots, a, ctas, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace tr
