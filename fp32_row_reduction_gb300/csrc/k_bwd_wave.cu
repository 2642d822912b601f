// Norm backward passes in one pass over x and dy (RMSNorm and LayerNorm,
// aligned rows of 1024 .. 8192 columns, both tree policies).
//
//   RMSNorm    r = 1 / sqrt(sum x^2 / N + eps), g = dy w, k = (sum g x / N) r r
//              dx = r (g - x k);                          dw_c = sum_rows (dy_c x_c) r
//   LayerNorm  xh = (x - mean) r, r = 1 / sqrt(var + eps), g = dy gamma,
//              a = sum g / N, b = sum g xh / N
//              dx = r ((g - a) - xh b);                   dgamma_c = sum_rows dy_c xh_c,
//                                                         dbeta_c = sum_rows dy_c
//
// A 256-thread CTA serves two consecutive rows, thread t owning the 16-byte
// slots t + 256 j of both (columns 1024 j + 4 t .. +3: the OT-1024 leaves
// 4t .. 4t+3 of every row sum, as in the forward wave kernels). x of both rows
// sits in registers; dy of both rows and the weight are copied into shared
// memory with cp.async when the CTA starts, so no global load waits in the
// passes. Independent row sums share one tree round (RMSNorm: one round;
// LayerNorm: the mean and sum g, then the variance, then, in the ordered
// policy, sum g xh; the unordered policy folds sum g (x - mean) into the
// variance round and scales it by r).
//
// Column gradients without a second pass over x and dy: the two CTAs of a
// cluster hold the four rows 4q .. 4q+3, one leaf quad of the column sums'
// OT-1024 tree (row i is leaf i). Each CTA forms (0 + t_2h) + (0 + t_2h+1) per
// column, the cluster adds rank 0's pair to rank 1's through distributed
// shared memory, which is the quad's value ((l0 + l1) + (l2 + l3)), and writes
// one partial per column and quad to the workspace; colsum_quads then runs the
// rest of the tree over the quads (the xor butterfly within each group of 32
// quads, the fixed top over the 8 groups). That is the ordered column sum for
// rows <= 1024, where every leaf holds one row; the unordered policy takes any
// number of rows and adds the groups of 256 quads first.
#include <cuda_runtime.h>

#include <algorithm>

#include "tr_device.cuh"
#include "tr_internal.h"
#include "tr_wave_kernels.cuh"

namespace tr {
namespace bwave {

constexpr int kThreads = 256;

// Binary32 steps: rounded one by one under the ordered policy, free to
// contract under the unordered one.
template <bool O>
__device__ __forceinline__ float add(float a, float b) { return O ? __fadd_rn(a, b) : a + b; }
template <bool O>
__device__ __forceinline__ float sub(float a, float b) { return O ? __fsub_rn(a, b) : a - b; }
template <bool O>
__device__ __forceinline__ float mul(float a, float b) { return O ? __fmul_rn(a, b) : a * b; }
template <bool O>
__device__ __forceinline__ float dvd(float a, float b) { return O ? __fdiv_rn(a, b) : __fdividef(a, b); }
// 1 / sqrt(v + eps)
template <bool O>
__device__ __forceinline__ float inv_root(float v, float eps) {
    return O ? __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(v, eps))) : rsqrtf(v + eps);
}

__device__ __forceinline__ float lane4(const float4& q, int e) { return e == 0 ? q.x : e == 1 ? q.y : e == 2 ? q.z : q.w; }

// Resident CTAs per SM each instantiation is compiled for: x of two rows is
// 8 K floats per thread.
template <int K>
constexpr int bwn_min_blocks() {
    return K <= 2 ? 6 : K <= 4 ? 4 : K <= 6 ? 3 : 2;
}

template <int OP, bool O, int K>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, bwn_min_blocks<K>())
    bwn_kernel(const BwArgs a, float* pg, float* pb) {
    using Add = typename std::conditional<O, wave::AddO, wave::AddU>::type;
    // dy of both rows at [r][j][t], then the weight at [j][t] (16-byte quads)
    extern __shared__ __align__(16) float4 sm[];
    __shared__ __align__(16) float part[2][4][8];
    const int t = threadIdx.x;
    const int cols = a.cols, nvec = cols >> 2;
    const float n = static_cast<float>(cols);
    const int64_t row0 = 2 * static_cast<int64_t>(blockIdx.x);
    bool has[2];
    has[0] = row0 < a.rows;
    has[1] = row0 + 1 < a.rows;
    bool okj[K];
#pragma unroll
    for (int j = 0; j < K; ++j) okj[j] = t + kThreads * j < nvec;
    auto dys = [&](int r, int j) -> float4& { return sm[(r * K + j) * kThreads + t]; };
    auto wsm = [&](int j) -> float4& { return sm[(2 * K + j) * kThreads + t]; };

    // staggered start, as in the forward wave kernels: launch rank k = blockIdx /
    // SMs requests its rows k x stagger_ns late (a cluster's two CTAs share a
    // rank: the SM count is even); one thread sleeps on the global timer
    if (a.stagger_ns > 0 && a.sms > 0) {
        const unsigned rank = blockIdx.x / static_cast<unsigned>(a.sms);
        if (rank > 0) {
            if (t == 0) {
                const unsigned long long t0 = global_ns();
                const unsigned long long d = static_cast<unsigned long long>(rank) * a.stagger_ns;
                while (global_ns() - t0 < d) __nanosleep(64);
            }
            __syncthreads();
        }
    }
    // ---- the CTA's inputs: dy and the weight by async copies, x into registers
#pragma unroll
    for (int r = 0; r < 2; ++r)
#pragma unroll
        for (int j = 0; j < K; ++j)
            if (okj[j]) {
                if (has[r]) wave::cp_async16(&dys(r, j), a.dy + (row0 + r) * cols + 4 * (t + kThreads * j));
                else dys(r, j) = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            }
    if (a.w)
#pragma unroll
        for (int j = 0; j < K; ++j)
            if (okj[j]) wave::cp_async16(&wsm(j), a.w + 4 * (t + kThreads * j));
    wave::cp_async_commit();
    float4 x[2][K];
#pragma unroll
    for (int r = 0; r < 2; ++r)
#pragma unroll
        for (int j = 0; j < K; ++j)
            x[r][j] = (has[r] && okj[j]) ? ld_stream4(a.x + (row0 + r) * cols + 4 * (t + kThreads * j))
                                         : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    wave::cp_async_wait_all();  // this thread's own quads
    // g = dy w of one quad (dy itself without a weight)
    auto grad = [&](int r, int j, int e) {
        const float d = lane4(dys(r, j), e);
        return a.w ? mul<O>(d, lane4(wsm(j), e)) : d;
    };
    // the thread's value of a row sum: its four leaves folded over j, then (l0 + l1) + (l2 + l3)
    auto row_sum = [&](auto&& term) {
        float l[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int j = 0; j < K; ++j)
            if (okj[j])
#pragma unroll
                for (int e = 0; e < 4; ++e) l[e] = add<O>(l[e], term(j, e));
        return add<O>(add<O>(l[0], l[1]), add<O>(l[2], l[3]));
    };
    int tb = 0;

    if constexpr (OP == BW_RMSNORM) {
        float v[4];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            v[2 * r] = row_sum([&](int j, int e) { const float xv = lane4(x[r][j], e); return mul<O>(xv, xv); });
            v[2 * r + 1] = row_sum([&](int j, int e) { return mul<O>(grad(r, j, e), lane4(x[r][j], e)); });
        }
        wave::tree_rows<Add, 4>(v, part[tb]);
        float inv[2], k[2];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            inv[r] = inv_root<O>(dvd<O>(v[2 * r], n), a.eps);
            k[r] = mul<O>(mul<O>(dvd<O>(v[2 * r + 1], n), inv[r]), inv[r]);
        }
#pragma unroll
        for (int j = 0; j < K; ++j) {
            if (!okj[j]) continue;
            const int c = 4 * (t + kThreads * j);
            float pw[4];
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                float o[4], term[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float xv = lane4(x[r][j], e);
                    o[e] = mul<O>(inv[r], sub<O>(grad(r, j, e), mul<O>(xv, k[r])));
                    term[e] = has[r] ? mul<O>(mul<O>(lane4(dys(r, j), e), xv), inv[r]) : 0.0f;
                }
                if (has[r]) st4(a.dx + (row0 + r) * cols + c, make_float4(o[0], o[1], o[2], o[3]));
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float leaf = has[r] ? add<O>(0.0f, term[e]) : 0.0f;  // a leaf starts at 0
                    pw[e] = r == 0 ? leaf : add<O>(pw[e], leaf);
                }
            }
            if (pg) dys(0, j) = make_float4(pw[0], pw[1], pw[2], pw[3]);  // dy of slot j is no longer read
        }
    } else {
        float mean[2], inv[2], ga[2], gb[2];
        {
            float v[4];
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                v[2 * r] = row_sum([&](int j, int e) { return lane4(x[r][j], e); });
                v[2 * r + 1] = row_sum([&](int j, int e) { return grad(r, j, e); });
            }
            wave::tree_rows<Add, 4>(v, part[tb]);
            tb ^= 1;
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                mean[r] = dvd<O>(v[2 * r], n);
                ga[r] = dvd<O>(v[2 * r + 1], n);
            }
        }
        if constexpr (O) {
            float v[2];
#pragma unroll
            for (int r = 0; r < 2; ++r)
                v[r] = row_sum([&](int j, int e) { const float c = sub<O>(lane4(x[r][j], e), mean[r]); return mul<O>(c, c); });
            wave::tree_rows<Add, 2>(v, part[tb]);
            tb ^= 1;
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                inv[r] = inv_root<O>(dvd<O>(v[r], n), a.eps);
                v[r] = row_sum([&](int j, int e) {
                    return mul<O>(grad(r, j, e), mul<O>(sub<O>(lane4(x[r][j], e), mean[r]), inv[r]));
                });
            }
            wave::tree_rows<Add, 2>(v, part[tb]);
#pragma unroll
            for (int r = 0; r < 2; ++r) gb[r] = dvd<O>(v[r], n);
        } else {
            // the variance and sum g (x - mean) in one round; sum g xh = r sum g (x - mean)
            float v[4];
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                v[2 * r] = row_sum([&](int j, int e) { const float c = lane4(x[r][j], e) - mean[r]; return c * c; });
                v[2 * r + 1] = row_sum([&](int j, int e) { return grad(r, j, e) * (lane4(x[r][j], e) - mean[r]); });
            }
            wave::tree_rows<Add, 4>(v, part[tb]);
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                inv[r] = inv_root<O>(v[2 * r] / n, a.eps);
                gb[r] = v[2 * r + 1] * inv[r] / n;
            }
        }
#pragma unroll
        for (int j = 0; j < K; ++j) {
            if (!okj[j]) continue;
            const int c = 4 * (t + kThreads * j);
            float pgm[4], pbt[4];
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                float o[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float xh = mul<O>(sub<O>(lane4(x[r][j], e), mean[r]), inv[r]);
                    const float d = lane4(dys(r, j), e);
                    o[e] = mul<O>(inv[r], sub<O>(sub<O>(grad(r, j, e), ga[r]), mul<O>(xh, gb[r])));
                    const float lg = has[r] ? add<O>(0.0f, mul<O>(d, xh)) : 0.0f;  // leaves start at 0
                    const float lb = has[r] ? add<O>(0.0f, d) : 0.0f;
                    pgm[e] = r == 0 ? lg : add<O>(pgm[e], lg);
                    pbt[e] = r == 0 ? lb : add<O>(pbt[e], lb);
                }
                if (has[r]) st4(a.dx + (row0 + r) * cols + c, make_float4(o[0], o[1], o[2], o[3]));
            }
            if (pg) {  // dy of slot j is no longer read
                dys(0, j) = make_float4(pgm[0], pgm[1], pgm[2], pgm[3]);
                dys(1, j) = make_float4(pbt[0], pbt[1], pbt[2], pbt[3]);
            }
        }
    }
    if (!pg) return;  // no column gradients asked for (uniform over the grid)

    // ---- the leaf quad of every column: rank 0's pair + rank 1's pair
    cg::cluster_group cl = cg::this_cluster();
    cl.sync();  // both CTAs' pairs are in shared memory
    const unsigned rank = cl.block_rank();
    const float4* p0 = cl.map_shared_rank(sm, 0);
    const float4* p1 = cl.map_shared_rank(sm, 1);
    const int64_t q = blockIdx.x >> 1;
    const int half = K * kThreads / 2;  // this CTA's slots: [rank * half, rank * half + half)
    for (int i = static_cast<int>(rank) * half + t; i < static_cast<int>(rank + 1) * half; i += kThreads) {
        if (i >= nvec) break;
        const float4 A = p0[i], B = p1[i];
        st4(pg + q * cols + 4 * i, make_float4(add<O>(A.x, B.x), add<O>(A.y, B.y), add<O>(A.z, B.z), add<O>(A.w, B.w)));
        if (OP == BW_LAYERNORM && pb) {
            const float4 C = p0[K * kThreads + i], D = p1[K * kThreads + i];
            st4(pb + q * cols + 4 * i, make_float4(add<O>(C.x, D.x), add<O>(C.y, D.y), add<O>(C.z, D.z), add<O>(C.w, D.w)));
        }
    }
    cl.sync();  // the peer has read this CTA's shared memory
}

// The column sums over Q quad partials (rows x cols -> Q = ceil(rows / 4) x
// cols): grid (ceil(cols / 32), vectors), 256 threads. Quad 32 w + l is lane l
// of warp w: the xor butterfly within each warp, then the fixed top over the 8
// warps, evaluated for 32 columns at a time (a 256 x 32 tile in shared
// memory). Quads past Q are 0 (leaves without rows). The unordered policy
// first adds the quads 256 m + i (any number of them) into tile row i.
template <bool O>
__global__ void __launch_bounds__(kThreads) colsum_quads(const float* pg, const float* pb, float* og, float* ob,
                                                         int64_t Q, int cols) {
    __shared__ float tile[kThreads][33];
    __shared__ float top[8][32];
    const float* p = blockIdx.y == 0 ? pg : pb;
    float* out = blockIdx.y == 0 ? og : ob;
    const int c0 = blockIdx.x * 32;
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    // (each (row, column) of the tile has one owner thread across the chunks;
    // 16-byte loads, eight per thread in flight: cols % 4 == 0 and c0 % 32 == 0)
    for (int64_t base = 0; base == 0 || base < Q; base += kThreads) {
        float4 v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int idx = t + kThreads * u, r = idx >> 3, c = 4 * (idx & 7);
            const int64_t qq = base + r;
            v[u] = (qq < Q && c0 + c < cols) ? *reinterpret_cast<const float4*>(p + qq * cols + c0 + c)
                                             : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int idx = t + kThreads * u, r = idx >> 3, c = 4 * (idx & 7);
            if (base == 0) {
                tile[r][c] = v[u].x; tile[r][c + 1] = v[u].y; tile[r][c + 2] = v[u].z; tile[r][c + 3] = v[u].w;
            } else if (base + r < Q) {
                tile[r][c] = add<O>(tile[r][c], v[u].x);
                tile[r][c + 1] = add<O>(tile[r][c + 1], v[u].y);
                tile[r][c + 2] = add<O>(tile[r][c + 2], v[u].z);
                tile[r][c + 3] = add<O>(tile[r][c + 3], v[u].w);
            }
        }
    }
    __syncthreads();
    // thread (w, c): the butterfly of group w for column c, evaluated in one
    // thread: lane 0's value after the xor steps 16, 8, 4, 2, 1 is
    // ((v0 + v16) + (v8 + v24)) + ... level by level, i.e. s[i] = s[i] + s[i + h]
    // for h = 16, 8, 4, 2, 1
    {
        const int c = lane, w = warp;
        float v[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = tile[32 * w + i][c];
#pragma unroll
        for (int h = 16; h >= 1; h >>= 1)
#pragma unroll
            for (int i = 0; i < h; ++i) v[i] = add<O>(v[i], v[i + h]);
        top[w][c] = v[0];
    }
    __syncthreads();
    if (t < 32 && c0 + t < cols) {
        const float s = add<O>(add<O>(add<O>(top[0][t], top[1][t]), add<O>(top[2][t], top[3][t])),
                               add<O>(add<O>(top[4][t], top[5][t]), add<O>(top[6][t], top[7][t])));
        out[c0 + t] = s;
    }
}

template <int OP, bool O, int K>
cudaError_t launch_k(const BwArgs& a, float* pg, float* pb, cudaStream_t stream) {
    const size_t smem = static_cast<size_t>(3) * K * kThreads * 16;  // dy of two rows, the weight
    static bool opted = false;
    if (!opted) {
        const cudaError_t e = cudaFuncSetAttribute(bwn_kernel<OP, O, K>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        opted = true;
    }
    static int resident = 0, sms = 0;
    if (resident == 0) {
        int dev = 0, per_sm = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e == cudaSuccess)
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, bwn_kernel<OP, O, K>, kThreads, smem);
        if (e != cudaSuccess) return e;
        resident = std::max(1, per_sm) * sms;
    }
    const int64_t pairs = (a.rows + 1) / 2;
    const int64_t ctas = (pairs + 1) / 2 * 2;  // whole clusters of two
    BwArgs b = a;
    b.sms = sms;
    // one launch rank's rows (x and dy) at the HBM rate, for grids of more than
    // one rank that the device holds at once and an even SM count
    b.stagger_ns = (ctas > sms && ctas <= resident && sms % 2 == 0)
                       ? static_cast<int>(std::min(4000.0, 0.95 * sms * 2.0 * a.cols * 8.0 / 7000.0))
                       : 0;
    bwn_kernel<OP, O, K><<<dim3(static_cast<unsigned>(ctas)), kThreads, smem, stream>>>(b, pg, pb);
    return cudaGetLastError();
}

template <int OP, bool O>
cudaError_t launch_slots(int K, const BwArgs& a, float* pg, float* pb, cudaStream_t stream) {
    switch (K) {
        case 2: return launch_k<OP, O, 2>(a, pg, pb, stream);
        case 4: return launch_k<OP, O, 4>(a, pg, pb, stream);
        case 6: return launch_k<OP, O, 6>(a, pg, pb, stream);
        case 8: return launch_k<OP, O, 8>(a, pg, pb, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace bwave

int bwn_slots(int64_t cols) {
    if (cols < 1024 || cols > 8192 || cols % 4 != 0) return 0;
    for (int k : {2, 4, 6, 8})
        if (cols <= 1024LL * k) return k;
    return 0;
}

cudaError_t launch_backward_wave(int op, bool ordered, const BwArgs& a, float* dw, float* db, float* partials,
                                 cudaStream_t stream) {
    const int K = bwn_slots(a.cols);
    if (K == 0 || (op != BW_RMSNORM && op != BW_LAYERNORM)) return cudaErrorInvalidValue;
    const int64_t Q = (a.rows + 3) / 4;
    float* pg = (dw || db) ? partials : nullptr;
    float* pb = (op == BW_LAYERNORM && pg) ? partials + Q * a.cols : nullptr;
    cudaError_t e;
    if (op == BW_RMSNORM)
        e = ordered ? bwave::launch_slots<BW_RMSNORM, true>(K, a, pg, pb, stream)
                    : bwave::launch_slots<BW_RMSNORM, false>(K, a, pg, pb, stream);
    else
        e = ordered ? bwave::launch_slots<BW_LAYERNORM, true>(K, a, pg, pb, stream)
                    : bwave::launch_slots<BW_LAYERNORM, false>(K, a, pg, pb, stream);
    if (e != cudaSuccess || !pg) return e;
    // the column gradients: dw (RMSNorm) or dgamma and dbeta (LayerNorm, either may be absent)
    const float* src_g = pg;
    const float* src_b = pb;
    float* out_g = op == BW_RMSNORM ? dw : dw;  // dw carries dgamma for LayerNorm
    const bool two = op == BW_LAYERNORM && dw && db;
    if (op == BW_LAYERNORM && !dw) {  // only dbeta: its partials are the second block
        src_g = pb;
        out_g = db;
    }
    dim3 grid(static_cast<unsigned>((a.cols + 31) / 32), two ? 2u : 1u);
    if (ordered)
        bwave::colsum_quads<true><<<grid, bwave::kThreads, 0, stream>>>(src_g, src_b, out_g, db, Q, a.cols);
    else
        bwave::colsum_quads<false><<<grid, bwave::kThreads, 0, stream>>>(src_g, src_b, out_g, db, Q, a.cols);
    return cudaGetLastError();
}

}  // namespace tr
