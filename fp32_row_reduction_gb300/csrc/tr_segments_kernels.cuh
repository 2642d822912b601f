// TR_PLAN_SEGMENTS: few long rows (unordered softmax and norms), every
// co-resident CTA owning one column segment of EVERY row.
//
// The split plan gives a CTA one segment of one row, so the CTAs of different
// rows that own the same columns each read that column range of the weight
// (and bias): at 16 x 1048576 a LayerNorm reads its 8 MB of parameters 16
// times from L2, as many bytes as the rows themselves. Here the roles are
// transposed: CTA g (of G, all resident at once, one per SM) owns quads
// [q0, q1) of every row, and thread t of it the quads q0 + t + 1024 i, i < I.
// A thread therefore sees the same columns in every row and keeps their
// weight and bias quads in registers for all rows: the parameters cross L2
// once per launch. The statistics of all rows meet in ONE exchange through
// the stream's workspace ("TIRx Metal reduction lowering" §4.2, the combine of
// cooperating workers one level above a CTA):
//   1. every row's segment streams through registers once, several rows'
//      loads in flight while the oldest is folded into per-row warp partials
//      (two passes over the lanes, not a merge per shuffle level);
//      the first nbuf rows are also kept, raw, in shared memory (the others
//      are read again in the epilogue: L2 evict-last until then);
//   2. the CTA publishes one partial per row, arrives once on the launch's
//      arrival word, and waits for all G CTAs (bounded); warp w then merges
//      rows w, w + 32, ... over the G partials in CTA order (row-major
//      partials, coalesced weak loads; approximate division in the moments
//      merges: the policy is unordered);
//   3. the epilogue writes every row's segment: cached rows from shared
//      memory, the others read again (evict-first), outputs evict-first.
// Requirements (checked by the plan selector): cols % 4 == 0, x, w and b
// 16-byte aligned, rows <= kSegMaxRows, rows * G partials fit the workspace,
// every segment fits I quads per thread.
#pragma once

#include "tr_split_kernels.cuh"

namespace tr {
namespace segments {

constexpr int kMaxRows = 32;

// One thread's fold of its valid quads (the first `n` of c) of one row, kept
// small so that the quads' registers take the next row's loads at once.
//   softmax: (m, s) about the thread's own maximum;
//   RMSNorm: the sum of squares;
//   LayerNorm: (n, mean, M2) about the thread's own mean (two passes over its
//   registers; n = 4 or 8 or ..., the mean by the reciprocal of n).
template <int OP>
struct ThreadFold;
template <>
struct ThreadFold<OP_SOFTMAX> { float m, s; };
template <>
struct ThreadFold<OP_RMSNORM> { float ss; };
template <>
struct ThreadFold<OP_LAYERNORM> { float n, mean, m2, sum; };

template <int OP, int I>
__device__ __forceinline__ ThreadFold<OP> fold_thread(const float4 (&c)[I], int n) {
    if constexpr (OP == OP_SOFTMAX) {
        float cm = MaxOp::id();
#pragma unroll
        for (int i = 0; i < I; ++i)
            if (i < n) cm = fmaxf(cm, max4(c[i]));
        if (cm == MaxOp::id()) return {cm, 0.0f};
        const float mb = mb_of(cm);
        float s = 0.0f;
#pragma unroll
        for (int i = 0; i < I; ++i)
            if (i < n)
                s += (ex2(fmaf(c[i].x, kL2E, -mb)) + ex2(fmaf(c[i].y, kL2E, -mb))) +
                     (ex2(fmaf(c[i].z, kL2E, -mb)) + ex2(fmaf(c[i].w, kL2E, -mb)));
        return {cm, s};
    } else if constexpr (OP == OP_RMSNORM) {
        float ss = 0.0f;
#pragma unroll
        for (int i = 0; i < I; ++i)
            if (i < n) ss = fmaf(c[i].x, c[i].x, fmaf(c[i].y, c[i].y, fmaf(c[i].z, c[i].z, fmaf(c[i].w, c[i].w, ss))));
        return {ss};
    } else {
        if (n <= 0) return {0.0f, 0.0f, 0.0f, 0.0f};
        float sm = 0.0f;
#pragma unroll
        for (int i = 0; i < I; ++i)
            if (i < n) sm += sum4(c[i]);
        const float cnt = 4.0f * n;
        const float mu = sm * __frcp_rn(cnt);
        float m2 = 0.0f;
#pragma unroll
        for (int i = 0; i < I; ++i)
            if (i < n) {
                const float dx = c[i].x - mu, dy = c[i].y - mu, dz = c[i].z - mu, dw = c[i].w - mu;
                m2 = fmaf(dx, dx, fmaf(dy, dy, fmaf(dz, dz, fmaf(dw, dw, m2))));
            }
        return {cnt, mu, m2, sm};
    }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
    return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, o));
    return v;
}

// The warp's statistic from its lanes' folds, in two passes over the lanes
// instead of a merge per shuffle level: softmax takes the warp maximum first
// and rescales each lane's sum to it once (one exponential per lane rather
// than two per level); LayerNorm sums first, divides once by the warp's count
// `nw`, and adds each lane's M2 to its squared offset from that mean times its
// count (the parallel-axis identity, exact in real arithmetic). Special
// values come out as from the pairwise merges: no finite element gives the
// identity, an infinite maximum a NaN sum.
template <int OP>
__device__ __forceinline__ SplitStat<OP> fold_warp(ThreadFold<OP> f, float nw) {
    if constexpr (OP == OP_SOFTMAX) {
        const float m = warp_max(f.m);
        if (m == MaxOp::id()) return MaxSum{m, 0.0f};
        return MaxSum{m, warp_sum(f.s * ex2(mb_of(f.m) - mb_of(m)))};
    } else if constexpr (OP == OP_RMSNORM) {
        return warp_sum(f.ss);
    } else {
        if (nw == 0.0f) return Moments{0.0f, 0.0f, 0.0f};
        const float mean = __fdiv_rn(warp_sum(f.sum), nw);
        const float d = f.mean - mean;
        return Moments{nw, mean, warp_sum(fmaf(f.n * d, d, f.m2))};
    }
}

// Merges of the unordered policy with the approximate division (Chan's
// moments): the exchange merges G partials per row, and the IEEE division of
// mo_merge would dominate it.
__device__ __forceinline__ float seg_merge(float a, float b) { return a + b; }
__device__ __forceinline__ MaxSum seg_merge(MaxSum a, MaxSum b) { return ms_merge(a, b); }
__device__ __forceinline__ Moments seg_merge(Moments a, Moments b) {
    const float n = a.n + b.n;
    if (n == 0.0f) return Moments{0.0f, 0.0f, 0.0f};
    const float d = b.mean - a.mean;
    const float fb = __fdividef(b.n, n);
    return Moments{n, fmaf(d, fb, a.mean), fmaf(d * d, a.n * fb, a.m2 + b.m2)};
}
template <class Stat>
__device__ __forceinline__ Stat seg_warp_merge(Stat v) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v = seg_merge(v, shfl_xor(v, o));
    return v;
}

// kThreads threads per CTA, I quads per thread and row, D rows in flight per thread.
template <int OP, int I, int kThreads = 1024, int D = 2>
__global__ void __launch_bounds__(kThreads, 1) segments_kernel(const RowArgs a) {
    using Stat = SplitStat<OP>;
    constexpr int kWarps = kThreads / 32;
    extern __shared__ __align__(16) float4 cache[];  // nbuf rows x sq quads (raw x)
    __shared__ float4 wpart[kWarps][kMaxRows];  // per warp, per row
    __shared__ float4 srow[kMaxRows];           // the rows' merged statistics
    __shared__ volatile int s_abort;
    const int G = gridDim.x, g = blockIdx.x, t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int R = static_cast<int>(a.rows);
    const int cols = a.cols;
    const int nq = cols >> 2;
    const int q0 = static_cast<int>(static_cast<int64_t>(g) * nq / G);
    const int q1 = static_cast<int>(static_cast<int64_t>(g + 1) * nq / G);
    const int sq = q1 - q0;
    const int rc = min(R, a.nbuf);                  // rows kept in shared memory
    // this thread's quads q0 + t + kThreads * i, the first `mine` of them valid
    const int mine = t < sq ? (sq - 1 - t) / kThreads + 1 : 0;
    // the elements this warp holds of every row (for LayerNorm's warp mean)
    float nw = 0.0f;
#pragma unroll
    for (int i = 0; i < I; ++i) nw += 4.0f * static_cast<float>(min(32, max(0, sq - 32 * warp - kThreads * i)));
    if (t == 0) s_abort = 0;
    __syncthreads();
    pdl_enter();
    uint64_t keep, drop;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(keep));
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(drop));
    auto row_ptr = [&](int r, int i) { return a.x + static_cast<int64_t>(r) * cols + 4 * (q0 + t + kThreads * i); };
    const float id = first_identity<OP>();
    auto load_row = [&](int r, float4 (&c)[I], uint64_t pol) {
#pragma unroll
        for (int i = 0; i < I; ++i) c[i] = i < mine ? ld_pol4(row_ptr(r, i), pol) : f4(id);
    };
    float4 buf[D][I];

    // ---- 1. every row streams through registers once, D rows in flight per
    // thread: a thread folds the oldest, reloads its registers with the row D
    // ahead, then its warp combines the folds; the first rc rows are also kept,
    // raw, in shared memory for the epilogue (the others are read again, L2
    // evict-last until then)
#pragma unroll
    for (int j = 0; j < D; ++j)
        if (j < R) load_row(j, buf[j], j < rc ? drop : keep);
    for (int r0 = 0; r0 < R; r0 += D) {
#pragma unroll
        for (int j = 0; j < D; ++j) {
            const int r = r0 + j;
            if (r < R) {
                if (r < rc)
#pragma unroll
                    for (int i = 0; i < I; ++i)
                        if (i < mine) cache[static_cast<int64_t>(r) * sq + t + kThreads * i] = buf[j][i];
                const ThreadFold<OP> f = fold_thread<OP, I>(buf[j], mine);
                if (r + D < R) load_row(r + D, buf[j], r + D < rc ? drop : keep);
                const Stat st = fold_warp<OP>(f, nw);
                if (lane == 0) wpart[warp][r] = pack(st);
            }
        }
    }
    __syncthreads();
    // the CTA's partial of each row (warp w merges rows w, w + kWarps, ...),
    // stored row-major: row r's G partials are contiguous
    for (int r = warp; r < R; r += kWarps) {
        const Stat v = seg_warp_merge(lane < kWarps ? unpack<Stat>(wpart[lane][r]) : identity_of<Stat>());
        if (lane == 0) a.sp_part[static_cast<int64_t>(r) * G + g] = pack(v);
    }
    // every partial of the CTA is stored before thread 0's release (cumulative
    // over the barrier) makes them visible with its arrival
    __syncthreads();

    // ---- 2. one arrival per CTA; wait for all G (bounded), then merge each row
    // over its G partials (CTA order, one fixed tree), warp w taking rows w,
    // w + kWarps, ...: a lane loads its partials (coalesced, weak L2 loads
    // ordered after the acquire by the barrier) before it merges them
    if (t == 0) red_add_release(a.sp_arrive, 1u);
    // the weight (and bias) quads of this thread's columns: in flight during the exchange
    float4 wq[I], bq[I];
#pragma unroll
    for (int i = 0; i < I; ++i) {
        const int c = 4 * (q0 + t + kThreads * i);
        wq[i] = (OP != OP_SOFTMAX && a.has_w && i < mine) ? ld_param4(a.w + c) : f4(1.0f);
        bq[i] = (OP == OP_LAYERNORM && a.has_b && i < mine) ? ld_param4(a.b + c) : f4(0.0f);
    }
    if (t < 32) {
        const unsigned long long t0 = global_ns();
        bool late = a.debug_flags & kDebugExpirePeers;  // (testing: gives up before it looks)
        while (!late) {
            if (ld_acquire(a.sp_arrive) >= static_cast<unsigned>(G)) break;
            if (static_cast<long long>(global_ns() - t0) > a.wait_ns) {
                late = true;
                break;
            }
            __nanosleep(32);
        }
        late = __any_sync(kFull, late);
        if (late && t == 0) {
            atomicOr(a.err, kErrWaitTimeout);
            s_abort = 1;
        }
    }
    __syncthreads();
    if (!s_abort) {
        constexpr int kPer = 5;  // partials per lane: G <= 160
        for (int r = warp; r < R; r += kWarps) {
            const float4* pr = a.sp_part + static_cast<int64_t>(r) * G;
            float4 pv[kPer];
#pragma unroll
            for (int m = 0; m < kPer; ++m) {
                const int k = lane + 32 * m;
                pv[m] = k < G ? __ldcg(pr + k) : pack(identity_of<Stat>());
            }
            Stat v = unpack<Stat>(pv[0]);
#pragma unroll
            for (int m = 1; m < kPer; ++m) v = seg_merge(v, unpack<Stat>(pv[m]));
            v = seg_warp_merge(v);
            if (lane == 0) srow[r] = pack(v);
        }
    }
    __syncthreads();  // every warp has read the partials it needs
    // the last CTA to leave clears the arrival word for the next launch
    if (t == 0 && atomicAdd(a.sp_depart, 1u) == static_cast<unsigned>(G - 1)) {
        *a.sp_arrive = 0u;
        *a.sp_depart = 0u;
        __threadfence();
    }
    if (s_abort) return;

    // ---- 3. the epilogue of every row
    auto out_row = [&](int r, const float4 (&c)[I]) {
        const Stat rs = unpack<Stat>(srow[r]);
        float scale, shift = 0.0f, mb = 0.0f;
        if constexpr (OP == OP_SOFTMAX) {
            mb = mb_of(rs.m);
            scale = 1.0f / rs.s;
        } else if constexpr (OP == OP_RMSNORM) {
            scale = rsqrtf(fmaf(rs, a.inv_cols, a.eps));
        } else {
            scale = rsqrtf(fmaf(rs.m2, a.inv_cols, a.eps));
            shift = rs.mean;
        }
        float* yr = a.y + static_cast<int64_t>(r) * cols + 4 * (q0 + t);
#pragma unroll
        for (int i = 0; i < I; ++i) {
            if (i >= mine) continue;
            float4 o = make_float4(split_out<OP>(c[i].x, scale, shift, mb), split_out<OP>(c[i].y, scale, shift, mb),
                                   split_out<OP>(c[i].z, scale, shift, mb), split_out<OP>(c[i].w, scale, shift, mb));
            if constexpr (OP != OP_SOFTMAX) {
                o.x *= wq[i].x; o.y *= wq[i].y; o.z *= wq[i].z; o.w *= wq[i].w;
            }
            if constexpr (OP == OP_LAYERNORM) {
                o.x += bq[i].x; o.y += bq[i].y; o.z += bq[i].z; o.w += bq[i].w;
            }
            st_out_pol(yr + 4 * kThreads * i, o, a.y_vec, drop);
        }
    };
    // the streamed rows first (their second read was kept in L2 most recently)
#pragma unroll
    for (int j = 0; j < D; ++j)
        if (rc + j < R) load_row(rc + j, buf[j], drop);
    for (int r0 = rc; r0 < R; r0 += D) {
#pragma unroll
        for (int j = 0; j < D; ++j) {
            const int r = r0 + j;
            if (r < R) {
                out_row(r, buf[j]);
                if (r + D < R) load_row(r + D, buf[j], drop);
            }
        }
    }
    for (int r = 0; r < rc; ++r) {
        float4 c[I];
#pragma unroll
        for (int i = 0; i < I; ++i) c[i] = i < mine ? cache[static_cast<int64_t>(r) * sq + t + kThreads * i] : f4(id);
        out_row(r, c);
    }
}

}  // namespace segments
}  // namespace tr
