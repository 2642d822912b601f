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
//   1. the first nbuf rows' segments are copied into shared memory by bulk
//      asynchronous copies issued at entry; the other rows' segments are
//      streamed (L2 evict-last: they are read again) while those land; each
//      warp folds every row's quads into per-row partials;
//   2. the CTA publishes one partial per row, arrives once on the launch's
//      arrival word, and waits for all G CTAs (bounded); warp w then merges
//      rows w, w + 32, ... over the G partials, in CTA order;
//   3. the epilogue writes every row's segment: cached rows from shared
//      memory, the others read again (evict-first), outputs evict-first.
// Requirements (checked by the plan selector): cols % 4 == 0, x, w and b
// 16-byte aligned, rows <= kSegMaxRows, rows * G partials fit the workspace,
// every segment fits I quads per thread.
#pragma once

#include "tr_split_kernels.cuh"

namespace tr {
namespace segments {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxRows = 32;

// Fold this thread's valid quads (the first `n` of c) into a statistic.
template <int OP, int I>
__device__ __forceinline__ SplitStat<OP> fold_quads(const float4 (&c)[I], int n) {
    if constexpr (OP == OP_SOFTMAX) {
        float cm = MaxOp::id();
#pragma unroll
        for (int i = 0; i < I; ++i)
            if (i < n) cm = fmaxf(cm, max4(c[i]));
        if (cm == MaxOp::id()) return MaxSum{cm, 0.0f};
        const float mb = mb_of(cm);
        float s = 0.0f;
#pragma unroll
        for (int i = 0; i < I; ++i)
            if (i < n)
                s += (ex2(fmaf(c[i].x, kL2E, -mb)) + ex2(fmaf(c[i].y, kL2E, -mb))) +
                     (ex2(fmaf(c[i].z, kL2E, -mb)) + ex2(fmaf(c[i].w, kL2E, -mb)));
        return MaxSum{cm, s};
    } else if constexpr (OP == OP_RMSNORM) {
        float ss = 0.0f;
#pragma unroll
        for (int i = 0; i < I; ++i)
            if (i < n) ss = fmaf(c[i].x, c[i].x, fmaf(c[i].y, c[i].y, fmaf(c[i].z, c[i].z, fmaf(c[i].w, c[i].w, ss))));
        return ss;
    } else {
        if (n <= 0) return Moments{0.0f, 0.0f, 0.0f};
        float sm = 0.0f;
#pragma unroll
        for (int i = 0; i < I; ++i)
            if (i < n) sm += sum4(c[i]);
        const float cnt = 4.0f * n;
        const float mu = __fdiv_rn(sm, cnt);
        float m2 = 0.0f;
#pragma unroll
        for (int i = 0; i < I; ++i)
            if (i < n) {
                const float dx = c[i].x - mu, dy = c[i].y - mu, dz = c[i].z - mu, dw = c[i].w - mu;
                m2 = fmaf(dx, dx, fmaf(dy, dy, fmaf(dz, dz, fmaf(dw, dw, m2))));
            }
        return Moments{cnt, mu, m2};
    }
}

template <int OP, int I>
__global__ void __launch_bounds__(kThreads, 1) segments_kernel(const RowArgs a) {
    using Stat = SplitStat<OP>;
    extern __shared__ __align__(16) float4 cache[];  // nbuf rows x sq quads
    __shared__ __align__(8) uint64_t bar;
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
    const int rc = min(R, a.nbuf);                  // rows cached in shared memory
    // this thread's quads q0 + t + kThreads * i, the first `mine` of them valid
    const int mine = t < sq ? (sq - 1 - t) / kThreads + 1 : 0;
    if (t == 0) {
        mbar_init(&bar, 1);
        s_abort = 0;
        fence_barrier_init();
    }
    __syncthreads();
    pdl_enter();
    uint64_t keep, drop;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(keep));
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(drop));
    if (t == 0) {
        if (rc > 0 && sq > 0) {
            mbar_arrive_expect_tx(&bar, static_cast<uint32_t>(rc) * static_cast<uint32_t>(sq) * 16u);
            for (int r = 0; r < rc; ++r)
                bulk_g2s_pol(cache + static_cast<int64_t>(r) * sq, a.x + static_cast<int64_t>(r) * cols + 4 * q0,
                             static_cast<uint32_t>(sq) * 16u, &bar, drop);
        } else {
            mbar_arrive(&bar);
        }
    }
    // the weight (and bias) quads of this thread's columns, for every row
    float4 wq[I], bq[I];
#pragma unroll
    for (int i = 0; i < I; ++i) {
        const int c = 4 * (q0 + t + kThreads * i);
        wq[i] = (OP != OP_SOFTMAX && a.has_w && i < mine) ? ld_param4(a.w + c) : f4(1.0f);
        bq[i] = (OP == OP_LAYERNORM && a.has_b && i < mine) ? ld_param4(a.b + c) : f4(0.0f);
    }
    auto row_ptr = [&](int r, int i) { return a.x + static_cast<int64_t>(r) * cols + 4 * (q0 + t + kThreads * i); };
    auto publish = [&](int r, Stat st) {  // warp partial of row r into shared memory
        st = warp_merge<Stat, 32>(st);
        if (lane == 0) wpart[warp][r] = pack(st);
    };

    // ---- 1. the streamed rows (two rows' loads in flight), then the cached rows
    float4 cur[I], nxt[I];
    const float id = first_identity<OP>();
    auto load_row = [&](int r, float4 (&c)[I], uint64_t pol) {
#pragma unroll
        for (int i = 0; i < I; ++i) c[i] = i < mine ? ld_pol4(row_ptr(r, i), pol) : f4(id);
    };
    if (rc < R) load_row(rc, cur, keep);
    for (int r = rc; r < R; ++r) {
        if (r + 1 < R) load_row(r + 1, nxt, keep);
        publish(r, fold_quads<OP, I>(cur, mine));
#pragma unroll
        for (int i = 0; i < I; ++i) cur[i] = nxt[i];
    }
    if (!mbar_wait_bounded(&bar, 0, a.wait_ns, a.err, a.debug_flags & kDebugExpireCopies)) s_abort = 1;
    __syncthreads();  // s_abort as every thread saw it
    const bool copied = !s_abort;
    for (int r = 0; r < rc; ++r) {
        float4 c[I];
#pragma unroll
        for (int i = 0; i < I; ++i)
            c[i] = (copied && i < mine) ? cache[static_cast<int64_t>(r) * sq + t + kThreads * i] : f4(id);
        publish(r, fold_quads<OP, I>(c, copied ? mine : 0));
    }
    __syncthreads();
    // the CTA's partial of each row: warp w merges rows w, w + kWarps, ...
    for (int r = warp; r < R; r += kWarps) {
        const Stat v = warp_merge<Stat, 32>(lane < kWarps ? unpack<Stat>(wpart[lane][r]) : identity_of<Stat>());
        if (lane == 0) {
            a.sp_part[static_cast<int64_t>(g) * R + r] = pack(v);
            __threadfence();  // visible at device scope before the CTA's arrival below
        }
    }
    __syncthreads();  // every partial of the CTA is stored before thread 0's release

    // ---- 2. one arrival per CTA; wait for all G (bounded), then merge each row over the G partials
    if (t == 0) red_add_release(a.sp_arrive, s_abort ? 1u + kSplitAbortUnit : 1u);
    if (t < 32) {
        const unsigned long long t0 = global_ns();
        bool late = a.debug_flags & kDebugExpirePeers, aborted = false;
        while (!late) {
            const unsigned v = ld_acquire(a.sp_arrive);
            if (v >= kSplitAbortUnit) {
                aborted = true;
                break;
            }
            if (v >= static_cast<unsigned>(G)) break;
            if (static_cast<long long>(global_ns() - t0) > a.wait_ns) {
                late = true;
                break;
            }
            __nanosleep(32);
        }
        late = __any_sync(kFull, late);
        aborted = __any_sync(kFull, aborted);
        if (late && t == 0) atomicOr(a.err, kErrWaitTimeout);
        if ((late || aborted) && t == 0) s_abort = 1;
    }
    __syncthreads();
    if (!s_abort) {
        (void)ld_acquire(a.sp_arrive);  // each reading thread acquires the arrivals itself
        for (int r = warp; r < R; r += kWarps) {
            Stat v = identity_of<Stat>();
            for (int k = lane; k < G; k += 32)
                v = split_merge(v, unpack<Stat>(ld_relaxed4(a.sp_part + static_cast<int64_t>(k) * R + r)));
            v = warp_merge<Stat, 32>(v);
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
    if (s_abort) {
        if (t == 0 && !copied) mbar_wait_bounded(&bar, 0, a.wait_ns, nullptr);  // drain the copies
        return;
    }

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
    if (rc < R) load_row(rc, cur, drop);
    for (int r = rc; r < R; ++r) {
        if (r + 1 < R) load_row(r + 1, nxt, drop);
        out_row(r, cur);
#pragma unroll
        for (int i = 0; i < I; ++i) cur[i] = nxt[i];
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
