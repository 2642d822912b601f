// TR_PLAN_SPLIT: few, long rows spread over every SM.
//
// A row is cut into C contiguous segments, one per CTA (C <= 32), and all
// rows * C CTAs are resident at once (cooperative launch), so a 16-row problem
// can use every SM instead of one cluster of at most 16 CTAs per row. Each CTA:
//   1. streams its whole segment through registers once, two chunks in
//      flight per thread, folding each chunk into its statistic as it lands;
//      the first part of the segment (up to its shared-memory share) is also
//      kept, raw, in shared memory;
//   2. reduces its segment to one partial statistic (softmax: the (max, sum
//      of exp) pair; RMSNorm: the sum of squares; LayerNorm: Chan moments),
//      publishes it to a global workspace and arrives on the row's counter;
//   3. waits (bounded in time) until the C segments of its row have arrived,
//      merges the C partials in a fixed order, and writes its segment: the
//      kept part from shared memory, the rest (the overflow) re-read from L2.
// This is the combine of "TIRx Metal reduction lowering" §4.2 (cooperative
// striping) one level up: the per-row partial array lives in global memory
// instead of on-chip memory, and a per-row arrival counter replaces the
// barrier. The last CTA to leave a row clears the row's counters, so launches
// that reuse one workspace in stream order (or graph replays) need no
// host-side reset.
#pragma once

#include <type_traits>

#include "tr_row_kernels.cuh"

namespace tr {

constexpr int kSplitU = 4;  // float4 per thread per streamed chunk
// A CTA that aborted before it arrived (the segments plan: its copy wait gave
// up) arrives with this weight on the arrival word, whose low 16 bits count
// arrivals.
constexpr unsigned kSplitAbortUnit = 1u << 16;

__device__ __forceinline__ float4 pack(float v) { return make_float4(v, 0.0f, 0.0f, 0.0f); }
__device__ __forceinline__ float4 pack(MaxSum v) { return make_float4(v.m, v.s, 0.0f, 0.0f); }
__device__ __forceinline__ float4 pack(Moments v) { return make_float4(v.n, v.mean, v.m2, 0.0f); }
template <class T>
__device__ __forceinline__ T unpack(float4 v);
template <>
__device__ __forceinline__ float unpack<float>(float4 v) { return v.x; }
template <>
__device__ __forceinline__ MaxSum unpack<MaxSum>(float4 v) { return MaxSum{v.x, v.y}; }
template <>
__device__ __forceinline__ Moments unpack<Moments>(float4 v) { return Moments{v.x, v.y, v.z}; }

template <int OP>
using SplitStat = typename std::conditional<
    OP == OP_SOFTMAX, MaxSum, typename std::conditional<OP == OP_LAYERNORM, Moments, float>::type>::type;

// Fold N float4 (all valid) into a running statistic.
template <int OP, int N>
__device__ __forceinline__ SplitStat<OP> fold_chunk(SplitStat<OP> st, const float4 (&c)[kSplitU]) {
    if constexpr (OP == OP_SOFTMAX) {
        float cm = MaxOp::id();
#pragma unroll
        for (int u = 0; u < N; ++u) cm = fmaxf(cm, max4(c[u]));
        const float m = fmaxf(st.m, cm);
        if (m == MaxOp::id()) return st;
        const float mb = mb_of(m);
        float s = st.s * ex2(mb_of(st.m) - mb);
#pragma unroll
        for (int u = 0; u < N; ++u)
            s += (ex2(fmaf(c[u].x, kL2E, -mb)) + ex2(fmaf(c[u].y, kL2E, -mb))) +
                 (ex2(fmaf(c[u].z, kL2E, -mb)) + ex2(fmaf(c[u].w, kL2E, -mb)));
        return MaxSum{m, s};
    } else if constexpr (OP == OP_RMSNORM) {
#pragma unroll
        for (int u = 0; u < N; ++u)
            st = fmaf(c[u].x, c[u].x, fmaf(c[u].y, c[u].y, fmaf(c[u].z, c[u].z, fmaf(c[u].w, c[u].w, st))));
        return st;
    } else {
        float sm = 0.0f;
#pragma unroll
        for (int u = 0; u < N; ++u) sm += sum4(c[u]);
        const float cnt = 4.0f * N;
        const float mu = __fdiv_rn(sm, cnt);
        float m2 = 0.0f;
#pragma unroll
        for (int u = 0; u < N; ++u) {
            const float dx = c[u].x - mu, dy = c[u].y - mu, dz = c[u].z - mu, dw = c[u].w - mu;
            m2 = fmaf(dx, dx, fmaf(dy, dy, fmaf(dz, dz, fmaf(dw, dw, m2))));
        }
        return mo_merge(st, Moments{cnt, mu, m2});
    }
}

// Fold one scalar (a head or tail element of the row).
template <int OP>
__device__ __forceinline__ SplitStat<OP> fold_one(SplitStat<OP> st, float x) {
    if constexpr (OP == OP_SOFTMAX) {
        return ms_merge(st, ms_single(x));
    } else if constexpr (OP == OP_RMSNORM) {
        return fmaf(x, x, st);
    } else {
        return mo_merge(st, Moments{1.0f, x, 0.0f});
    }
}

// Arrival on a row counter: the release orders this thread's earlier stores
// (the partial) before the increment; no value comes back.
__device__ __forceinline__ void red_add_release(unsigned* p, unsigned v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ float4 ld_relaxed4(const float4* p) {
    float4 v;
    asm volatile("ld.relaxed.gpu.global.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(p)
                 : "memory");
    return v;
}

// Merge of two statistics (the sum for RMSNorm's float).
__device__ __forceinline__ float split_merge(float a, float b) { return a + b; }
__device__ __forceinline__ MaxSum split_merge(MaxSum a, MaxSum b) { return ms_merge(a, b); }
__device__ __forceinline__ Moments split_merge(Moments a, Moments b) { return mo_merge(a, b); }

// Epilogue of one element for the row statistic (scale, shift, mb) and the
// element's parameters.
template <int OP>
__device__ __forceinline__ float split_out(float x, float scale, float shift, float mb) {
    if constexpr (OP == OP_SOFTMAX) {
        return ex2(fmaf(x, kL2E, -mb)) * scale;
    } else {
        return (x - shift) * scale;
    }
}

// 16-byte load and store under an L2 eviction policy (createpolicy).
__device__ __forceinline__ float4 ld_pol4(const float* p, uint64_t pol) {
    float4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.f32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(p), "l"(pol));
    return v;
}
// Bulk copy global -> shared under an L2 eviction policy.
__device__ __forceinline__ void bulk_g2s_pol(void* dst, const void* src, uint32_t bytes, uint64_t* bar, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(pol)
        : "memory");
}
__device__ __forceinline__ void st_out_pol(float* p, float4 o, bool vec, uint64_t pol) {
    if (vec) {
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

template <int OP>
__global__ void __launch_bounds__(1024) split_kernel(const RowArgs a) {
    using Stat = SplitStat<OP>;
    extern __shared__ __align__(16) float4 cache[];
    __shared__ float4 part[2][32];
    __shared__ volatile int s_abort;
    const int C = a.C;
    const int64_t row = static_cast<int64_t>(blockIdx.x) / C;
    const int seg = static_cast<int>(blockIdx.x - row * C);
    const int T = blockDim.x, t = threadIdx.x;
    const float* xr = a.x + row * a.cols;
    float* yr = a.y + row * a.cols;
    const RowGeom g = row_geom(xr, a.cols);
    const int per = (g.nvec + C - 1) / C;
    const int v0 = min(g.nvec, seg * per), v1 = min(g.nvec, v0 + per);
    const int nsm = min(v1 - v0, a.slot_floats / 4);  // slots [v0, v0 + nsm) are kept in shared memory
    const float* xb = xr + g.head;
    float* yb = yr + g.head;
    const bool own_h = seg == 0 && t < g.head;
    const bool own_t = seg == C - 1 && t < g.tail;
    const int ti = g.head + 4 * g.nvec + t;
    if (t == 0) s_abort = 0;
    __syncthreads();
    pdl_enter();
    // L2 policies: the overflow is read again after the exchange (keep); the
    // kept part, the re-read and the outputs are on their last use (drop)
    uint64_t keep, drop;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(keep));
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(drop));

    // ---- 1. statistics: every slot streams through registers once, the next
    // chunk's loads in flight while this one is folded. (A bulk copy of the
    // kept part landed together with the streamed loads, at the end of the
    // read phase, and its fold from shared memory then ran after the reads.)
    Stat st = identity_of<Stat>();
    const int vk = v0 + nsm;  // slots below vk are kept
    auto load_chunk = [&](int base, float4 (&c)[kSplitU]) {
#pragma unroll
        for (int u = 0; u < kSplitU; ++u) c[u] = ld_pol4(xb + 4 * (base + u * T), base + u * T < vk ? drop : keep);
    };
    int i = v0 + t;
    bool have = i + (kSplitU - 1) * T < v1;
    float4 cur[kSplitU];
    if (have) load_chunk(i, cur);
    while (have) {
        const int inext = i + kSplitU * T;
        const bool hnext = inext + (kSplitU - 1) * T < v1;
        float4 nxt[kSplitU];
        if (hnext) load_chunk(inext, nxt);
#pragma unroll
        for (int u = 0; u < kSplitU; ++u)
            if (i + u * T < vk) cache[i + u * T - v0] = cur[u];
        st = fold_chunk<OP, kSplitU>(st, cur);
#pragma unroll
        for (int u = 0; u < kSplitU; ++u) cur[u] = nxt[u];
        i = inext;
        have = hnext;
    }
    for (; i < v1; i += T) {
        float4 c[kSplitU];
        c[0] = ld_pol4(xb + 4 * i, i < vk ? drop : keep);
        if (i < vk) cache[i - v0] = c[0];
        st = fold_chunk<OP, 1>(st, c);
    }
    float hv = 0.0f, tv = 0.0f;
    if (own_h) {
        hv = ld_stream1(xr + t);
        st = fold_one<OP>(st, hv);
    }
    if (own_t) {
        tv = ld_stream1(xr + ti);
        st = fold_one<OP>(st, tv);
    }
    RowPos p;
    p.w = t;
    p.W = T;
    p.q = 0;
    p.s = t >> 5;
    p.S = T >> 5;
    p.lane = t & 31;
    int buf = 0;
    st = cta_row_merge<Stat, 32>(st, p, part, buf);  // every thread holds the CTA's partial

    // ---- 2. publish the partial; warp 0 waits for the row's C partials and
    // merges them in lane order (the same in every CTA of the row)
    __shared__ float4 s_row;
    if (t == 0) {
        a.sp_part[blockIdx.x] = pack(st);
        red_add_release(a.sp_arrive + row, 1u);
    }
    if (t < 32) {
        const unsigned long long t0 = global_ns();
        // (testing: every CTA's wait gives up before it looks)
        bool late = a.debug_flags & kDebugExpirePeers;
        while (!late) {
            if (ld_acquire(a.sp_arrive + row) >= static_cast<unsigned>(C)) break;
            if (static_cast<long long>(global_ns() - t0) > a.wait_ns) {
                late = true;
                break;
            }
            __nanosleep(20);
        }
        late = __any_sync(kFull, late);
        if (late && t == 0) {
            atomicOr(a.err, kErrWaitTimeout);
            s_abort = 1;
        }
        const Stat v = warp_merge<Stat, 32>(p.lane < C ? unpack<Stat>(ld_relaxed4(a.sp_part + row * C + p.lane))
                                                       : identity_of<Stat>());
        if (t == 0) s_row = pack(v);
    }
    __syncthreads();
    const Stat rs = unpack<Stat>(s_row);
    // the last CTA to leave the row clears its counters for the next launch;
    // every CTA has read the partials once its warp 0 is past the merge
    auto depart = [&]() {
        if (t == 0 && atomicAdd(a.sp_depart + row, 1u) == static_cast<unsigned>(C - 1)) {
            a.sp_arrive[row] = 0u;
            a.sp_depart[row] = 0u;
            __threadfence();
        }
    };
    if (s_abort) {
        depart();
        return;
    }

    // ---- 4. epilogue: the overflow re-read first (most recently in L2), then the cached part
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
    const bool wv = a.has_w && aligned16(a.w + g.head);
    const bool bv = a.has_b && aligned16(a.b + g.head);
    auto params = [&](float4 o, int j) -> float4 {
        if constexpr (OP != OP_SOFTMAX) {
            if (a.has_w) {
                const float4 w4 = ld_param(a.w + g.head + 4 * j, wv);
                o.x *= w4.x; o.y *= w4.y; o.z *= w4.z; o.w *= w4.w;
            }
            if constexpr (OP == OP_LAYERNORM) {
                if (a.has_b) {
                    const float4 b4 = ld_param(a.b + g.head + 4 * j, bv);
                    o.x += b4.x; o.y += b4.y; o.z += b4.z; o.w += b4.w;
                }
            }
        }
        return o;
    };
    auto out4 = [&](float4 c) -> float4 {
        return make_float4(split_out<OP>(c.x, scale, shift, mb), split_out<OP>(c.y, scale, shift, mb),
                           split_out<OP>(c.z, scale, shift, mb), split_out<OP>(c.w, scale, shift, mb));
    };
    // the weight and bias loads of the norms issue with the row's, not after them
    auto pload = [&](const float* p, int j, bool vec, float dflt) {
        return p ? ld_param(p + g.head + 4 * j, vec) : f4(dflt);
    };
    const float* pw = a.has_w ? a.w : nullptr;
    const float* pb = (OP == OP_LAYERNORM && a.has_b) ? a.b : nullptr;
    // the norms sweep their whole blocks of T slots starting at a per-row
    // rotation, so that the CTAs of the rows sharing a segment read different
    // weight lines at a time instead of all the same ones
    const int ob = OP == OP_SOFTMAX ? 0 : (v1 - (v0 + nsm)) / T;  // whole blocks of the overflow
    const int orot = ob > 0 ? static_cast<int>(row % ob) : 0;
    auto oslot = [&](int b) { return v0 + nsm + ((b + orot) % ob) * T + t; };
    if constexpr (OP != OP_SOFTMAX) {
        int b = 0;
        for (; b + kSplitU - 1 < ob; b += kSplitU) {
            float4 c[kSplitU], w4[kSplitU], b4[kSplitU];
#pragma unroll
            for (int u = 0; u < kSplitU; ++u) {
                const int k = oslot(b + u);
                c[u] = ld_pol4(xb + 4 * k, drop);
                w4[u] = pload(pw, k, wv, 1.0f);
                b4[u] = pload(pb, k, bv, 0.0f);
            }
#pragma unroll
            for (int u = 0; u < kSplitU; ++u) {
                float4 o = out4(c[u]);
                o.x = fmaf(o.x, w4[u].x, b4[u].x);
                o.y = fmaf(o.y, w4[u].y, b4[u].y);
                o.z = fmaf(o.z, w4[u].z, b4[u].z);
                o.w = fmaf(o.w, w4[u].w, b4[u].w);
                st_out_pol(yb + 4 * oslot(b + u), o, a.y_vec, drop);
            }
        }
        for (; b < ob; ++b) st_out_pol(yb + 4 * oslot(b), params(out4(ld_pol4(xb + 4 * oslot(b), drop)), oslot(b)), a.y_vec, drop);
    }
    i = OP == OP_SOFTMAX ? v0 + nsm + t : v0 + nsm + ob * T + t;  // the norms: the part block
    for (; i + (kSplitU - 1) * T < v1; i += kSplitU * T) {
        float4 c[kSplitU];
        if constexpr (OP == OP_SOFTMAX) {
#pragma unroll
            for (int u = 0; u < kSplitU; ++u) c[u] = ld_pol4(xb + 4 * (i + u * T), drop);
#pragma unroll
            for (int u = 0; u < kSplitU; ++u) st_out_pol(yb + 4 * (i + u * T), out4(c[u]), a.y_vec, drop);
        } else {
            float4 w4[kSplitU], b4[kSplitU];
#pragma unroll
            for (int u = 0; u < kSplitU; ++u) {
                c[u] = ld_pol4(xb + 4 * (i + u * T), drop);
                w4[u] = pload(pw, i + u * T, wv, 1.0f);
                b4[u] = pload(pb, i + u * T, bv, 0.0f);
            }
#pragma unroll
            for (int u = 0; u < kSplitU; ++u) {
                float4 o = out4(c[u]);
                o.x = fmaf(o.x, w4[u].x, b4[u].x);
                o.y = fmaf(o.y, w4[u].y, b4[u].y);
                o.z = fmaf(o.z, w4[u].z, b4[u].z);
                o.w = fmaf(o.w, w4[u].w, b4[u].w);
                st_out_pol(yb + 4 * (i + u * T), o, a.y_vec, drop);
            }
        }
    }
    for (; i < v1; i += T) st_out_pol(yb + 4 * i, params(out4(ld_pol4(xb + 4 * i, drop)), i), a.y_vec, drop);
    if constexpr (OP == OP_SOFTMAX) {
        for (int j = t; j < nsm; j += T) st_out_pol(yb + 4 * (v0 + j), out4(cache[j]), a.y_vec, drop);
    } else {
        // kSplitU slots at a time, so that their weight/bias loads are in flight
        // together; whole blocks of T slots from the per-row rotation, as above
        const int cb = nsm / T;
        const int crot = cb > 0 ? static_cast<int>(row % cb) : 0;
        auto cslot = [&](int bb) { return ((bb + crot) % cb) * T + t; };
        int bb = 0;
        for (; bb + kSplitU - 1 < cb; bb += kSplitU) {
            float4 w4[kSplitU], b4[kSplitU];
#pragma unroll
            for (int u = 0; u < kSplitU; ++u) {
                w4[u] = pload(pw, v0 + cslot(bb + u), wv, 1.0f);
                b4[u] = pload(pb, v0 + cslot(bb + u), bv, 0.0f);
            }
#pragma unroll
            for (int u = 0; u < kSplitU; ++u) {
                float4 o = out4(cache[cslot(bb + u)]);
                o.x = fmaf(o.x, w4[u].x, b4[u].x);
                o.y = fmaf(o.y, w4[u].y, b4[u].y);
                o.z = fmaf(o.z, w4[u].z, b4[u].z);
                o.w = fmaf(o.w, w4[u].w, b4[u].w);
                st_out_pol(yb + 4 * (v0 + cslot(bb + u)), o, a.y_vec, drop);
            }
        }
        for (; bb < cb; ++bb) st_out_pol(yb + 4 * (v0 + cslot(bb)), params(out4(cache[cslot(bb)]), v0 + cslot(bb)), a.y_vec, drop);
        int j = cb * T + t;  // the part block
        for (; j + (kSplitU - 1) * T < nsm; j += kSplitU * T) {
            float4 w4[kSplitU], b4[kSplitU];
#pragma unroll
            for (int u = 0; u < kSplitU; ++u) {
                w4[u] = pload(pw, v0 + j + u * T, wv, 1.0f);
                b4[u] = pload(pb, v0 + j + u * T, bv, 0.0f);
            }
#pragma unroll
            for (int u = 0; u < kSplitU; ++u) {
                float4 o = out4(cache[j + u * T]);
                o.x = fmaf(o.x, w4[u].x, b4[u].x);
                o.y = fmaf(o.y, w4[u].y, b4[u].y);
                o.z = fmaf(o.z, w4[u].z, b4[u].z);
                o.w = fmaf(o.w, w4[u].w, b4[u].w);
                st_out_pol(yb + 4 * (v0 + j + u * T), o, a.y_vec, drop);
            }
        }
        for (; j < nsm; j += T) st_out_pol(yb + 4 * (v0 + j), params(out4(cache[j]), v0 + j), a.y_vec, drop);
    }
    auto params1 = [&](float o, int col) -> float {
        if constexpr (OP != OP_SOFTMAX) {
            if (a.has_w) o *= __ldg(a.w + col);
            if (OP == OP_LAYERNORM && a.has_b) o += __ldg(a.b + col);
        }
        return o;
    };
    if (own_h) yr[t] = params1(split_out<OP>(hv, scale, shift, mb), t);
    if (own_t) yr[ti] = params1(split_out<OP>(tv, scale, shift, mb), ti);
    depart();
}

}  // namespace tr
