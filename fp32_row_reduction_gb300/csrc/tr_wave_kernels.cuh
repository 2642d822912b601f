// TR_PLAN_WAVE: rows whose 16-byte-aligned body fits 256 threads x K slots,
// all resident in one wave, both reduction policies.
//
// Mapping ("TIRx Metal reduction lowering" §4.4, blocked-cyclic ownership with
// V = 4): a 256-thread CTA serves R consecutive rows; thread t owns the
// 16-byte slots t, t + 256, ..., t + 256 (K - 1) of EVERY one of its rows, so
// the same thread sees the same columns R times. That is what the norms need:
// a weight (and bias) quad is loaded once per thread and applied to R rows,
// which divides the epilogue's L1 parameter traffic by R, the cost that keeps
// one-row-per-thread norm kernels below the copy bandwidth at 768 x 6144.
//
// The layout is also the OT-1024 leaf layout: the slots t + 256 j, j = 0..K-1,
// are the columns 1024 j + 4 t .. 1024 j + 4 t + 3, i.e. the leaves 4t .. 4t+3,
// each folded over j in increasing column order. The ordered policy therefore
// runs in the same kernel with IEEE round-to-nearest steps, the fixed tree
// above the leaves (quad pairing, xor butterfly 16..1, the fixed top over the
// eight warps) and the library's own exp, and gives the bits of every other
// OT-1024 realisation. The unordered policy uses the same tree shape with
// contracted arithmetic and the hardware exp2.
//
// Requirements (checked by the plan selector): cols % 4 == 0, x 16-byte
// aligned, cols <= 1024 K (y at another 16-byte phase takes scalar stores). All loads of a CTA are issued before any
// reduction; every CTA of the grid is resident at once when the plan is chosen
// for a single wave.
#pragma once

#include <type_traits>

#include "tr_device.cuh"
#include "tr_internal.h"
#include "tr_ot.cuh"

namespace tr {
namespace wave {

constexpr int kThreads = 256;

// Resident CTAs per SM each instantiation is compiled for (register budget of
// 4 K R cached floats plus addresses and statistics): K = 6 gives 6, 3 and 2
// CTAs for R = 1, 2, 3, i.e. 912 rows resident on 152 SMs in every case.
// Smaller stripes also stop at six (40 registers): at eight (32) the norms'
// epilogues spilled.
template <int K, int R>
constexpr int min_blocks() {
    return K * R <= 6 ? 6 : K * R <= 8 ? 4 : K * R <= 12 ? 3 : K * R <= 18 ? 2 : 1;
}

// Reducers. The ordered ones round every step; max is the hardware maxNum in
// both policies (see the ordered kernels: it changes no output bit).
struct AddU {
    static __device__ __forceinline__ float f(float a, float b) { return a + b; }
};
struct AddO {
    static __device__ __forceinline__ float f(float a, float b) { return __fadd_rn(a, b); }
};
struct MaxR {
    static __device__ __forceinline__ float f(float a, float b) { return fmaxf(a, b); }
};

// The tree above each thread's value for R rows at once: xor butterfly with
// offsets 16, 8, 4, 2, 1, one shared-memory exchange of the 8 warp values
// (one barrier for all R rows), then ((p0+p1)+(p2+p3)) + ((p4+p5)+(p6+p7)),
// evaluated identically by every thread. `part` is this tree's own [R][8]
// slot block, so consecutive trees never share a slot.
template <class Rd, int R>
__device__ __forceinline__ void tree_rows(float (&v)[R], float (*part)[8]) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1)
#pragma unroll
        for (int r = 0; r < R; ++r) v[r] = Rd::f(v[r], __shfl_xor_sync(kFull, v[r], o));
    if ((threadIdx.x & 31) == 0)
#pragma unroll
        for (int r = 0; r < R; ++r) part[r][threadIdx.x >> 5] = v[r];
    __syncthreads();
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const float4 lo = *reinterpret_cast<const float4*>(&part[r][0]);
        const float4 hi = *reinterpret_cast<const float4*>(&part[r][4]);
        v[r] = Rd::f(Rd::f(Rd::f(lo.x, lo.y), Rd::f(lo.z, lo.w)), Rd::f(Rd::f(hi.x, hi.y), Rd::f(hi.z, hi.w)));
    }
}

// A thread's value from its four leaves of one row: (l0 + l1) + (l2 + l3).
template <class Rd>
__device__ __forceinline__ float quad_top(float4 l) {
    return Rd::f(Rd::f(l.x, l.y), Rd::f(l.z, l.w));
}

// 16-byte asynchronous copy global -> shared (cp.async: no register is held
// while it is in flight, and the later shared-memory reads do not queue behind
// the row loads in the SM's global-load path).
__device__ __forceinline__ void cp_async16(void* dst, const float* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// LayerNorm's parameter staging: the weight quads t + 256 j of the row in
// psm[t + 256 j], the bias quads in psm[256 K + t + 256 j]; each thread copies
// exactly the quads its own epilogue reads, so a thread's wait for its own
// copies is all the synchronisation there is.
template <int K>
__device__ __forceinline__ void stage_params(const RowArgs& a, float4* psm) {
    const int t = threadIdx.x, nvec = a.cols >> 2;
#pragma unroll
    for (int j = 0; j < K; ++j) {
        const int q = t + kThreads * j;
        if (q >= nvec) continue;
        if (a.has_w) cp_async16(&psm[q], a.w + 4 * q);
        if (a.has_b) cp_async16(&psm[K * kThreads + q], a.b + 4 * q);
    }
    cp_async_commit();
}

__device__ __forceinline__ float4 param4(const float* p, bool vec) {
    if (vec) return ld_param4(p);
    return make_float4(__ldg(p), __ldg(p + 1), __ldg(p + 2), __ldg(p + 3));
}

// y rows may sit at another 16-byte phase than x rows: then scalar stores.
__device__ __forceinline__ void store4(float* p, float4 o, bool vec) {
    if (vec) {
        st4(p, o);
    } else {
        p[0] = o.x;
        p[1] = o.y;
        p[2] = o.z;
        p[3] = o.w;
    }
}

// Quad arithmetic on the packed binary32 instructions: each float4 is two
// float2 lanes, and every lane rounds exactly like the scalar _rn form, so the
// ordered policy keeps its bits while issuing half the instructions. One rule
// for the ordered policy: a product that feeds an addition is formed with the
// scalar __fmul_rn (prod4_rn), never a packed multiply. The scalar _rn forms
// are never fused, but a packed multiply whose result fed a packed add was
// seen fused into one rounding inside these kernels, which changed bits.
__device__ __forceinline__ float2 lo2(float4 v) { return make_float2(v.x, v.y); }
__device__ __forceinline__ float2 hi2(float4 v) { return make_float2(v.z, v.w); }
__device__ __forceinline__ float4 cat2(float2 a, float2 b) { return make_float4(a.x, a.y, b.x, b.y); }
__device__ __forceinline__ float2 dup2(float s) { return make_float2(s, s); }
__device__ __forceinline__ float4 add4(float4 a, float4 b) {
    return cat2(__fadd2_rn(lo2(a), lo2(b)), __fadd2_rn(hi2(a), hi2(b)));
}
__device__ __forceinline__ float4 mul4(float4 a, float4 b) {
    return cat2(__fmul2_rn(lo2(a), lo2(b)), __fmul2_rn(hi2(a), hi2(b)));
}
__device__ __forceinline__ float4 mul4s(float4 a, float s) {
    return cat2(__fmul2_rn(lo2(a), dup2(s)), __fmul2_rn(hi2(a), dup2(s)));
}
// a - s, exactly a + (-s)
__device__ __forceinline__ float4 sub4s(float4 a, float s) {
    return cat2(__fadd2_rn(lo2(a), dup2(-s)), __fadd2_rn(hi2(a), dup2(-s)));
}
__device__ __forceinline__ float4 fma4(float4 a, float4 b, float4 c) {
    return cat2(__ffma2_rn(lo2(a), lo2(b), lo2(c)), __ffma2_rn(hi2(a), hi2(b), hi2(c)));
}
// a * b per element with the scalar round-to-nearest multiply (never fused)
__device__ __forceinline__ float4 prod4_rn(float4 a, float4 b) {
    return make_float4(__fmul_rn(a.x, b.x), __fmul_rn(a.y, b.y), __fmul_rn(a.z, b.z), __fmul_rn(a.w, b.w));
}
// the packed running sum of squares (unordered: any association)
__device__ __forceinline__ float2 sq_acc(float2 acc, float4 v) {
    acc = __ffma2_rn(lo2(v), lo2(v), acc);
    return __ffma2_rn(hi2(v), hi2(v), acc);
}

// One group of nr <= R rows starting at row0 (rows r >= nr repeat row0 and
// are not stored). `part` holds two [R][8] slot blocks;
// the group's trees use part[tb], part[tb ^ 1], ... alternately, continuing
// from the previous group (the caller passes the next block index in tb).
template <int OP, bool ORD, int K, int R>
__device__ __forceinline__ void wave_group(const RowArgs& a, int64_t row0, int nr_in, float (*part)[R][8],
                                           const float4* psm, int& tb) {
    using Add = typename std::conditional<ORD, AddO, AddU>::type;
    const int nr = R == 1 ? 1 : nr_in;  // (a constant for one-row groups)
    const int t = threadIdx.x;
    const int nvec = a.cols >> 2;
    // slots past the end of the row hold the reducer's identity (folded last,
    // where they change no bit of an ordered leaf)
    bool okj[K];
#pragma unroll
    for (int j = 0; j < K; ++j) okj[j] = t + kThreads * j < nvec;
    const float kId = OP == OP_SOFTMAX ? -__int_as_float(0x7f800000) : 0.0f;
    float4 v[R][K];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int64_t row = r < nr ? row0 + r : row0;  // (a repeated row is served by L2, not stored)
        const float* xr = a.x + row * a.cols + 4 * t;
#pragma unroll
        for (int j = 0; j < K; ++j) v[r][j] = okj[j] ? ld_stream4(xr + 4 * kThreads * j) : make_float4(kId, kId, kId, kId);
    }
    if constexpr (OP == OP_RMSNORM) {
        // The epilogue's weight quads, into L1 while the rows load: by the
        // first CTA on each SM (the block scheduler gives CTAs 0 .. SMs - 1 one
        // SM each); the SM's later CTAs then find them in L1. One prefetch per
        // 128-byte line: from the thread whose quad starts the line, and from
        // thread 0 (a vector need not start on a line).
        if (blockIdx.x < a.pf_ctas) {
#pragma unroll
            for (int j = 0; j < K; ++j) {
                if (!okj[j]) continue;
                const int c = 4 * (t + kThreads * j);
                if (a.has_w && (t == 0 || (reinterpret_cast<uintptr_t>(a.w + c) & 127) < 16)) prefetch_l1(a.w + c);
            }
        }
    }
    const float n = a.cols_f;

    if constexpr (OP == OP_SOFTMAX) {
        float m[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            float4 l = v[r][0];
#pragma unroll
            for (int j = 1; j < K; ++j) {
                l.x = fmaxf(l.x, v[r][j].x);
                l.y = fmaxf(l.y, v[r][j].y);
                l.z = fmaxf(l.z, v[r][j].z);
                l.w = fmaxf(l.w, v[r][j].w);
            }
            m[r] = quad_top<MaxR>(l);
        }
        tree_rows<MaxR, R>(m, part[tb]);
        tb ^= 1;
        float s[R];
        if constexpr (ORD) {
            // e = exp_ot(x - m) in place. The differences of a finite row lie in
            // (-86, 0] almost always: then the whole thread takes the packed,
            // branch-free form; otherwise (a huge spread, infinities, NaN) every
            // element takes the general form. Padding slots end up 0.
            bool fast = true;
#pragma unroll
            for (int r = 0; r < R; ++r)
#pragma unroll
                for (int j = 0; j < K; ++j)
                    if (okj[j]) {
                        v[r][j] = sub4s(v[r][j], m[r]);
                        fast &= ordered::exp_ot_in_fast_range(v[r][j].x) & ordered::exp_ot_in_fast_range(v[r][j].y) &
                                ordered::exp_ot_in_fast_range(v[r][j].z) & ordered::exp_ot_in_fast_range(v[r][j].w);
                    }
            if (fast) {
#pragma unroll
                for (int r = 0; r < R; ++r)
#pragma unroll
                    for (int j = 0; j < K; ++j)
                        if (okj[j]) v[r][j] = cat2(ordered::exp_ot_fast2(lo2(v[r][j])), ordered::exp_ot_fast2(hi2(v[r][j])));
            } else {
#pragma unroll
                for (int r = 0; r < R; ++r)
#pragma unroll
                    for (int j = 0; j < K; ++j)
                        if (okj[j]) {
                            v[r][j].x = ordered::exp_ot(v[r][j].x);
                            v[r][j].y = ordered::exp_ot(v[r][j].y);
                            v[r][j].z = ordered::exp_ot(v[r][j].z);
                            v[r][j].w = ordered::exp_ot(v[r][j].w);
                        }
            }
#pragma unroll
            for (int j = 0; j < K; ++j)
                if (!okj[j])
#pragma unroll
                    for (int r = 0; r < R; ++r) v[r][j] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        } else {
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const float4 nmb = make_float4(-mb_of(m[r]), -mb_of(m[r]), -mb_of(m[r]), -mb_of(m[r]));
                const float4 l2e = make_float4(kL2E, kL2E, kL2E, kL2E);
#pragma unroll
                for (int j = 0; j < K; ++j) {  // padding: ex2(-inf) = 0
                    const float4 t4 = fma4(v[r][j], l2e, nmb);
                    v[r][j] = make_float4(ex2(t4.x), ex2(t4.y), ex2(t4.z), ex2(t4.w));
                }
            }
        }
#pragma unroll
        for (int r = 0; r < R; ++r) {
            float4 l = v[r][0];
#pragma unroll
            for (int j = 1; j < K; ++j) l = add4(l, v[r][j]);
            s[r] = quad_top<Add>(l);
        }
        tree_rows<Add, R>(s, part[tb]);
        tb ^= 1;
#pragma unroll
        for (int r = 0; r < R; ++r) {
            if (r >= nr) break;
            const float inv = ORD ? __fdiv_rn(1.0f, s[r]) : 1.0f / s[r];
            float* yr = a.y + (row0 + r) * a.cols + 4 * t;
#pragma unroll
            for (int j = 0; j < K; ++j)
                if (okj[j]) store4(yr + 4 * kThreads * j, mul4s(v[r][j], inv), a.y_vec);
        }
    } else if constexpr (OP == OP_RMSNORM) {
        float ss[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            if constexpr (ORD) {
                float4 l = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
                for (int j = 0; j < K; ++j) l = add4(l, prod4_rn(v[r][j], v[r][j]));
                ss[r] = quad_top<AddO>(l);
            } else {
                float2 acc = make_float2(0.0f, 0.0f);
#pragma unroll
                for (int j = 0; j < K; ++j) acc = sq_acc(acc, v[r][j]);
                ss[r] = acc.x + acc.y;
            }
        }
        tree_rows<Add, R>(ss, part[tb]);
        tb ^= 1;
        float sc[R];
#pragma unroll
        for (int r = 0; r < R; ++r)
            sc[r] = ORD ? __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ss[r], n), a.eps)))
                        : rsqrtf(fmaf(ss[r], a.inv_cols, a.eps));
        const bool wv = a.has_w && aligned16(a.w);
#pragma unroll
        for (int j = 0; j < K; ++j) {
            if (!okj[j]) continue;
            const int c = 4 * (t + kThreads * j);
            const float4 w = a.has_w ? param4(a.w + c, wv) : make_float4(1.0f, 1.0f, 1.0f, 1.0f);
#pragma unroll
            for (int r = 0; r < R; ++r) {
                if (r >= nr) break;
                float4 o = mul4s(v[r][j], sc[r]);
                if (ORD) {
                    if (a.has_w) o = mul4(o, w);
                } else {
                    o = mul4(o, w);
                }
                store4(a.y + (row0 + r) * a.cols + c, o, a.y_vec);
            }
        }
    } else {  // OP_LAYERNORM: mean, then the centred sum of squares on the cached row
        float mu[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            float4 l = v[r][0];
#pragma unroll
            for (int j = 1; j < K; ++j) l = add4(l, v[r][j]);
            mu[r] = quad_top<Add>(l);
        }
        tree_rows<Add, R>(mu, part[tb]);
        tb ^= 1;
        float q[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            // one rounded division (a contracted x - sum * (1/N) would leave a
            // constant row at ~1e-7 instead of 0)
            mu[r] = __fdiv_rn(mu[r], n);
            if constexpr (ORD) {
                float4 l = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
                for (int j = 0; j < K; ++j) {
                    if (!okj[j]) continue;  // padding is no column of the row
                    const float4 c = sub4s(v[r][j], mu[r]);
                    l = add4(l, prod4_rn(c, c));
                }
                q[r] = quad_top<AddO>(l);
            } else {
                float2 acc = make_float2(0.0f, 0.0f);
#pragma unroll
                for (int j = 0; j < K; ++j)
                    if (okj[j]) acc = sq_acc(acc, sub4s(v[r][j], mu[r]));
                q[r] = acc.x + acc.y;
            }
        }
        tree_rows<Add, R>(q, part[tb]);
        tb ^= 1;
        float sc[R];
#pragma unroll
        for (int r = 0; r < R; ++r)
            sc[r] = ORD ? __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(q[r], n), a.eps)))
                        : rsqrtf(fmaf(q[r], a.inv_cols, a.eps));
        cp_async_wait_all();  // this thread's own parameter quads (copied at entry)
#pragma unroll
        for (int j = 0; j < K; ++j) {
            if (!okj[j]) continue;
            const int c = 4 * (t + kThreads * j);
            const float4 w = a.has_w ? psm[t + kThreads * j] : make_float4(1.0f, 1.0f, 1.0f, 1.0f);
            const float4 b = a.has_b ? psm[K * kThreads + t + kThreads * j] : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
            for (int r = 0; r < R; ++r) {
                if (r >= nr) break;
                float4 o = mul4s(sub4s(v[r][j], mu[r]), sc[r]);
                if (ORD) {
                    if (a.has_w) o = a.has_b ? prod4_rn(o, w) : mul4(o, w);
                    if (a.has_b) o = add4(o, b);
                } else {
                    o = fma4(o, w, b);
                }
                store4(a.y + (row0 + r) * a.cols + c, o, a.y_vec);
            }
        }
    }
}

// Groups blockIdx.x, blockIdx.x + gridDim.x, ... (one group per CTA when the
// grid covers the rows). A block index alternates over consecutive trees, so a
// tree never writes a slot block that a thread may still be reading: between
// two uses of one block lies the other tree's barrier.
template <int OP, bool ORD, int K, int R>
__global__ void __launch_bounds__(kThreads, min_blocks<K, R>()) wave_kernel(const RowArgs a) {
    __shared__ __align__(16) float part[2][R][8];
    // LayerNorm: its weight and bias quads, 2 x 256 K of them (dynamic shared memory)
    extern __shared__ __align__(16) float4 psm[];
    int tb = 0;
    pdl_enter();
    if constexpr (OP == OP_LAYERNORM) {
        // Every CTA copies the weight and bias quads its threads will use into
        // shared memory before it requests its rows. Read from global memory in
        // the epilogue, they would wait behind the other CTAs' row loads still
        // outstanding on the SM, even as L1 or L2 hits; from shared memory they
        // are there when the statistics are, and the SM's stores start early.
        stage_params<K>(a, psm);
    }
    if constexpr (OP != OP_SOFTMAX) {
        // The norms read their weight (and bias) quads only in the epilogue, and
        // in a stream of launches those vectors have usually left L2, so the
        // first read per SM would wait on DRAM after the merges. CTA 0 asks L2
        // for both vectors now (one prefetch per 128-byte line, two per
        // thread at 6144 columns): they land while the rows load, and each
        // SM's epilogue finds them in L2 or, after its first CTA, in L1.
        // Prefetching from every CTA measured slower: the redundant requests
        // compete with the row loads.
        if (blockIdx.x == 0) {
            // 128-byte steps over one vector, plus its last element (a vector
            // need not start on a line); every address lies inside the vector
            const int lines = (a.cols + 31) / 32 + 1;
            const int nvecs = (a.has_w ? 1 : 0) + (OP == OP_LAYERNORM && a.has_b ? 1 : 0);
            for (int i = threadIdx.x; i < nvecs * lines; i += kThreads) {
                const float* base = (a.has_w && i < lines) ? a.w : a.b;
                prefetch_l2(base + min(32 * (i < lines ? i : i - lines), a.cols - 1));
            }
        }
    }
    // Staggered start. The block scheduler gives CTAs 0 .. SMs - 1 one SM each,
    // the next SMs CTAs one more each, and so on: CTA b is of launch rank
    // k = b / SMs. Issued all at once, every CTA's loads would be served
    // interleaved and land together at the end of the read phase, and all
    // epilogues would follow it at once, each SM storing its five or six rows
    // while DRAM idles. A CTA of rank k instead requests its rows k x
    // stagger_ns late, about the time DRAM takes to serve one rank: the ranks'
    // rows land one after another, and each rank's reductions and stores run
    // while the next ranks' rows stream in. (Host-set for grids that are
    // resident in one wave; the wait is one thread's bounded sleep on the
    // global timer, the others wait at the barrier.)
    if (a.stagger_ns > 0) {
        const unsigned rank = blockIdx.x / static_cast<unsigned>(a.pf_ctas);
        if (rank > 0) {
            if (threadIdx.x == 0) {
                const unsigned long long t0 = global_ns();
                const unsigned long long d = static_cast<unsigned long long>(rank) * a.stagger_ns;
                while (global_ns() - t0 < d) __nanosleep(64);
            }
            __syncthreads();
        }
    }
    if constexpr (R == 2) {
        // One wave of every resident CTA (the selector's choice when the rows
        // outnumber the CTAs the device holds but not twice over): CTAs
        // 0 .. rows - G - 1 take two rows, the others one, so that an SM holds
        // five or six rows rather than four or six.
        const int64_t G = gridDim.x;
        if (G < a.rows && 2 * G > a.rows) {
            const int64_t pairs = a.rows - G, g = blockIdx.x;
            wave_group<OP, ORD, K, R>(a, g < pairs ? 2 * g : pairs + g, g < pairs ? 2 : 1, part, psm, tb);
            return;
        }
    }
    for (int64_t g = blockIdx.x; g * R < a.rows; g += gridDim.x)
        wave_group<OP, ORD, K, R>(a, g * R, a.rows - g * R < R ? static_cast<int>(a.rows - g * R) : R, part, psm, tb);
}

}  // namespace wave
}  // namespace tr
