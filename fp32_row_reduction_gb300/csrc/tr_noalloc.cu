// The no-allocation entry point: the split-row plan over a fixed scratch area.
//
// Callers that cannot allocate device memory at call time use it. Examples:
// code that runs inside a pre-sized memory arena where every byte is
// accounted for, and latency-critical loops where cudaMalloc is not
// acceptable, because it may synchronise the device and can fail under memory
// pressure. The existing entry points allocate a split-plan workspace on a
// stream's first split launch. This one uses a file-scope device array instead,
// sized for at most kNoAllocMaxParts row segments and kNoAllocMaxRows rows, and
// performs no device allocation on any call.
//
// Zero state: the arrival and departure counters must be zero before a launch.
// The array is zero when the module loads, and every complete launch leaves
// the counters at zero: the last CTA to leave a row clears the row's counters,
// and every CTA of a grid leaves eventually, even one whose wait gave up.
//
// Concurrency: one scratch area per device, shared by all streams and host
// threads. Two calls whose kernels overlap in time (different streams, or host
// threads without ordering) race on the counters and partials. Callers must
// order such calls, for example by issuing them on one stream.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>

#include "tr.h"
#include "tr_internal.h"

constexpr int kNoAllocMaxRows = 256;
constexpr int kNoAllocMaxParts = 1024;
constexpr size_t kNoAllocScratchBytes = kNoAllocMaxParts * 16 + 2 * kNoAllocMaxRows * sizeof(unsigned);  // 18 KB

// The scratch: partials (kNoAllocMaxParts x 16 bytes), then the arrival and
// departure counters (kNoAllocMaxRows each). Zero when the module loads.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace tr {

namespace {

constexpr int kNoAllocThreads = 512;  // threads per CTA
constexpr int kNoAllocMaxSlots = 13;  // 16-byte slots cached per thread (two CTAs per SM fit)
constexpr int kMaxDevices = 64;

struct NoAllocDevice {
    bool ready;
    unsigned char* scratch;  // device address of g_noalloc_scratch
    unsigned* err;           // device address of the library's error word
    int sm_count;
    int ctas_per_sm[3];      // resident CTAs per SM at the largest cache, per operator
};
NoAllocDevice g_na[kMaxDevices];
std::mutex g_na_mu;

const void* split_fn(int op) {
    switch (op) {
        case TR_OP_SOFTMAX: return kernel_softmax(TR_PLAN_SPLIT, 32, 1, 0);
        case TR_OP_RMSNORM: return kernel_rmsnorm(TR_PLAN_SPLIT, 32, 1, 0);
        case TR_OP_LAYERNORM: return kernel_layernorm(TR_PLAN_SPLIT, 32, 1, 0);
    }
    return nullptr;
}

// Report a CUDA error and clear it from the runtime's sticky last-error slot,
// so that a failed set-up does not surface in the caller's next CUDA call.
tr_status cuda_err(cudaError_t e, const char* what) {
    set_last_error(what, cudaGetErrorString(e));
    cudaGetLastError();
    return TR_ERR_CUDA;
}

// One-time set-up per device: symbol addresses, the kernels' shared-memory
// limit and their residency. Done on the first call on each device.
tr_status setup(int dev, NoAllocDevice** out) {
    if (dev < 0 || dev >= kMaxDevices) {
        set_last_error("no-alloc entry point", "device ordinal out of range");
        return TR_ERR_UNSUPPORTED;
    }
    NoAllocDevice& d = g_na[dev];
    if (!d.ready) {
        void* p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return cuda_err(e, "cudaGetSymbolAddress(no-alloc scratch)");
        d.scratch = static_cast<unsigned char*>(p);
        e = device_error_symbol(&p);
        if (e != cudaSuccess) return cuda_err(e, "cudaGetSymbolAddress(device error word)");
        d.err = static_cast<unsigned*>(p);
        e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return cuda_err(e, "cudaDeviceGetAttribute");
        const size_t smem = static_cast<size_t>(kNoAllocMaxSlots) * kNoAllocThreads * 16;
        int optin = 0;
        e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if (e != cudaSuccess) return cuda_err(e, "cudaDeviceGetAttribute");
        for (int op = 0; op < 3; ++op) {
            const void* fn = split_fn(op);
            // the dynamic limit is what the per-CTA opt-in maximum leaves beside
            // the kernel's static shared memory (as for the other entry points)
            cudaFuncAttributes fa;
            e = cudaFuncGetAttributes(&fa, fn);
            if (e != cudaSuccess) return cuda_err(e, "cudaFuncGetAttributes");
            const int budget = std::min<int>(kStagedSmemBudget, optin - static_cast<int>(fa.sharedSizeBytes));
            if (budget < static_cast<int>(smem)) {
                set_last_error("no-alloc entry point", "the segment cache does not fit this device's shared memory");
                return TR_ERR_UNSUPPORTED;
            }
            e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, budget);
            if (e != cudaSuccess) return cuda_err(e, "cudaFuncSetAttribute(shared memory)");
            int n = 0;
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, kNoAllocThreads, smem);
            if (e != cudaSuccess) return cuda_err(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
            d.ctas_per_sm[op] = n;
        }
        d.ready = true;
    }
    *out = &d;
    return TR_OK;
}

bool overlap(const void* a, size_t na, const void* b, size_t nb) {
    if (!a || !b || na == 0 || nb == 0) return false;
    const uintptr_t pa = reinterpret_cast<uintptr_t>(a), pb = reinterpret_cast<uintptr_t>(b);
    return pa < pb + nb && pb < pa + na;
}

bool mis4(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 3u) != 0; }

}  // namespace
}  // namespace tr

using namespace tr;

extern "C" tr_status tr_split_rows_noalloc_f32(int32_t op, const float* x, const float* w, const float* b, float* y,
                                               int64_t rows, int64_t cols, float eps, cudaStream_t stream) {
    if (op != TR_OP_SOFTMAX && op != TR_OP_RMSNORM && op != TR_OP_LAYERNORM) {
        set_last_error("no-alloc entry point", "op must be TR_OP_SOFTMAX, TR_OP_RMSNORM or TR_OP_LAYERNORM");
        return TR_ERR_INVALID_ARG;
    }
    if (rows < 0 || cols < 1 || cols >= (1LL << 24) || (rows > 0 && rows > INT64_MAX / cols / 4)) {
        set_last_error("no-alloc entry point", "rows must be >= 0 and cols in [1, 2^24 - 1]");
        return TR_ERR_INVALID_ARG;
    }
    if (op != TR_OP_SOFTMAX && (!std::isfinite(eps) || eps < 0.0f)) {
        set_last_error("no-alloc entry point", "eps must be finite and >= 0");
        return TR_ERR_INVALID_ARG;
    }
    if ((op == TR_OP_SOFTMAX && (w || b)) || (op == TR_OP_RMSNORM && b)) {
        set_last_error("no-alloc entry point", "softmax takes no w or b, RMSNorm no b");
        return TR_ERR_INVALID_ARG;
    }
    if (rows == 0) return TR_OK;
    if (!x || !y) {
        set_last_error("no-alloc entry point", "x and y must not be null");
        return TR_ERR_INVALID_ARG;
    }
    if (mis4(x) || mis4(y) || mis4(w) || mis4(b)) {
        set_last_error("no-alloc entry point", "x, y, w and b must be 4-byte aligned");
        return TR_ERR_INVALID_ARG;
    }
    const size_t n = static_cast<size_t>(rows) * static_cast<size_t>(cols) * 4;
    const size_t nv = static_cast<size_t>(cols) * 4;
    if (overlap(x, n, y, n) || overlap(w, nv, y, n) || overlap(b, nv, y, n)) {
        set_last_error("no-alloc entry point", "the output overlaps an input");
        return TR_ERR_INVALID_ARG;
    }
    if (rows > kNoAllocMaxRows) {
        set_last_error("no-alloc entry point", "at most 256 rows (the fixed scratch holds 256 row counters)");
        return TR_ERR_UNSUPPORTED;
    }
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_err(e, "cudaGetDevice");
    NoAllocDevice* d = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_na_mu);
        tr_status s = setup(dev, &d);
        if (s != TR_OK) return s;
    }
    // C co-resident CTAs per row: as many as the device holds at once, at most 32
    const int64_t cap = std::min<int64_t>(static_cast<int64_t>(d->ctas_per_sm[op]) * d->sm_count, kNoAllocMaxParts);
    const int64_t C = std::min<int64_t>(kSplitMaxCtas, cap / rows);
    if (C < 2) {
        set_last_error("no-alloc entry point",
                       "too many rows: each row needs 2 co-resident CTAs (at most half the device's resident CTAs)");
        return TR_ERR_UNSUPPORTED;
    }
    const int64_t n4 = (cols + 3) / 4;
    const int64_t per = (n4 + C - 1) / C;
    const int K = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>((per + kNoAllocThreads - 1) / kNoAllocThreads,
                                                                           kNoAllocMaxSlots)));
    RowArgs a;
    std::memset(&a, 0, sizeof a);
    a.x = x;
    a.y = y;
    a.w = w;
    a.b = b;
    a.rows = rows;
    a.cols = static_cast<int>(cols);
    a.eps = eps;
    a.inv_cols = 1.0f / static_cast<float>(cols);
    a.cols_f = static_cast<float>(cols);
    a.S = kNoAllocThreads / 32;
    a.C = static_cast<int>(C);
    a.y_vec = ((reinterpret_cast<uintptr_t>(x) - reinterpret_cast<uintptr_t>(y)) & 15u) == 0;
    a.has_w = w != nullptr;
    a.has_b = b != nullptr;
    a.err = d->err;
    a.wait_ns = 2000000000LL;
    a.debug_flags = debug_flags_now();
    a.slot_floats = 4 * K * kNoAllocThreads;
    a.sp_part = reinterpret_cast<float4*>(d->scratch);
    a.sp_arrive = reinterpret_cast<unsigned*>(d->scratch + kNoAllocMaxParts * 16);
    a.sp_depart = a.sp_arrive + kNoAllocMaxRows;
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof cfg);
    cfg.gridDim = dim3(static_cast<unsigned>(rows * C));
    cfg.blockDim = dim3(kNoAllocThreads);
    cfg.dynamicSmemBytes = static_cast<size_t>(K) * kNoAllocThreads * 16;
    cfg.stream = stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeCooperative;  // every CTA waits for its row's other segments
    attr.val.cooperative = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    void* args[] = {&a};
    e = cudaLaunchKernelExC(&cfg, split_fn(op), args);
    if (e != cudaSuccess) return cuda_err(e, "kernel launch");
    return TR_OK;
}
