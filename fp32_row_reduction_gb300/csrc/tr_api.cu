// The C-ABI of libtr: argument validation, plan selection and caching, launch.
//
// Contracts ("TIRx Metal reduction lowering"): noalias arguments (§3 "Semantic
// domain and fail-closed admission"), explicit errors rather than clamping or
// fallback (§1, §6), guarded out-of-range labels selecting 0 (§5.2). Every
// step of the hot path runs in this library's kernels; there is no CPU path.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <tuple>
#include <vector>

#include "tr.h"
#include "tr_internal.h"
#include "tr_plan.h"

namespace tr {

// Device error word: set by a bounded device-side wait that gives up, read and
// cleared by tr_last_device_error().
__device__ unsigned int g_device_error = 0;

namespace {

thread_local std::string t_last_error;

tr_status fail(tr_status s, const std::string& msg) {
    t_last_error = msg;
    return s;
}
tr_status cuda_fail(cudaError_t e, const char* what) {
    return fail(TR_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

struct DeviceState {
    bool ready = false;
    tr_device_desc desc{};
    unsigned* err = nullptr;  // device address of g_device_error on this device
    std::map<std::tuple<int, int64_t, int64_t, int, int>, tr_plan> plans;  // (op, rows, cols, order, align16)
    std::map<std::tuple<const void*, int, int, size_t>, int64_t> occ;  // (kernel, threads, cluster, smem) -> resident CTAs
    std::map<const void*, bool> smem_opt_in;                        // kernels allowed large dynamic smem
    std::map<const void*, bool> wide_cluster;                       // kernels allowed clusters above 8 CTAs
    std::map<cudaStream_t, void*> split_ws;                         // split-plan workspace per stream
};

std::mutex g_mu;
std::map<int, DeviceState> g_devices;
constexpr int kOps = TR_OP_ROW_MINMAX + 1;
bool g_override_set[kOps] = {};
tr_plan g_override[kOps];
int g_debug_flags = 0;
// Launch with programmatic stream serialization (dependent launches overlap
// their launch latency with the previous kernel's tail); TR_DISABLE_PDL=1 turns it off.
const bool g_pdl = [] {
    const char* v = std::getenv("TR_DISABLE_PDL");
    return !(v && v[0] == '1');
}();
constexpr long long kWaitNs = 2000000000LL;  // a bounded device wait gives up after 2 s

// The start delay per launch rank of a wave plan (see the wave kernel): the
// time the device's HBM takes to deliver one rank's rows (SMs x rows_per_cta
// rows), scaled per operator (against 6800 GB/s: 0.92, and 1.0 for RMSNorm,
// which an A/B at 768 x 6144 preferred by 0.05 us; 1.6 lost everywhere), for
// grids of more than one rank that are resident in one wave; 0 (no delay)
// otherwise.
int wave_stagger_ns(const tr_device_desc& d, const tr_plan& p, int64_t cols) {
    if (p.kind != TR_PLAN_WAVE || d.sm_count < 1 || d.hbm_gbs <= 0.0) return 0;
    const int64_t resident = p.resident_ctas > 0 ? p.resident_ctas : static_cast<int64_t>(p.ctas_per_sm) * d.sm_count;
    if (p.grid_ctas <= d.sm_count || p.grid_ctas > resident) return 0;
    const double scale = p.op == TR_OP_RMSNORM ? 1.0 : 0.92;
    const double rank_bytes = static_cast<double>(d.sm_count) * p.rows_per_cta * static_cast<double>(cols) * 4.0;
    return static_cast<int>(std::min(4000.0, scale * rank_bytes / 6800.0));  // 6800 GB/s = bytes per ns
}

// Allow a kernel the full dynamic shared memory budget (once per kernel and
// device), less what its static shared memory takes of the per-CTA limit.
bool opt_in_smem(DeviceState& st, const void* fn) {
    auto it = st.smem_opt_in.find(fn);
    if (it != st.smem_opt_in.end()) return it->second;
    cudaFuncAttributes fa;
    int dev = 0, optin = 0;
    bool ok = cudaFuncGetAttributes(&fa, fn) == cudaSuccess && cudaGetDevice(&dev) == cudaSuccess &&
              cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) == cudaSuccess;
    if (ok) {
        const int budget = std::min<int>(kStagedSmemBudget, optin - static_cast<int>(fa.sharedSizeBytes));
        ok = budget > 0 && cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, budget) == cudaSuccess;
    }
    if (!ok) cudaGetLastError();
    st.smem_opt_in[fn] = ok;
    return ok;
}

tr_status device_state(int dev, DeviceState** out) {
    DeviceState& st = g_devices[dev];
    if (!st.ready) {
        tr_device_desc d = gb300_desc();
        int v = 0;
        cudaError_t e;
#define TR_ATTR(attr, field)                                      \
    e = cudaDeviceGetAttribute(&v, attr, dev);                    \
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute"); \
    d.field = v;
        TR_ATTR(cudaDevAttrMultiProcessorCount, sm_count)
        TR_ATTR(cudaDevAttrMaxThreadsPerMultiProcessor, max_threads_per_sm)
        TR_ATTR(cudaDevAttrMaxBlocksPerMultiprocessor, max_ctas_per_sm)
        TR_ATTR(cudaDevAttrMaxRegistersPerMultiprocessor, regs_per_sm)
        TR_ATTR(cudaDevAttrMaxSharedMemoryPerMultiprocessor, smem_per_sm)
#undef TR_ATTR
        e = cudaDeviceGetAttribute(&v, cudaDevAttrL2CacheSize, dev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
        d.l2_bytes = v;
        e = cudaDeviceGetAttribute(&v, cudaDevAttrClusterLaunch, dev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
        d.max_cluster_ctas = v ? 16 : 1;  // sizes above 8 are non-portable: checked per kernel
        if (const char* bw = std::getenv("TR_HBM_GBS")) d.hbm_gbs = std::atof(bw);
        void* errp = nullptr;
        e = cudaGetSymbolAddress(&errp, g_device_error);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(device error word)");
        st.err = static_cast<unsigned*>(errp);
        st.desc = d;
        st.ready = true;
    }
    *out = &st;
    return TR_OK;
}

// Allow a kernel clusters of more than 8 CTAs (non-portable sizes, up to 16).
bool opt_in_wide_cluster(DeviceState& st, const void* fn) {
    auto it = st.wide_cluster.find(fn);
    if (it != st.wide_cluster.end()) return it->second;
    const bool ok = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess;
    if (!ok) cudaGetLastError();
    st.wide_cluster[fn] = ok;
    return ok;
}

// CTAs of a plan's kernel resident at once on the device (0 = cannot run).
// Cluster plans: the device's concurrent clusters times C.
int64_t query_occupancy(DeviceState& st, const tr_plan& p, size_t smem) {
    const void* fn = kernel_for(p);
    if (!fn) return 0;
    const int C = (p.kind == TR_PLAN_CLUSTER || p.kind == TR_PLAN_STREAM || p.kind == TR_PLAN_ORDERED) ? p.cluster_ctas : 1;
    const auto key = std::make_tuple(fn, p.block_threads, C, smem);
    auto it = st.occ.find(key);
    if (it != st.occ.end()) return it->second;
    int n = 0;
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, fn) != cudaSuccess || fa.maxThreadsPerBlock < p.block_threads) {
        cudaGetLastError();
        st.occ[key] = 0;
        return 0;
    }
    if ((smem > 0 && !opt_in_smem(st, fn)) || (C > 8 && !opt_in_wide_cluster(st, fn))) {
        st.occ[key] = 0;
        return 0;
    }
    if (C == 1) {
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, p.block_threads, smem) != cudaSuccess) n = 0;
        n *= st.desc.sm_count;
    } else {
        cudaLaunchConfig_t cfg;
        std::memset(&cfg, 0, sizeof cfg);
        cfg.gridDim = dim3(static_cast<unsigned>(C) * 64u);
        cfg.blockDim = dim3(p.block_threads);
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeClusterDimension;
        attr.val.clusterDim.x = C;
        attr.val.clusterDim.y = 1;
        attr.val.clusterDim.z = 1;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        int clusters = 0;
        if (cudaOccupancyMaxActiveClusters(&clusters, fn, &cfg) != cudaSuccess) clusters = 0;
        n = clusters > 0 ? clusters * C : 0;
    }
    cudaGetLastError();
    st.occ[key] = n;
    return n;
}

// The split-plan workspace of `stream` (kSplitWorkspaceBytes, counters zero),
// allocated and cleared in stream order on the stream's first split launch.
// Launches on one stream run one at a time, so they can share it; another
// stream gets its own. Allocation is refused while the stream is being
// captured: make one split call on the stream before capturing it.
tr_status split_workspace(DeviceState& st, cudaStream_t stream, void** out) {
    auto it = st.split_ws.find(stream);
    if (it != st.split_ws.end()) {
        *out = it->second;
        return TR_OK;
    }
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(stream, &cap);
    if (e != cudaSuccess || cap != cudaStreamCaptureStatusNone) {
        cudaGetLastError();
        return fail(TR_ERR_UNSUPPORTED,
                    "a split plan's workspace is allocated on the stream's first call, which must not be captured: "
                    "run one call on this stream before capturing it");
    }
    void* ws = nullptr;
    e = cudaMalloc(&ws, kSplitWorkspaceBytes);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc(split workspace)");
    e = cudaMemsetAsync(ws, 0, kSplitWorkspaceBytes, stream);
    if (e != cudaSuccess) {
        cudaFree(ws);
        return cuda_fail(e, "cudaMemsetAsync(split workspace)");
    }
    st.split_ws.emplace(stream, ws);
    *out = ws;
    return TR_OK;
}

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
    if (!a || !b || na == 0 || nb == 0) return false;
    const uintptr_t pa = reinterpret_cast<uintptr_t>(a), pb = reinterpret_cast<uintptr_t>(b);
    return pa < pb + nb && pb < pa + na;
}

bool misaligned(const void* p, uintptr_t a) { return p && (reinterpret_cast<uintptr_t>(p) % a) != 0; }

struct Call {
    int op;
    RowArgs a;
    int order;
};

// The operators (softmax, the norms, cross-entropy, their fused and backward
// forms) take rows of fewer than 2^24 columns, so that (float)cols, by which
// the norms divide, is exact; the standalone row reductions divide by nothing
// and take rows of up to 2^31 - 1 columns.
constexpr int64_t kMaxOperatorCols = (1LL << 24) - 1;
constexpr int64_t kMaxReductionCols = 0x7fffffffLL;

tr_status validate_common(int64_t rows, int64_t cols, int order, int64_t max_cols = kMaxOperatorCols) {
    if (order != TR_ORDER_UNORDERED_TREE && order != TR_ORDER_ORDERED_TREE && !fold_order(order))
        return fail(TR_ERR_INVALID_ARG, "order must be one of the tr_order values");
    if (rows < 0) return fail(TR_ERR_INVALID_ARG, "rows must be >= 0");
    if (cols < 1 || cols > max_cols)
        return fail(TR_ERR_INVALID_ARG, max_cols == kMaxOperatorCols ? "cols must be in [1, 2^24 - 1]"
                                                                      : "cols must be in [1, 2^31 - 1]");
    if (rows > 0 && rows > INT64_MAX / cols / 4) return fail(TR_ERR_INVALID_ARG, "rows * cols too large");
    return TR_OK;
}

tr_status validate_eps(float eps) {
    if (!std::isfinite(eps) || eps < 0.0f) return fail(TR_ERR_INVALID_ARG, "eps must be finite and >= 0");
    return TR_OK;
}

// The fold policies' single realisation (TR_PLAN_FOLD): a warp per row.
static tr_plan fold_plan(int op, int64_t rows, int order) {
    tr_plan p;
    std::memset(&p, 0, sizeof p);
    p.op = op;
    p.order = order;
    p.kind = TR_PLAN_FOLD;
    p.lanes_per_row = 32;
    p.warps_per_row = 1;
    p.rows_per_cta = 2;
    p.cluster_ctas = 1;
    p.block_threads = 64;
    p.grid_ctas = (rows + 1) / 2;
    p.candidates = 1;
    return p;
}

tr_status run(Call& c, cudaStream_t stream) {
    RowArgs& a = c.a;
    if (a.rows == 0) return TR_OK;
    if (fold_order(c.order)) {
        if (!fold_supported(c.op)) return fail(TR_ERR_UNSUPPORTED, "the fold policies cover the four operators and the row reductions");
        const cudaError_t fe = launch_fold(c.op, c.order == TR_ORDER_FOLD_RIGHT, a, stream);
        if (fe != cudaSuccess) return cuda_fail(fe, "fold launch");
        return TR_OK;
    }
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    const bool align16 = (a.cols % 4 == 0) && (reinterpret_cast<uintptr_t>(a.x) % 16 == 0) &&
                         (reinterpret_cast<uintptr_t>(a.w) % 16 == 0) && (reinterpret_cast<uintptr_t>(a.b) % 16 == 0);
    tr_plan plan;
    DeviceState* split_dev = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        DeviceState* st = nullptr;
        tr_status s = device_state(dev, &st);
        if (s != TR_OK) return s;
        OccupancyFn occ = [st](const tr_plan& p, size_t smem) { return query_occupancy(*st, p, smem); };
        a.err = st->err;
        split_dev = st;
        if (g_override_set[c.op]) {
            plan = g_override[c.op];
            plan.op = c.op;
            plan.order = c.order;
            const char* why = "";
            s = check_plan(st->desc, occ, &plan, a.rows, a.cols, align16, &why);
            if (s != TR_OK) return fail(TR_ERR_UNSUPPORTED, std::string("plan override rejected: ") + why);
            plan.est_us = estimate_us(st->desc, plan, a.rows, a.cols, align16);
        } else {
            const auto key = std::make_tuple(c.op, a.rows, static_cast<int64_t>(a.cols), c.order, align16 ? 1 : 0);
            auto it = st->plans.find(key);
            if (it == st->plans.end()) {
                s = select_plan(st->desc, occ, c.op, a.rows, a.cols, c.order, align16, &plan);
                if (s != TR_OK) return fail(s, "no legal plan for this shape on this device");
                st->plans.emplace(key, plan);
            } else {
                plan = it->second;
            }
        }
    }
    const void* fn = kernel_for(plan);
    if (!fn) return fail(TR_ERR_UNSUPPORTED, "plan has no kernel in this build");
    a.S = plan.warps_per_row;
    a.C = plan.cluster_ctas;
    a.wait_ns = kWaitNs;
    a.debug_flags = g_debug_flags;
    a.pf_ctas = split_dev->desc.sm_count;  // about one CTA per SM: the first the block scheduler places there
    a.stagger_ns = wave_stagger_ns(split_dev->desc, plan, a.cols);
    a.nbuf = (plan.kind == TR_PLAN_STAGED || plan.kind == TR_PLAN_ORDERED_STAGED) ? plan.rows_per_cta : 0;
    a.slot_floats = staged_slot_floats(a.cols);
    const bool split = plan.kind == TR_PLAN_SPLIT;
    const bool segs = plan.kind == TR_PLAN_SEGMENTS;
    if (split || segs) {
        void* ws = nullptr;
        {
            std::lock_guard<std::mutex> lock(g_mu);
            tr_status s = split_workspace(*split_dev, stream, &ws);
            if (s != TR_OK) return s;
        }
        a.sp_part = static_cast<float4*>(ws);
        a.sp_arrive = reinterpret_cast<unsigned*>(static_cast<char*>(ws) + kSplitMaxParts * 16);
        a.sp_depart = a.sp_arrive + kSplitMaxRows;
        a.slot_floats = 4 * plan.vec_slots * plan.block_threads;
        if (segs) a.nbuf = seg_cached_rows(a.rows, a.cols, plan.grid_ctas);
    }
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof cfg);
    cfg.gridDim = dim3(static_cast<unsigned>(plan.grid_ctas));
    cfg.blockDim = dim3(plan.block_threads);
    cfg.dynamicSmemBytes = plan_dynamic_smem(plan, a.cols);
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    unsigned nattr = 0;
    if (plan.cluster_ctas > 1 && !split && !segs) {
        attr[nattr].id = cudaLaunchAttributeClusterDimension;
        attr[nattr].val.clusterDim.x = plan.cluster_ctas;
        attr[nattr].val.clusterDim.y = 1;
        attr[nattr].val.clusterDim.z = 1;
        ++nattr;
    }
    if (split || segs) {
        // every CTA waits for the other segments of its row(s): all must be resident
        attr[nattr].id = cudaLaunchAttributeCooperative;
        attr[nattr].val.cooperative = 1;
        ++nattr;
    } else if (g_pdl) {
        attr[nattr].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[nattr].val.programmaticStreamSerializationAllowed = 1;
        ++nattr;
    }
    cfg.attrs = attr;
    cfg.numAttrs = nattr;
    void* args[] = {&a};
    e = cudaLaunchKernelExC(&cfg, fn, args);
    if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
    return TR_OK;
}

RowArgs blank_args(const float* x, int64_t rows, int64_t cols) {
    RowArgs a;
    std::memset(&a, 0, sizeof a);
    a.x = x;
    a.rows = rows;
    a.cols = static_cast<int>(cols);
    a.inv_cols = 1.0f / static_cast<float>(cols);
    a.cols_f = static_cast<float>(cols);
    a.S = 1;
    a.C = 1;
    return a;
}

}  // namespace

void set_last_error(const char* what, const char* detail) { t_last_error = std::string(what) + ": " + detail; }

cudaError_t device_error_symbol(void** out) { return cudaGetSymbolAddress(out, g_device_error); }

int debug_flags_now() {
    std::lock_guard<std::mutex> lock(g_mu);
    return g_debug_flags;
}

}  // namespace tr

using namespace tr;

extern "C" {

tr_status tr_softmax_f32(const float* x, float* y, int64_t rows, int64_t cols, tr_order order,
                         cudaStream_t stream) {
    tr_status s = validate_common(rows, cols, order);
    if (s != TR_OK) return s;
    if (rows == 0) return TR_OK;
    if (!x || !y) return fail(TR_ERR_INVALID_ARG, "x and y must not be null");
    if (misaligned(x, 4) || misaligned(y, 4)) return fail(TR_ERR_INVALID_ARG, "x and y must be 4-byte aligned");
    const size_t n = static_cast<size_t>(rows) * static_cast<size_t>(cols) * 4;
    if (overlaps(x, n, y, n)) return fail(TR_ERR_INVALID_ARG, "x and y overlap (in-place is not supported)");
    Call c{TR_OP_SOFTMAX, blank_args(x, rows, cols), order};
    c.a.y = y;
    c.a.y_vec = ((reinterpret_cast<uintptr_t>(x) - reinterpret_cast<uintptr_t>(y)) & 15u) == 0;
    return run(c, stream);
}

tr_status tr_rmsnorm_f32(const float* x, const float* w, float* y, int64_t rows, int64_t cols, float eps,
                         tr_order order, cudaStream_t stream) {
    tr_status s = validate_common(rows, cols, order);
    if (s != TR_OK) return s;
    s = validate_eps(eps);
    if (s != TR_OK) return s;
    if (rows == 0) return TR_OK;
    if (!x || !y) return fail(TR_ERR_INVALID_ARG, "x and y must not be null");
    if (misaligned(x, 4) || misaligned(y, 4) || misaligned(w, 4))
        return fail(TR_ERR_INVALID_ARG, "x, y and w must be 4-byte aligned");
    const size_t n = static_cast<size_t>(rows) * static_cast<size_t>(cols) * 4;
    if (overlaps(x, n, y, n) || overlaps(w, cols * 4, y, n))
        return fail(TR_ERR_INVALID_ARG, "the output overlaps an input");
    Call c{TR_OP_RMSNORM, blank_args(x, rows, cols), order};
    c.a.y = y;
    c.a.w = w;
    c.a.has_w = w != nullptr;
    c.a.eps = eps;
    c.a.y_vec = ((reinterpret_cast<uintptr_t>(x) - reinterpret_cast<uintptr_t>(y)) & 15u) == 0;
    return run(c, stream);
}

tr_status tr_layernorm_f32(const float* x, const float* gamma, const float* beta, float* y, int64_t rows,
                           int64_t cols, float eps, tr_order order, cudaStream_t stream) {
    tr_status s = validate_common(rows, cols, order);
    if (s != TR_OK) return s;
    s = validate_eps(eps);
    if (s != TR_OK) return s;
    if (rows == 0) return TR_OK;
    if (!x || !y) return fail(TR_ERR_INVALID_ARG, "x and y must not be null");
    if (misaligned(x, 4) || misaligned(y, 4) || misaligned(gamma, 4) || misaligned(beta, 4))
        return fail(TR_ERR_INVALID_ARG, "x, y, gamma and beta must be 4-byte aligned");
    const size_t n = static_cast<size_t>(rows) * static_cast<size_t>(cols) * 4;
    if (overlaps(x, n, y, n) || overlaps(gamma, cols * 4, y, n) || overlaps(beta, cols * 4, y, n))
        return fail(TR_ERR_INVALID_ARG, "the output overlaps an input");
    Call c{TR_OP_LAYERNORM, blank_args(x, rows, cols), order};
    c.a.y = y;
    c.a.w = gamma;
    c.a.b = beta;
    c.a.has_w = gamma != nullptr;
    c.a.has_b = beta != nullptr;
    c.a.eps = eps;
    c.a.y_vec = ((reinterpret_cast<uintptr_t>(x) - reinterpret_cast<uintptr_t>(y)) & 15u) == 0;
    return run(c, stream);
}

tr_status tr_cross_entropy_f32(const float* logits, const int64_t* labels, float* losses, int64_t rows,
                               int64_t cols, tr_order order, cudaStream_t stream) {
    tr_status s = validate_common(rows, cols, order);
    if (s != TR_OK) return s;
    if (rows == 0) return TR_OK;
    if (!logits || !labels || !losses) return fail(TR_ERR_INVALID_ARG, "logits, labels and losses must not be null");
    if (misaligned(logits, 4) || misaligned(losses, 4) || misaligned(labels, 8))
        return fail(TR_ERR_INVALID_ARG, "logits/losses must be 4-byte and labels 8-byte aligned");
    const size_t n = static_cast<size_t>(rows) * static_cast<size_t>(cols) * 4;
    if (overlaps(logits, n, losses, rows * 4) || overlaps(labels, rows * 8, losses, rows * 4))
        return fail(TR_ERR_INVALID_ARG, "losses overlap an input");
    Call c{TR_OP_CROSS_ENTROPY, blank_args(logits, rows, cols), order};
    c.a.labels = labels;
    c.a.loss = losses;
    return run(c, stream);
}

// Fused residual norms: validation common to both, then the norm's own fields.
static tr_status residual_call(int op, const float* x, const float* residual, const float* w, const float* b,
                               float* y, float* h, int64_t rows, int64_t cols, float eps, tr_order order,
                               cudaStream_t stream) {
    tr_status s = validate_common(rows, cols, order);
    if (s != TR_OK) return s;
    s = validate_eps(eps);
    if (s != TR_OK) return s;
    if (rows == 0) return TR_OK;
    if (!x || !residual || !y) return fail(TR_ERR_INVALID_ARG, "x, residual and y must not be null");
    if (misaligned(x, 4) || misaligned(residual, 4) || misaligned(y, 4) || misaligned(h, 4) || misaligned(w, 4) ||
        misaligned(b, 4))
        return fail(TR_ERR_INVALID_ARG, "x, residual, y, h, w and b must be 4-byte aligned");
    const size_t n = static_cast<size_t>(rows) * static_cast<size_t>(cols) * 4;
    const size_t nv = static_cast<size_t>(cols) * 4;
    const bool bad = overlaps(x, n, y, n) || overlaps(residual, n, y, n) || overlaps(w, nv, y, n) ||
                     overlaps(b, nv, y, n) || overlaps(h, n, x, n) || overlaps(h, n, residual, n) ||
                     overlaps(h, n, y, n) || overlaps(h, n, w, nv) || overlaps(h, n, b, nv);
    if (bad) return fail(TR_ERR_INVALID_ARG, "an output overlaps an input or the other output");
    Call c{op, blank_args(x, rows, cols), order};
    c.a.y = y;
    c.a.w = w;
    c.a.b = b;
    c.a.has_w = w != nullptr;
    c.a.has_b = b != nullptr;
    c.a.eps = eps;
    c.a.r = residual;
    c.a.h = h;
    c.a.y_vec = ((reinterpret_cast<uintptr_t>(x) - reinterpret_cast<uintptr_t>(y)) & 15u) == 0;
    c.a.r_vec = ((reinterpret_cast<uintptr_t>(x) - reinterpret_cast<uintptr_t>(residual)) & 15u) == 0;
    c.a.h_vec = h && ((reinterpret_cast<uintptr_t>(x) - reinterpret_cast<uintptr_t>(h)) & 15u) == 0;
    return run(c, stream);
}

// Standalone row reductions: out[r] (and out2[r]) per row.
static tr_status reduce_call(int op, const float* x, float* out, float* out2, int64_t rows, int64_t cols,
                             tr_order order, cudaStream_t stream) {
    tr_status s = validate_common(rows, cols, order, kMaxReductionCols);
    if (s != TR_OK) return s;
    if (rows == 0) return TR_OK;
    if (!x || !out || (op == TR_OP_ROW_MINMAX && !out2))
        return fail(TR_ERR_INVALID_ARG, "x and the outputs must not be null");
    if (misaligned(x, 4) || misaligned(out, 4) || misaligned(out2, 4))
        return fail(TR_ERR_INVALID_ARG, "x and the outputs must be 4-byte aligned");
    const size_t n = static_cast<size_t>(rows) * static_cast<size_t>(cols) * 4;
    const size_t no = static_cast<size_t>(rows) * 4;
    if (overlaps(x, n, out, no) || overlaps(x, n, out2, no) || overlaps(out, no, out2, no))
        return fail(TR_ERR_INVALID_ARG, "an output overlaps the input or the other output");
    Call c{op, blank_args(x, rows, cols), order};
    c.a.loss = out;
    c.a.out2 = out2;
    return run(c, stream);
}

tr_status tr_row_sum_f32(const float* x, float* out, int64_t rows, int64_t cols, tr_order order,
                         cudaStream_t stream) {
    return reduce_call(TR_OP_ROW_SUM, x, out, nullptr, rows, cols, order, stream);
}

tr_status tr_row_max_f32(const float* x, float* out, int64_t rows, int64_t cols, tr_order order,
                         cudaStream_t stream) {
    return reduce_call(TR_OP_ROW_MAX, x, out, nullptr, rows, cols, order, stream);
}

tr_status tr_row_min_f32(const float* x, float* out, int64_t rows, int64_t cols, tr_order order,
                         cudaStream_t stream) {
    return reduce_call(TR_OP_ROW_MIN, x, out, nullptr, rows, cols, order, stream);
}

tr_status tr_row_minmax_f32(const float* x, float* out_min, float* out_max, int64_t rows, int64_t cols,
                            tr_order order, cudaStream_t stream) {
    return reduce_call(TR_OP_ROW_MINMAX, x, out_min, out_max, rows, cols, order, stream);
}

// Splits of the reduced axis: the most (a power of two, at most 32) that keep
// the launch within one wave of the CTAs per SM its kernel is built for, with
// at least 32 rows per split, within the workspace's partial and ticket
// capacity.
int axis_splits(int64_t tiles, int64_t extent, int values, int tile_cols, int ctas_per_sm, int sm_count) {
    const int64_t wave = static_cast<int64_t>(ctas_per_sm) * sm_count;
    int S = 1;
    while (S < kAxisMaxSplits && tiles * 2 * S <= wave && extent >= 64 * static_cast<int64_t>(S)) S *= 2;
    while (S > 1 && (tiles > kAxisMaxTickets || tiles * S * tile_cols * values > kAxisMaxPartFloats)) S /= 2;
    return S;
}

// Columns per thread: four when every column quad is one aligned float4 of a
// row, except for the ordered sum, whose tree keeps one column per thread.
int axis_vec(int op, int order, int64_t inner, bool x_aligned16) {
    if (op == TR_OP_ROW_SUM && order == TR_ORDER_ORDERED_TREE) return 1;
    return (inner % 4 == 0 && x_aligned16) ? 4 : 1;
}

int axis_ctas_per_sm(int op, int order) {
    return (op == TR_OP_ROW_SUM && order == TR_ORDER_ORDERED_TREE) ? kAxisCtasTree : kAxisCtasFree;
}

static tr_status axis_run(int op, const float* x, float* out, float* out2, int64_t extent, int64_t inner,
                          int64_t ncols, tr_order order, cudaStream_t stream);

// Splits of the staged ordered column sum (a reduced axis of at most 1024 rows,
// each CTA staging at most 256 of them), or 0 where it does not apply.
int axis_staged_splits(int64_t rows, int64_t tiles, int arrays, int sm_count) {
    if (rows > kAxisStagedMaxRows) return 0;
    const int64_t per = kAxisStagedRowsPerCta / arrays;  // rows per CTA: 32 KB of shared memory
    int S = rows <= per ? 1 : static_cast<int>(kAxisStagedMaxRows / per);
    if (S > 1 && S < 8 && tiles * 2 * S <= 6LL * sm_count) S *= 2;  // few tiles: more CTAs per tile
    if (S > 1 && (tiles > kAxisMaxTickets || tiles * S * kAxisCols > kAxisMaxPartFloats)) return 0;
    return S;
}

// Arrays the staged tree copies per row: x and dy for the two-input terms.
static int staged_arrays(int term) {
    return term == AXIS_RMS_W || term == AXIS_LN_GAMMA || term == AXIS_LN_BOTH ? 2 : 1;
}

// Launch an axis sum / max / min (term AXIS_PLAIN) or the column sum of a
// backward term over `tiles` column tiles: the staged tree for ordered sums of
// at most 1024 rows, otherwise the splits that fill one wave.
static tr_status axis_dispatch(int op, int term, AxisArgs a, tr_order order, int vec, int64_t tiles,
                               cudaStream_t stream) {
    const bool ordered = order == TR_ORDER_ORDERED_TREE;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    int S = 1, staged = 0;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        DeviceState* st = nullptr;
        tr_status s = device_state(dev, &st);
        if (s != TR_OK) return s;
        const int sm = st->desc.sm_count;
        staged = (ordered && op == TR_OP_ROW_SUM) ? axis_staged_splits(a.extent, tiles, staged_arrays(term), sm) : 0;
        if (staged > 0) {
            S = staged;
        } else if (term == AXIS_LN_BOTH && ordered) {
            S = 0;  // the ordered pair runs as two single-term sums (below, outside the lock)
        } else {
            // ordered max and min keep two keys per column; the LayerNorm pair two sums
            const int values = (op == TR_OP_ROW_SUM && term != AXIS_LN_BOTH) ? 1 : 2;
            const int ctas = term == AXIS_PLAIN ? axis_ctas_per_sm(op, order) : (ordered ? kAxisCtasTree : kAxisCtasFree);
            S = axis_splits(tiles, a.extent, values, kAxisCols * vec, ctas, sm);
        }
        if (S > 1) {
            void* ws = nullptr;
            s = split_workspace(*st, stream, &ws);
            if (s != TR_OK) return s;
            a.part = reinterpret_cast<float*>(static_cast<char*>(ws) + kAxisPartOffset);
            a.ticket = reinterpret_cast<unsigned*>(static_cast<char*>(ws) + kAxisTicketOffset);
        }
    }
    if (S == 0) {
        AxisArgs g = a, b = a;
        g.out2 = nullptr;
        b.out = a.out2;
        b.out2 = nullptr;
        tr_status s = axis_dispatch(op, AXIS_LN_GAMMA, g, order, vec, tiles, stream);
        return s != TR_OK ? s : axis_dispatch(op, AXIS_LN_BETA, b, order, vec, tiles, stream);
    }
    if (staged > 0) {
        const int64_t rows_per = a.extent < kAxisStagedMaxRows / S ? a.extent : kAxisStagedMaxRows / S;
        e = launch_axis_staged(term, a, tiles, S,
                               static_cast<size_t>(rows_per) * kAxisCols * sizeof(float) * staged_arrays(term), stream);
    } else if (term == AXIS_PLAIN) {
        e = launch_axis(op, ordered, a, vec, tiles, S, stream);
    } else {
        e = launch_axis_term(term, ordered, a, vec, tiles, S, stream);
    }
    if (e != cudaSuccess) return cuda_fail(e, "axis reduction launch");
    return TR_OK;
}

static tr_status axis_call(int op, const float* x, float* out, float* out2, int64_t outer, int64_t extent,
                           int64_t inner, tr_order order, cudaStream_t stream) {
    if (fold_order(order)) return fail(TR_ERR_UNSUPPORTED, "the axis reductions take the tree policies");
    if (order != TR_ORDER_UNORDERED_TREE && order != TR_ORDER_ORDERED_TREE)
        return fail(TR_ERR_INVALID_ARG, "order must be one of the tr_order values");
    if (outer < 0 || extent < 1 || inner < 1)
        return fail(TR_ERR_INVALID_ARG, "need outer >= 0, extent >= 1 and inner >= 1");
    if (outer == 0) return TR_OK;
    if (extent > INT64_MAX / 4 / inner || outer > INT64_MAX / 4 / inner / extent)
        return fail(TR_ERR_INVALID_ARG, "outer * extent * inner too large");
    const int64_t ncols = outer * inner;
    const int vec = axis_vec(op, order, inner, !misaligned(x, 16));
    const int64_t tiles = (ncols + kAxisCols * vec - 1) / (kAxisCols * vec);
    if (tiles > 0x7fffffffLL) return fail(TR_ERR_UNSUPPORTED, "more output columns than one launch covers");
    if (!x || !out || (op == TR_OP_ROW_MINMAX && !out2))
        return fail(TR_ERR_INVALID_ARG, "x and the outputs must not be null");
    if (misaligned(x, 4) || misaligned(out, 4) || misaligned(out2, 4))
        return fail(TR_ERR_INVALID_ARG, "x and the outputs must be 4-byte aligned");
    const size_t n = static_cast<size_t>(outer) * static_cast<size_t>(extent) * static_cast<size_t>(inner) * 4;
    const size_t no = static_cast<size_t>(ncols) * 4;
    if (overlaps(x, n, out, no) || overlaps(x, n, out2, no) || overlaps(out, no, out2, no))
        return fail(TR_ERR_INVALID_ARG, "an output overlaps the input or the other output");
    return axis_run(op, x, out, out2, extent, inner, ncols, order, stream);
}

// The axis reduction of validated arguments (also the second step of the
// column gradients of the norm backward passes).
static tr_status axis_run(int op, const float* x, float* out, float* out2, int64_t extent, int64_t inner,
                          int64_t ncols, tr_order order, cudaStream_t stream) {
    const int vec = axis_vec(op, order, inner, !misaligned(x, 16));
    const int64_t tiles = (ncols + kAxisCols * vec - 1) / (kAxisCols * vec);
    AxisArgs a{x, out, out2, extent, inner, ncols, nullptr, nullptr};
    return axis_dispatch(op, AXIS_PLAIN, a, order, vec, tiles, stream);
}

tr_status tr_axis_launch_shape(int32_t sm_count, int32_t op, tr_order order, int64_t outer, int64_t extent,
                               int64_t inner, int32_t* splits, int64_t* tiles) {
    if (!splits || !tiles) return fail(TR_ERR_INVALID_ARG, "splits and tiles must not be null");
    if (sm_count < 1) return fail(TR_ERR_INVALID_ARG, "sm_count must be >= 1");
    if (op < TR_OP_ROW_SUM || op > TR_OP_ROW_MINMAX) return fail(TR_ERR_INVALID_ARG, "op must be a row reduction");
    if (order != TR_ORDER_UNORDERED_TREE && order != TR_ORDER_ORDERED_TREE)
        return fail(TR_ERR_INVALID_ARG, "order must be TR_ORDER_UNORDERED_TREE or TR_ORDER_ORDERED_TREE");
    if (outer < 0 || extent < 1 || inner < 1) return fail(TR_ERR_INVALID_ARG, "need outer >= 0, extent >= 1, inner >= 1");
    if (outer > 0 && outer > INT64_MAX / inner) return fail(TR_ERR_INVALID_ARG, "outer * inner too large");
    const int vec = axis_vec(op, order, inner, true);
    *tiles = (outer * inner + kAxisCols * vec - 1) / (kAxisCols * vec);
    const int staged = (order == TR_ORDER_ORDERED_TREE && op == TR_OP_ROW_SUM && *tiles > 0)
                           ? axis_staged_splits(extent, *tiles, 1, sm_count) : 0;
    *splits = staged > 0 ? staged
            : *tiles > 0 ? axis_splits(*tiles, extent, op == TR_OP_ROW_SUM ? 1 : 2, kAxisCols * vec,
                                       axis_ctas_per_sm(op, order), sm_count)
                         : 1;
    return TR_OK;
}

tr_status tr_axis_sum_f32(const float* x, float* out, int64_t outer, int64_t extent, int64_t inner, tr_order order,
                          cudaStream_t stream) {
    return axis_call(TR_OP_ROW_SUM, x, out, nullptr, outer, extent, inner, order, stream);
}

tr_status tr_axis_max_f32(const float* x, float* out, int64_t outer, int64_t extent, int64_t inner, tr_order order,
                          cudaStream_t stream) {
    return axis_call(TR_OP_ROW_MAX, x, out, nullptr, outer, extent, inner, order, stream);
}

tr_status tr_axis_min_f32(const float* x, float* out, int64_t outer, int64_t extent, int64_t inner, tr_order order,
                          cudaStream_t stream) {
    return axis_call(TR_OP_ROW_MIN, x, out, nullptr, outer, extent, inner, order, stream);
}

tr_status tr_axis_minmax_f32(const float* x, float* out_min, float* out_max, int64_t outer, int64_t extent,
                             int64_t inner, tr_order order, cudaStream_t stream) {
    return axis_call(TR_OP_ROW_MINMAX, x, out_min, out_max, outer, extent, inner, order, stream);
}

// ---- backward passes -------------------------------------------------------

// Cached quads per thread: the fewest that hold the row, 0 beyond 8192 columns.
static int bw_slots(int64_t cols) {
    for (int k : kBwSlots)
        if (k > 0 && cols <= 1024LL * k) return k;
    return 0;
}

// CTAs of a backward launch: one per row (capped; the CTAs loop over the rest).
static int64_t bw_ctas(int64_t rows) { return rows < (1LL << 20) ? rows : (1LL << 20); }

tr_status tr_norm_backward_workspace_bytes(int64_t rows, int64_t cols, size_t* bytes) {
    if (!bytes) return fail(TR_ERR_INVALID_ARG, "bytes must not be null");
    tr_status s = validate_common(rows, cols, TR_ORDER_UNORDERED_TREE);
    if (s != TR_OK) return s;
    // two statistics per row, or the one-pass kernel's column partials: two
    // vectors of ceil(rows / 4) x cols floats
    const size_t stats = static_cast<size_t>(rows) * 2 * sizeof(float);
    const size_t quads = bwn_slots(cols) > 0 ? static_cast<size_t>((rows + 3) / 4) * static_cast<size_t>(cols) * 2 * sizeof(float) : 0;
    *bytes = std::max(stats, quads);
    return TR_OK;
}

// The column sum over the rows of a norm backward term (see AxisTerm).
static tr_status term_sum(int term, const BwArgs& b, float* out, float* out2, tr_order order, cudaStream_t stream) {
    const int64_t rows = b.rows, cols = b.cols;
    const bool ordered = order == TR_ORDER_ORDERED_TREE;
    const int vec = (!ordered && cols % 4 == 0 && !misaligned(b.x, 16) && !misaligned(b.dy, 16)) ? 4 : 1;
    const int64_t tiles = (cols + kAxisCols * vec - 1) / (kAxisCols * vec);
    AxisArgs a{b.x, out, out2, rows, cols, cols, nullptr, nullptr, b.dy, b.stat_a, b.stat_b};
    return axis_dispatch(TR_OP_ROW_SUM, term, a, order, vec, tiles, stream);
}

static tr_status bw_run(int op, BwArgs a, tr_order order, float* dw, float* db, void* ws, size_t ws_bytes,
                        cudaStream_t stream) {
    if (a.rows == 0) return TR_OK;
    // the norms' one-pass kernel: aligned rows of 1024 .. 8192 columns (and, for
    // the ordered column sums, at most 1024 rows: one row per tree leaf)
    const bool one_pass = (op == BW_RMSNORM || op == BW_LAYERNORM) && bwn_slots(a.cols) > 0 &&
                          !(order == TR_ORDER_ORDERED_TREE && a.rows > 1024) && !misaligned(a.x, 16) &&
                          !misaligned(a.dy, 16) && !misaligned(a.dx, 16) && !misaligned(a.w, 16);
    if (one_pass) {
        float* partials = nullptr;
        if (dw || db) {
            size_t need = 0;  // the contract: at least tr_norm_backward_workspace_bytes
            tr_norm_backward_workspace_bytes(a.rows, a.cols, &need);
            if (!ws || ws_bytes < need)
                return fail(TR_ERR_INVALID_ARG,
                            "the workspace is missing or smaller than tr_norm_backward_workspace_bytes");
            partials = static_cast<float*>(ws);
        }
        const cudaError_t e = launch_backward_wave(op, order == TR_ORDER_ORDERED_TREE, a, dw, db, partials, stream);
        if (e != cudaSuccess) return cuda_fail(e, "backward launch");
        return TR_OK;
    }
    if (dw || db) {
        const size_t need = static_cast<size_t>(a.rows) * 2 * sizeof(float);
        if (!ws || ws_bytes < need)
            return fail(TR_ERR_INVALID_ARG, "the workspace is missing or smaller than tr_norm_backward_workspace_bytes");
        a.stat_a = static_cast<float*>(ws);
        a.stat_b = a.stat_a + a.rows;
    }
    const bool ordered = order == TR_ORDER_ORDERED_TREE;
    // unordered cross-entropy rows too long for registers: the 1024-thread streaming kernel
    const bool xent_stream = op == BW_XENT && !ordered && bw_slots(a.cols) == 0;
    if (xent_stream) {
        int dev = 0;
        cudaError_t de = cudaGetDevice(&dev);
        if (de != cudaSuccess) return cuda_fail(de, "cudaGetDevice");
        std::lock_guard<std::mutex> lock(g_mu);
        DeviceState* st = nullptr;
        tr_status ss = device_state(dev, &st);
        if (ss != TR_OK) return ss;
        a.err = st->err;
    }
    cudaError_t e = xent_stream ? launch_xent_backward_stream(a, stream)
                                : launch_backward(op, ordered, bw_slots(a.cols), a, static_cast<int>(bw_ctas(a.rows)), stream);
    if (e != cudaSuccess) return cuda_fail(e, "backward launch");
    if (dw && db) return term_sum(AXIS_LN_BOTH, a, dw, db, order, stream);  // one pass over x and dy
    if (dw) return term_sum(op == BW_RMSNORM ? AXIS_RMS_W : AXIS_LN_GAMMA, a, dw, nullptr, order, stream);
    if (db) return term_sum(AXIS_LN_BETA, a, db, nullptr, order, stream);
    return TR_OK;
}

static BwArgs bw_blank(const float* x, float* dx, int64_t rows, int64_t cols) {
    BwArgs a;
    std::memset(&a, 0, sizeof a);
    a.x = x;
    a.dx = dx;
    a.rows = rows;
    a.cols = static_cast<int>(cols);
    return a;
}

tr_status tr_softmax_backward_f32(const float* y, const float* dy, float* dx, int64_t rows, int64_t cols,
                                  tr_order order, cudaStream_t stream) {
    tr_status s = validate_common(rows, cols, order);
    if (s != TR_OK) return s;
    if (fold_order(order)) return fail(TR_ERR_UNSUPPORTED, "the backward passes take the tree policies");
    if (rows == 0) return TR_OK;
    if (!y || !dy || !dx) return fail(TR_ERR_INVALID_ARG, "y, dy and dx must not be null");
    if (misaligned(y, 4) || misaligned(dy, 4) || misaligned(dx, 4))
        return fail(TR_ERR_INVALID_ARG, "y, dy and dx must be 4-byte aligned");
    const size_t n = static_cast<size_t>(rows) * static_cast<size_t>(cols) * 4;
    if (overlaps(dx, n, y, n) || overlaps(dx, n, dy, n)) return fail(TR_ERR_INVALID_ARG, "dx overlaps an input");
    BwArgs a = bw_blank(y, dx, rows, cols);
    a.dy = dy;
    return bw_run(BW_SOFTMAX, a, order, nullptr, nullptr, nullptr, 0, stream);
}

tr_status tr_cross_entropy_backward_f32(const float* logits, const int64_t* labels, const float* dloss,
                                        float* dlogits, int64_t rows, int64_t cols, tr_order order,
                                        cudaStream_t stream) {
    tr_status s = validate_common(rows, cols, order);
    if (s != TR_OK) return s;
    if (fold_order(order)) return fail(TR_ERR_UNSUPPORTED, "the backward passes take the tree policies");
    if (rows == 0) return TR_OK;
    if (!logits || !labels || !dlogits) return fail(TR_ERR_INVALID_ARG, "logits, labels and dlogits must not be null");
    if (misaligned(logits, 4) || misaligned(dlogits, 4) || misaligned(dloss, 4) || misaligned(labels, 8))
        return fail(TR_ERR_INVALID_ARG, "misaligned pointer");
    const size_t n = static_cast<size_t>(rows) * static_cast<size_t>(cols) * 4;
    if (overlaps(dlogits, n, logits, n) || overlaps(dlogits, n, labels, static_cast<size_t>(rows) * 8) ||
        overlaps(dlogits, n, dloss, static_cast<size_t>(rows) * 4))
        return fail(TR_ERR_INVALID_ARG, "dlogits overlaps an input");
    BwArgs a = bw_blank(logits, dlogits, rows, cols);
    a.labels = labels;
    a.dloss = dloss;
    return bw_run(BW_XENT, a, order, nullptr, nullptr, nullptr, 0, stream);
}

static tr_status norm_bw_call(int op, const float* x, const float* w, const float* dy, float* dx, float* dw,
                              float* db, int64_t rows, int64_t cols, float eps, tr_order order, void* ws,
                              size_t ws_bytes, cudaStream_t stream) {
    tr_status s = validate_common(rows, cols, order);
    if (s != TR_OK) return s;
    if (fold_order(order)) return fail(TR_ERR_UNSUPPORTED, "the backward passes take the tree policies");
    s = validate_eps(eps);
    if (s != TR_OK) return s;
    if (rows == 0) return TR_OK;
    if (!x || !dy || !dx) return fail(TR_ERR_INVALID_ARG, "x, dy and dx must not be null");
    if (misaligned(x, 4) || misaligned(dy, 4) || misaligned(dx, 4) || misaligned(w, 4) || misaligned(dw, 4) ||
        misaligned(db, 4) || misaligned(ws, 16))
        return fail(TR_ERR_INVALID_ARG, "misaligned pointer (the workspace must be 16-byte aligned)");
    const size_t n = static_cast<size_t>(rows) * static_cast<size_t>(cols) * 4;
    const size_t nc = static_cast<size_t>(cols) * 4;
    const void* ins[] = {x, dy, w};
    const size_t in_n[] = {n, n, nc};
    float* outs[] = {dx, dw, db};
    const size_t out_n[] = {n, nc, nc};
    for (int o = 0; o < 3; ++o) {
        for (int i = 0; i < 3; ++i)
            if (overlaps(outs[o], out_n[o], ins[i], in_n[i])) return fail(TR_ERR_INVALID_ARG, "an output overlaps an input");
        for (int p = o + 1; p < 3; ++p)
            if (overlaps(outs[o], out_n[o], outs[p], out_n[p])) return fail(TR_ERR_INVALID_ARG, "two outputs overlap");
        if (overlaps(outs[o], out_n[o], ws, ws_bytes)) return fail(TR_ERR_INVALID_ARG, "an output overlaps the workspace");
    }
    for (int i = 0; i < 3; ++i)
        if ((dw || db) && overlaps(ws, ws_bytes, ins[i], in_n[i]))
            return fail(TR_ERR_INVALID_ARG, "the workspace overlaps an input");
    BwArgs a = bw_blank(x, dx, rows, cols);
    a.dy = dy;
    a.w = w;
    a.eps = eps;
    return bw_run(op, a, order, dw, db, ws, ws_bytes, stream);
}

tr_status tr_rmsnorm_backward_f32(const float* x, const float* w, const float* dy, float* dx, float* dw,
                                  int64_t rows, int64_t cols, float eps, tr_order order, void* workspace,
                                  size_t workspace_bytes, cudaStream_t stream) {
    return norm_bw_call(BW_RMSNORM, x, w, dy, dx, dw, nullptr, rows, cols, eps, order, workspace, workspace_bytes,
                        stream);
}

tr_status tr_layernorm_backward_f32(const float* x, const float* gamma, const float* dy, float* dx, float* dgamma,
                                    float* dbeta, int64_t rows, int64_t cols, float eps, tr_order order,
                                    void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    return norm_bw_call(BW_LAYERNORM, x, gamma, dy, dx, dgamma, dbeta, rows, cols, eps, order, workspace,
                        workspace_bytes, stream);
}

tr_status tr_add_rmsnorm_f32(const float* x, const float* residual, const float* w, float* y, float* h,
                             int64_t rows, int64_t cols, float eps, tr_order order, cudaStream_t stream) {
    return residual_call(TR_OP_ADD_RMSNORM, x, residual, w, nullptr, y, h, rows, cols, eps, order, stream);
}

tr_status tr_add_layernorm_f32(const float* x, const float* residual, const float* gamma, const float* beta,
                               float* y, float* h, int64_t rows, int64_t cols, float eps, tr_order order,
                               cudaStream_t stream) {
    return residual_call(TR_OP_ADD_LAYERNORM, x, residual, gamma, beta, y, h, rows, cols, eps, order, stream);
}

tr_status tr_plan_describe(int32_t op, int64_t rows, int64_t cols, tr_order order, tr_plan* out) {
    if (!out) return fail(TR_ERR_INVALID_ARG, "out must not be null");
    if (op < TR_OP_SOFTMAX || op > TR_OP_ROW_MINMAX) return fail(TR_ERR_INVALID_ARG, "bad op");
    tr_status s = validate_common(rows, cols, order);
    if (s != TR_OK) return s;
    if (rows < 1) return fail(TR_ERR_INVALID_ARG, "rows must be >= 1 to describe a plan");
    if (fold_order(order)) {
        if (!fold_supported(op)) return fail(TR_ERR_UNSUPPORTED, "no fold plan for this operator");
        *out = fold_plan(op, rows, order);
        return TR_OK;
    }
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState* st = nullptr;
    s = device_state(dev, &st);
    if (s != TR_OK) return s;
    OccupancyFn occ = [st](const tr_plan& p, size_t smem) { return query_occupancy(*st, p, smem); };
    if (g_override_set[op]) {
        tr_plan p = g_override[op];
        p.op = op;
        p.order = order;
        const char* why = "";
        s = check_plan(st->desc, occ, &p, rows, cols, cols % 4 == 0, &why);
        if (s != TR_OK) return fail(TR_ERR_UNSUPPORTED, std::string("plan override rejected: ") + why);
        p.est_us = estimate_us(st->desc, p, rows, cols, cols % 4 == 0);
        *out = p;
        return TR_OK;
    }
    s = select_plan(st->desc, occ, op, rows, cols, order, cols % 4 == 0, out);
    if (s != TR_OK) return fail(s, "no legal plan for this shape on this device");
    return TR_OK;
}

tr_status tr_plan_select_for(const tr_device_desc* dev, int32_t op, int64_t rows, int64_t cols, tr_order order,
                             int32_t align16, tr_plan* out) {
    if (!dev || !out) return fail(TR_ERR_INVALID_ARG, "dev and out must not be null");
    if (op < TR_OP_SOFTMAX || op > TR_OP_ROW_MINMAX) return fail(TR_ERR_INVALID_ARG, "bad op");
    tr_status s = validate_common(rows, cols, order);
    if (s != TR_OK) return s;
    if (rows < 1) return fail(TR_ERR_INVALID_ARG, "rows must be >= 1 to select a plan");
    if (dev->sm_count < 1 || dev->max_threads_per_sm < 32 || dev->regs_per_sm < 1 || dev->hbm_gbs <= 0)
        return fail(TR_ERR_INVALID_ARG, "malformed device description");
    if (fold_order(order)) {
        if (!fold_supported(op)) return fail(TR_ERR_UNSUPPORTED, "no fold plan for this operator");
        *out = fold_plan(op, rows, order);
        return TR_OK;
    }
    s = select_plan(*dev, OccupancyFn(), op, rows, cols, order, align16 != 0, out);
    if (s != TR_OK) return fail(s, "no legal plan for this shape on this device");
    return TR_OK;
}

tr_status tr_plan_check_for(const tr_device_desc* dev, tr_plan* plan, int64_t rows, int64_t cols, int32_t align16) {
    if (!dev || !plan) return fail(TR_ERR_INVALID_ARG, "dev and plan must not be null");
    if (dev->sm_count < 1 || dev->max_threads_per_sm < 32 || dev->regs_per_sm < 1 || dev->hbm_gbs <= 0)
        return fail(TR_ERR_INVALID_ARG, "malformed device description");
    const char* why = "";
    tr_status s = check_plan(*dev, OccupancyFn(), plan, rows, cols, align16 != 0, &why);
    if (s != TR_OK) return fail(s, why);
    plan->est_us = estimate_us(*dev, *plan, rows, cols, align16 != 0);
    return TR_OK;
}

tr_status tr_plan_cost_constants(double* out, int32_t n) {
    if (!out || n != kCostConstantCount) return fail(TR_ERR_INVALID_ARG, "out must hold TR_COST_CONSTANTS doubles");
    static_assert(sizeof(CostConstants) == kCostConstantCount * sizeof(double), "constants are doubles");
    std::memcpy(out, &kCostDefaults, sizeof(CostConstants));
    return TR_OK;
}

tr_status tr_plan_estimate_with(const tr_device_desc* dev, const tr_plan* plan, int64_t rows, int64_t cols,
                                int32_t align16, const double* constants, double* out_us) {
    if (!dev || !plan || !out_us) return fail(TR_ERR_INVALID_ARG, "dev, plan and out_us must not be null");
    if (rows < 1 || cols < 1) return fail(TR_ERR_INVALID_ARG, "rows and cols must be >= 1");
    if (dev->sm_count < 1 || dev->hbm_gbs <= 0) return fail(TR_ERR_INVALID_ARG, "malformed device description");
    if (plan->grid_ctas < 1 || (plan->ctas_per_sm < 1 && plan->resident_ctas < 1) || plan->block_threads < 1)
        return fail(TR_ERR_INVALID_ARG, "plan needs grid_ctas, resident_ctas (or ctas_per_sm) and block_threads");
    CostConstants c = kCostDefaults;
    if (constants) std::memcpy(&c, constants, sizeof c);
    *out_us = estimate_us(*dev, *plan, rows, cols, align16 != 0 && cols % 4 == 0, c);
    return TR_OK;
}

tr_status tr_plan_candidates(int32_t op, int64_t rows, int64_t cols, tr_order order, int32_t align16, tr_plan* out,
                             int32_t cap, int32_t* count) {
    if (!count || (cap > 0 && !out)) return fail(TR_ERR_INVALID_ARG, "count (and out when cap > 0) must not be null");
    if (op < TR_OP_SOFTMAX || op > TR_OP_ROW_MINMAX) return fail(TR_ERR_INVALID_ARG, "bad op");
    tr_status s = validate_common(rows, cols, order);
    if (s != TR_OK) return s;
    if (rows < 1) return fail(TR_ERR_INVALID_ARG, "rows must be >= 1");
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState* st = nullptr;
    s = device_state(dev, &st);
    if (s != TR_OK) return s;
    OccupancyFn occ = [st](const tr_plan& p, size_t smem) { return query_occupancy(*st, p, smem); };
    std::vector<tr_plan> legal;
    enumerate_plans(st->desc, occ, op, rows, cols, order, align16 != 0, &legal);
    *count = static_cast<int32_t>(legal.size());
    for (int32_t i = 0; i < cap && i < *count; ++i) out[i] = legal[i];
    return TR_OK;
}

tr_status tr_plan_override(const tr_plan* plan) {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!plan) {
        for (bool& b : g_override_set) b = false;
        return TR_OK;
    }
    if (plan->op < TR_OP_SOFTMAX || plan->op > TR_OP_ROW_MINMAX) return fail(TR_ERR_INVALID_ARG, "bad op");
    if ((plan->kind < TR_PLAN_ROWS || plan->kind > TR_PLAN_SPLIT) && plan->kind != TR_PLAN_WAVE &&
        plan->kind != TR_PLAN_SEGMENTS)
        return fail(TR_ERR_INVALID_ARG, "bad plan kind");
    g_override[plan->op] = *plan;
    g_override_set[plan->op] = true;
    return TR_OK;
}

tr_status tr_debug_force_wait_timeout(int32_t mode) {
    if (mode & ~kDebugModes) return fail(TR_ERR_INVALID_ARG, "mode is a mask of 1, 2 and 4");
    std::lock_guard<std::mutex> lock(g_mu);
    g_debug_flags = mode;
    return TR_OK;
}

tr_status tr_last_device_error(void) {
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
    unsigned int word = 0;
    e = cudaMemcpyFromSymbol(&word, g_device_error, sizeof word);
    if (e != cudaSuccess) return cuda_fail(e, "reading the device error word");
    if (word != 0) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(g_device_error, &zero, sizeof zero);
        if (e != cudaSuccess) return cuda_fail(e, "clearing the device error word");
        // Nothing else needs resetting: every CTA of a split launch arrives and
        // departs exactly once, also when a wait gave up, and the last to depart
        // zeroes its row's counters, so workspaces and the no-allocation scratch
        // are left ready for the next launch.
        if (word & kErrAccessCheck)
            return fail(TR_ERR_CUDA, "a kernel's own access check found an out-of-range or misaligned access and skipped it");
        return fail(TR_ERR_DEVICE_TIMEOUT, "a bounded device-side wait gave up");
    }
    return TR_OK;
}

const char* tr_status_string(tr_status status) {
    switch (status) {
        case TR_OK: return "TR_OK";
        case TR_ERR_INVALID_ARG: return "TR_ERR_INVALID_ARG";
        case TR_ERR_UNSUPPORTED: return "TR_ERR_UNSUPPORTED";
        case TR_ERR_CUDA: return "TR_ERR_CUDA";
        case TR_ERR_DEVICE_TIMEOUT: return "TR_ERR_DEVICE_TIMEOUT";
    }
    return "unknown tr_status";
}

const char* tr_last_error_message(void) { return t_last_error.c_str(); }

int32_t tr_version(void) { return 200; }

}  // extern "C"
