// Internal host/device interface of the library (not installed).
#pragma once

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime.h>

#include "tr.h"

namespace tr {

// Kernel parameter block shared by every row kernel (passed by value).
struct RowArgs {
    const float* x;
    float* y;
    const float* w;         // weight / gamma (has_w == 0: weight 1)
    const float* b;         // beta (has_b == 0: bias 0)
    const int64_t* labels;  // cross-entropy
    float* loss;            // cross-entropy
    int64_t rows;
    int cols;
    float eps;
    float inv_cols;  // 1 / cols
    float cols_f;    // (float) cols
    int S;           // warps per row (lanes_per_row == 32)
    int C;           // CTAs per row (cluster / stream plans)
    int y_vec;       // y rows have the same 16-byte phase as x rows
    int has_w, has_b;
    unsigned* err;         // device error word (bounded waits record timeouts here)
    long long wait_ns;     // a bounded wait gives up after this many nanoseconds
    int nbuf;              // staged plans: row slots in the shared-memory ring
    int slot_floats;       // staged plans: floats per ring slot (multiple of 4)
    int debug_flags;       // testing: kDebugForceTimeout makes one bounded wait expire
    float4* sp_part;       // split plans: per (row, segment) partial statistic, rows * C entries
    unsigned* sp_arrive;   // split plans: per-row arrival counters (zero between launches)
    unsigned* sp_depart;   // split plans: per-row departure counters (zero between launches)
    const float* r;        // fused residual norms: the residual added to x before the norm
    float* h;              // fused residual norms: x + r written out (null: not written)
    int r_vec;             // r rows have the same 16-byte phase as x rows
    int h_vec;             // h rows have the same 16-byte phase as x rows
    float* out2;           // row min/max: the maxima (loss receives the minima)
    int pf_ctas;           // wave plans: the SM count (CTAs below it prefetch the norm parameters into L1)
    int stagger_ns;        // wave plans: a CTA of launch rank k = blockIdx / pf_ctas starts k x this late
};

// Testing modes (tr_debug_force_wait_timeout), a bit mask in RowArgs::debug_flags:
constexpr int kDebugForceTimeout = 1;  // one extra wait on a barrier nothing completes (1 ms limit)
constexpr int kDebugExpireCopies = 2;  // waits for bulk copies (staged rings) give up at once
constexpr int kDebugExpirePeers = 4;   // a split CTA's wait for the other CTAs of its row gives up at once
constexpr int kDebugModes = kDebugForceTimeout | kDebugExpireCopies | kDebugExpirePeers;
// The testing modes in force now (for launches that build their own arguments).
int debug_flags_now();
constexpr int kMaxRing = 8;                // staged plans: most rows in flight per CTA
constexpr int kStagedSmemBudget = 225 * 1024;  // dynamic shared memory per CTA (bytes; 2 KB left for static)

// Split plans: at most 32 CTAs per row (the partials are merged by one warp);
// the workspace holds kSplitMaxParts partials and kSplitMaxRows counter pairs.
constexpr int kSplitMaxCtas = 32;
constexpr int kSplitMaxParts = 4096;
constexpr int kSplitMaxRows = 2048;
// Axis reductions (a non-last axis of [outer, extent, inner]): 256 threads
// per CTA over 32 output columns (32 column quads when inner is a multiple of
// 4 and x is 16-byte aligned); a launch with splits > 1 keeps its per-CTA
// partials and per-tile tickets after the split-plan region of the workspace.
constexpr int kAxisThreads = 256;
constexpr int kAxisCols = 32;
constexpr int kAxisMaxSplits = 32;
constexpr int kAxisCtasFree = 4;  // resident CTAs per SM the free and key kernels are built for
constexpr int kAxisCtasTree = 3;  // the same for the ordered sum
constexpr int kAxisMaxTickets = 2048;
constexpr int kAxisMaxPartFloats = 1 << 20;
constexpr size_t kAxisPartOffset = kSplitMaxParts * 16 + 2 * kSplitMaxRows * sizeof(unsigned);
constexpr size_t kAxisTicketOffset = kAxisPartOffset + kAxisMaxPartFloats * sizeof(float);
constexpr size_t kSplitWorkspaceBytes = kAxisTicketOffset + kAxisMaxTickets * sizeof(unsigned);

struct AxisArgs {
    const float* x;   // [outer, extent, inner], contiguous
    float* out;       // [outer * inner]: sums, maxima, minima (min and max together: the minima)
    float* out2;      // min and max together: the maxima
    int64_t extent;   // length of the reduced axis
    int64_t inner;    // elements after the reduced axis
    int64_t ncols;    // outer * inner output columns
    float* part;      // splits > 1: per-CTA partials (tiles * splits * values * columns of a tile)
    unsigned* ticket; // splits > 1: per-tile arrival tickets (zero between launches)
    // column gradients of the norm backward passes (term != AXIS_PLAIN): the
    // reduced element of row r is a term of x, dy (same layout as x) and the
    // row's statistics sa[r], sb[r]
    const float* dy;
    const float* sa;
    const float* sb;
};

// The element an axis sum reduces: x itself, or a term of a norm backward pass.
enum AxisTerm : int {
    AXIS_PLAIN = 0,
    AXIS_RMS_W = 1,   // (dy x) r,              sa = r = 1 / rms
    AXIS_LN_GAMMA = 2,  // dy ((x - mean) r),   sa = mean, sb = r = 1 / sigma
    AXIS_LN_BETA = 3,   // dy
    AXIS_LN_BOTH = 4    // the LayerNorm's two column gradients at once: out = dgamma, out2 = dbeta
};

// Launch the ordered column sum (plain or of a term) of a reduced axis of at
// most 1024 rows with the split's rows staged in `smem` bytes of shared memory
// (splits 1, 2, 4 or 8).
cudaError_t launch_axis_staged(int term, const AxisArgs& a, int64_t tiles, int splits, size_t smem,
                               cudaStream_t stream);
constexpr int kAxisStagedMaxRows = 1024;
constexpr int kAxisStagedRowsPerCta = 256;  // rows one CTA stages (32 KB for 32 columns)

// Launch the column sum of a norm backward term (AXIS_RMS_W .. AXIS_LN_BETA).
cudaError_t launch_axis_term(int term, bool ordered, const AxisArgs& a, int vec, int64_t tiles, int splits,
                             cudaStream_t stream);

// Floats of one ring slot for rows of `cols` floats: the row's 16-byte-aligned
// body plus one partial 16-byte chunk on each side.
inline int staged_slot_floats(int64_t cols) { return static_cast<int>((cols + 3) / 4 * 4 + 8); }

// Launch the axis reduction `op` (TR_OP_ROW_SUM .. TR_OP_ROW_MINMAX) over (tiles, splits) CTAs,
// each thread on `vec` (1 or 4) adjacent columns.
cudaError_t launch_axis(int op, bool ordered, const AxisArgs& a, int vec, int64_t tiles, int splits,
                        cudaStream_t stream);

// Set the calling thread's last-error text to "what: detail" (tr_last_error_message).
void set_last_error(const char* what, const char* detail);
// Device address of the library's error word on the current device.
cudaError_t device_error_symbol(void** out);

// Kernel entry for a plan, or nullptr when this build has no such
// instantiation (the plan is then unsupported). One table per operator.
const void* kernel_softmax(int kind, int lanes, int slots, int flags);
const void* kernel_rmsnorm(int kind, int lanes, int slots, int flags);
const void* kernel_layernorm(int kind, int lanes, int slots, int flags);
const void* kernel_xent(int kind, int lanes, int slots, int flags);
const void* kernel_ordered(int op, int slots);
const void* kernel_ordered_residual(int op, int slots);
const void* kernel_add_rmsnorm(int kind, int lanes, int slots, int flags);
const void* kernel_add_layernorm(int kind, int lanes, int slots, int flags);
const void* kernel_reduce(int op, int kind, int lanes, int slots, int flags);
const void* kernel_ordered_staged(int op, int slots);
// OT-1024 for few long rows: a cluster of kOtClusterCtas CTAs per row, one per group of the tree.
const void* kernel_ordered_cluster(int op);
constexpr int kOtClusterCtas = 8;
constexpr size_t kOtClusterSmemMax = 200 * 1024;  // a group's share of the row staged in shared memory
inline size_t ot_cluster_smem(int64_t cols) { return static_cast<size_t>((cols + 1023) / 1024) * 32 * 16; }
// Wave kernels (TR_PLAN_WAVE): softmax, RMSNorm, LayerNorm; vec_slots 2, 4, 6, 8;
// rows_per_cta 1 or 2.
const void* kernel_wave_unordered(int op, int slots, int rows_per_cta);
const void* kernel_wave_ordered(int op, int slots, int rows_per_cta);
constexpr int kWaveSlots[] = {2, 4, 6, 8};
constexpr int kWaveThreads = 256;
// Segments kernels (TR_PLAN_SEGMENTS): softmax, RMSNorm, LayerNorm; vec_slots 1, 2.
const void* kernel_segments(int op, int slots);
constexpr int kSegSlots[] = {1, 2};
constexpr int kSegThreads = 1024;
constexpr int kSegMaxRows = 32;
constexpr int kSegSmem = 200 * 1024;  // dynamic shared memory of a segments CTA (one CTA per SM)
// Rows of a segments launch whose segment is cached in shared memory.
inline int seg_cached_rows(int64_t rows, int64_t cols, int64_t grid) {
    const int64_t sq = (cols / 4 + grid - 1) / grid;
    const int64_t n = sq > 0 ? kSegSmem / (sq * 16) : rows;
    return static_cast<int>(n < rows ? n : rows);
}
// Dynamic shared memory a plan's kernel needs (0 for all but staged plans).
size_t plan_dynamic_smem(const tr_plan& p, int64_t cols);

inline const void* kernel_for(const tr_plan& p) {
    if (p.op == TR_OP_ADD_RMSNORM || p.op == TR_OP_ADD_LAYERNORM) {
        if (p.kind == TR_PLAN_ORDERED) return p.flags ? nullptr : kernel_ordered_residual(p.op, p.vec_slots);
        return p.op == TR_OP_ADD_RMSNORM ? kernel_add_rmsnorm(p.kind, p.lanes_per_row, p.vec_slots, p.flags)
                                         : kernel_add_layernorm(p.kind, p.lanes_per_row, p.vec_slots, p.flags);
    }
    if (p.op >= TR_OP_ROW_SUM && p.op <= TR_OP_ROW_MINMAX) {
        if (p.kind == TR_PLAN_ORDERED) return p.flags ? nullptr : kernel_ordered(p.op, p.vec_slots);
        return kernel_reduce(p.op, p.kind, p.lanes_per_row, p.vec_slots, p.flags);
    }
    if (p.kind == TR_PLAN_SEGMENTS) return p.flags || p.order != TR_ORDER_UNORDERED_TREE ? nullptr
                                                                                         : kernel_segments(p.op, p.vec_slots);
    if (p.kind == TR_PLAN_WAVE) {
        if (p.flags) return nullptr;
        return p.order == TR_ORDER_ORDERED_TREE ? kernel_wave_ordered(p.op, p.vec_slots, p.rows_per_cta)
                                                : kernel_wave_unordered(p.op, p.vec_slots, p.rows_per_cta);
    }
    if (p.kind == TR_PLAN_ORDERED && p.cluster_ctas == kOtClusterCtas)
        return p.flags ? nullptr : kernel_ordered_cluster(p.op);
    if (p.kind == TR_PLAN_ORDERED) return p.flags ? nullptr : kernel_ordered(p.op, p.vec_slots);
    if (p.kind == TR_PLAN_ORDERED_STAGED) return p.flags ? nullptr : kernel_ordered_staged(p.op, p.vec_slots);
    switch (p.op) {
        case TR_OP_SOFTMAX: return kernel_softmax(p.kind, p.lanes_per_row, p.vec_slots, p.flags);
        case TR_OP_RMSNORM: return kernel_rmsnorm(p.kind, p.lanes_per_row, p.vec_slots, p.flags);
        case TR_OP_LAYERNORM: return kernel_layernorm(p.kind, p.lanes_per_row, p.vec_slots, p.flags);
        case TR_OP_CROSS_ENTROPY: return kernel_xent(p.kind, p.lanes_per_row, p.vec_slots, p.flags);
    }
    return nullptr;
}

// Instantiated K values (16-byte slots per worker).
constexpr int kRowsSlotsSub[] = {1, 2, 4};           // lanes_per_row 4, 8, 16
constexpr int kRowsSlotsWarp[] = {1, 2, 4, 6, 8, 16};  // lanes_per_row 32
constexpr int kRowsSlotsShared[] = {2, 4, 6, 8};       // lanes_per_row 32, weights in shared memory
constexpr int kRowsSlotsPair[] = {2, 4, 6};            // lanes_per_row 32, two rows per group
constexpr int kClusterSlots[] = {4, 8, 16};
constexpr int kStagedSlots[] = {1, 2, 4, 8};
constexpr int kOrderedSlots[] = {0, 1, 2, 4, 6, 8, 12, 16}; // 0: re-read plan
constexpr int kOrderedStagedSlots[] = {1, 2, 4, 8};
constexpr int kOrderedThreads = 256;                  // OT-1024: 256 workers x 4 leaves

// The fold policies: one warp per row, 2 rows per CTA (op: TR_OP_SOFTMAX ..
// TR_OP_CROSS_ENTROPY or TR_OP_ROW_SUM .. TR_OP_ROW_MINMAX; right: fold_right).
cudaError_t launch_fold(int op, bool right, const RowArgs& a, cudaStream_t stream);
inline bool fold_order(int order) { return order == TR_ORDER_FOLD_LEFT || order == TR_ORDER_FOLD_RIGHT; }
inline bool fold_supported(int op) {
    return (op >= TR_OP_SOFTMAX && op <= TR_OP_CROSS_ENTROPY) || (op >= TR_OP_ROW_SUM && op <= TR_OP_ROW_MINMAX);
}

// Backward passes: one CTA of 256 threads per row in the OT-1024 layout (thread
// t owns columns 1024j + 4t .. +3); CTA c takes rows c, c + G, c + 2G, ...
enum BwOp : int { BW_SOFTMAX = 0, BW_XENT = 1, BW_RMSNORM = 2, BW_LAYERNORM = 3 };
constexpr int kBwSlots[] = {0, 1, 2, 4, 6, 8};  // 0: rows longer than 8192 columns, read again per pass

struct BwArgs {
    const float* x;          // softmax: y (the forward output); cross-entropy: logits; norms: x
    const float* dy;         // softmax, norms: the upstream gradient (rows x cols)
    const float* w;          // norms: weight / gamma (null: 1)
    const int64_t* labels;   // cross-entropy
    const float* dloss;      // cross-entropy: per-row upstream gradient (null: 1)
    float* dx;               // rows x cols
    float* stat_a;           // norms: per-row statistic for the column gradients, RMSNorm 1/rms,
                             // LayerNorm the mean (null: not written)
    float* stat_b;           // LayerNorm: per-row 1/sigma (null: not written)
    int64_t rows;
    int cols;
    float eps;
    unsigned* err;           // device error word (kernels that check their own accesses record here)
    int sms;                 // one-pass norm backward: the SM count (launch rank = blockIdx / sms)
    int stagger_ns;          // one-pass norm backward: a CTA of launch rank k starts k x this late
};

// Device error word bit: a kernel's own access check skipped a bad access
// (bit 1, kErrWaitTimeout, is a bounded wait that gave up).
constexpr unsigned kErrAccessCheck = 2u;

// Launch backward op `op` (BwOp) with K cached quads per thread (0: re-read) on G CTAs.
cudaError_t launch_backward(int op, bool ordered, int slots, const BwArgs& a, int ctas, cudaStream_t stream);
// The one-pass norm backward (RMSNorm, LayerNorm) of aligned rows of 1024 .. 8192
// columns: quads per thread (2, 4, 6, 8), 0 where it does not apply.
int bwn_slots(int64_t cols);
// dx, and the column gradients asked for (dw: dw or dgamma; db: dbeta) through
// `partials`, ceil(rows / 4) x cols floats per gradient vector (both blocks for
// LayerNorm). The ordered policy needs rows <= 1024.
cudaError_t launch_backward_wave(int op, bool ordered, const BwArgs& a, float* dw, float* db, float* partials,
                                 cudaStream_t stream);
// Unordered cross-entropy backward of rows longer than the cached kernels take
// (more than 8192 columns): a 1024-thread CTA per row, the row read twice.
cudaError_t launch_xent_backward_stream(const BwArgs& a, cudaStream_t stream);

}  // namespace tr
