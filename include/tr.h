/*
 * tr.h — FP32 row reductions with fused epilogues for one GB300 (sm_103a).
 *
 * Four operators, each a per-row reduction followed by an elementwise
 * epilogue over the same row ("TIRx Metal reduction lowering", §1 "The
 * frontend stays execution-first": row softmax and cross-entropy programs;
 * §5.1: LayerNorm mean/variance; RMSNorm is named on the "Whole-launch
 * reduction cost policy" page and read here as x / sqrt(mean(x^2) + eps) * w).
 *
 * Layout: every matrix is row-major and contiguous, element (r, c) at
 * ptr[r * cols + c]; weights and biases are vectors of `cols` floats; labels
 * are `rows` int64 values; losses are `rows` floats.
 *
 * Sizes: rows >= 0 (0 does nothing and returns TR_OK). The operators
 * (softmax, RMSNorm, LayerNorm, cross-entropy, the fused residual norms, the
 * backward passes and the no-allocation entry point) take 1 <= cols < 2^24,
 * so that (float)cols, by which the norms divide, is exact; the standalone row
 * reductions take 1 <= cols < 2^31. Other sizes: TR_ERR_INVALID_ARG.
 *
 * Pointers are DEVICE pointers owned by the caller. They must be 4-byte
 * aligned; 16-byte alignment of the row starts is not required (unaligned
 * heads and tails are peeled), but is faster. Inputs and outputs must not
 * overlap (the noalias contract of §3 "Semantic domain and fail-closed
 * admission"): in-place calls are rejected, not silently serialised.
 * The library allocates no memory per call. Calls are asynchronous on
 * `stream` (0 = the legacy default stream) and do not synchronise.
 *
 * Reduction order (§1, ReductionPolicy): TR_ORDER_UNORDERED_TREE lets the
 * library pick any tree and plan (results within a max relative error of
 * 2e-6 plus an absolute 1e-6 of the exact FP64 values); TR_ORDER_ORDERED_TREE
 * always uses the canonical fixed tree OT-1024 with IEEE round-to-nearest
 * arithmetic, IEEE division and square root and the library's own exp/log, so
 * that results are bit-identical across plans, runs and launch
 * configurations. Unsupported requests are errors, never a fallback (§1:
 * "missing support is an explicit compile error, not a tolerance change or
 * CPU fallback").
 *
 * Errors: every entry point returns a tr_status. Argument errors are detected
 * on the host before anything is launched. TR_ERR_CUDA reports a CUDA launch
 * error (the message is in tr_last_error_message()). Kernels never trap: a
 * bounded device-side wait that gives up records TR_ERR_DEVICE_TIMEOUT in a
 * device error word, which tr_last_device_error() reads and clears (a kernel
 * that checks its own accesses records a skipped access there too).
 */
#ifndef TR_H
#define TR_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum tr_status {
    TR_OK = 0,
    TR_ERR_INVALID_ARG = 1,    /* null pointer, bad size, overlap, bad eps or enum */
    TR_ERR_UNSUPPORTED = 2,    /* a legal request this build cannot realise (e.g. an illegal plan override) */
    TR_ERR_CUDA = 3,           /* a CUDA runtime error (launch, attribute, device query) */
    TR_ERR_DEVICE_TIMEOUT = 4  /* a bounded device-side wait gave up (reported by tr_last_device_error) */
} tr_status;

typedef enum tr_order {
    TR_ORDER_UNORDERED_TREE = 0,  /* default: any reassociation / permutation of the reduction */
    TR_ORDER_ORDERED_TREE = 1,    /* canonical OT-1024 fixed tree, bit-exact */
    /* §1 ReductionPolicy fold_left / fold_right: every row reduction one
     * sequential fold over the columns, in increasing order with the
     * accumulator on the left, or in decreasing order with the accumulator on
     * the right, from the identity; otherwise the ordered tree's op sequences,
     * bit-identical to the CPU emulation. For the four operators and the row
     * reductions; other entry points return TR_ERR_UNSUPPORTED. A fold is one
     * chain of dependent additions per row, so it runs far below bandwidth. */
    TR_ORDER_FOLD_LEFT = 2,
    TR_ORDER_FOLD_RIGHT = 3
} tr_order;

typedef enum tr_op {
    TR_OP_SOFTMAX = 0,
    TR_OP_RMSNORM = 1,
    TR_OP_LAYERNORM = 2,
    TR_OP_CROSS_ENTROPY = 3,
    TR_OP_ADD_RMSNORM = 4,   /* fused residual: y = RMSNorm(x + r) (tr_add_rmsnorm_f32) */
    TR_OP_ADD_LAYERNORM = 5, /* fused residual: y = LayerNorm(x + r) (tr_add_layernorm_f32) */
    TR_OP_ROW_SUM = 6,       /* standalone row reductions (tr_row_sum_f32, ...) */
    TR_OP_ROW_MAX = 7,
    TR_OP_ROW_MIN = 8,
    TR_OP_ROW_MINMAX = 9
} tr_op;

/* How a row is mapped onto the GPU (the build's counterpart of the page's
 * GroupPlan, §2 "Where the optimization lives"). */
typedef enum tr_plan_kind {
    TR_PLAN_ROWS = 0,     /* a row per lane group (4/8/16 lanes) or per S warps of a CTA; Q rows per CTA; row cached in registers */
    TR_PLAN_CLUSTER = 1,  /* a row per cluster of C CTAs; slices cached in registers; partials combined through distributed shared memory */
    TR_PLAN_STREAM = 2,   /* a row per C CTAs (C >= 1); no cache: statistics pass, then the row is re-read (from L2 when it fits) */
    TR_PLAN_XENT = 3,     /* cross-entropy: one streaming pass with an online (max, sum of exp) pair */
    TR_PLAN_ORDERED = 4,  /* OT-1024: 256 threads per row; cached (vec_slots > 0) or re-read (vec_slots == 0) */
    TR_PLAN_STAGED = 5,   /* persistent CTAs; rows_per_cta rows in flight in a shared-memory ring filled by
                             bulk asynchronous copies (TMA); each row reduced by the whole CTA from registers */
    TR_PLAN_ORDERED_STAGED = 6, /* OT-1024 on persistent 256-thread CTAs fed by the same ring (rows_per_cta slots) */
    TR_PLAN_SPLIT = 7,    /* a row per cluster_ctas co-resident CTAs (cooperative launch, 2..32); each CTA caches
                             vec_slots * block_threads 16-byte slots of its segment in shared memory (one bulk
                             asynchronous copy) and streams the rest; partials meet in a per-stream global
                             workspace allocated on first use (per stream and device) */
    TR_PLAN_FOLD = 8,     /* fold policies: a warp per row, 2 rows per 64-thread CTA */
    TR_PLAN_WAVE = 9,     /* softmax and the norms on 16-byte-aligned rows (cols % 4 == 0) of at most
                             1024 * vec_slots columns, both tree policies: a 256-thread CTA per
                             rows_per_cta rows (1 or 2), thread t caching the 16-byte slots t + 256 j
                             (j < vec_slots, 2/4/6/8) of each of its rows, which is the OT-1024 leaf
                             layout; meant for grids that are resident in one wave */
    TR_PLAN_SEGMENTS = 10 /* few long rows, unordered softmax and norms on 16-byte-aligned rows: grid_ctas
                             co-resident CTAs (cooperative launch, one per SM) of 1024 threads, CTA g owning
                             one column segment of EVERY row (rows_per_cta = rows, at most 32), vec_slots
                             16-byte slots per thread per row (1 or 2); a thread keeps its columns' weight and
                             bias in registers for all rows; the rows' partials meet once in the stream's
                             workspace (allocated on first use, as for the split plan). The selector
                             considers it for RMSNorm and LayerNorm, and for softmax with fewer rows than
                             SMs / 32 (beyond that the split plans fill the GPU) */
} tr_plan_kind;

typedef struct tr_plan {
    int32_t op;              /* tr_op */
    int32_t order;           /* tr_order */
    int32_t kind;            /* tr_plan_kind */
    int32_t lanes_per_row;   /* 4, 8, 16 (a row inside a warp) or 32 (a row spans warps_per_row warps) */
    int32_t warps_per_row;   /* S: warps of one CTA cooperating on a row (1 when lanes_per_row < 32) */
    int32_t rows_per_cta;    /* Q: independent rows packed into one CTA (staged plans: ring slots in flight) */
    int32_t cluster_ctas;    /* C: CTAs cooperating on one row (1 = no cluster) */
    int32_t vec_slots;       /* K: 16-byte row slots cached per thread (0 = not cached) */
    int32_t block_threads;   /* threads per CTA */
    int32_t ctas_per_sm;     /* resident CTAs per SM assumed by the cost model */
    int64_t grid_ctas;       /* CTAs launched for the problem this plan was selected for */
    double est_us;           /* cost-model estimate in microseconds (a prior, not a measurement) */
    int32_t candidates;      /* legal candidates the selector ranked */
    int32_t flags;           /* TR_PLAN_FLAG_* */
    int64_t resident_ctas;   /* CTAs of this plan the device holds at once (from the occupancy query) */
} tr_plan;

/* Staged norm plans: each worker keeps the weight (and bias) values of its
 * columns in registers for all the rows of its CTA. Requires 16-byte-aligned
 * rows (cols % 4 == 0, aligned x) and 16-byte-aligned weight/bias vectors. */
#define TR_PLAN_FLAG_PARAMS_IN_REGISTERS 1
/* Row plans (lanes_per_row 32) of the norms: the CTA copies the whole weight
 * (and bias) vector into shared memory with bulk asynchronous copies issued
 * when it starts, so the epilogue needs no dependent global load. Requires
 * 16-byte-aligned rows and weight/bias vectors; uses cols * 4 bytes of shared
 * memory per vector. */
#define TR_PLAN_FLAG_PARAMS_IN_SHARED 2
/* Warp-row plans (lanes_per_row 32, vec_slots 2, 4 or 6): each of the CTA's
 * rows_per_cta worker groups handles two consecutive rows in sequence, loading
 * both before reducing the first (the CTA covers 2 * rows_per_cta rows). */
#define TR_PLAN_FLAG_TWO_ROWS 4

/* A device as the plan selector sees it (for host-only planning and tests). */
typedef struct tr_device_desc {
    int32_t sm_count;              /* 152 on GB300 */
    int32_t max_threads_per_sm;    /* 2048 */
    int32_t max_ctas_per_sm;       /* 32 */
    int32_t regs_per_sm;           /* 65536 */
    int32_t smem_per_sm;           /* bytes */
    int32_t max_cluster_ctas;      /* 16 on GB300 (sizes above 8 are non-portable) */
    int64_t l2_bytes;
    double hbm_gbs;                /* DRAM bandwidth, GB/s */
} tr_device_desc;

/* ---- the four operators ------------------------------------------------ */

/* y[r, :] = softmax(x[r, :]): m = max, e = exp(x - m), y = e / sum(e).
 * x, y: rows x cols. */
tr_status tr_softmax_f32(const float* x, float* y, int64_t rows, int64_t cols,
                         tr_order order, cudaStream_t stream);

/* y[r, c] = x[r, c] / sqrt(sum_c x[r, c]^2 / cols + eps) * w[c].
 * w may be NULL (weight 1). eps must be finite and >= 0. */
tr_status tr_rmsnorm_f32(const float* x, const float* w, float* y,
                         int64_t rows, int64_t cols, float eps,
                         tr_order order, cudaStream_t stream);

/* mean = sum(x)/cols, var = sum((x - mean)^2)/cols (population),
 * y = (x - mean) / sqrt(var + eps) * gamma + beta.
 * gamma may be NULL (1), beta may be NULL (0). eps finite and >= 0. */
tr_status tr_layernorm_f32(const float* x, const float* gamma, const float* beta,
                           float* y, int64_t rows, int64_t cols, float eps,
                           tr_order order, cudaStream_t stream);

/* loss[r] = log(sum_c exp(x[r, c] - m)) + m - selected, m = max_c x[r, c],
 * selected = x[r, labels[r]] if 0 <= labels[r] < cols, else 0 (§5.2 "Guarded
 * immutable views and dynamic gather": an out-of-range label is not an error).
 * logits: rows x cols; labels: rows int64; losses: rows floats. */
tr_status tr_cross_entropy_f32(const float* logits, const int64_t* labels, float* losses,
                               int64_t rows, int64_t cols, tr_order order, cudaStream_t stream);

/* ---- fused residual norms ----------------------------------------------
 * "TIRx Metal reduction lowering" §5.1 (Shared SSA is not a physical
 * allocation decision): LayerNorm over combined = X + residual, where the
 * combined row is kept as a worker stripe so that each input element is
 * loaded once. With gamma = beta = NULL and h = NULL this is the page's
 * example exactly. h = x + residual (one rounded FP32 add per
 * element), y = RMSNorm(h) or LayerNorm(h) exactly as tr_rmsnorm_f32 /
 * tr_layernorm_f32 define them on h, and h is written to `h` unless it is NULL
 * (the updated residual stream). x, residual, y, h: rows x cols; w / gamma /
 * beta: cols or NULL. No output may overlap an input or the other output.
 * Runs on the cached row, cluster and cached ordered plans: rows longer than
 * a cluster's register stripes (unordered) or 16384 columns (ordered) return
 * TR_ERR_UNSUPPORTED. */
tr_status tr_add_rmsnorm_f32(const float* x, const float* residual, const float* w, float* y, float* h,
                             int64_t rows, int64_t cols, float eps, tr_order order, cudaStream_t stream);
tr_status tr_add_layernorm_f32(const float* x, const float* residual, const float* gamma, const float* beta,
                               float* y, float* h, int64_t rows, int64_t cols, float eps, tr_order order,
                               cudaStream_t stream);

/* ---- standalone row reductions -----------------------------------------
 * "TIRx Metal reduction lowering" §8 (its test list: row sums at widths 127,
 * 257, 1024 and 4096; minimum and maximum together at 7x1024). x: rows x cols;
 * out (out_min, out_max): rows floats. Unordered policy: a tree in worker
 * order for the sum; max and min are exact in any order and skip NaN elements
 * (NaN only when every element of the row is NaN). Ordered policy: the OT-1024 tree with IEEE
 * adds, and for max/min the canonical select (a NaN wins, +0 over -0 for the
 * max, -0 over +0 for the min), bit-identical to its CPU emulation (a sum
 * that becomes NaN has no portable NaN payload). */
tr_status tr_row_sum_f32(const float* x, float* out, int64_t rows, int64_t cols, tr_order order,
                         cudaStream_t stream);
tr_status tr_row_max_f32(const float* x, float* out, int64_t rows, int64_t cols, tr_order order,
                         cudaStream_t stream);
tr_status tr_row_min_f32(const float* x, float* out, int64_t rows, int64_t cols, tr_order order,
                         cudaStream_t stream);
tr_status tr_row_minmax_f32(const float* x, float* out_min, float* out_max, int64_t rows, int64_t cols,
                            tr_order order, cudaStream_t stream);

/* ---- backward passes --------------------------------------------------------
 * The gradients of the four row operators (the pages define the forward
 * operators only; these are the next rows of the same row-reduction family).
 * All tensors are device memory, row major; rows x cols unless stated.
 *
 *   softmax        dx = y * (dy - sum_j dy_j y_j), y = the forward output
 *   cross-entropy  dlogits = dloss_r * (softmax(logits) - onehot(label)); a
 *                  label outside [0, cols) has no one-hot term; dloss: rows
 *                  floats, or NULL for 1
 *   RMSNorm        dx = r (g - x r^2 mean(g x)), g = dy w, r = 1/sqrt(mean(x^2)+eps);
 *                  dw = sum over rows of dy x r (cols floats, or NULL)
 *   LayerNorm      dx = r (g - mean(g) - xh mean(g xh)), xh = (x - mean) r,
 *                  g = dy gamma; dgamma = sum over rows of dy xh, dbeta = sum
 *                  over rows of dy (each cols floats, or NULL)
 *
 * w / gamma may be NULL (weight 1). Outputs may overlap no input, no other
 * output and not the workspace. Under TR_ORDER_ORDERED_TREE every row sum and
 * every column sum is OT-1024 with each binary32 step rounded in the order
 * written above, bit-identical to the CPU emulation; unordered results meet a
 * rounding bound. The column gradients need a caller-owned, 16-byte-aligned
 * device workspace of at least tr_norm_backward_workspace_bytes(rows, cols)
 * bytes (none when dw, dgamma and dbeta are NULL): two statistics per row, or,
 * for rows of 1024 .. 8192 columns with cols % 4 == 0, the one-pass kernel's
 * column partials, two vectors of ceil(rows / 4) x cols floats, whichever is
 * larger. The norms take that one-pass kernel when x, dy, dx and the weight
 * are 16-byte aligned (and, ordered, rows <= 1024); otherwise the column
 * gradients are column sums over the rows of their per-element terms, which may
 * use the stream's library workspace, allocated on the first such call on the
 * stream, which therefore must not be captured. */
tr_status tr_softmax_backward_f32(const float* y, const float* dy, float* dx, int64_t rows, int64_t cols,
                                  tr_order order, cudaStream_t stream);
tr_status tr_cross_entropy_backward_f32(const float* logits, const int64_t* labels, const float* dloss,
                                        float* dlogits, int64_t rows, int64_t cols, tr_order order,
                                        cudaStream_t stream);
tr_status tr_rmsnorm_backward_f32(const float* x, const float* w, const float* dy, float* dx, float* dw,
                                  int64_t rows, int64_t cols, float eps, tr_order order, void* workspace,
                                  size_t workspace_bytes, cudaStream_t stream);
tr_status tr_layernorm_backward_f32(const float* x, const float* gamma, const float* dy, float* dx, float* dgamma,
                                    float* dbeta, int64_t rows, int64_t cols, float eps, tr_order order,
                                    void* workspace, size_t workspace_bytes, cudaStream_t stream);
/* Host only: workspace bytes of a norm backward pass of rows x cols. */
tr_status tr_norm_backward_workspace_bytes(int64_t rows, int64_t cols, size_t* bytes);

/* ---- reductions over a non-last axis --------------------------------------
 * "TIRx Metal reduction lowering", Reductions inside composed groups: the
 * reduced axis need not be the last memory dimension. x is a contiguous
 * [outer, extent, inner] array (device memory, row major); the result has
 * outer * inner floats, out[o * inner + i] = reduce over r of x[o, r, i]
 * (min and max together: minima to out_min, maxima to out_max). extent >= 1,
 * inner >= 1, outer >= 0 (0: nothing to do). Policies as for the row
 * reductions: unordered sums in any order, max / min skip NaN elements;
 * ordered applies the OT-1024 tree to each column vector x[o, :, i], giving
 * the bits tr_row_*_f32 gives for that vector. Outputs may not overlap x or
 * each other. A launch that splits the reduced axis over several CTAs uses the
 * stream's library workspace (allocated on the first such call on the stream,
 * which therefore must not be captured into a graph). */
tr_status tr_axis_sum_f32(const float* x, float* out, int64_t outer, int64_t extent, int64_t inner, tr_order order,
                          cudaStream_t stream);
tr_status tr_axis_max_f32(const float* x, float* out, int64_t outer, int64_t extent, int64_t inner, tr_order order,
                          cudaStream_t stream);
tr_status tr_axis_min_f32(const float* x, float* out, int64_t outer, int64_t extent, int64_t inner, tr_order order,
                          cudaStream_t stream);
tr_status tr_axis_minmax_f32(const float* x, float* out_min, float* out_max, int64_t outer, int64_t extent,
                             int64_t inner, tr_order order, cudaStream_t stream);
/* Host only: the launch an axis reduction of a 16-byte-aligned x gets on a
 * device with `sm_count` SMs: `tiles` CTAs of 32 output columns (128 when
 * inner is a multiple of 4, except for the ordered sum), and `splits` CTAs per
 * tile along the reduced axis (a power of two, at most 32, sized to one wave).
 * op is one of TR_OP_ROW_SUM .. TR_OP_ROW_MINMAX. */
tr_status tr_axis_launch_shape(int32_t sm_count, int32_t op, tr_order order, int64_t outer, int64_t extent,
                               int64_t inner, int32_t* splits, int64_t* tiles);

/* ---- no-allocation entry point ----------------------------------------- */

/* Softmax, RMSNorm or LayerNorm of few long rows with no device allocation on
 * any call. The pages have no counterpart: it exists for callers that cannot
 * allocate device memory at call time, such as code running inside a
 * pre-sized arena in which every byte is accounted for, or latency-critical
 * loops in which cudaMalloc (which may synchronise the device and can fail
 * under memory pressure) is not acceptable. The other entry points allocate a
 * small workspace on a stream's first split-row launch; this one always runs
 * the split-row plan (TR_PLAN_SPLIT, unordered policy) over a fixed 18 KB
 * scratch array compiled into the library.
 *
 * op: TR_OP_SOFTMAX (w and b must be NULL), TR_OP_RMSNORM (w optional, b
 * NULL) or TR_OP_LAYERNORM (w = gamma, b = beta, each optional); x, y:
 * rows x cols row-major device pointers, 4-byte aligned, y not overlapping an
 * input; eps finite and >= 0 (ignored by softmax). The library owns nothing
 * the caller passes.
 *
 * Limits: rows <= 256, and each row gets C = min(32, R / rows) CTAs, where R
 * is the number of CTAs the device holds at once (two per SM at 512 threads),
 * capped at the scratch's 1024 row segments, so rows <= R / 2 (152 rows on a
 * 152-SM device). Larger inputs return TR_ERR_UNSUPPORTED with the reason in
 * tr_last_error_message(); nothing is launched. Results are within the
 * unordered tolerance of the FP64 definitions and run-to-run deterministic.
 *
 * Set-up: the first call on each device looks up the scratch and error-word
 * addresses, sets the kernels' shared-memory limit and queries their
 * residency. Make that first call before capturing a stream into a graph.
 *
 * State and concurrency: the scratch's counters must be zero before a launch.
 * They are zero when the library loads, and every launch leaves them at zero,
 * also one in which a bounded wait gave up: every CTA of a row arrives and
 * departs exactly once, and the last to depart clears the row's counters
 * (nothing is reset on the host). There is one scratch per device, shared by
 * all streams and host threads: calls whose kernels may overlap in time race
 * on it, so order them (for example, one stream). */
tr_status tr_split_rows_noalloc_f32(int32_t op, const float* x, const float* w, const float* b, float* y,
                                    int64_t rows, int64_t cols, float eps, cudaStream_t stream);

/* ---- plans, errors, introspection -------------------------------------- */

/* The plan the next call with these arguments would use on the current
 * device (16-byte-aligned rows assumed when cols % 4 == 0). */
tr_status tr_plan_describe(int32_t op, int64_t rows, int64_t cols, tr_order order, tr_plan* out);

/* Host-only selection for a described device (no GPU needed). align16 = 1
 * when every row start and the weight/bias vectors are 16-byte aligned. */
tr_status tr_plan_select_for(const tr_device_desc* dev, int32_t op, int64_t rows, int64_t cols,
                             tr_order order, int32_t align16, tr_plan* out);

/* Host-only legality check of `plan` for a described device (occupancy from
 * the device description's register and shared-memory model). Fills
 * plan->grid_ctas, ctas_per_sm and est_us when legal. Returns TR_OK or
 * TR_ERR_UNSUPPORTED / TR_ERR_INVALID_ARG with the reason in
 * tr_last_error_message(); nothing is launched. */
tr_status tr_plan_check_for(const tr_device_desc* dev, tr_plan* plan, int64_t rows, int64_t cols,
                            int32_t align16);

/* ---- cost-model calibration and audit (host side) ----------------------
 * The model's constants, in this order: launch, latency, cta_barrier,
 * cluster_barrier, l2_over_hbm, staged_row, one_wave_alu, wave, slot_pass,
 * param_trip, clock_ghz, split_sync, pair_overlap, wave_slot_pass, wave_row_share,
 * seg_row (microseconds unless stated). They are
 * fixed in the library; these calls exist so that an offline calibration can
 * score the model on measured plan sweeps ("Whole-launch reduction cost
 * policy": measurement calibrates priors, never selects a plan). */
#define TR_COST_CONSTANTS 16

/* Copy the library's constants into out[0 .. n-1] (n must be TR_COST_CONSTANTS). */
tr_status tr_plan_cost_constants(double* out, int32_t n);

/* The model's estimate for a plan whose grid_ctas and ctas_per_sm are already
 * filled (for example, as described on a device), with the given constants
 * (NULL: the library's). No legality check; nothing is launched. */
tr_status tr_plan_estimate_with(const tr_device_desc* dev, const tr_plan* plan, int64_t rows, int64_t cols,
                                int32_t align16, const double* constants, double* out_us);

/* Every legal candidate for these arguments on the current device (occupancy
 * from the CUDA occupancy API), with its estimate: up to `cap` plans are
 * written to out, and *count receives the number of legal candidates. */
tr_status tr_plan_candidates(int32_t op, int64_t rows, int64_t cols, tr_order order, int32_t align16,
                             tr_plan* out, int32_t cap, int32_t* count);

/* Force the next calls of plan->op to use exactly this plan (kind,
 * lanes_per_row, warps_per_row, rows_per_cta, cluster_ctas, vec_slots,
 * block_threads). NULL clears. A plan that is illegal for a later call's
 * shape makes that call return TR_ERR_UNSUPPORTED: constraints are never
 * clamped or reinterpreted (§6 "Cost model and finite solver"). The override
 * is process-wide and meant for tests and offline plan audits. */
tr_status tr_plan_override(const tr_plan* plan);

/* Synchronises the current device, then reads and clears its device error
 * word: TR_OK; TR_ERR_CUDA if a kernel that checks its own accesses (the
 * unordered cross-entropy backward of rows over 8192 columns) found one out of
 * range or misaligned and skipped it; else TR_ERR_DEVICE_TIMEOUT if a bounded
 * wait gave up. */
tr_status tr_last_device_error(void);

/* Static text for a status. */
const char* tr_status_string(tr_status status);

/* Text describing the last error returned on the calling thread ("" if none). */
const char* tr_last_error_message(void);

/* Testing hook: makes bounded device-side waits give up, so that their
 * give-up paths run and tr_last_device_error() reports TR_ERR_DEVICE_TIMEOUT,
 * without a GPU fault or hang. `mode` is a bit mask (0 turns everything off):
 *   1  every launch of a plan with bounded waits (staged plans) also waits on
 *      a barrier that nothing completes, with a 1 ms limit; results stay correct;
 *   2  waits for bulk asynchronous copies give up at once: in the staged
 *      plans every ring slot (that row's outputs are undefined); a CTA still
 *      waits for its copies, with the normal limit, before it exits. The split
 *      and segments plans stream their segments through registers and have no
 *      such wait;
 *   4  every split (and segments) CTA's wait for the other CTAs of its row
 *      gives up at once: no CTA of the row writes outputs.
 * Applies to the launches made while it is set, including
 * tr_split_rows_noalloc_f32. A launch that gave up leaves every workspace and
 * the no-allocation scratch ready for the next launch. Other bits:
 * TR_ERR_INVALID_ARG. */
tr_status tr_debug_force_wait_timeout(int32_t mode);

/* Library version, major * 10000 + minor * 100 + patch. */
int32_t tr_version(void);

#ifdef __cplusplus
}
#endif

#endif /* TR_H */
