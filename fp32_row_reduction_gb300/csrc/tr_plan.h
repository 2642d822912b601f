// Plan selection (host only, no CUDA calls): legality first, then a fixed
// cost model ("TIRx Metal reduction lowering" §6 "Cost model and finite
// solver": legality is decided before profitability, candidates are few
// enough to enumerate exhaustively, exact constraints are never clamped).
#pragma once

#include <functional>
#include <stdint.h>
#include <vector>

#include "tr.h"

namespace tr {

// CTAs of a fully specified plan (using `smem` bytes of dynamic shared memory)
// that the whole device holds at once, or 0 if it cannot run. For cluster
// launches: the clusters the device can hold times the cluster size.
using OccupancyFn = std::function<int64_t(const tr_plan&, size_t smem)>;

// Host-only occupancy model from a register estimate (used without a GPU).
int model_occupancy(const tr_device_desc& d, const tr_plan& p, size_t smem);

// Fill grid_ctas and check every legality rule of `p` for this shape.
// Returns TR_OK, TR_ERR_UNSUPPORTED (illegal for the shape or not built) or
// TR_ERR_INVALID_ARG (malformed fields). `why` receives a reason.
tr_status check_plan(const tr_device_desc& d, const OccupancyFn& occ, tr_plan* p, int64_t rows, int64_t cols,
                     bool align16, const char** why);

// The cost model's constants (microseconds unless stated).
struct CostConstants {
    double launch, latency, cta_barrier, cluster_barrier, l2_over_hbm, staged_row, one_wave_alu, wave, slot_pass,
        param_trip, clock_ghz, split_sync, pair_overlap, wave_slot_pass, wave_row_share, seg_row;
};
constexpr int kCostConstantCount = 16;
extern const CostConstants kCostDefaults;

// Cost-model estimate in microseconds for a legal plan (grid_ctas and
// ctas_per_sm filled).
double estimate_us(const tr_device_desc& d, const tr_plan& p, int64_t rows, int64_t cols, bool align16,
                   const CostConstants& c = kCostDefaults);

// Every legal candidate of the family, with its estimate.
void enumerate_plans(const tr_device_desc& d, const OccupancyFn& occ, int32_t op, int64_t rows, int64_t cols,
                     int32_t order, bool align16, std::vector<tr_plan>* legal);

// Enumerate every legal candidate and return the cheapest.
tr_status select_plan(const tr_device_desc& d, const OccupancyFn& occ, int32_t op, int64_t rows, int64_t cols,
                      int32_t order, bool align16, tr_plan* out);

// Default description of a GB300 (used by tests and host-only planning).
tr_device_desc gb300_desc();

}  // namespace tr
