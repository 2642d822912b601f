// Kernel tables: the instantiations a plan can name, per operator.
#pragma once

#include "tr_split_kernels.cuh"

namespace tr {

template <int OP, int G, bool RES = false>
const void* rows_table(int slots) {
    switch (slots) {
        case 1: return reinterpret_cast<const void*>(rows_cached_kernel<OP, G, 1, false, RES>);
        case 2: return reinterpret_cast<const void*>(rows_cached_kernel<OP, G, 2, false, RES>);
        case 4: return reinterpret_cast<const void*>(rows_cached_kernel<OP, G, 4, false, RES>);
    }
    if constexpr (G == 32) {
        switch (slots) {
            case 6: return reinterpret_cast<const void*>(rows_cached_kernel<OP, 32, 6, false, RES>);
            case 8: return reinterpret_cast<const void*>(rows_cached_kernel<OP, 32, 8, false, RES>);
            case 16: return reinterpret_cast<const void*>(rows_cached_kernel<OP, 32, 16, false, RES>);
        }
    }
    return nullptr;
}

// Staged kernels holding the weights in registers (norms, aligned rows).
template <int OP>
const void* staged_pre_table(int slots) {
    if constexpr (OP == OP_SOFTMAX) {
        return nullptr;
    } else {
        switch (slots) {
            case 1: return reinterpret_cast<const void*>(staged_kernel<OP, 1, true>);
            case 2: return reinterpret_cast<const void*>(staged_kernel<OP, 2, true>);
            case 4: return reinterpret_cast<const void*>(staged_kernel<OP, 4, true>);
            case 8: return reinterpret_cast<const void*>(staged_kernel<OP, 8, true>);
        }
        return nullptr;
    }
}

// Row kernels of the norms with the weights staged in shared memory.
template <int OP>
const void* rows_sp_table(int slots) {
    if constexpr (OP == OP_SOFTMAX) {
        return nullptr;
    } else {
        switch (slots) {
            case 2: return reinterpret_cast<const void*>(rows_cached_kernel<OP, 32, 2, true>);
            case 4: return reinterpret_cast<const void*>(rows_cached_kernel<OP, 32, 4, true>);
            case 6: return reinterpret_cast<const void*>(rows_cached_kernel<OP, 32, 6, true>);
            case 8: return reinterpret_cast<const void*>(rows_cached_kernel<OP, 32, 8, true>);
        }
        return nullptr;
    }
}

// Two rows per worker group in sequence (optionally with the weights in shared memory).
template <int OP, bool SP>
const void* rows_pair_table(int slots) {
    if constexpr (SP && OP == OP_SOFTMAX) {
        return nullptr;
    } else {
        switch (slots) {
            case 2: return reinterpret_cast<const void*>(rows_pair_kernel<OP, 2, SP>);
            case 4:
                // norms with global weights fetch them early for K <= 4: two rows of
                // that spill, so only the shared-memory-weight form is built
                if constexpr (OP != OP_SOFTMAX && !SP) return nullptr;
                else return reinterpret_cast<const void*>(rows_pair_kernel<OP, 4, SP>);
            case 6: return reinterpret_cast<const void*>(rows_pair_kernel<OP, 6, SP>);
        }
        return nullptr;
    }
}

template <int OP>
const void* unordered_table(int kind, int lanes, int slots, int flags) {
    if (flags & TR_PLAN_FLAG_TWO_ROWS) {
        if (kind != TR_PLAN_ROWS || lanes != 32) return nullptr;
        if (flags == TR_PLAN_FLAG_TWO_ROWS) return rows_pair_table<OP, false>(slots);
        if (flags == (TR_PLAN_FLAG_TWO_ROWS | TR_PLAN_FLAG_PARAMS_IN_SHARED)) return rows_pair_table<OP, true>(slots);
        return nullptr;
    }
    if (flags & TR_PLAN_FLAG_PARAMS_IN_REGISTERS)
        return kind == TR_PLAN_STAGED ? staged_pre_table<OP>(slots) : nullptr;
    if (flags & TR_PLAN_FLAG_PARAMS_IN_SHARED)
        return (kind == TR_PLAN_ROWS && lanes == 32) ? rows_sp_table<OP>(slots) : nullptr;
    if (flags) return nullptr;
    switch (kind) {
        case TR_PLAN_ROWS:
            switch (lanes) {
                case 4: return rows_table<OP, 4>(slots);
                case 8: return rows_table<OP, 8>(slots);
                case 16: return rows_table<OP, 16>(slots);
                case 32: return rows_table<OP, 32>(slots);
            }
            return nullptr;
        case TR_PLAN_CLUSTER:
            switch (slots) {
                case 4: return reinterpret_cast<const void*>(cluster_cached_kernel<OP, 4>);
                case 8: return reinterpret_cast<const void*>(cluster_cached_kernel<OP, 8>);
                case 16: return reinterpret_cast<const void*>(cluster_cached_kernel<OP, 16>);
            }
            return nullptr;
        case TR_PLAN_STREAM:
            return slots == 0 ? reinterpret_cast<const void*>(stream_kernel<OP>) : nullptr;
        case TR_PLAN_SPLIT:
            return lanes == 32 ? reinterpret_cast<const void*>(split_kernel<OP>) : nullptr;
        case TR_PLAN_STAGED:
            switch (slots) {
                case 1: return reinterpret_cast<const void*>(staged_kernel<OP, 1, false>);
                case 2: return reinterpret_cast<const void*>(staged_kernel<OP, 2, false>);
                case 4: return reinterpret_cast<const void*>(staged_kernel<OP, 4, false>);
                case 8: return reinterpret_cast<const void*>(staged_kernel<OP, 8, false>);
            }
            return nullptr;
    }
    return nullptr;
}

// Fused residual norms (y = norm(x + r), h = x + r): the cached row and
// cluster plans, with the weights in shared memory for aligned warp rows.
template <int OP>
const void* residual_table(int kind, int lanes, int slots, int flags) {
    if (kind == TR_PLAN_ROWS && flags == TR_PLAN_FLAG_PARAMS_IN_SHARED) {
        if (lanes != 32) return nullptr;
        switch (slots) {
            case 2: return reinterpret_cast<const void*>(rows_cached_kernel<OP, 32, 2, true, true>);
            case 4: return reinterpret_cast<const void*>(rows_cached_kernel<OP, 32, 4, true, true>);
            case 6: return reinterpret_cast<const void*>(rows_cached_kernel<OP, 32, 6, true, true>);
            case 8: return reinterpret_cast<const void*>(rows_cached_kernel<OP, 32, 8, true, true>);
        }
        return nullptr;
    }
    if (flags) return nullptr;
    switch (kind) {
        case TR_PLAN_ROWS:
            switch (lanes) {
                case 4: return rows_table<OP, 4, true>(slots);
                case 8: return rows_table<OP, 8, true>(slots);
                case 16: return rows_table<OP, 16, true>(slots);
                case 32: return rows_table<OP, 32, true>(slots);
            }
            return nullptr;
        case TR_PLAN_CLUSTER:
            switch (slots) {
                case 4: return reinterpret_cast<const void*>(cluster_cached_kernel<OP, 4, true>);
                case 8: return reinterpret_cast<const void*>(cluster_cached_kernel<OP, 8, true>);
                case 16: return reinterpret_cast<const void*>(cluster_cached_kernel<OP, 16, true>);
            }
            return nullptr;
    }
    return nullptr;
}

}  // namespace tr
