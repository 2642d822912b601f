// Segments kernels (TR_PLAN_SEGMENTS): few long rows, every co-resident CTA
// owning one column segment of every row (unordered policy).
#include "tr_segments_kernels.cuh"

namespace tr {

template <int OP>
static const void* segments_table(int slots) {
    switch (slots) {
        case 1: return reinterpret_cast<const void*>(segments::segments_kernel<OP, 1>);
        case 2: return reinterpret_cast<const void*>(segments::segments_kernel<OP, 2>);
    }
    return nullptr;
}

const void* kernel_segments(int op, int slots) {
    switch (op) {
        case TR_OP_SOFTMAX: return segments_table<OP_SOFTMAX>(slots);
        case TR_OP_RMSNORM: return segments_table<OP_RMSNORM>(slots);
        case TR_OP_LAYERNORM: return segments_table<OP_LAYERNORM>(slots);
    }
    return nullptr;
}

}  // namespace tr
