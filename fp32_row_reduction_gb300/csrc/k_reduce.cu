// Standalone row reductions (sum, max, min, min and max together): the
// instantiations of the streaming reduction kernel.
#include "tr_row_kernels.cuh"

namespace tr {
namespace {
template <int OP>
const void* reduce_table(int kind, int lanes, int slots, int flags) {
    if (kind != TR_PLAN_XENT || flags) return nullptr;
    switch (lanes) {
        case 4: return slots == 2 ? reinterpret_cast<const void*>(reduce_kernel<OP, 4, 2>) : nullptr;
        case 8: return slots == 2 ? reinterpret_cast<const void*>(reduce_kernel<OP, 8, 2>) : nullptr;
        case 16: return slots == 2 ? reinterpret_cast<const void*>(reduce_kernel<OP, 16, 2>) : nullptr;
        case 32:
            switch (slots) {
                case 2: return reinterpret_cast<const void*>(reduce_kernel<OP, 32, 2>);
                case 4: return reinterpret_cast<const void*>(reduce_kernel<OP, 32, 4>);
                case 8: return reinterpret_cast<const void*>(reduce_kernel<OP, 32, 8>);
            }
    }
    return nullptr;
}
}  // namespace

const void* kernel_reduce(int op, int kind, int lanes, int slots, int flags) {
    switch (op) {
        case TR_OP_ROW_SUM: return reduce_table<OP_RSUM>(kind, lanes, slots, flags);
        case TR_OP_ROW_MAX: return reduce_table<OP_RMAX>(kind, lanes, slots, flags);
        case TR_OP_ROW_MIN: return reduce_table<OP_RMIN>(kind, lanes, slots, flags);
        case TR_OP_ROW_MINMAX: return reduce_table<OP_RMINMAX>(kind, lanes, slots, flags);
    }
    return nullptr;
}
}  // namespace tr
