// Unordered softmax kernels: the instantiations of the row kernel family.
#include "tr_dispatch.cuh"

namespace tr {
const void* kernel_softmax(int kind, int lanes, int slots, int flags) {
    return unordered_table<OP_SOFTMAX>(kind, lanes, slots, flags);
}
}  // namespace tr
