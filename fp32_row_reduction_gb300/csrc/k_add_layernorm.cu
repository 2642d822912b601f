// Fused residual LayerNorm kernels (y = LayerNorm(x + r), optionally h = x + r): the
// instantiations of the cached row and cluster kernels with the residual added
// at load time.
#include "tr_dispatch.cuh"

namespace tr {
const void* kernel_add_layernorm(int kind, int lanes, int slots, int flags) {
    return residual_table<OP_LAYERNORM>(kind, lanes, slots, flags);
}
}  // namespace tr
