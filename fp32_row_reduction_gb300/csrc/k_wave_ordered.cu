// Wave kernels (TR_PLAN_WAVE) under the ordered policy (OT-1024). Built with every binary32
// step rounded: no FMA contraction, IEEE division and square root, no flush to zero.
#include "tr_wave_kernels.cuh"

namespace tr {

template <int OP>
static const void* wave_ordered(int slots, int rows_per_cta) {
#define TR_WAVE_CASE(K)                                                                               \
    case K:                                                                                           \
        return rows_per_cta == 1 ? reinterpret_cast<const void*>(wave::wave_kernel<OP, true, K, 1>)  \
               : rows_per_cta == 2 ? reinterpret_cast<const void*>(wave::wave_kernel<OP, true, K, 2>) \
                                   : nullptr;
    switch (slots) {
        TR_WAVE_CASE(2)
        TR_WAVE_CASE(4)
        TR_WAVE_CASE(6)
        TR_WAVE_CASE(8)
    }
#undef TR_WAVE_CASE
    return nullptr;
}

const void* kernel_wave_ordered(int op, int slots, int rows_per_cta) {
    switch (op) {
        case TR_OP_SOFTMAX: return wave_ordered<OP_SOFTMAX>(slots, rows_per_cta);
        case TR_OP_RMSNORM: return wave_ordered<OP_RMSNORM>(slots, rows_per_cta);
        case TR_OP_LAYERNORM: return wave_ordered<OP_LAYERNORM>(slots, rows_per_cta);
    }
    return nullptr;
}

}  // namespace tr
