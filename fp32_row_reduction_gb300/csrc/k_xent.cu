// Unordered cross-entropy kernels (one streaming pass per row).
#include "tr_row_kernels.cuh"

namespace tr {
const void* kernel_xent(int kind, int lanes, int slots, int flags) {
    if (kind != TR_PLAN_XENT || flags) return nullptr;
    switch (lanes) {
        case 4: return slots == 2 ? reinterpret_cast<const void*>(xent_kernel<4, 2>) : nullptr;
        case 8: return slots == 2 ? reinterpret_cast<const void*>(xent_kernel<8, 2>) : nullptr;
        case 16: return slots == 2 ? reinterpret_cast<const void*>(xent_kernel<16, 2>) : nullptr;
        case 32:
            switch (slots) {
                case 2: return reinterpret_cast<const void*>(xent_kernel<32, 2>);
                case 4: return reinterpret_cast<const void*>(xent_kernel<32, 4>);
                case 8: return reinterpret_cast<const void*>(xent_kernel<32, 8>);
            }
    }
    return nullptr;
}
}  // namespace tr
