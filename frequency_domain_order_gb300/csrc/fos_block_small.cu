// fos_block_small.cu -- instantiations of the fused block kernel for N = 64 .. 512.
#include "fos_block.cuh"

namespace fos {

KernelEntry block_kernel_small(int logn, bool real) {
    switch (logn) {
        case 6: return real ? block_entry<6, true>() : block_entry<6, false>();
        case 7: return real ? block_entry<7, true>() : block_entry<7, false>();
        case 8: return real ? block_entry<8, true>() : block_entry<8, false>();
        case 9: return real ? block_entry<9, true>() : block_entry<9, false>();
        default: return KernelEntry{};
    }
}

}  // namespace fos
