// fos_block_large.cu -- instantiations of the fused block kernel for N = 1024 .. 8192.
#include "fos_block.cuh"

namespace fos {

KernelEntry block_kernel_large(int logn, bool real) {
    switch (logn) {
        case 10: return real ? block_entry<10, true>() : block_entry<10, false>();
        case 11: return real ? block_entry<11, true>() : block_entry<11, false>();
        case 12: return real ? block_entry<12, true>() : block_entry<12, false>();
        case 13: return real ? block_entry<13, true>() : block_entry<13, false>();
        default: return KernelEntry{};
    }
}

}  // namespace fos
