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

int pass_twiddle_entries(int logn) {
    switch (logn) {
        case 6: return FftShape<6>::TW_ENTRIES;
        case 7: return FftShape<7>::TW_ENTRIES;
        case 8: return FftShape<8>::TW_ENTRIES;
        case 9: return FftShape<9>::TW_ENTRIES;
        case 10: return FftShape<10>::TW_ENTRIES;
        case 11: return FftShape<11>::TW_ENTRIES;
        case 12: return FftShape<12>::TW_ENTRIES;
        case 13: return FftShape<13>::TW_ENTRIES;
        default: return 0;
    }
}

}  // namespace fos
