// fos_kernels.h -- host-side view of the block kernels (internal to libfir_os.so).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace fos {

// Arguments of one block-kernel launch (passed by value).
struct BlockParams {
    const void *x;         // n input samples (float or float2)
    void *y;               // n output samples
    void *state;           // M-1 samples of S0 in, S0' out (NULL when M == 1)
    const float2 *H;       // N bins, H / N: natural order, or c-major (H[c + C d] at [c P + d])
                           // for the resident kernel
    const float2 *tw;      // Stockham pass twiddles of the per-CTA transform
    const float2 *twa;     // resident / pair kernels: W_N^r at [r] (r < 128), then W_N^{128 m}
                           // at [128 + m] (m < 32): the two factors of W_N^b, b = r + 128 m
    const float2 *btc;     // tensor-core variant: the split 16-point DFT matrices (fos_tc.cuh),
                           // forward hi, forward lo, inverse hi, inverse lo, 4 KB each
    int *err;              // device error word (set to 1 when a bounded wait ran out)
    uint64_t wait_ns;      // limit of one bounded wait for a bulk copy (0: every wait runs out)
    int64_t n;             // samples in this call (per channel)
    int64_t nunits;        // work units of all channels (block groups / blocks / block pairs)
    int64_t upc;           // work units per channel; unit u is unit u mod upc of channel u / upc
    int64_t x_stride;      // samples between channels' x, y and state (0 for one channel)
    int64_t y_stride;
    int64_t s_stride;
    int M;                 // taps
    int L;                 // block length N - M + 1
    int fuse_state;        // the kernel writes S0' itself (else a state kernel follows)
    int no_bulk;           // gather every unit with plain loads (x in page-locked host memory)
};

// The buffers of one channel of a (possibly multi-channel) call.
struct Chan {
    const void *x;
    void *y;
    void *state;
};

#ifdef __CUDACC__
// Channel of work unit u, and lu, the unit's index within that channel.  Kernels keep only this
// index alive and form the channel's pointers (chan) where they use them.  Everything else a
// kernel needs (n, M, L, ...) is the same for every channel and stays in BlockParams.
template <bool MULTI = true>
__device__ __forceinline__ int channel_of(const BlockParams &p, int64_t u, int64_t &lu) {
    if constexpr (!MULTI) {  // a single-channel instantiation: channel 0, nothing to compute
        lu = u;
        return 0;
    }
    const int64_t ch = u / p.upc;
    lu = u - ch * p.upc;
    return (int)ch;
}
template <bool REAL>
__device__ __forceinline__ Chan chan(const BlockParams &p, int ch) {
    constexpr int64_t SB = REAL ? 4 : 8;
    Chan c;
    c.x = static_cast<const char *>(p.x) + (int64_t)ch * p.x_stride * SB;
    c.y = static_cast<char *>(p.y) + (int64_t)ch * p.y_stride * SB;
    c.state = p.state ? static_cast<char *>(p.state) + (int64_t)ch * p.s_stride * SB : nullptr;
    return c;
}
#endif

struct KernelEntry {
    const void *func = nullptr;  // __global__ function
    const void *func_multi = nullptr;  // the same for calls of more than one channel, if separate
    const void *func_short = nullptr;  // the variant for calls of less than one wave, if any
    int smem_short = 0;                // its dynamic shared memory per CTA (bytes)
    const void *func_tc = nullptr;     // the variant with its 16-point DFTs on the tensor cores, if any
    const void *func_multi_tc = nullptr;  // the tensor-core variant for several channels, if separate
    int smem_tc = 0;                   // its dynamic shared memory per CTA (bytes)
    int threads = 0;             // threads per CTA
    int smem = 0;                // dynamic shared memory per CTA (bytes)
    int cluster = 1;             // CTAs per cluster (1 = no cluster)
    int units_per_cta = 1;       // blocks (complex) or block pairs (real) per work unit
    int groups = 1;              // independent thread groups per CTA, each taking work units
    int fft_logn = 0;            // log2 of the per-CTA transform size (twiddle table shape)
    int split_c = 0;             // resident kernel: C = N / 2^fft_logn (H c-major, twa as above)
    int state_from_x = 0;        // the fused state write reads x only (needs n >= M - 1)
};

// Single-CTA kernels, N = 2^logn, logn in [6, 13].
KernelEntry block_kernel_small(int logn, bool real);   // logn 6..9
KernelEntry block_kernel_large(int logn, bool real);   // logn 10..13
// One block resident in one SM's Tensor Memory, N = 2^logn, logn in [14, 15].
KernelEntry resident_kernel(int logn, bool real);
// One block in the Tensor Memory of a two-CTA cluster, N = 2^16.
KernelEntry pair_kernel(int logn, bool real);

}  // namespace fos
