// fos_chan.h -- host-side view of the channelizer kernel (internal to libfir_os.so).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace fos {

// Arguments of one channelizer launch (passed by value).
struct ChanParams {
    const void *x;       // n input samples (float or float2)
    float2 *y;           // nout x K outputs, y[m K + q]
    const void *state;   // Nh - 1 samples before x[0] (oldest first); NULL when Nh == 1
    const float *h;      // prototype, P K floats (zero beyond Nh)
    const float2 *tw;    // Stockham pass twiddles of the K-point transform
    int64_t nout;        // output vectors: n / D
    int64_t nunits;      // work units of F transforms
    int K, D, Nh, P;     // channels, decimation, taps, taps per branch (ceil(Nh / K))
    int pack;            // real input: 1 = two output vectors per transform, 2 = four per slot (K = 2D)
};

struct ChanEntry {
    const void *func = nullptr;
    int threads = 0;
    int groups = 1;      // groups per CTA, each taking units
    int per_unit = 1;    // transforms per unit (F), each one output vector or (packed) two
    int smem_fixed = 0;  // dynamic shared memory before the prototype
    int tw_entries = 0;  // pass-twiddle table entries
};

// K = 2^logk, logk in [6, 12].
ChanEntry chan_kernel(int logk, bool real);

}  // namespace fos
