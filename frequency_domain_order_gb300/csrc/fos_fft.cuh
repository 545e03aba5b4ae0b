// fos_fft.cuh -- N-point complex FFT held by N/16 threads of one CTA (N = 64 .. 8192).
//
// Layout: thread j of the transform holds v[e] = z[j + e*T], T = N/16, e = 0..15, both on
// input and on output (natural order, no bit reversal).  The transform is a Stockham
// auto-sort sequence of passes: a first pass of radix R0 = 2^(log2 N mod 4) (16 when that is
// 0) done entirely in registers, then radix-16 passes.  Pass p reads z[j + e*T] from the
// exchange buffer, multiplies by W_{16 Ns}^{(j mod Ns) r}, does a 16-point DFT and writes
// element r to (j / Ns) * 16 Ns + (j mod Ns) + r Ns; the last pass writes nothing because
// those indices are exactly j + r*T, i.e. the result is already where the multiply by H
// (step 4 of the claim in "一种基于GPU的高阶数字FIR滤波器频域并行处理实现方法",
// zl.czvv.com/42398539.html) and the inverse transform want it.
//
// Twiddles for pass p (p >= 1) come from a float32 table (computed in float64 on the host)
// laid out as tw[twoff(p) + (r-1) * Ns + m] = e^{-2 pi i m r / (16 Ns)}, m = 0..Ns-1, so that
// consecutive threads read consecutive entries.  The inverse uses their conjugates.
#pragma once

#include "fos_device.cuh"

namespace fos {

__host__ __device__ constexpr int ilog2c(int v) { return v <= 1 ? 0 : 1 + ilog2c(v / 2); }

template <int LOGN>
struct FftShape {
    static constexpr int N = 1 << LOGN;
    static constexpr int T = N / 16;
    static constexpr int REM = LOGN % 4;
    static constexpr int R0 = REM == 0 ? 16 : (1 << REM);
    static constexpr int NPASS = 1 + (LOGN - ilog2c(R0)) / 4;
    __host__ __device__ static constexpr int ns(int p) { return p == 0 ? 1 : R0 << (4 * (p - 1)); }
    __host__ __device__ static constexpr int twoff(int p) {
        int o = 0;
        for (int q = 1; q < p; ++q) o += 15 * ns(q);
        return o;
    }
    static constexpr int TW_ENTRIES = twoff(NPASS);
    static_assert(LOGN >= 6 && LOGN <= 13, "one CTA holds 64 .. 8192 points");
};

template <int LOGN, int DIR, int P>
__device__ __forceinline__ void fft_pass(float2 (&v)[16], float2 *ex, const float2 *__restrict__ tw, int j) {
    using S = FftShape<LOGN>;
    if constexpr (P < S::NPASS) {
        constexpr int T = S::T;
        constexpr int Ns = S::ns(P);
        constexpr bool last = (P == S::NPASS - 1);
#pragma unroll
        for (int e = 0; e < 16; ++e) v[e] = ex[xpad(j + e * T)];
        if constexpr (!last) __syncthreads();  // every read done before the buffer is rewritten
        const int m = j & (Ns - 1);
        const float2 *twp = tw + S::twoff(P) + m;
#pragma unroll
        for (int r = 1; r < 16; ++r) v[r] = ctw<DIR>(v[r], __ldg(twp + (r - 1) * Ns));
        dft<16, DIR>(v);
        if constexpr (!last) {
            const int base = (j / Ns) * (16 * Ns) + m;
#pragma unroll
            for (int r = 0; r < 16; ++r) ex[xpad(base + r * Ns)] = v[r];
            __syncthreads();
        }
        fft_pass<LOGN, DIR, P + 1>(v, ex, tw, j);
    }
}

// Transform v in place (layout above).  `ex` is this transform's N-element exchange buffer.
// sync_first: the buffer may still be read by other threads of the CTA (a previous transform),
// so barrier before the first write.
template <int LOGN, int DIR>
__device__ __forceinline__ void fft_regs(float2 (&v)[16], float2 *ex, const float2 *__restrict__ tw, int j,
                                         bool sync_first) {
    using S = FftShape<LOGN>;
    constexpr int T = S::T, R0 = S::R0, G = 16 / R0;
    // pass 0: radix R0 on groups g = j + q T; element r of group g is z[g + r N/R0] = v[q + r G]
#pragma unroll
    for (int q = 0; q < G; ++q) {
        float2 a[R0];
#pragma unroll
        for (int r = 0; r < R0; ++r) a[r] = v[q + r * G];
        dft<R0, DIR>(a);
#pragma unroll
        for (int r = 0; r < R0; ++r) v[q + r * G] = a[r];
    }
    if (sync_first) __syncthreads();
#pragma unroll
    for (int q = 0; q < G; ++q)
#pragma unroll
        for (int r = 0; r < R0; ++r) ex[xpad((j + q * T) * R0 + r)] = v[q + r * G];
    __syncthreads();
    fft_pass<LOGN, DIR, 1>(v, ex, tw, j);
}

}  // namespace fos
