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
//
// Compile-time variants, each chosen per kernel by measurement (the same change sped one kernel
// up and slowed another): PQ, the quarter-turn form of the radix-4 butterflies; FS, the 16-point
// DFT's second stage with its sqrt(1/2) factors folded into fused multiply-adds; TWMIN, the
// smallest Ns at which a shared-memory pass loads 4 of its 15 twiddles and forms the rest by
// products; TC, the 16-point DFTs on the tensor cores (fos_tc.cuh).  All give results within the
// same float32 rounding; they differ in instruction mix, not in what is computed.
#pragma once

#include "fos_device.cuh"
#include "fos_tc.cuh"

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

// Where the twiddles of each pass of the Tensor-Memory variant below live: passes with
// Ns <= SMAX read a small shared-memory table (entry r-1 of pass p at
// smem_off(p) + (r-1) Ns + m, m = j mod Ns), the others 32 Tensor-Memory columns of the thread's
// lane starting at tmem_col(p) (entry r-1 at columns 2(r-1), 2(r-1)+1).  Columns 0..31 hold the
// thread's 16 bins of H; TMEM_COLS is the first column after the twiddles.
template <int LOGN, int SMAX>
struct TwLayout {
    using S = FftShape<LOGN>;
    __host__ __device__ static constexpr bool in_smem(int p) { return S::ns(p) <= SMAX; }
    __host__ __device__ static constexpr int smem_off(int p) {
        int o = 0;
        for (int q = 1; q < p; ++q)
            if (in_smem(q)) o += 15 * S::ns(q);
        return o;
    }
    __host__ __device__ static constexpr int tmem_col(int p) {
        int c = 32;
        for (int q = 1; q < p; ++q)
            if (!in_smem(q)) c += 32;
        return c;
    }
    static constexpr int SMEM_ENTRIES = smem_off(S::NPASS);
    static constexpr int TMEM_COLS = tmem_col(S::NPASS);
};

// ---------------------------------------------------------------------------------------
// The transform, with per-thread twiddles in Tensor Memory (or, for passes with Ns <= SMAX, in
// the shared table `stw`), laid out as TwLayout<LOGN, SMAX> describes.  The passes alternate between two
// exchange buffers, so each pass needs one barrier: pass p of the forward transform
// (INV = false) writes buffer (p mod 2) and reads buffer ((p-1) mod 2); the inverse transform
// is shifted by NPASS + 1 so that its first write never lands in the buffer the forward
// transform's last pass reads.  Every buffer is xpad_len(N) elements of this transform.

template <int LOGN, int SMAX, int P, bool INV, bool PQ, bool TC, bool FS, int TWMIN, class Bar>
__device__ __forceinline__ void fft_tm_pass(float2 (&v)[16], float2 *b0, float2 *b1, const float2 *stw,
                                            uint32_t tm, int j, const Bar &bar, const TcCtx *tc,
                                            uint32_t *tcpar) {
    using S = FftShape<LOGN>;
    if constexpr (P < S::NPASS) {
        constexpr int T = S::T;
        constexpr int Ns = S::ns(P);
        constexpr bool last = (P == S::NPASS - 1);
        constexpr int DIR = INV ? 1 : -1;
        constexpr int SH = INV ? S::NPASS + 1 : 0;
        float2 *rd = ((P - 1 + SH) % 2 == 0) ? b0 : b1;
        float2 *wr = ((P + SH) % 2 == 0) ? b0 : b1;
        if constexpr (T % 16 == 0) {
            const float2 *src = rd + xpad(j);
#pragma unroll
            for (int e = 0; e < 16; ++e) v[e] = src[e * xpad_len(T)];
        } else {
#pragma unroll
            for (int e = 0; e < 16; ++e) v[e] = rd[xpad(j + e * T)];
        }
        const int m = j & (Ns - 1);
        using TL = TwLayout<LOGN, SMAX>;
        if constexpr (TL::in_smem(P) && Ns >= TWMIN) {
            // load W^m, W^{2m}, W^{4m}, W^{8m} and form the other eleven twiddles by products (no
            // power more than three products from the loaded ones): 11 shared-memory loads per
            // thread traded for 44 FP32 operations, in the passes with Ns >= TWMIN (chosen per
            // kernel by measurement)
            const float2 *t = stw + TL::smem_off(P) + m;
            float2 w[16];
            w[1] = t[0];
            w[2] = t[Ns];
            w[4] = t[3 * Ns];
            w[8] = t[7 * Ns];
            w[3] = cmul(w[1], w[2]);
            w[5] = cmul(w[4], w[1]);
            w[6] = cmul(w[4], w[2]);
            w[7] = cmul(w[4], w[3]);
#pragma unroll
            for (int r = 9; r < 16; ++r) w[r] = cmul(w[8], w[r - 8]);
#pragma unroll
            for (int r = 1; r < 16; ++r) v[r] = ctw<DIR>(v[r], w[r]);
        } else if constexpr (TL::in_smem(P)) {
            const float2 *t = stw + TL::smem_off(P) + m;
#pragma unroll
            for (int r = 1; r < 16; ++r) v[r] = ctw<DIR>(v[r], t[(r - 1) * Ns]);
        } else {
            float tw[16];
            tmem_ld16(tm + (uint32_t)TL::tmem_col(P), tw);
            tmem_wait_ld();
#pragma unroll
            for (int r = 1; r <= 8; ++r) v[r] = ctw<DIR>(v[r], make_float2(tw[2 * r - 2], tw[2 * r - 1]));
            tmem_ld16(tm + (uint32_t)TL::tmem_col(P) + 16u, tw);
            tmem_wait_ld();
#pragma unroll
            for (int r = 9; r < 16; ++r) v[r] = ctw<DIR>(v[r], make_float2(tw[2 * r - 18], tw[2 * r - 17]));
        }
        if constexpr (TC) tc_dft16<DIR>(v, *tc, bar, *tcpar);
        else dft<16, DIR, PQ, FS>(v);
        if constexpr (!last) {
            const int base = (j / Ns) * (16 * Ns) + m;
            if constexpr (Ns % 16 == 0) {
                float2 *dst = wr + xpad(base);
#pragma unroll
                for (int r = 0; r < 16; ++r) dst[r * xpad_len(Ns)] = v[r];
            } else {
#pragma unroll
                for (int r = 0; r < 16; ++r) wr[xpad(base + r * Ns)] = v[r];
            }
            bar.sync();
        }
        fft_tm_pass<LOGN, SMAX, P + 1, INV, PQ, TC, FS, TWMIN>(v, b0, b1, stw, tm, j, bar, tc, tcpar);
    }
}

// Transform v in place (layout z[j + e T] -> Z[j + e T]).  `bar` synchronises the threads that
// share the two buffers.  No barrier is needed before the first write: see the buffer rotation
// above and the callers' barrier placement.  PQ: the quarter-turn form of dft4 (fos_device.cuh).
// TC: every radix-16 DFT on the tensor cores (fos_tc.cuh; tc and tcpar are then the group's
// context and MMA-barrier phase, and the tile region may overlap b0 and b1).  FS: the folded
// second stage of the 16-point DFTs (fos_device.cuh).  TWMIN: shared-memory passes with Ns >= TWMIN
// form most of their twiddles by products of four loaded ones.
template <int LOGN, int SMAX, bool INV, bool PQ = false, bool TC = false, bool FS = false, int TWMIN = 256,
          class Bar>
__device__ __forceinline__ void fft_tm(float2 (&v)[16], float2 *b0, float2 *b1, const float2 *stw, uint32_t tm,
                                       int j, const Bar &bar, const TcCtx *tc = nullptr,
                                       uint32_t *tcpar = nullptr) {
    using S = FftShape<LOGN>;
    constexpr int T = S::T, R0 = S::R0, G = 16 / R0;
    constexpr int DIR = INV ? 1 : -1;
    constexpr int SH = INV ? S::NPASS + 1 : 0;
    float2 *wr = (SH % 2 == 0) ? b0 : b1;
    if constexpr (TC && R0 == 16) {
        tc_dft16<DIR>(v, *tc, bar, *tcpar);
    } else {
#pragma unroll
        for (int q = 0; q < G; ++q) {
            float2 a[R0];
#pragma unroll
            for (int r = 0; r < R0; ++r) a[r] = v[q + r * G];
            dft<R0, DIR, PQ, FS>(a);
#pragma unroll
            for (int r = 0; r < R0; ++r) v[q + r * G] = a[r];
        }
    }
    if constexpr ((T * R0) % 16 == 0) {
        float2 *dst = wr + j * R0 + ((j * R0) >> 4);
#pragma unroll
        for (int q = 0; q < G; ++q)
#pragma unroll
            for (int r = 0; r < R0; ++r) dst[q * (T * R0 + (T * R0) / 16) + r] = v[q + r * G];
    } else {
#pragma unroll
        for (int q = 0; q < G; ++q)
#pragma unroll
            for (int r = 0; r < R0; ++r) wr[xpad((j + q * T) * R0 + r)] = v[q + r * G];
    }
    bar.sync();
    fft_tm_pass<LOGN, SMAX, 1, INV, PQ, TC, FS, TWMIN>(v, b0, b1, stw, tm, j, bar, tc, tcpar);
}

}  // namespace fos
