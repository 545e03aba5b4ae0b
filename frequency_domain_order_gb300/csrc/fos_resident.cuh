// fos_resident.cuh -- pieces shared by the kernels that keep a whole block (or half of one)
// in one SM's Tensor Memory: the 32x32b lane layout, the gather of one input point, the L2
// prefetch of a block's input window, and the P = 4096-point filtering of phase B.
//
// Lane l of the Tensor Memory holds the values with b mod 128 = l (b = l + 128 m,
// m = 0..31) of every local sub-transform c', at complex slot q(c', m) = 32 c' + 16 (m & 1) +
// (m >> 1), columns 2q and 2q + 1.
#pragma once

#include "fos_fft.cuh"
#include "fos_kernels.h"

namespace fos {

// w[c] = g^c for c = 1 .. C-1 (C = 4, 8 or 16; w[0] is not written): the twiddles W_N^{bc} of
// one point set from g = W_N^b, by squarings and products, so that no power is more than four
// complex multiplications from g.
template <int C>
__device__ __forceinline__ void twiddle_powers(float2 g, float2 (&w)[C]) {
    static_assert(C == 4 || C == 8 || C == 16, "C-point stages of 4, 8 or 16");
    w[1] = g;
    w[2] = cmul(g, g);
    w[3] = cmul(w[2], g);
    if constexpr (C > 4) {
        w[4] = cmul(w[2], w[2]);
        w[5] = cmul(w[4], g);
        w[6] = cmul(w[4], w[2]);
        w[7] = cmul(w[4], w[3]);
    }
    if constexpr (C > 8) {
        w[8] = cmul(w[4], w[4]);
#pragma unroll
        for (int c = 9; c < 16; ++c) w[c] = cmul(w[8], w[c - 8]);
    }
}

// Complex slot pair of steps i0 and i0 + 2 of thread row s: columns of q(c, 8 s + i0) and
// q(c, 8 s + i0 + 2) = that + 1, relative to c's 64 columns.
__device__ __forceinline__ uint32_t step_col(int s, int i0) {
    return 2u * (uint32_t)(16 * (i0 & 1) + 4 * s + (i0 >> 1));
}

// xt[t] of the first block of the unit (and, for real data, of the second block at t + L) in
// channel ch: x inside [0, n), S0 in front of it, zeros after it.
template <bool REAL>
__device__ __forceinline__ float2 load_point(const BlockParams &p, const Chan &ch, int64_t t, bool interior) {
    if constexpr (REAL) {
        const float *x = static_cast<const float *>(ch.x);
        if (interior) return make_float2(x[t], x[t + p.L]);
        const float *s0 = static_cast<const float *>(ch.state);
        float v[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int64_t q = t + (h ? p.L : 0);
            v[h] = 0.f;
            if (q >= 0) {
                if (q < p.n) v[h] = x[q];
            } else if (q >= -(int64_t)(p.M - 1)) {
                v[h] = s0[p.M - 1 + q];
            }
        }
        return make_float2(v[0], v[1]);
    } else {
        const float2 *x = static_cast<const float2 *>(ch.x);
        if (interior) return x[t];
        if (t >= 0) return t < p.n ? x[t] : make_float2(0.f, 0.f);
        if (t >= -(int64_t)(p.M - 1)) return static_cast<const float2 *>(ch.state)[p.M - 1 + t];
        return make_float2(0.f, 0.f);
    }
}

// v[a] = xt[t0 + P a] for a < NA (load_point of each), with the test for a window that lies
// inside x taken once: there every point is a plain load at a constant offset from one pointer.
template <bool REAL, int NA, int P>
__device__ __forceinline__ void load_points(const BlockParams &p, const Chan &ch, int64_t t0, bool interior,
                                            float2 (&v)[NA]) {
    if (interior) {
        if constexpr (REAL) {
            const float *x = static_cast<const float *>(ch.x) + t0;
            const float *x2 = x + p.L;
#pragma unroll
            for (int a = 0; a < NA; ++a) v[a] = make_float2(x[P * a], x2[P * a]);
        } else {
            const float2 *x = static_cast<const float2 *>(ch.x) + t0;
#pragma unroll
            for (int a = 0; a < NA; ++a) v[a] = x[P * a];
        }
    } else {
#pragma unroll
        for (int a = 0; a < NA; ++a) v[a] = load_point<REAL>(p, ch, t0 + (int64_t)P * a, false);
    }
}

// Bulk L2 prefetch of part `part` of `parts` of the input window of unit u of channel ch (the
// part of the window inside x), split over 128 threads (pieces of ~2 KB: a few large prefetches
// are fetched far slower than many small ones, measured 1 / 16 / 32 / 128 pieces).
template <int N, bool REAL>
__device__ __forceinline__ void prefetch_window(const BlockParams &p, const Chan &ch, int64_t u, int tid,
                                                int part = 0, int parts = 1) {
    constexpr int SB = REAL ? 4 : 8;
    constexpr int NPF = 128;
    if (tid >= NPF) return;
    const int64_t blk = REAL ? 2 * u : u;
    const int64_t w0 = blk * p.L - (p.M - 1);
    const int64_t wlen = N + (REAL ? p.L : 0);
    int64_t lo = w0 + wlen * part / parts;
    int64_t hi = w0 + wlen * (part + 1) / parts;
    if (lo < 0) lo = 0;
    if (hi > p.n) hi = p.n;
    if (hi <= lo) return;
    // rounded inwards to 16 bytes, so the range stays inside x
    const uintptr_t xb = reinterpret_cast<uintptr_t>(ch.x);
    const uintptr_t a0 = (xb + (uintptr_t)lo * SB + 15) & ~uintptr_t(15);
    const uintptr_t a1 = (xb + (uintptr_t)hi * SB) & ~uintptr_t(15);
    if (a1 <= a0) return;
    const uintptr_t piece = ((a1 - a0) / NPF + 15) & ~uintptr_t(15);
    const uintptr_t b = a0 + (uintptr_t)tid * piece;
    if (b >= a1) return;
    const uintptr_t e = b + piece < a1 ? b + piece : a1;
    prefetch_l2_bulk(reinterpret_cast<const void *>(b), (uint32_t)(e - b));
}

// Phase B: P-point FFT, multiply by H, inverse FFT for the CL local sub-transforms
// c' = g, g + 2, ... (Tensor Memory columns 64 c'), whose bins are H[c + C d] with
// c = hoff + hstride c'.  col0 = 32 (j >> 7), passed in by the caller as a warp-uniform value.
// TC: the 16-point DFTs of the P-point transforms on the tensor cores (fos_tc.cuh).  Their
// accumulators are the sub-transform's own 64 columns, free while its values are in registers:
// tile t (the vectors of threads j = 128 t .. 128 t + 127) at columns 64 c' + 32 t of every lane,
// so thread j reads its DFT back from its own columns.  tc->a_base, b_base, row_off, mbar, err and
// leader are set by the caller (the A tiles overlap b0 and b1).
template <int CL, bool PQ = false, bool FS = false, int TWMIN = 256, bool TC = false>
__device__ __forceinline__ void phase_b(const BlockParams &p, uint32_t tlane, int g, int j, float2 *b0,
                                        float2 *b1, const float2 *stw, const GroupBarrier<256> &gbar, int hoff,
                                        int hstride, uint32_t col0, TcCtx *tc = nullptr, uint32_t *tcpar = nullptr) {
    constexpr int LOGP = 12, P = 1 << LOGP;
#pragma unroll 1
    for (int c = g; c < CL; c += 2) {
        const uint32_t ta = tlane + 64u * (uint32_t)c + col0;
        if constexpr (TC) {
            tc->d_row = ta;
            tc->d_tile = (tlane & 0xFFFFu) + 64u * (uint32_t)c;  // lane 0, the sub-transform's first column
        }
        float2 v[16];
        {
            float f0[16], f1[16];
            tmem_ld16(ta, f0);
            tmem_ld16(ta + 16u, f1);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                v[e] = make_float2(f0[2 * e], f0[2 * e + 1]);
                v[8 + e] = make_float2(f1[2 * e], f1[2 * e + 1]);
            }
        }
        fft_tm<LOGP, 256, false, PQ, TC, FS, TWMIN>(v, b0, b1, stw, 0u, j, gbar, tc, tcpar);
        const float2 *hp = p.H + (hoff + hstride * c) * P + j;
        float2 h[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) h[e] = __ldg(hp + 256 * e);
#pragma unroll
        for (int e = 0; e < 16; ++e) v[e] = cmul(v[e], h[e]);
        fft_tm<LOGP, 256, true, PQ, TC, FS, TWMIN>(v, b0, b1, stw, 0u, j, gbar, tc, tcpar);
        {
            float f0[16], f1[16];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                f0[2 * e] = v[e].x;
                f0[2 * e + 1] = v[e].y;
                f1[2 * e] = v[8 + e].x;
                f1[2 * e + 1] = v[8 + e].y;
            }
            tmem_st16(ta, f0);
            tmem_st16(ta + 16u, f1);
        }
    }
    tmem_wait_st();
}

}  // namespace fos
