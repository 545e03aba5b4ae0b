// fos_chan.cu -- the polyphase DFT channelizer of "GPU加速短波信道化：多相滤波器组的并行重构与
// CUDA实现": a K-channel analysis filter bank decimated by D,
//
//   y[m][q] = sum_{l < Nh} h[l] e^{-2 pi i q l / K} xt[t_m - l],   t_m = m D + D - 1,
//
// computed as the page's three steps: the input is dealt into K branches (branch k of output
// m reads xt[t_m - k - r K], r = 0, 1, ...), each branch is filtered by its polyphase component
// h_k(r) = h[r K + k], and a K-point DFT across the branches gives the K channels:
//
//   v_k(m) = sum_r h[r K + k] xt[t_m - r K - k],   y[m][q] = sum_k v_k(m) e^{-2 pi i q k / K}.
//
// Real input, long calls (p.pack): two consecutive output vectors m, m+1 share one complex
// transform, their branch sums as the real and imaginary parts (each h[r K + k] read once for
// both); the two spectra are separated after the transform through Z[K - q]
// (Y_m[q] = (Z[q] + conj Z[K-q]) / 2, Y_{m+1}[q] = (Z[q] - conj Z[K-q]) / 2i), read back from
// shared memory.  With K = 2D (the page's 50%-overlapping channels) a thread computes four
// consecutive vectors, two transforms, whose taps share half their samples (quad_taps).  Short
// calls, which are latency-bound, keep one vector per transform: more transforms in flight,
// fewer serial loads per thread.
//
// Thread j of a transform computes v_k for k = j + (K/16) e, e = 0..15 -- exactly the register
// layout of the K-point Stockham FFT of fos_fft.cuh, which then runs with its twiddles in
// shared memory (no Tensor Memory: the prototype, not per-thread constants, fills shared
// memory).  A group of max(64, K/16) threads transforms F = max(1, 64 / (K/16)) consecutive
// output vectors; a CTA of 512 threads holds 512 / group groups, each with two exchange
// buffers per transform; the (zero-padded) prototype h[r K + k] lives once per CTA in shared
// memory.  Grid: persistent, one CTA per SM; work units of F transform slots (each one, two or
// four output vectors) in a contiguous range per CTA, its groups taking them in turn.  The
// input is read through L1/L2 (each sample feeds ceil(Nh / D) output vectors).
#include <type_traits>

#include "fos_chan.h"
#include "fos_fft.cuh"

namespace fos {

template <int LOGK, bool REAL>
struct ChanCfg {
    using S = FftShape<LOGK>;
    static constexpr int K = S::N;
    static constexpr int T = S::T;                // threads of one transform
    static constexpr int F = T >= 64 ? 1 : 64 / T;
    static constexpr int GT = F * T;              // threads of one group
    static constexpr int THREADS = 512;
    static constexpr int GROUPS = THREADS / GT;
    using TL = TwLayout<LOGK, (1 << 30)>;         // every pass twiddle in shared memory
    static constexpr int EX = xpad_len(K);        // elements of one exchange buffer
    static constexpr int OFF_TW = 0;
    static constexpr int OFF_BUF = (8 * TL::SMEM_ENTRIES + 127) / 128 * 128;
    static constexpr int OFF_H = OFF_BUF + GROUPS * F * 2 * 8 * EX;  // then P K floats of h
    static constexpr int smem_bytes(int P) { return OFF_H + 4 * P * K; }
    using Bar = GroupBarrier<GT>;
};

// v[e] += sum over taps r0 .. r0 + NR - 1 of h[r K + k] xt[t_m - r K - k], k = j + T e: all
// 16 NR loads are issued before the first multiply-add.  INTERIOR: every index lies in the
// array that x points into (x itself, or the state when x is passed as the state's end), so the
// loads are one base pointer with constant offsets through the read-only path; otherwise each
// index is checked and the state (or zero) read in front of x.
template <int NR, int K, int T, bool INTERIOR, typename T_>
__device__ __forceinline__ void branch_taps(float2 (&v)[16], const float *hs, const T_ *x, const T_ *s0,
                                            int64_t hist, int64_t tm, int r0, int j) {
    T_ xv[NR][16];
    if constexpr (INTERIOR) {
        const T_ *xb = x + (tm - (int64_t)r0 * K - j);
#pragma unroll
        for (int q = 0; q < NR; ++q)
#pragma unroll
            for (int e = 0; e < 16; ++e) xv[q][e] = __ldg(xb - (q * K + T * e));
    } else {
#pragma unroll
        for (int q = 0; q < NR; ++q) {
            const int64_t tb = tm - (int64_t)(r0 + q) * K - j;
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const int64_t t = tb - T * e;
                if (t >= 0) xv[q][e] = x[t];
                else xv[q][e] = t >= -hist ? s0[hist + t] : T_{};
            }
        }
    }
    const float *hb = hs + r0 * K + j;
#pragma unroll
    for (int q = 0; q < NR; ++q)
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            const float hr = hb[q * K + T * e];
            if constexpr (std::is_same<T_, float>::value) {
                v[e].x = fmaf(hr, xv[q][e], v[e].x);
            } else {
                v[e].x = fmaf(hr, xv[q][e].x, v[e].x);
                v[e].y = fmaf(hr, xv[q][e].y, v[e].y);
            }
        }
}

// Real input, two output vectors: v[e].x += taps of the vector at t_m = tm, v[e].y += taps of the
// one at tm + d1 (d1 = D, or 0 when that vector does not exist: it then repeats the first and is
// not stored), both with the same h[r K + k].  INTERIOR as above, for the first vector.
template <int NR, int K, int T, bool INTERIOR>
__device__ __forceinline__ void pair_taps(float2 (&v)[16], const float *hs, const float *x, const float *s0,
                                          int64_t hist, int64_t tm, int d1, int r0, int j) {
    float xa[NR][16], xb[NR][16];
    if constexpr (INTERIOR) {
        const float *pa = x + (tm - (int64_t)r0 * K - j);
        const float *pb = pa + d1;
#pragma unroll
        for (int q = 0; q < NR; ++q)
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                xa[q][e] = __ldg(pa - (q * K + T * e));
                xb[q][e] = __ldg(pb - (q * K + T * e));
            }
    } else {
#pragma unroll
        for (int q = 0; q < NR; ++q) {
            const int64_t tb = tm - (int64_t)(r0 + q) * K - j;
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const int64_t ta = tb - T * e, tc = ta + d1;
                xa[q][e] = ta >= 0 ? x[ta] : (ta >= -hist ? s0[hist + ta] : 0.f);
                xb[q][e] = tc >= 0 ? x[tc] : (tc >= -hist ? s0[hist + tc] : 0.f);
            }
        }
    }
    const float *hb = hs + r0 * K + j;
#pragma unroll
    for (int q = 0; q < NR; ++q)
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            const float hr = hb[q * K + T * e];
            v[e].x = fmaf(hr, xa[q][e], v[e].x);
            v[e].y = fmaf(hr, xb[q][e], v[e].y);
        }
}

// K = 2D, four vectors m0 .. m0+3 (t = tm + i D): vector m0 + i reads at tap r
// X(i - 2r) = xt[tm + D (i - 2r) - k], so X(2 - 2r) and X(3 - 2r) are what vectors m0 and m0 + 1
// read at tap r - 1: each tap loads two new samples and one coefficient per branch for four
// multiply-adds.  v[e] accumulates vectors m0 (x) and m0 + 1 (y), w[e] vectors m0 + 2 and m0 + 3,
// each in the same order as pair_taps (taps ascending), so the sums are the pair path's bit for
// bit.  Every index is inside x (the caller checks).  The branches are taken eight at a time to
// bound the registers.
template <int K, int T>
__device__ __forceinline__ void quad_taps(float2 (&v)[16], float2 (&w)[16], const float *hs, const float *x,
                                          int64_t tm, int D, int P, int j) {
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
        const float *pb = x + (tm - j - (int64_t)T * 8 * hf);  // X(a) of branch e = 8 hf + i: pb[D a - T i]
        const float *hb = hs + j + T * 8 * hf;
        float c0[8], c1[8];                                    // X(2 - 2r), X(3 - 2r)
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            c0[i] = __ldg(pb + 2 * D - T * i);
            c1[i] = __ldg(pb + 3 * D - T * i);
        }
#pragma unroll 1
        for (int r = 0; r < P; ++r) {
            const float *pr = pb - (int64_t)r * K;
            float n0[8], n1[8], hr[8];                         // X(-2r), X(1 - 2r), h[r K + k]
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                n0[i] = __ldg(pr - T * i);
                n1[i] = __ldg(pr + D - T * i);
                hr[i] = hb[r * K + T * i];
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int e = 8 * hf + i;
                v[e].x = fmaf(hr[i], n0[i], v[e].x);
                v[e].y = fmaf(hr[i], n1[i], v[e].y);
                w[e].x = fmaf(hr[i], c0[i], w[e].x);
                w[e].y = fmaf(hr[i], c1[i], w[e].y);
                c0[i] = n0[i];
                c1[i] = n1[i];
            }
        }
    }
}

// Branch sums of the real-input vectors m (x parts) and m + 1 (y parts) into v, which is zero;
// nothing for m >= nout, and the second repeats the first when m + 1 >= nout.  NRI taps in
// flight at a time while no branch reaches the state.
template <int NRI, int K, int T>
__device__ __forceinline__ void pair_sums(float2 (&v)[16], const float *hs, const float *x, const float *s0,
                                          int64_t hist, int64_t m, int64_t nout, int D, int P, int j) {
    if (m >= nout) return;
    const int64_t tm = m * D + D - 1;
    const int d1 = m + 1 < nout ? D : 0;
    int r = 0;
    if (tm - (int64_t)P * K + 1 >= 0) {
#pragma unroll 1
        for (; r + NRI <= P; r += NRI) pair_taps<NRI, K, T, true>(v, hs, x, s0, hist, tm, d1, r, j);
#pragma unroll 1
        for (; r < P; ++r) pair_taps<1, K, T, true>(v, hs, x, s0, hist, tm, d1, r, j);
    } else {
#pragma unroll 1
        for (; r < P; ++r) pair_taps<1, K, T, false>(v, hs, x, s0, hist, tm, d1, r, j);
    }
}

template <int LOGK, bool REAL>
__global__ void __launch_bounds__(512, 1) fos_chan_kernel(const ChanParams p) {
    using C = ChanCfg<LOGK, REAL>;
    using T_ = typename std::conditional<REAL, float, float2>::type;
    constexpr int K = C::K, T = C::T;
    extern __shared__ __align__(128) unsigned char smem[];
    const int tid = threadIdx.x;
    const int g = tid / C::GT, tg = tid % C::GT;
    const int f = tg / T, j = tg % T;
    float2 *stw = reinterpret_cast<float2 *>(smem + C::OFF_TW);
    float2 *b0 = reinterpret_cast<float2 *>(smem + C::OFF_BUF) + (g * C::F + f) * 2 * C::EX;
    float2 *b1 = b0 + C::EX;
    float *hs = reinterpret_cast<float *>(smem + C::OFF_H);
    const typename C::Bar gbar{1 + g};

    griddep_launch_dependents();  // the next call's kernel may start its own set-up
    // plan constants into shared memory: every load of a batch is issued before its stores, so
    // the latencies overlap (a short call pays this set-up once per CTA)
    for (int i0 = tid; i0 < C::TL::SMEM_ENTRIES; i0 += 4 * C::THREADS) {
        float2 t[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int i = i0 + q * C::THREADS;
            t[q] = i < C::TL::SMEM_ENTRIES ? p.tw[i] : make_float2(0.f, 0.f);
        }
#pragma unroll
        for (int q = 0; q < 4; ++q)
            if (i0 + q * C::THREADS < C::TL::SMEM_ENTRIES) stw[i0 + q * C::THREADS] = t[q];
    }
    {
        // the prototype, P K floats (zero-padded by the plan), as 16-byte pieces
        const float4 *h4 = reinterpret_cast<const float4 *>(p.h);
        float4 *hs4 = reinterpret_cast<float4 *>(hs);
        const int n4 = p.P * K / 4;
        for (int i0 = tid; i0 < n4; i0 += 8 * C::THREADS) {
            float4 t[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const int i = i0 + q * C::THREADS;
                t[q] = i < n4 ? __ldg(h4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int q = 0; q < 8; ++q)
                if (i0 + q * C::THREADS < n4) hs4[i0 + q * C::THREADS] = t[q];
        }
    }
    __syncthreads();
    // the set-up read plan memory only; x, y and the state may belong to the previous kernel
    griddep_wait();

    const T_ *x = static_cast<const T_ *>(p.x);
    const T_ *s0 = static_cast<const T_ *>(p.state);
    float2 *y = p.y;
    const int64_t hist = p.Nh - 1;
    // each CTA takes a contiguous range of units (the launch has at most one CTA per unit), its
    // groups taking them in turn, so that the groups of an SM read overlapping windows
    const int64_t uend = (blockIdx.x + 1) * p.nunits / gridDim.x;
    for (int64_t u = blockIdx.x * p.nunits / gridDim.x + g; u < uend; u += C::GROUPS) {
        // branch sums of this slot's transforms (v, and w for the second of a four-vector slot),
        // then one code path for every transform: a single copy of the FFT in the kernel keeps
        // its instruction footprint small, which short calls (cold instruction caches) feel
        float2 v[16], w[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) v[e] = w[e] = make_float2(0.f, 0.f);
        int64_t m;    // the slot's first output vector
        int ntr = 1;  // its transforms
        if (REAL && p.pack) {
            const float *xr = static_cast<const float *>(p.x), *sr = static_cast<const float *>(p.state);
            if (p.pack == 2) {  // K = 2D: vectors m .. m + 3, two transforms
                m = (u * C::F + f) * 4;
                ntr = 2;
                const int64_t tm = m * p.D + p.D - 1;
                if (m + 3 < p.nout && tm - (int64_t)p.P * K + 1 >= 0) {
                    quad_taps<K, T>(v, w, hs, xr, tm, p.D, p.P, j);
                } else {
                    // the second pair first, kept in w, then the first pair
#pragma unroll 1
                    for (int t = 1; t >= 0; --t) {
#pragma unroll
                        for (int e = 0; e < 16; ++e) v[e] = make_float2(0.f, 0.f);
                        pair_sums<1, K, T>(v, hs, xr, sr, hist, m + 2 * t, p.nout, p.D, p.P, j);
                        if (t == 1) {
#pragma unroll
                            for (int e = 0; e < 16; ++e) w[e] = v[e];
                        }
                    }
                }
            } else {  // vectors m, m + 1
                m = (u * C::F + f) * 2;
                pair_sums<2, K, T>(v, hs, xr, sr, hist, m, p.nout, p.D, p.P, j);
            }
        } else {
            m = u * C::F + f;
            const int64_t tm = m * p.D + p.D - 1;
            if (m < p.nout) {  // a partial last unit: the spare transforms idle
                // v[e] = v_k(m), k = j + T e; several taps of every branch in flight at a time
                // (four for real input, two for complex), then one tap at a time
                constexpr int NR = REAL ? 4 : 2;
                int r = 0;
                if (tm - (int64_t)p.P * K + 1 >= 0) {  // no branch reaches the state
#pragma unroll 1
                    for (; r + NR <= p.P; r += NR) branch_taps<NR, K, T, true>(v, hs, x, s0, hist, tm, r, j);
#pragma unroll 1
                    for (; r < p.P; ++r) branch_taps<1, K, T, true>(v, hs, x, s0, hist, tm, r, j);
                } else {
                    // the window reaches the state.  Tap r reads xt[tm - rK - (K-1) .. tm - rK]:
                    // taps below rx lie inside x, tap rx may straddle x[0], the taps below rs lie
                    // inside the state (read with the same batched loads, from the state's end),
                    // and only the straddling tap and taps reaching below the state (prototype
                    // padding) take checked loads
                    const int rx = (int)((tm + 1) / K);
                    const int rs = (int)((tm + hist + 1) / K) < p.P ? (int)((tm + hist + 1) / K) : p.P;
                    const T_ *se = s0 + hist;  // xt[t] = se[t] for -hist <= t < 0
#pragma unroll 1
                    for (; r + NR <= rx; r += NR) branch_taps<NR, K, T, true>(v, hs, x, s0, hist, tm, r, j);
#pragma unroll 1
                    for (; r < rx; ++r) branch_taps<1, K, T, true>(v, hs, x, s0, hist, tm, r, j);
                    if (r < p.P && tm - (int64_t)r * K >= 0) {
                        branch_taps<1, K, T, false>(v, hs, x, s0, hist, tm, r, j);
                        ++r;
                    }
#pragma unroll 1
                    for (; r + NR <= rs; r += NR) branch_taps<NR, K, T, true>(v, hs, se, s0, hist, tm, r, j);
#pragma unroll 1
                    for (; r < rs; ++r) branch_taps<1, K, T, true>(v, hs, se, s0, hist, tm, r, j);
#pragma unroll 1
                    for (; r < p.P; ++r) branch_taps<1, K, T, false>(v, hs, x, s0, hist, tm, r, j);
                }
            }
        }
#pragma unroll 1
        for (int t = 0; t < ntr; ++t) {
            if (t == 1) {
#pragma unroll
                for (int e = 0; e < 16; ++e) v[e] = w[e];
            }
            const int64_t mt = m + 2 * t;
            // the K-point DFT across the branches (forward, unscaled): Z[j + T e] in v[e]
            fft_tm<LOGK, (1 << 30), false>(v, b0, b1, stw, 0u, j, gbar);
            if (REAL && p.pack) {
                // Z[K - q] through shared memory: the transform's last pass reads the other
                // buffer; this one was last read before that pass's barrier
                float2 *bz = ((C::S::NPASS - 1) % 2 == 0) ? b0 : b1;
#pragma unroll
                for (int e = 0; e < 16; ++e) bz[xpad(j + T * e)] = v[e];
                gbar.sync();
                if (mt < p.nout) {
                    const bool live1 = mt + 1 < p.nout;
                    float2 *ym = y + mt * K + j;
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const float2 zc = bz[xpad((K - j - T * e) & (K - 1))];
                        st_cs(ym + T * e, make_float2(0.5f * (v[e].x + zc.x), 0.5f * (v[e].y - zc.y)));
                        if (live1)
                            st_cs(ym + K + T * e, make_float2(0.5f * (v[e].y + zc.y), 0.5f * (zc.x - v[e].x)));
                    }
                }
            } else if (mt < p.nout) {
                float2 *ym = y + mt * K + j;
#pragma unroll
                for (int e = 0; e < 16; ++e) st_cs(ym + T * e, v[e]);
            }
            gbar.sync();  // the next transform's first pass may write the buffers read here
        }
    }
}

template <int LOGK, bool REAL>
ChanEntry chan_entry() {
    using C = ChanCfg<LOGK, REAL>;
    ChanEntry k;
    k.func = reinterpret_cast<const void *>(&fos_chan_kernel<LOGK, REAL>);
    k.threads = C::THREADS;
    k.groups = C::GROUPS;
    k.per_unit = C::F;
    k.smem_fixed = C::OFF_H;
    k.tw_entries = C::TL::SMEM_ENTRIES;
    return k;
}

ChanEntry chan_kernel(int logk, bool real) {
    switch (logk) {
        case 6: return real ? chan_entry<6, true>() : chan_entry<6, false>();
        case 7: return real ? chan_entry<7, true>() : chan_entry<7, false>();
        case 8: return real ? chan_entry<8, true>() : chan_entry<8, false>();
        case 9: return real ? chan_entry<9, true>() : chan_entry<9, false>();
        case 10: return real ? chan_entry<10, true>() : chan_entry<10, false>();
        case 11: return real ? chan_entry<11, true>() : chan_entry<11, false>();
        case 12: return real ? chan_entry<12, true>() : chan_entry<12, false>();
        default: return ChanEntry{};
    }
}

}  // namespace fos
