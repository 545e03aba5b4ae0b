/*
 * fir_oracle.c -- float64 CPU oracle for frequency-domain overlap-save FIR filtering.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or call this
 * file; it exists so that tests, the smoke check and the benchmark's CPU-baseline leg
 * can check the CUDA library against a slow, plainly written definition.  It shares no
 * code, header, table or constant with the CUDA library.
 *
 * Source of the method: "一种基于GPU的高阶数字FIR滤波器频域并行处理实现方法"
 * (zl.czvv.com/42398539.html), claim (主权项), steps 1-6.
 *
 * Samples are complex float64, stored interleaved (re, im).  Real signals are passed
 * with im = 0.  Every function here is single-purpose and unblocked:
 *
 *   fo_direct        y[j] = sum_{m<M} h[m] * xt[j-m]                (the plain definition)
 *   fo_direct_at     the same sum at caller-chosen output indices only
 *   fo_state_next    S0' = last M-1 samples of concat(S0, x)          (step 3, state carry)
 *   fo_dft           X[k] = sum_n x[n] e^{-+2 pi i n k / N}           (textbook O(N^2) DFT)
 *   fo_fft           iterative radix-2 FFT, same convention as fo_dft
 *   fo_freq_response H = FFT_N(h zero-padded to N)                    (step 1)
 *   fo_overlap_save  steps 2-5 of the claim, written out block by block with fo_fft
 *   fo_channelize    a K-channel DFT analysis filter bank decimated by D (the polyphase
 *                    channelizer of "GPU加速短波信道化：多相滤波器组的并行重构与CUDA实现"),
 *                    written as its defining sum; fo_channelize_at at chosen output times
 *
 * Conventions (the page states neither the DFT sign nor its scaling): the forward
 * transform uses e^{-2 pi i nk/N} unscaled, the inverse e^{+2 pi i nk/N} scaled by 1/N.
 * With that reading H = FFT(h) as step 1 says, and the product of step 4 is a linear
 * convolution with h (not a correlation).
 *
 * xt[t] is the extended input of step 3: xt[t] = x[t] for 0 <= t < n, the initial state
 * S0 for -(M-1) <= t < 0 (xt[t] = S0[M-1+t], S0[M-2] the newest sample), 0 for t >= n.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

static const double FO_PI = 3.14159265358979323846264338327950288;

/* xt[t] (step 3's extended input) as a (re, im) pair. */
static void fo_xt(const double *x, int64_t n, const double *s0, int M, int64_t t,
                  double *re, double *im)
{
    if (t >= 0 && t < n) {
        *re = x[2 * t];
        *im = x[2 * t + 1];
    } else if (t < 0 && t >= -(int64_t)(M - 1)) {
        int64_t s = (int64_t)(M - 1) + t;
        *re = s0 ? s0[2 * s] : 0.0;
        *im = s0 ? s0[2 * s + 1] : 0.0;
    } else {
        *re = 0.0;
        *im = 0.0;
    }
}

/* One output of the definition: y[j] = sum_{m=0}^{M-1} h[m] * xt[j-m]. */
static void fo_one(const double *x, int64_t n, const double *h, int M, const double *s0,
                   int64_t j, double *yr, double *yi)
{
    double ar = 0.0, ai = 0.0;
    for (int m = 0; m < M; ++m) {
        double xr, xi;
        fo_xt(x, n, s0, M, j - m, &xr, &xi);
        double hr = h[2 * m], hi = h[2 * m + 1];
        ar += hr * xr - hi * xi;
        ai += hr * xi + hi * xr;
    }
    *yr = ar;
    *yi = ai;
}

/* Linear convolution with carried state, every output.  Parallel over outputs only;
 * each output is the same sequential sum over m, so the result does not depend on the
 * thread count. */
int fo_direct(const double *x, int64_t n, const double *h, int M, const double *s0,
              double *y)
{
    if (n < 0 || M < 1) return -1;
#pragma omp parallel for schedule(static, 4096)
    for (int64_t j = 0; j < n; ++j) fo_one(x, n, h, M, s0, j, &y[2 * j], &y[2 * j + 1]);
    return 0;
}

/* The definition evaluated only at idx[0..nidx-1] (each in [0, n)). */
int fo_direct_at(const double *x, int64_t n, const double *h, int M, const double *s0,
                 const int64_t *idx, int64_t nidx, double *y_at)
{
    if (n < 0 || M < 1) return -1;
    for (int64_t q = 0; q < nidx; ++q)
        if (idx[q] < 0 || idx[q] >= n) return -2;
#pragma omp parallel for schedule(dynamic, 64)
    for (int64_t q = 0; q < nidx; ++q)
        fo_one(x, n, h, M, s0, idx[q], &y_at[2 * q], &y_at[2 * q + 1]);
    return 0;
}

/* Step 3's carry: the state for the next call is the newest M-1 samples seen so far,
 * i.e. the last M-1 entries of concat(S0, x).  For n >= M-1 this is D_{k-1} when the
 * blocks tile x exactly; for a partial last block it is the last real samples, never
 * padding zeros. */
int fo_state_next(const double *x, int64_t n, const double *s0, int M, double *s_out)
{
    if (n < 0 || M < 1) return -1;
    for (int t = 0; t < M - 1; ++t) {
        /* position t of the new state is sample (n - (M-1) + t) of the extended input */
        double re, im;
        fo_xt(x, n, s0, M, n - (int64_t)(M - 1) + t, &re, &im);
        s_out[2 * t] = re;
        s_out[2 * t + 1] = im;
    }
    return 0;
}

/* Textbook DFT, O(N^2).  sign = -1 forward (unscaled), +1 inverse (scaled by 1/N).
 * The angle is reduced exactly with integer arithmetic (n*k mod N) before cos/sin. */
int fo_dft(const double *in, int64_t N, int sign, double *out)
{
    if (N < 1 || N > (1LL << 31) || (sign != -1 && sign != 1)) return -1;
#pragma omp parallel for schedule(static)
    for (int64_t k = 0; k < N; ++k) {
        double ar = 0.0, ai = 0.0;
        for (int64_t nn = 0; nn < N; ++nn) {
            int64_t e = (nn * k) % N; /* exact: nn, k < N <= 2^31 */
            double ang = sign * 2.0 * FO_PI * (double)e / (double)N;
            double c = cos(ang), s = sin(ang);
            double xr = in[2 * nn], xi = in[2 * nn + 1];
            ar += xr * c - xi * s;
            ai += xr * s + xi * c;
        }
        if (sign == 1) {
            ar /= (double)N;
            ai /= (double)N;
        }
        out[2 * k] = ar;
        out[2 * k + 1] = ai;
    }
    return 0;
}

/* In-place iterative radix-2 FFT (bit-reversal permutation, then log2 N butterfly
 * stages), same sign and scaling convention as fo_dft.  N must be a power of two. */
int fo_fft(double *z, int64_t N, int sign)
{
    if (N < 1 || (N & (N - 1)) != 0 || (sign != -1 && sign != 1)) return -1;
    /* bit-reversal permutation */
    for (int64_t i = 1, j = 0; i < N; ++i) {
        int64_t bit = N >> 1;
        for (; j & bit; bit >>= 1) j ^= bit;
        j ^= bit;
        if (i < j) {
            double tr = z[2 * i], ti = z[2 * i + 1];
            z[2 * i] = z[2 * j];
            z[2 * i + 1] = z[2 * j + 1];
            z[2 * j] = tr;
            z[2 * j + 1] = ti;
        }
    }
    /* butterflies; the twiddle of each butterfly is taken directly from cos/sin */
    for (int64_t len = 2; len <= N; len <<= 1) {
        int64_t half = len >> 1;
        for (int64_t start = 0; start < N; start += len) {
            for (int64_t q = 0; q < half; ++q) {
                double ang = sign * 2.0 * FO_PI * (double)q / (double)len;
                double wr = cos(ang), wi = sin(ang);
                int64_t a = start + q, b = a + half;
                double br = z[2 * b] * wr - z[2 * b + 1] * wi;
                double bi = z[2 * b] * wi + z[2 * b + 1] * wr;
                double ar = z[2 * a], ai = z[2 * a + 1];
                z[2 * a] = ar + br;
                z[2 * a + 1] = ai + bi;
                z[2 * b] = ar - br;
                z[2 * b + 1] = ai - bi;
            }
        }
    }
    if (sign == 1) {
        for (int64_t i = 0; i < 2 * N; ++i) z[i] /= (double)N;
    }
    return 0;
}

/* Step 1: the M taps of h, zero-padded at the tail to length N, transformed by an
 * N-point forward FFT: H = {H(0), ..., H(N-1)}. */
int fo_freq_response(const double *h, int M, int64_t N, double *H)
{
    if (M < 1 || N < M) return -1;
    memset(H, 0, sizeof(double) * 2 * (size_t)N);
    memcpy(H, h, sizeof(double) * 2 * (size_t)M);
    return fo_fft(H, N, -1);
}

/* Steps 2-5 of the claim for one call, in the page's order and notation:
 *   step 2  X = {B_0 .. B_{k-1}}, blocks of L = N-M+1 samples; the last block is
 *           zero-padded past n (the claim assumes Nblk = k*L exactly)
 *   step 3  E_0 = {S0, B_0}, E_i = {D_{i-1}, B_i}: N samples starting M-1 before B_i
 *   step 4  F_i = FFT(E_i), I_i = F_i * H, R_i = IFFT(I_i)
 *   step 5  R_i = {Z_i, Y_i}; Z_i (first M-1) is dropped, Y_i = R_i[M-1 .. M-1+L)
 * H is passed in (fo_freq_response of h, or a given response).  The new state is
 * written by fo_state_next. */
int fo_overlap_save(const double *x, int64_t n, const double *H, int M, int64_t N,
                    const double *s0, double *y)
{
    if (n < 0 || M < 1 || N < M || (N & (N - 1)) != 0) return -1;
    int64_t L = N - M + 1;
    int64_t k = (n + L - 1) / L;
    double *E = (double *)malloc(sizeof(double) * 2 * (size_t)N);
    if (!E) return -3;
    for (int64_t i = 0; i < k; ++i) {
        /* step 3: E_i starts M-1 samples before B_i (i*L) */
        for (int64_t t = 0; t < N; ++t)
            fo_xt(x, n, s0, M, i * L - (M - 1) + t, &E[2 * t], &E[2 * t + 1]);
        /* step 4 */
        fo_fft(E, N, -1);
        for (int64_t t = 0; t < N; ++t) {
            double fr = E[2 * t], fi = E[2 * t + 1];
            double hr = H[2 * t], hi = H[2 * t + 1];
            E[2 * t] = fr * hr - fi * hi;
            E[2 * t + 1] = fr * hi + fi * hr;
        }
        fo_fft(E, N, +1);
        /* step 5: keep R_i[M-1 .. M-1+L), clipped to the n real outputs */
        for (int64_t j = 0; j < L; ++j) {
            int64_t o = i * L + j;
            if (o >= n) break;
            y[2 * o] = E[2 * (M - 1 + j)];
            y[2 * o + 1] = E[2 * (M - 1 + j) + 1];
        }
    }
    free(E);
    return 0;
}

/*
 * Channelizer.  The page describes the filter bank by its polyphase steps (decimate into
 * branches, filter each branch with its polyphase component h_k(n) = h(nK + k), DFT across the
 * branches) with K channels and decimation D = K/2 (50% overlapping channels); those steps
 * compute the K modulated filters h_q(l) = h(l) e^{-2 pi i q l / K} applied to x and sampled
 * every D inputs.  The oracle is that definition, not the polyphase algorithm:
 *
 *   y[m][q] = sum_{l < Nh} h[l] e^{-2 pi i q l / K} xt[m D + D - 1 - l],   q < K, m < n / D
 *
 * Output vector m follows the m-th hop of D new input samples.  xt[t] = x[t] for t >= 0 and
 * the state S0 (Nh - 1 samples, newest last) for -(Nh-1) <= t < 0.  The angle is reduced
 * exactly, (q l) mod K, before the cosine and sine.  y is m-major: y[m K + q].
 */
static void fo_chan_one(const double *x, int64_t n, const double *h, int Nh, int K, int D, const double *s0,
                        int64_t m, double *ym) {
    const int64_t t0 = m * D + D - 1;
    for (int q = 0; q < K; ++q) {
        double re = 0.0, im = 0.0;
        for (int l = 0; l < Nh; ++l) {
            double a[2];
            fo_xt(x, n, s0, Nh, t0 - l, &a[0], &a[1]);
            const int64_t e = ((int64_t)q * l) % K;
            const double ang = -2.0 * FO_PI * (double)e / (double)K;
            const double wr = cos(ang), wi = sin(ang);
            /* h[l] w */
            const double hr = h[2 * l] * wr - h[2 * l + 1] * wi, hi = h[2 * l] * wi + h[2 * l + 1] * wr;
            re += hr * a[0] - hi * a[1];
            im += hr * a[1] + hi * a[0];
        }
        ym[2 * q] = re;
        ym[2 * q + 1] = im;
    }
}

int fo_channelize(const double *x, int64_t n, const double *h, int Nh, int K, int D, const double *s0,
                  double *y) {
    if (n < 0 || Nh < 1 || K < 1 || D < 1 || n % D != 0) return -1;
    const int64_t mo = n / D;
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < mo; ++m) fo_chan_one(x, n, h, Nh, K, D, s0, m, y + 2 * m * K);
    return 0;
}

int fo_channelize_at(const double *x, int64_t n, const double *h, int Nh, int K, int D, const double *s0,
                     const int64_t *ms, int64_t count, double *y) {
    if (n < 0 || Nh < 1 || K < 1 || D < 1 || n % D != 0) return -1;
    for (int64_t i = 0; i < count; ++i)
        if (ms[i] < 0 || ms[i] >= n / D) return -2;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < count; ++i) fo_chan_one(x, n, h, Nh, K, D, s0, ms[i], y + 2 * i * K);
    return 0;
}

int fo_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
