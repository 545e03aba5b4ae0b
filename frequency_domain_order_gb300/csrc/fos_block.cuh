// fos_block.cuh -- the fused overlap-save block kernel for N <= 8192 (one CTA per block group).
//
// One launch performs steps 3, 4 and 5 of the claim in "一种基于GPU的高阶数字FIR滤波器
// 频域并行处理实现方法" (zl.czvv.com/42398539.html, 主权项) for every block of one call, and
// the state carry of step 3:
//   gather   E_i = xt[i L - (M-1) .. i L - (M-1) + N) into shared memory.  Interior
//            groups of blocks arrive by one bulk (TMA) copy issued while the previous group
//            is being transformed (double-buffered); groups that touch the state S0 or run
//            past the input are gathered with plain loads (S0 in front, zeros behind).
//   FFT      F_i = FFT_N(E_i) in registers + the exchange buffer (fos_fft.cuh)
//   multiply I_i = F_i * H with H / N held in shared memory for the life of the CTA
//   IFFT     R_i = IFFT_N(I_i), again natural order in registers
//   discard  Y_i = R_i[M-1 .. M-1+L) stored straight from registers, masked to n outputs
//   state    the CTA holding block 0 writes S0' = last M-1 samples of concat(S0, x)
//            after it has read S0 (no other CTA reads S0 when fuse_state is set)
// Real input packs two consecutive blocks into one complex transform (E_{2p} as real part,
// E_{2p+1} as imaginary part); with a real h the two outputs come back as the real and
// imaginary parts of R.
//
// Grid: persistent, at most (SMs x resident CTAs) CTAs; CTA c takes work units c, c + grid,
// ...  A work unit is F consecutive blocks (complex) or F consecutive block pairs (real),
// F = max(1, 256 / (N/16)), each handled by N/16 threads.
#pragma once

#include <type_traits>

#include "fos_fft.cuh"
#include "fos_kernels.h"

namespace fos {

template <int LOGN, bool REAL>
struct BlockCfg {
    using S = FftShape<LOGN>;
    static constexpr int N = S::N;
    static constexpr int T = S::T;
    static constexpr int F = T >= 256 ? 1 : 256 / T;
    static constexpr int THREADS = F * T;
    static constexpr int SB = REAL ? 4 : 8;  // bytes per sample
    // F blocks' gather windows (complex: (F-1)L + N samples; real: (2F-1)L + N floats) fit in
    // 8 F N bytes; +32 covers rounding the bulk copy out to 16-byte boundaries at both ends.
    // The same buffer then serves as the F padded exchange buffers (8 F xpad_len(N) bytes).
    static constexpr int EX_BYTES = 8 * F * xpad_len(N);
    static constexpr int BUF_BYTES = (((8 * F * N + 32) > EX_BYTES ? (8 * F * N + 32) : EX_BYTES) + 127) / 128 * 128;
    static constexpr int H_BYTES = 8 * N;
    static constexpr int SMEM_BYTES = 128 + H_BYTES + 2 * BUF_BYTES;
    static constexpr int MIN_BLOCKS = THREADS <= 256 ? 2 : 1;
};

// Gather the input window of work unit u into `buf`.  Returns the element offset of
// xt[start] inside the buffer.  A bulk copy is used (issued by thread 0, completing on
// `bar`; used_tma = true) when the 16-byte-rounded byte range lies inside x; otherwise every
// thread gathers with plain loads and the CTA synchronises (used_tma = false).
template <int LOGN, bool REAL>
__device__ __forceinline__ int stage_unit(const BlockParams &p, int64_t u, unsigned char *buf, uint64_t *bar,
                                          bool allow_tma, bool &used_tma) {
    using C = BlockCfg<LOGN, REAL>;
    constexpr int SB = C::SB;
    const int64_t span = (int64_t)C::F * p.L * (REAL ? 2 : 1);
    const int64_t start = u * span - (p.M - 1);
    const int64_t len = (int64_t)(REAL ? 2 * C::F - 1 : C::F - 1) * p.L + C::N;
    if (allow_tma && start >= 0) {
        const uintptr_t xb = reinterpret_cast<uintptr_t>(p.x);
        const uintptr_t a0 = xb + (uintptr_t)start * SB, a1 = a0 + (uintptr_t)len * SB;
        const uintptr_t b0 = a0 & ~uintptr_t(15), b1 = (a1 + 15) & ~uintptr_t(15);
        if (b0 >= xb && b1 <= xb + (uintptr_t)p.n * SB) {
            if (threadIdx.x == 0) {
                fence_proxy_async_smem();
                mbar_arrive_expect_tx(bar, (uint32_t)(b1 - b0));
                bulk_g2s(buf, reinterpret_cast<const void *>(b0), (uint32_t)(b1 - b0), bar);
            }
            used_tma = true;
            return (int)((a0 - b0) / SB);
        }
    }
    used_tma = false;
    const int64_t hist = p.M - 1;
    if constexpr (REAL) {
        const float *x = static_cast<const float *>(p.x);
        const float *s0 = static_cast<const float *>(p.state);
        float *dst = reinterpret_cast<float *>(buf);
        for (int64_t i = threadIdx.x; i < len; i += C::THREADS) {
            const int64_t t = start + i;
            float v = 0.f;
            if (t >= 0) {
                if (t < p.n) v = x[t];
            } else if (t >= -hist) {
                v = s0[hist + t];
            }
            dst[i] = v;
        }
    } else {
        const float2 *x = static_cast<const float2 *>(p.x);
        const float2 *s0 = static_cast<const float2 *>(p.state);
        float2 *dst = reinterpret_cast<float2 *>(buf);
        for (int64_t i = threadIdx.x; i < len; i += C::THREADS) {
            const int64_t t = start + i;
            float2 v = make_float2(0.f, 0.f);
            if (t >= 0) {
                if (t < p.n) v = x[t];
            } else if (t >= -hist) {
                v = s0[hist + t];
            }
            dst[i] = v;
        }
    }
    __syncthreads();
    return 0;
}

// S0' = xt[n-(M-1) .. n): samples of x, or (when n < M-1) of S0, which the gather of unit 0
// left at buffer index (t + M - 1) for xt[t], t < 0.
template <int LOGN, bool REAL>
__device__ __forceinline__ void write_state(const BlockParams &p, const unsigned char *buf) {
    using C = BlockCfg<LOGN, REAL>;
    using T_ = typename std::conditional<REAL, float, float2>::type;
    const T_ *x = static_cast<const T_ *>(p.x);
    const T_ *stg = reinterpret_cast<const T_ *>(buf);
    T_ *st = static_cast<T_ *>(p.state);
    const int hist = p.M - 1;
    for (int t = threadIdx.x; t < hist; t += C::THREADS) {
        const int64_t src = p.n - hist + t;
        st[t] = src >= 0 ? x[src] : stg[src + hist];
    }
}

template <int LOGN, bool REAL>
__global__ void __launch_bounds__(BlockCfg<LOGN, REAL>::THREADS, BlockCfg<LOGN, REAL>::MIN_BLOCKS)
    fos_block_kernel(const BlockParams p) {
    using C = BlockCfg<LOGN, REAL>;
    constexpr int T = C::T;
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem);
    float2 *hs = reinterpret_cast<float2 *>(smem + 128);  // H / N, natural order
    unsigned char *bufs[2] = {smem + 128 + C::H_BYTES, smem + 128 + C::H_BYTES + C::BUF_BYTES};
    const int tid = threadIdx.x;
    const int f = tid / T;  // transform slot within the CTA
    const int j = tid % T;  // thread within the transform

    if (tid == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        fence_mbar_init();
    }
    // H / N stays in shared memory for every block this CTA filters
    for (int i = tid; i < C::N; i += C::THREADS) hs[i] = __ldg(p.H + i);
    __syncthreads();

    // double buffering: `cur` holds the unit being filtered, `nxt` the one being fetched
    unsigned char *cur = bufs[0], *nxt = bufs[1];
    uint64_t *bcur = &bars[0], *bnxt = &bars[1];
    uint32_t pcur = 0u, pnxt = 0u;  // mbarrier phase parity to wait for
    bool ucur = false, unxt = false;  // filled by a bulk copy (else by plain loads)
    int ocur = 0, onxt = 0;           // element offset of the window in the buffer
    bool allow_tma = true;

    int64_t u = blockIdx.x;
    if (u < p.nunits) ocur = stage_unit<LOGN, REAL>(p, u, cur, bcur, allow_tma, ucur);

    for (; u < p.nunits; u += gridDim.x) {
        const int64_t un = u + gridDim.x;
        if (un < p.nunits) onxt = stage_unit<LOGN, REAL>(p, un, nxt, bnxt, allow_tma, unxt);
        if (ucur) {
            const bool ok = mbar_wait_bounded(bcur, pcur);
            pcur ^= 1u;
            if (__syncthreads_or(!ok)) {
                // the copy did not arrive in time: report it, stop using bulk copies and
                // gather this unit with plain loads instead
                if (tid == 0) atomicExch(p.err, 1);
                allow_tma = false;
                ocur = stage_unit<LOGN, REAL>(p, u, cur, bcur, false, ucur);
            }
        }

        // gather E_i (step 3) from the staged window into registers: v[e] = E[j + e T]
        float2 v[16];
        if constexpr (REAL) {
            const float *sr = reinterpret_cast<const float *>(cur) + ocur + 2 * f * p.L;
#pragma unroll
            for (int e = 0; e < 16; ++e) v[e] = make_float2(sr[j + e * T], sr[p.L + j + e * T]);
        } else {
            const float2 *sc = reinterpret_cast<const float2 *>(cur) + ocur + f * p.L;
#pragma unroll
            for (int e = 0; e < 16; ++e) v[e] = sc[j + e * T];
        }
        if (p.fuse_state && u == 0) write_state<LOGN, REAL>(p, cur);
        __syncthreads();  // the window is consumed; the buffer becomes the exchange buffer

        // step 4: FFT, multiply by H, IFFT
        float2 *ex = reinterpret_cast<float2 *>(cur) + f * xpad_len(C::N);
        fft_regs<LOGN, -1>(v, ex, p.tw, j, false);
#pragma unroll
        for (int e = 0; e < 16; ++e) v[e] = cmul(v[e], hs[j + e * T]);
        fft_regs<LOGN, +1>(v, ex, p.tw, j, true);

        // step 5: drop R[0 .. M-2], store R[M-1 .. N) as Y_i
        const int64_t blk = REAL ? 2 * (u * C::F + f) : (u * C::F + f);
        const int64_t obase = blk * p.L - (p.M - 1);
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            const int t = j + e * T;
            if (t >= p.M - 1) {
                const int64_t o = obase + t;
                if constexpr (REAL) {
                    float *y = static_cast<float *>(p.y);
                    if (o < p.n) st_cs(y + o, v[e].x);
                    if (o + p.L < p.n) st_cs(y + o + p.L, v[e].y);
                } else {
                    float2 *y = static_cast<float2 *>(p.y);
                    if (o < p.n) st_cs(y + o, v[e]);
                }
            }
        }
        __syncthreads();  // `cur` is free for the copy issued at the top of the next iteration
        unsigned char *tb = cur; cur = nxt; nxt = tb;
        uint64_t *tm = bcur; bcur = bnxt; bnxt = tm;
        uint32_t tp = pcur; pcur = pnxt; pnxt = tp;
        bool tu = ucur; ucur = unxt; unxt = tu;
        int to = ocur; ocur = onxt; onxt = to;
    }
}

template <int LOGN, bool REAL>
KernelEntry block_entry() {
    using C = BlockCfg<LOGN, REAL>;
    KernelEntry k;
    k.func = reinterpret_cast<const void *>(&fos_block_kernel<LOGN, REAL>);
    k.threads = C::THREADS;
    k.smem = C::SMEM_BYTES;
    k.cluster = 1;
    k.units_per_cta = C::F;
    k.fft_logn = LOGN;
    return k;
}

}  // namespace fos
