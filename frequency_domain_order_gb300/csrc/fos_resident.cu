// fos_resident.cu -- the fused overlap-save block kernel for N = 16384 and 32768: one block
// resident in one SM's Tensor Memory.
//
// Steps 3-5 of the claim in "一种基于GPU的高阶数字FIR滤波器频域并行处理实现方法"
// (zl.czvv.com/42398539.html, 主权项) for N = C x P, P = 4096, C = N / P (4 or 8), computed
// with the split n = P a + b, k = c + C d of the DFT:
//
//   X[c + C d] = sum_b W_P^{bd} [ W_N^{bc} sum_a x[P a + b] W_C^{ac} ]
//   R[P a + b] = sum_c W_C^{-ac} [ W_N^{-bc} sum_d W_P^{-bd} (X H / N)[c + C d] ]
//
// A block of N complex values (256 KB at N = 32768) is more than a CTA's shared memory but
// fits one SM's Tensor Memory (128 lanes x 512 columns).  Lane l holds every (b, c) with
// b mod 128 = l, that is b = l + 128 m, m = 0..31, at complex slot
// q(c, m) = 32 c + 16 (m & 1) + (m >> 1) (columns 2q and 2q + 1).  Threads t, t + 128,
// t + 256 and t + 384 of the CTA share lane t mod 128, so every regrouping the split needs
// stays inside a lane and no data crosses between threads through shared memory outside the
// P-point transforms themselves:
//
//   phase A  thread (s, r) = (t / 128, t mod 128) owns b = r + 128 (8 s + i), i = 0..7.  It
//            loads xt[blk L - (M-1) + P a + b] for every a (the window was prefetched into L2
//            while the previous block was being transformed), does the C-point DFTs over a,
//            multiplies by W_N^{bc} (the powers of W_N^b = W_N^r W_N^{128 m}) and writes (b, c)
//            to its lane.
//   phase B  two groups of 256 threads; group g transforms c = g, g + 2, ...  Thread j of a
//            group holds b = j + 256 e, e = 0..15 (32 contiguous columns of lane j mod 128)
//            and runs the P-point FFT of fos_fft.cuh (twiddles in shared memory), the
//            multiply by H[c + C d] / N (stored c-major at plan time), the inverse FFT, and
//            writes the result back to the same columns.  Meanwhile the next block's input
//            window is prefetched into L2.
//   phase C  the ownership of phase A: multiply by W_N^{-bc}; the C-point inverse DFTs over
//            c give R[P a + b] for every a; R[t] with t >= M - 1 is stored (step 5).
//
// Phase A of a thread writes exactly the columns that its phase C reads, so phase C of one
// block and phase A of the next run fused, step by step, with the next block's loads issued
// first; two CTA barriers per block order A -> B -> C.  Real input packs two consecutive blocks into one complex transform, as
// in the other kernels.  Grid: persistent, one CTA per SM (the Tensor Memory allocation),
// blocks taken round-robin.  The kernel has no waits on other CTAs or on copies.
#include <type_traits>

#include "fos_resident.cuh"

namespace fos {

template <int LOGN, bool REAL>
struct ResidentCfg {
    static constexpr int N = 1 << LOGN;
    static constexpr int LOGP = 12;
    static constexpr int P = 1 << LOGP;
    static constexpr int C = N / P;          // 4 or 8
    static constexpr int THREADS = 512;
    static constexpr int GT = 256;           // threads of one phase-B group
    static constexpr int TM_COLS = 64 * C;   // 32 C complex slots per lane
    using TL = TwLayout<LOGP, 256>;          // every pass twiddle of the P-point FFT in shared memory
    static constexpr int BUF = xpad_len(P);  // elements of one exchange buffer
    // shared memory: 128-byte header (Tensor Memory address), pass twiddles, W_N^{128 m} (m < 32),
    // W_N^r (r < 128), then two exchange buffers per group
    static constexpr int OFF_TW = 128;
    static constexpr int OFF_HI = OFF_TW + 8 * TL::SMEM_ENTRIES;
    static constexpr int OFF_WR = OFF_HI + 8 * 32;
    static constexpr int OFF_BUF = (OFF_WR + 8 * 128 + 127) / 128 * 128;
    static constexpr int SMEM_BYTES = OFF_BUF + 2 * 2 * 8 * BUF;
    // the tensor-core variant: the four 4 KB DFT-matrix tiles after the buffers, and one
    // MMA-completion mbarrier per group in the header; a group's A tiles (64 KB) overlap its
    // two exchange buffers
    static constexpr int OFF_BTC = (SMEM_BYTES + 1023) / 1024 * 1024;
    static constexpr int SMEM_TC = OFF_BTC + 4 * (int)kTcBTileBytes;
    static constexpr int OFF_TCBAR = 64;
    static_assert(C == 4 || C == 8, "N = 16384 or 32768");
    static_assert(2 * 8 * BUF >= 4 * (int)kTcTileBytes && SMEM_TC <= 227 * 1024 && OFF_TCBAR + 16 <= OFF_TW,
                  "tensor-core variant layout");
    static_assert(TL::SMEM_ENTRIES == FftShape<LOGP>::TW_ENTRIES, "all pass twiddles in shared memory");
};

// Phase C of unit uc (when uc >= 0) and phase A of unit ua (when ua >= 0), fused step by
// step.  Phase A writes exactly the Tensor Memory columns of this thread that its phase C
// reads, so each step first issues the loads of unit ua, then reads unit uc's values, does the
// inverse twiddle, the C-point inverse DFTs and the discard-and-store (step 5), and finally
// the C-point DFTs over a and the forward twiddle of unit ua into the same columns: the load
// latency overlaps the inverse work and the stores.
template <int LOGN, bool REAL>
__device__ __forceinline__ void phase_ca(const BlockParams &p, int64_t uc, void *yc, int64_t ua, const Chan &cha,
                                         uint32_t tlane, int s, int r, const float2 *hi_s, const float2 *wr_s) {
    using R_ = ResidentCfg<LOGN, REAL>;
    constexpr int C = R_::C, P = R_::P;
    // uc, ua: unit indices within their channels; yc: uc's channel's output, cha: ua's channel
    const int64_t sc = (REAL ? 2 * uc : uc) * p.L - (p.M - 1);  // output index of R[0] of unit uc
    const bool whole = sc + R_::N + (REAL ? p.L : 0) <= p.n;
    const int keep = p.M - 1;
    // outputs R[t] of unit uc with t < lim exist (t = P a + b < N, so lim is capped to an int)
    const int lim = p.n - sc > (int64_t)R_::N + p.L ? R_::N + p.L : (int)(p.n - sc);
    const int64_t sa = (REAL ? 2 * ua : ua) * p.L - (p.M - 1);  // xt index of E[0] of unit ua
    const bool interior = sa >= 0 && sa + R_::N + (REAL ? p.L : 0) <= p.n;
    const float2 wr1 = wr_s[r];  // W_N^r
#pragma unroll 1
    for (int st = 0; st < 4; ++st) {
        const int i0 = (st & 1) + 4 * (st >> 1);  // 0, 1, 4, 5: steps i0 and i0 + 2
        const uint32_t col = step_col(s, i0);
        float2 xa[2][C];
        if (ua >= 0) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int b = r + 128 * (8 * s + i0 + 2 * h);
                load_points<REAL, C, P>(p, cha, sa + b, interior, xa[h]);
            }
        }
        if (uc >= 0) {
            float2 v[2][C];
#pragma unroll
            for (int c = 0; c < C; ++c) tmem_ld4(tlane + 64u * c + col, v[0][c], v[1][c]);
            tmem_wait_ld();
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int m = 8 * s + i0 + 2 * h;
                float2 w[C];  // W_N^{bc}: W_N^b = W_N^r W_N^{128 m} (m < 32 < N / 128), then its powers
                twiddle_powers<C>(cmul(wr1, hi_s[m]), w);
#pragma unroll
                for (int c = 1; c < C; ++c) v[h][c] = cmulc(v[h][c], w[c]);
                dft<C, +1>(v[h]);
                const int b = r + 128 * m;
                // y[sc + b + P a] at a constant offset from one pointer (dereferenced only for t >= keep)
#pragma unroll
                for (int a = 0; a < C; ++a) {
                    const int t = P * a + b;
                    if (t < keep) continue;
                    if constexpr (REAL) {
                        float *yb = static_cast<float *>(yc) + sc + b;
                        if (whole || t < lim) st_cs(yb + P * a, v[h][a].x);
                        if (whole || t + p.L < lim) st_cs(yb + p.L + P * a, v[h][a].y);
                    } else {
                        float2 *yb = static_cast<float2 *>(yc) + sc + b;
                        if (whole || t < lim) st_cs(yb + P * a, v[h][a]);
                    }
                }
            }
        }
        if (ua >= 0) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int m = 8 * s + i0 + 2 * h;
                dft<C, -1>(xa[h]);
                float2 w[C];
                twiddle_powers<C>(cmul(wr1, hi_s[m]), w);
#pragma unroll
                for (int c = 1; c < C; ++c) xa[h][c] = cmul(xa[h][c], w[c]);
            }
#pragma unroll
            for (int c = 0; c < C; ++c) tmem_st4(tlane + 64u * c + col, xa[0][c], xa[1][c]);
        }
    }
    if (ua >= 0) tmem_wait_st();
}

// TC: the P-point transforms' 16-point DFTs on the tensor cores (the optional engine)
template <int LOGN, bool REAL, bool MULTI, bool TC = false>
__global__ void __launch_bounds__(512, 1) fos_resident_kernel(const BlockParams p) {
    using R_ = ResidentCfg<LOGN, REAL>;
    extern __shared__ __align__(128) unsigned char smem[];
    const int tid = threadIdx.x;
    // the warp index broadcast from lane 0, so that the compiler knows it (and s, g, the Tensor
    // Memory addresses derived from it) to be the same in every lane of a warp
    const int warp = __shfl_sync(0xffffffffu, tid >> 5, 0);
    const int s = warp >> 2, r = tid & 127;  // phases A and C: s = tid / 128
    const int g = warp >> 3, j = tid & 255;  // phase B: g = tid / 256
    uint32_t *tm_slot = reinterpret_cast<uint32_t *>(smem);
    float2 *stw = reinterpret_cast<float2 *>(smem + R_::OFF_TW);
    float2 *hi_s = reinterpret_cast<float2 *>(smem + R_::OFF_HI);
    float2 *wr_s = reinterpret_cast<float2 *>(smem + R_::OFF_WR);
    float2 *b0 = reinterpret_cast<float2 *>(smem + R_::OFF_BUF) + g * 2 * R_::BUF;
    float2 *b1 = b0 + R_::BUF;
    const GroupBarrier<R_::GT> gbar{1 + g};

    griddep_launch_dependents();  // the next call's kernel may start its own set-up
    int64_t u = blockIdx.x, lu = 0, lun = 0;
    int chu = u < p.nunits ? channel_of<MULTI>(p, u, lu) : 0;  // unit u's channel
    if (u < p.nunits && !p.no_bulk) prefetch_window<R_::N, REAL>(p, chan<REAL>(p, chu), lu, tid);  // a hint only
    if (warp == 0) {
        tmem_alloc(tm_slot, R_::TM_COLS);
        tmem_relinquish();
    }
    for (int k = tid; k < R_::TL::SMEM_ENTRIES; k += R_::THREADS) stw[k] = p.tw[k];
    for (int k = tid; k < 32; k += R_::THREADS) hi_s[k] = p.twa[128 + k];
    for (int k = tid; k < 128; k += R_::THREADS) wr_s[k] = p.twa[k];
    uint64_t *tcbar = reinterpret_cast<uint64_t *>(smem + R_::OFF_TCBAR) + g;
    if constexpr (TC) {  // the split DFT matrices (read by the tensor cores) and the MMA barriers
        float2 *bt = reinterpret_cast<float2 *>(smem + R_::OFF_BTC);
        for (int k = tid; k < 4 * (int)kTcBTileBytes / 8; k += R_::THREADS) bt[k] = p.btc[k];
        fence_proxy_async_smem();
        if (j == 0) {
            mbar_init(tcbar, 1);
            fence_mbar_init();
        }
    }
    tmem_fence_before_sync();
    __syncthreads();
    tmem_fence_after_sync();
    const uint32_t tlane = __shfl_sync(0xffffffffu, *tm_slot, 0) + ((uint32_t)(32 * (warp & 3)) << 16);
    TcCtx tc{};
    uint32_t tcpar = 0u;
    if constexpr (TC) {
        tc.a_base = smem_addr(b0);
        tc.b_base = smem_addr(smem + R_::OFF_BTC);
        tc.row_off = (uint32_t)(j >> 7) * 2u * kTcTileBytes + tc_offset(j & 127, 0);
        tc.mbar = tcbar;
        tc.err = p.err;
        tc.leader = j == 0;
    }
    // the set-up read plan memory only; x, y and the state may belong to the previous kernel
    griddep_wait();

    if (u < p.nunits)  // phase A of the first unit
        phase_ca<LOGN, REAL>(p, -1, nullptr, lu, chan<REAL>(p, chu), tlane, s, r, hi_s, wr_s);
    for (; u < p.nunits; u += gridDim.x) {
        tmem_fence_before_sync();
        __syncthreads();  // every (b, c) of the block is in Tensor Memory; S0 has been read
        tmem_fence_after_sync();
        if (p.fuse_state && lu == 0) {
            // only the channel's unit 0 reads its S0 (fuse_state), and n >= M - 1: S0' = the
            // last M-1 samples of the channel's x
            using T_ = typename std::conditional<REAL, float, float2>::type;
            const Chan cu = chan<REAL>(p, chu);
            const T_ *x = static_cast<const T_ *>(cu.x);
            T_ *st = static_cast<T_ *>(cu.state);
            for (int t = tid; t < p.M - 1; t += R_::THREADS) st[t] = x[p.n - (p.M - 1) + t];
        }
        const int64_t un = u + gridDim.x;
        const int chn = un < p.nunits ? channel_of<MULTI>(p, un, lun) : chu;
        if (un < p.nunits && !p.no_bulk) prefetch_window<R_::N, REAL>(p, chan<REAL>(p, chn), lun, tid);
        // (the packed quarter turn in the P-point transforms: C3 -2.3% measured, the pair kernel
        // +2.4%; the twiddles of both twiddled passes formed from four loaded ones: C3 -2.4%,
        // the pair kernel +3.9%)
        phase_b<R_::C, true, false, 16, TC>(p, tlane, g, j, b0, b1, stw, gbar, 0, 1, 32u * (uint32_t)((warp >> 2) & 1),
                                            &tc, &tcpar);
        tmem_fence_before_sync();
        __syncthreads();  // every c has been filtered
        tmem_fence_after_sync();
        // phase C of this unit with phase A of the next (un is resident in L2 by now)
        phase_ca<LOGN, REAL>(p, lu, chan<REAL>(p, chu).y, un < p.nunits ? lun : -1, chan<REAL>(p, chn), tlane, s,
                             r, hi_s, wr_s);
        chu = chn;
        lu = lun;
    }

    tmem_fence_before_sync();
    __syncthreads();
    tmem_fence_after_sync();
    if (warp == 0) tmem_dealloc(*tm_slot, R_::TM_COLS);
}

template <int LOGN, bool REAL>
KernelEntry resident_entry() {
    using R_ = ResidentCfg<LOGN, REAL>;
    KernelEntry k;
    k.func = reinterpret_cast<const void *>(&fos_resident_kernel<LOGN, REAL, false>);
    k.func_multi = reinterpret_cast<const void *>(&fos_resident_kernel<LOGN, REAL, true>);
    k.func_tc = reinterpret_cast<const void *>(&fos_resident_kernel<LOGN, REAL, false, true>);
    k.func_multi_tc = reinterpret_cast<const void *>(&fos_resident_kernel<LOGN, REAL, true, true>);
    k.smem_tc = R_::SMEM_TC;
    k.threads = R_::THREADS;
    k.smem = R_::SMEM_BYTES;
    k.cluster = 1;
    k.units_per_cta = 1;
    k.groups = 1;
    k.fft_logn = R_::LOGP;
    k.split_c = R_::C;
    k.state_from_x = 1;
    return k;
}

KernelEntry resident_kernel(int logn, bool real) {
    switch (logn) {
        case 14: return real ? resident_entry<14, true>() : resident_entry<14, false>();
        case 15: return real ? resident_entry<15, true>() : resident_entry<15, false>();
        default: return KernelEntry{};
    }
}

}  // namespace fos
