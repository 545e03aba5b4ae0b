// fos_pair.cu -- the fused overlap-save block kernel for N = 65536: one block held by a
// cluster of two CTAs, half of it in each SM's Tensor Memory.
//
// Steps 3-5 of the claim in "一种基于GPU的高阶数字FIR滤波器频域并行处理实现方法"
// (zl.czvv.com/42398539.html, 主权项) with the split n = P a + b, k = c + 16 d (P = 4096,
// a, c < 16).  CTA kappa (0 or 1, its rank in the cluster) computes the bins with c = kappa + 2 c',
// c' < 8, so that the 16-point DFT over a falls apart into a radix-2 step and an 8-point DFT:
//
//   X[c + 16 d] = sum_b W_P^{bd} W_N^{bc} sum_{a<8} W_8^{a c'} [ W_16^{a kappa} (x[P a + b] + (-1)^kappa x[P (a+8) + b]) ]
//
// and the inverse splits the same way: with P_kappa[a', b] = sum_{c'} W_8^{-a'c'} W_N^{-bc} Z_c[b]
// (Z_c the filtered sub-transform c after its inverse P-point FFT),
//
//   R[P (a' + 8 h) + b] = P_0[a', b] + (-1)^h W_16^{-a'} P_1[a', b],   a' < 8, h < 2.
//
// Each CTA therefore holds N/2 = 32768 values (its whole Tensor Memory, laid out as in
// fos_resident.cuh with c' as the sub-transform index), reads the whole input window (from L2;
// each CTA prefetches half of the next window), and exchanges P values once per block:
//
//   phase A   thread (s, r) takes b = r + 128 m for m = 16 rho + 4 s + i (rho < 2, i < 4):
//             loads the 16 points of every b, the radix-2 step for its kappa, the 8-point DFTs,
//             the twiddles W_N^{bc}.
//   phase B   the P-point filtering of fos_resident.cuh for its 8 sub-transforms.
//   [cluster barrier: both CTAs are done with phase B, so each may write into the other's
//    exchange buffers]
//   phase C1  thread (s, r) takes m = 8 s + i (i < 8): W_N^{-bc} and the 8-point inverse DFT
//             over c' give P_kappa[a', b].  CTA kappa finishes the outputs for b in
//             [2048 kappa, 2048 kappa + 2048) (m in [16 kappa, 16 kappa + 16)): rows
//             s = 2 kappa, 2 kappa + 1 keep their P values in their lane, the other rows store
//             theirs into the other CTA's shared memory (128 KB, distributed shared memory).
//   [cluster barrier: the values have landed]
//   phase C2  with phase A's assignment of m: for its 4 values of m in this CTA's range each
//             thread combines P_0 and P_1 and stores R[t] for t >= M - 1 (step 5).  Phase A of
//             the next block runs fused with it: every m starts with the next block's loads,
//             and the slots a thread combines are the ones it then refills.
//
// The two cluster barriers are the only waits on the other CTA; both CTAs take the same
// blocks (one per cluster, round-robin) and so pass the same barriers.  Real input packs two
// consecutive blocks into one complex transform, as in the other kernels.
#include <type_traits>

#include "fos_resident.cuh"

namespace fos {

template <bool REAL>
struct PairCfg {
    static constexpr int LOGN = 16;
    static constexpr int N = 1 << LOGN;
    static constexpr int P = 4096;
    static constexpr int CL = 8;             // local sub-transforms per CTA
    static constexpr int THREADS = 512;
    static constexpr int TM_COLS = 512;
    using TL = TwLayout<12, 256>;
    static constexpr int BUF = xpad_len(P);
    static constexpr int OFF_TW = 128;
    static constexpr int OFF_HI = OFF_TW + 8 * TL::SMEM_ENTRIES;  // W_N^{128 m}, m < 32
    static constexpr int OFF_WR = OFF_HI + 8 * 32;                 // W_N^r, r < 128
    static constexpr int OFF_BUF = (OFF_WR + 8 * 128 + 127) / 128 * 128;
    static constexpr int SMEM_BYTES = OFF_BUF + 2 * 2 * 8 * BUF;
    // the tensor-core variant (as in fos_resident.cu): DFT-matrix tiles after the buffers, one
    // MMA-completion mbarrier per group in the header, A tiles over the group's exchange buffers
    static constexpr int OFF_BTC = (SMEM_BYTES + 1023) / 1024 * 1024;
    static constexpr int SMEM_TC = OFF_BTC + 4 * (int)kTcBTileBytes;
    static constexpr int OFF_TCBAR = 64;
    static_assert(2 * 8 * BUF >= 4 * (int)kTcTileBytes && SMEM_TC <= 227 * 1024 && OFF_TCBAR + 16 <= OFF_TW,
                  "tensor-core variant layout");
    // phase C receive buffer (reuses the exchange buffers): P_other[a'][m mod 16][r]
    static constexpr int RECV_ELEMS = 8 * 16 * 128;
    static_assert(8 * RECV_ELEMS <= 2 * 2 * 8 * BUF, "receive buffer inside the exchange buffers");
};

__device__ __forceinline__ int recv_index(int a, int m, int r) { return (a * 16 + (m & 15)) * 128 + r; }

// w[c'] = W_N^{b c} for this CTA's bins c = KAPPA + 2 c', c' < 8 (w[0] = 1 for KAPPA = 0 is not
// written), from g = W_N^b by squarings and products: no power is more than four complex
// multiplications from g.
template <int KAPPA>
__device__ __forceinline__ void pair_twiddles(float2 g, float2 (&w)[8]) {
    const float2 h = cmul(g, g);  // W_N^{2b}
    if constexpr (KAPPA == 0) {
        w[1] = h;
        w[2] = cmul(h, h);
        w[3] = cmul(w[2], h);
        w[4] = cmul(w[2], w[2]);
        w[5] = cmul(w[4], h);
        w[6] = cmul(w[4], w[2]);
        w[7] = cmul(w[4], w[3]);
    } else {
        const float2 h2 = cmul(h, h), h4 = cmul(h2, h2);  // W_N^{4b}, W_N^{8b}
        w[0] = g;
        w[1] = cmul(g, h);
        w[2] = cmul(g, h2);
        w[3] = cmul(w[1], h2);
        w[4] = cmul(g, h4);
        w[5] = cmul(w[1], h4);
        w[6] = cmul(w[2], h4);
        w[7] = cmul(w[3], h4);
    }
}

template <bool REAL, int KAPPA>
__device__ __forceinline__ void pair_phase_c1(uint32_t tlane, int s, int r, const float2 *hi_s, float2 wr1,
                                              uint32_t peer_recv) {
    const bool own = (s >> 1) == KAPPA;
#pragma unroll 1
    for (int st = 0; st < 4; ++st) {
        const int i0 = (st & 1) + 4 * (st >> 1);
        const uint32_t col = step_col(s, i0);
        float2 v[2][8];
#pragma unroll
        for (int c = 0; c < 8; ++c) tmem_ld4(tlane + 64u * c + col, v[0][c], v[1][c]);
        tmem_wait_ld();
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int m = 8 * s + i0 + 2 * h;
            float2 w[8];  // W_N^b = W_N^r W_N^{128 m} (m < 32), then its powers
            pair_twiddles<KAPPA>(cmul(wr1, hi_s[m]), w);
#pragma unroll
            for (int c = KAPPA == 0 ? 1 : 0; c < 8; ++c) v[h][c] = cmulc(v[h][c], w[c]);
            dft<8, +1>(v[h]);
        }
        if (own) {
            // P_kappa[a', b] back into the slots the c' values came from
#pragma unroll
            for (int a = 0; a < 8; ++a) tmem_st4(tlane + 64u * a + col, v[0][a], v[1][a]);
        } else {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int m = 8 * s + i0 + 2 * h;
#pragma unroll
                for (int a = 0; a < 8; ++a) st_cluster(peer_recv + 8u * (uint32_t)recv_index(a, m, r), v[h][a]);
            }
        }
    }
    tmem_wait_st();
}

// Phase C2 of unit uc (when uc >= 0) fused with phase A of unit ua (when ua >= 0).  Thread
// (s, r) takes the 8 values of m = 16 rho + 4 s + i (rho = 0, 1; i < 4): for those in this
// CTA's range (rho = kappa) it first combines P_0 and P_1 and stores R (step 5), reading the
// slots (a', m) that it then overwrites with unit ua's values (c', m); the other range's slots
// were freed by phase C1.  Each m starts with unit ua's 16 loads, so their latency overlaps the
// combine and the stores.
template <bool REAL, int KAPPA>
__device__ __forceinline__ void pair_phase_c2a(const BlockParams &p, int64_t uc, void *yc, int64_t ua,
                                               const Chan &cha, uint32_t tlane, int s, int r,
                                               const float2 *hi_s, float2 wr1, const float2 *recv) {
    using Q = PairCfg<REAL>;
    constexpr int P = Q::P;
    // uc, ua: unit indices within their channels; yc: uc's channel's output, cha: ua's channel
    const int64_t sc = (REAL ? 2 * uc : uc) * p.L - (p.M - 1);  // output index of R[0] of unit uc
    const bool whole = sc + Q::N + (REAL ? p.L : 0) <= p.n;
    const int keep = p.M - 1;
    // outputs R[t] of unit uc with t < lim exist (t < N, so lim is capped to an int)
    const int lim = p.n - sc > (int64_t)Q::N + p.L ? Q::N + p.L : (int)(p.n - sc);
    const int64_t sa = (REAL ? 2 * ua : ua) * p.L - (p.M - 1);  // xt index of E[0] of unit ua
    const bool interior = sa >= 0 && sa + Q::N + (REAL ? p.L : 0) <= p.n;
#pragma unroll 1
    for (int q = 0; q < 8; ++q) {
        const int rho = (q < 4) ? KAPPA : 1 - KAPPA;
        const int m = 16 * rho + 4 * s + (q & 3);
        const int b = r + 128 * m;
        const uint32_t col = 2u * (uint32_t)(16 * (m & 1) + (m >> 1));  // slot (0, m); + 64 per a' or c'
        float2 x[16];
        if (ua >= 0) load_points<REAL, 16, P>(p, cha, sa + b, interior, x);
        if (q < 4 && uc >= 0) {
            float2 pown[8];
#pragma unroll
            for (int a = 0; a < 8; ++a) tmem_ld2(tlane + 64u * a + col, pown[a]);
            tmem_wait_ld();
#pragma unroll
            for (int a = 0; a < 8; ++a) {
                const float2 other = recv[recv_index(a, m, r)];
                const float2 p0 = KAPPA == 0 ? pown[a] : other;
                const float2 p1 = KAPPA == 0 ? other : pown[a];
                const float2 w = ctw_dyn<16, +1>(p1, a);  // W_16^{-a'} P_1
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const float2 val = h == 0 ? cadd(p0, w) : csub(p0, w);
                    const int t = P * (a + 8 * h) + b;
                    if (t < keep) continue;
                    // y[sc + b + P (a + 8 h)] at a constant offset from one pointer
                    if constexpr (REAL) {
                        float *yb = static_cast<float *>(yc) + sc + b;
                        if (whole || t < lim) st_cs(yb + P * (a + 8 * h), val.x);
                        if (whole || t + p.L < lim) st_cs(yb + p.L + P * (a + 8 * h), val.y);
                    } else {
                        float2 *yb = static_cast<float2 *>(yc) + sc + b;
                        if (whole || t < lim) st_cs(yb + P * (a + 8 * h), val);
                    }
                }
            }
        }
        if (ua >= 0) {
            float2 v[8];
            if constexpr (KAPPA == 0) {
#pragma unroll
                for (int a = 0; a < 8; ++a) v[a] = cadd(x[a], x[a + 8]);
            } else {
#pragma unroll
                for (int a = 0; a < 8; ++a) v[a] = ctw_dyn<16, -1>(csub(x[a], x[a + 8]), a);
            }
            dft<8, -1>(v);
            float2 w[8];
            pair_twiddles<KAPPA>(cmul(wr1, hi_s[m]), w);
#pragma unroll
            for (int c = KAPPA == 0 ? 1 : 0; c < 8; ++c) v[c] = cmul(v[c], w[c]);
#pragma unroll
            for (int c = 0; c < 8; ++c) tmem_st2(tlane + 64u * c + col, v[c]);
        }
    }
    if (ua >= 0) tmem_wait_st();
}

// The block loop of CTA KAPPA of a cluster (a copy per rank, so that every rank-dependent choice
// is made at compile time).
template <bool REAL, bool MULTI, int KAPPA, bool TC>
__device__ __forceinline__ void pair_loop(const BlockParams &p, int64_t u, int64_t uend, int tid, int warp, int s,
                                          int r, int g, int j, uint32_t tlane, const float2 *stw,
                                          const float2 *hi_s, float2 wr1, float2 *bufs, float2 *b0, float2 *b1,
                                          uint32_t peer_recv, const GroupBarrier<256> &gbar, TcCtx *tc,
                                          uint32_t *tcpar) {
    using Q = PairCfg<REAL>;
    int64_t lu = 0, lun = 0;
    int chu = u < uend ? channel_of<MULTI>(p, u, lu) : 0;  // unit u's channel
    if (u < uend)  // phase A of the first unit
        pair_phase_c2a<REAL, KAPPA>(p, -1, nullptr, lu, chan<REAL>(p, chu), tlane, s, r, hi_s, wr1, bufs);
    for (; u < uend; ++u) {
        tmem_fence_before_sync();
        __syncthreads();
        tmem_fence_after_sync();
        const int64_t un = u + 1;
        const int chn = un < uend ? channel_of<MULTI>(p, un, lun) : chu;
        if (un < uend && !p.no_bulk) prefetch_window<Q::N, REAL>(p, chan<REAL>(p, chn), lun, tid, KAPPA, 2);
        // (the folded 16-point DFT stage: C5 -2.4% measured)
        phase_b<8, false, true, 256, TC>(p, tlane, g, j, b0, b1, stw, gbar, KAPPA, 2,
                                         32u * (uint32_t)((warp >> 2) & 1), tc, tcpar);
        tmem_fence_before_sync();
        cluster_sync();  // both CTAs are past phase B (and past every read of S0)
        tmem_fence_after_sync();
        if (KAPPA == 0 && p.fuse_state && lu == 0) {
            // only the channel's unit 0 reads its S0 (fuse_state), and n >= M - 1: S0' = the
            // last M-1 samples of the channel's x
            using T_ = typename std::conditional<REAL, float, float2>::type;
            const Chan cu = chan<REAL>(p, chu);
            const T_ *x = static_cast<const T_ *>(cu.x);
            T_ *st = static_cast<T_ *>(cu.state);
            for (int t = tid; t < p.M - 1; t += Q::THREADS) st[t] = x[p.n - (p.M - 1) + t];
        }
        pair_phase_c1<REAL, KAPPA>(tlane, s, r, hi_s, wr1, peer_recv);
        tmem_fence_before_sync();
        cluster_sync();  // the other CTA's P values have landed in bufs
        tmem_fence_after_sync();
        pair_phase_c2a<REAL, KAPPA>(p, lu, chan<REAL>(p, chu).y, un < uend ? lun : -1, chan<REAL>(p, chn), tlane, s,
                                    r, hi_s, wr1, bufs);
        chu = chn;
        lu = lun;
    }
}

// TC: the 4096-point transforms' 16-point DFTs on the tensor cores (the optional engine)
template <bool REAL, bool MULTI, bool TC = false>
__global__ void __launch_bounds__(512, 1) fos_pair_kernel(const BlockParams p) {
    using Q = PairCfg<REAL>;
    extern __shared__ __align__(128) unsigned char smem[];
    const int tid = threadIdx.x;
    // the warp index broadcast from lane 0, so that the compiler knows it (and s, g, the Tensor
    // Memory addresses derived from it) to be the same in every lane of a warp
    const int warp = __shfl_sync(0xffffffffu, tid >> 5, 0);
    const int s = warp >> 2, r = tid & 127;  // phases A and C: s = tid / 128
    const int g = warp >> 3, j = tid & 255;  // phase B: g = tid / 256
    const uint32_t kappa = cluster_ctarank();
    uint32_t *tm_slot = reinterpret_cast<uint32_t *>(smem);
    float2 *stw = reinterpret_cast<float2 *>(smem + Q::OFF_TW);
    float2 *hi_s = reinterpret_cast<float2 *>(smem + Q::OFF_HI);
    float2 *wr_s = reinterpret_cast<float2 *>(smem + Q::OFF_WR);
    float2 *bufs = reinterpret_cast<float2 *>(smem + Q::OFF_BUF);
    float2 *b0 = bufs + g * 2 * Q::BUF;
    float2 *b1 = b0 + Q::BUF;
    const uint32_t peer_recv = map_rank(smem_addr(bufs), kappa ^ 1u);
    const GroupBarrier<256> gbar{1 + g};

    griddep_launch_dependents();  // the next call's kernel may start its own set-up
    // a contiguous range of units per cluster (at most one cluster per unit); both CTAs of a
    // cluster take the same units
    const int64_t ncl = nclusters_x();
    const int64_t u = (int64_t)cluster_id_x() * p.nunits / ncl;
    const int64_t uend = ((int64_t)cluster_id_x() + 1) * p.nunits / ncl;
    if (u < uend && !p.no_bulk) {  // a hint
        int64_t lu = 0;
        const int chu = channel_of<MULTI>(p, u, lu);
        prefetch_window<Q::N, REAL>(p, chan<REAL>(p, chu), lu, tid, (int)kappa, 2);
    }
    if (warp == 0) {
        tmem_alloc(tm_slot, Q::TM_COLS);
        tmem_relinquish();
    }
    for (int k = tid; k < Q::TL::SMEM_ENTRIES; k += Q::THREADS) stw[k] = p.tw[k];
    for (int k = tid; k < 32; k += Q::THREADS) hi_s[k] = p.twa[128 + k];
    for (int k = tid; k < 128; k += Q::THREADS) wr_s[k] = p.twa[k];
    uint64_t *tcbar = reinterpret_cast<uint64_t *>(smem + Q::OFF_TCBAR) + g;
    if constexpr (TC) {  // the split DFT matrices (read by the tensor cores) and the MMA barriers
        float2 *bt = reinterpret_cast<float2 *>(smem + Q::OFF_BTC);
        for (int k = tid; k < 4 * (int)kTcBTileBytes / 8; k += Q::THREADS) bt[k] = p.btc[k];
        fence_proxy_async_smem();
        if (j == 0) {
            mbar_init(tcbar, 1);
            fence_mbar_init();
        }
    }
    tmem_fence_before_sync();
    cluster_sync();  // both CTAs are running (and set up) before any remote store
    tmem_fence_after_sync();
    const uint32_t tlane = __shfl_sync(0xffffffffu, *tm_slot, 0) + ((uint32_t)(32 * (warp & 3)) << 16);
    TcCtx tc{};
    uint32_t tcpar = 0u;
    if constexpr (TC) {
        tc.a_base = smem_addr(b0);
        tc.b_base = smem_addr(smem + Q::OFF_BTC);
        tc.row_off = (uint32_t)(j >> 7) * 2u * kTcTileBytes + tc_offset(j & 127, 0);
        tc.mbar = tcbar;
        tc.err = p.err;
        tc.leader = j == 0;
    }
    const float2 wr1 = wr_s[r];  // W_N^r
    // the set-up read plan memory only; x, y and the state may belong to the previous kernel
    griddep_wait();

    if (kappa == 0)
        pair_loop<REAL, MULTI, 0, TC>(p, u, uend, tid, warp, s, r, g, j, tlane, stw, hi_s, wr1, bufs, b0, b1,
                                      peer_recv, gbar, &tc, &tcpar);
    else
        pair_loop<REAL, MULTI, 1, TC>(p, u, uend, tid, warp, s, r, g, j, tlane, stw, hi_s, wr1, bufs, b0, b1,
                                      peer_recv, gbar, &tc, &tcpar);

    tmem_fence_before_sync();
    __syncthreads();
    tmem_fence_after_sync();
    if (warp == 0) tmem_dealloc(*tm_slot, Q::TM_COLS);
}

template <bool REAL>
KernelEntry pair_entry() {
    using Q = PairCfg<REAL>;
    KernelEntry k;
    k.func = reinterpret_cast<const void *>(&fos_pair_kernel<REAL, false>);
    k.func_multi = reinterpret_cast<const void *>(&fos_pair_kernel<REAL, true>);
    k.func_tc = reinterpret_cast<const void *>(&fos_pair_kernel<REAL, false, true>);
    k.func_multi_tc = reinterpret_cast<const void *>(&fos_pair_kernel<REAL, true, true>);
    k.smem_tc = Q::SMEM_TC;
    k.threads = Q::THREADS;
    k.smem = Q::SMEM_BYTES;
    k.cluster = 2;
    k.units_per_cta = 1;
    k.groups = 1;
    k.fft_logn = 12;
    k.split_c = 16;
    k.state_from_x = 1;
    return k;
}

KernelEntry pair_kernel(int logn, bool real) {
    if (logn != 16) return KernelEntry{};
    return real ? pair_entry<true>() : pair_entry<false>();
}

}  // namespace fos
