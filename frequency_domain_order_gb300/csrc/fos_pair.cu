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
//   phase A   thread (s, r) owns b = r + 128 (8 s + i), i = 0..7: loads the 16 points of every
//             b, the radix-2 step for its kappa, the 8-point DFTs, the twiddles W_N^{bc}.
//   phase B   the P-point filtering of fos_resident.cuh for its 8 sub-transforms.
//   [cluster barrier: both CTAs are done with phase B, so each may write into the other's
//    exchange buffers]
//   phase C1  W_N^{-bc} and the 8-point inverse DFT over c' give P_kappa[a', b].  CTA kappa
//             finishes the outputs for b in [2048 kappa, 2048 kappa + 2048): rows s = 2 kappa,
//             2 kappa + 1 keep their P values in their lane, the other rows store theirs into
//             the other CTA's shared memory (128 KB, distributed shared memory).
//   [cluster barrier: the values have landed]
//   phase C2  all 512 threads combine P_0 and P_1 for the CTA's 2048 values of b (4 values of
//             m per thread) and store R[t] for t >= M - 1 (step 5).
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
    static constexpr int HI = N / 128;       // period of W_N^{128 m c} in m c
    static constexpr int THREADS = 512;
    static constexpr int TM_COLS = 512;
    using TL = TwLayout<12, 256>;
    static constexpr int BUF = xpad_len(P);
    static constexpr int OFF_TW = 128;
    static constexpr int OFF_HI = OFF_TW + 8 * TL::SMEM_ENTRIES;
    static constexpr int OFF_WR = OFF_HI + 8 * HI;
    static constexpr int OFF_BUF = (OFF_WR + 8 * 16 * 128 + 127) / 128 * 128;
    static constexpr int SMEM_BYTES = OFF_BUF + 2 * 2 * 8 * BUF;
    // phase C receive buffer (reuses the exchange buffers): P_other[a'][m mod 16][r]
    static constexpr int RECV_ELEMS = 8 * 16 * 128;
    static_assert(8 * RECV_ELEMS <= 2 * 2 * 8 * BUF, "receive buffer inside the exchange buffers");
};

__device__ __forceinline__ int recv_index(int a, int m, int r) { return (a * 16 + (m & 15)) * 128 + r; }

template <bool REAL>
__device__ __forceinline__ void pair_phase_a(const BlockParams &p, int64_t u, uint32_t kappa, uint32_t tlane,
                                             int s, int r, const float2 *hi_s, const float2 *wr_s) {
    using Q = PairCfg<REAL>;
    constexpr int P = Q::P, HI = Q::HI;
    const int64_t blk = REAL ? 2 * u : u;
    const int64_t start = blk * p.L - (p.M - 1);
    const bool interior = start >= 0 && start + Q::N + (REAL ? p.L : 0) <= p.n;
    float2 wr[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) wr[c] = wr_s[(kappa + 2 * c) * 128 + r];
#pragma unroll 1
    for (int st = 0; st < 4; ++st) {
        const int i0 = (st & 1) + 4 * (st >> 1);
        float2 v[2][8];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int b = r + 128 * (8 * s + i0 + 2 * h);
            float2 x[16];
#pragma unroll
            for (int a = 0; a < 16; ++a) x[a] = load_point<REAL>(p, start + P * a + b, interior);
            if (kappa == 0) {
#pragma unroll
                for (int a = 0; a < 8; ++a) v[h][a] = cadd(x[a], x[a + 8]);
            } else {
#pragma unroll
                for (int a = 0; a < 8; ++a) v[h][a] = ctw_dyn<16, -1>(csub(x[a], x[a + 8]), a);
            }
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int m = 8 * s + i0 + 2 * h;
            dft<8, -1>(v[h]);
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const int cc = (int)kappa + 2 * c;
                if (cc != 0) v[h][c] = cmul(v[h][c], cmul(wr[c], hi_s[(m * cc) & (HI - 1)]));
            }
        }
        const uint32_t col = step_col(s, i0);
#pragma unroll
        for (int c = 0; c < 8; ++c) tmem_st4(tlane + 64u * c + col, v[0][c], v[1][c]);
    }
    tmem_wait_st();
}

template <bool REAL>
__device__ __forceinline__ void pair_phase_c1(uint32_t kappa, uint32_t tlane, int s, int r, const float2 *hi_s,
                                              const float2 *wr_s, uint32_t peer_recv) {
    using Q = PairCfg<REAL>;
    constexpr int HI = Q::HI;
    const bool own = (uint32_t)(s >> 1) == kappa;
    float2 wr[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) wr[c] = wr_s[(kappa + 2 * c) * 128 + r];
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
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const int cc = (int)kappa + 2 * c;
                if (cc != 0) v[h][c] = cmulc(v[h][c], cmul(wr[c], hi_s[(m * cc) & (HI - 1)]));
            }
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

template <bool REAL>
__device__ __forceinline__ void pair_phase_c2(const BlockParams &p, int64_t u, uint32_t kappa, uint32_t tlane,
                                              int s, int r, const float2 *recv) {
    using Q = PairCfg<REAL>;
    constexpr int P = Q::P;
    const int64_t blk = REAL ? 2 * u : u;
    const int64_t start = blk * p.L - (p.M - 1);  // output index of R[0]
    const bool whole = start + Q::N + (REAL ? p.L : 0) <= p.n;
    const int keep = p.M - 1;
    // this thread: m = 16 kappa + 4 s + i, i = 0..3, taken as the slot pairs (i, i + 2)
#pragma unroll 1
    for (int i0 = 0; i0 < 2; ++i0) {
        const int m0 = 16 * (int)kappa + 4 * s + i0;  // and m0 + 2
        const uint32_t col = 2u * (uint32_t)(16 * (m0 & 1) + (m0 >> 1));
        float2 pown[2][8];
#pragma unroll
        for (int a = 0; a < 8; ++a) tmem_ld4(tlane + 64u * a + col, pown[0][a], pown[1][a]);
        tmem_wait_ld();
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
            const int m = m0 + 2 * h2;
            const int b = r + 128 * m;
#pragma unroll
            for (int a = 0; a < 8; ++a) {
                const float2 other = recv[recv_index(a, m, r)];
                const float2 p0 = kappa == 0 ? pown[h2][a] : other;
                const float2 p1 = kappa == 0 ? other : pown[h2][a];
                const float2 q = ctw_dyn<16, +1>(p1, a);  // W_16^{-a} P_1
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const float2 val = h == 0 ? cadd(p0, q) : csub(p0, q);
                    const int t = P * (a + 8 * h) + b;
                    if (t < keep) continue;
                    const int64_t o = start + t;
                    if constexpr (REAL) {
                        float *y = static_cast<float *>(p.y);
                        if (whole || o < p.n) st_cs(y + o, val.x);
                        if (whole || o + p.L < p.n) st_cs(y + o + p.L, val.y);
                    } else {
                        float2 *y = static_cast<float2 *>(p.y);
                        if (whole || o < p.n) st_cs(y + o, val);
                    }
                }
            }
        }
    }
}

template <bool REAL>
__global__ void __launch_bounds__(512, 1) fos_pair_kernel(const BlockParams p) {
    using Q = PairCfg<REAL>;
    extern __shared__ __align__(128) unsigned char smem[];
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int s = tid >> 7, r = tid & 127;
    const int g = tid >> 8, j = tid & 255;
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
    int64_t u = cluster_id_x();
    const int64_t ncl = nclusters_x();
    if (u < p.nunits && !p.no_bulk) prefetch_window<Q::N, REAL>(p, u, tid, (int)kappa, 2);  // a hint
    if (warp == 0) {
        tmem_alloc(tm_slot, Q::TM_COLS);
        tmem_relinquish();
    }
    for (int k = tid; k < Q::TL::SMEM_ENTRIES; k += Q::THREADS) stw[k] = p.tw[k];
    for (int k = tid; k < Q::HI; k += Q::THREADS) hi_s[k] = p.twa[16 * 128 + k];
    for (int k = tid; k < 16 * 128; k += Q::THREADS) wr_s[k] = p.twa[k];
    tmem_fence_before_sync();
    cluster_sync();  // both CTAs are running (and set up) before any remote store
    tmem_fence_after_sync();
    const uint32_t tlane = *tm_slot + ((uint32_t)(32 * (warp & 3)) << 16);
    // the set-up read plan memory only; x, y and the state may belong to the previous kernel
    griddep_wait();

    for (; u < p.nunits; u += ncl) {
        pair_phase_a<REAL>(p, u, kappa, tlane, s, r, hi_s, wr_s);
        tmem_fence_before_sync();
        __syncthreads();
        tmem_fence_after_sync();
        const int64_t un = u + ncl;
        if (un < p.nunits && !p.no_bulk) prefetch_window<Q::N, REAL>(p, un, tid, (int)kappa, 2);
        phase_b<8>(p, tlane, g, j, b0, b1, stw, gbar, (int)kappa, 2);
        tmem_fence_before_sync();
        cluster_sync();  // both CTAs are past phase B (and past every read of S0)
        tmem_fence_after_sync();
        if (p.fuse_state && u == 0 && kappa == 0) {
            // only unit 0 reads S0 (fuse_state), and n >= M - 1: S0' = the last M-1 samples of x
            using T_ = typename std::conditional<REAL, float, float2>::type;
            const T_ *x = static_cast<const T_ *>(p.x);
            T_ *st = static_cast<T_ *>(p.state);
            for (int t = tid; t < p.M - 1; t += Q::THREADS) st[t] = x[p.n - (p.M - 1) + t];
        }
        pair_phase_c1<REAL>(kappa, tlane, s, r, hi_s, wr_s, peer_recv);
        tmem_fence_before_sync();
        cluster_sync();  // the other CTA's P values have landed in bufs
        tmem_fence_after_sync();
        pair_phase_c2<REAL>(p, u, kappa, tlane, s, r, bufs);
    }

    tmem_fence_before_sync();
    __syncthreads();
    tmem_fence_after_sync();
    if (warp == 0) tmem_dealloc(*tm_slot, Q::TM_COLS);
}

template <bool REAL>
KernelEntry pair_entry() {
    using Q = PairCfg<REAL>;
    KernelEntry k;
    k.func = reinterpret_cast<const void *>(&fos_pair_kernel<REAL>);
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
