// fos_cluster.cu -- the fused overlap-save block kernel for N = 16384 .. 65536.
//
// An N-point block does not fit one CTA's shared memory (N = 32768 complex64 is 256 KB), so a
// thread-block cluster of C = N / 4096 CTAs (4, 8 or 16) filters one block at a time, the
// CTAs exchanging data through distributed shared memory.  Steps 3-5 of the claim in
// "一种基于GPU的高阶数字FIR滤波器频域并行处理实现方法" (zl.czvv.com/42398539.html, 主权项) are
// computed with the N = C x P (P = 4096) split of the DFT:
//
//   n = P a + b, k = c + C d:   X[c + C d] = sum_b W_P^{bd} [ W_N^{bc} sum_a x[P a + b] W_C^{ac} ]
//
//   phase A  CTA r owns b in [r Q, (r+1) Q), Q = P / C.  It gathers E[P a + b] for its b and
//            all a (C runs of Q contiguous samples; interior blocks by bulk copy, prefetched
//            during the previous block), does the C-point DFTs over a, multiplies by
//            W_N^{bc} and stores element (b, c) into CTA c's receive buffer at b.
//   phase B  CTA c now holds all P values for its c: a P-point FFT over b (fos_fft.cuh)
//            gives X[c + C d] in registers; multiply by H[c + C d] / N (registers); P-point
//            inverse FFT back to b; multiply by W_N^{-bc}; send element b to the CTA owning b.
//   phase C  CTA r holds, for its b, all C values: C-point inverse DFTs over c give
//            R[P a + b] for every a; outputs with P a + b >= M - 1 are stored (step 5).
//
// Two cluster barriers per block order the exchanges; they are the only cross-CTA waits and
// every CTA of a cluster passes through the same sequence of them.  Real input packs two
// blocks into one complex transform exactly as the single-CTA kernel does.
#include <type_traits>

#include "fos_fft.cuh"
#include "fos_kernels.h"

namespace fos {

template <int LOGN, bool REAL>
struct ClusterCfg {
    static constexpr int N = 1 << LOGN;
    static constexpr int LOGP = 12;
    static constexpr int P = 1 << LOGP;  // points per CTA
    static constexpr int C = N / P;       // CTAs per cluster
    static constexpr int T = P / 16;      // threads per CTA (256)
    static constexpr int Q = P / C;       // b values owned by one CTA
    static constexpr int QT = 16 / C;     // b values per thread
    static constexpr int SB = REAL ? 4 : 8;
    static constexpr int NSEG = REAL ? 2 * C : C;                 // gather runs per block
    static constexpr int SEG_BYTES = (Q * SB + 32 + 15) / 16 * 16;  // one run + 16-byte rounding
    static constexpr int STG_BYTES = (NSEG * SEG_BYTES + 127) / 128 * 128;
    static constexpr int RECV1_BYTES = (8 * xpad_len(P) + 127) / 128 * 128;  // phase B buffer
    static constexpr int RECV2_BYTES = 8 * P;                                  // phase C buffer
    static constexpr int SMEM_BYTES = 128 + RECV1_BYTES + RECV2_BYTES + STG_BYTES;
    static_assert(C >= 2 && C <= 16, "cluster of 2..16 CTAs");
};

// Gather the C runs (2C for real data) of block-or-pair `u` that CTA `rank` needs.  Returns
// the element offsets of the runs inside their staging slots (run a of the first block at
// a * SEG_BYTES + offA, of the second block of a real pair at (C + a) * SEG_BYTES + offB).
template <int LOGN, bool REAL>
__device__ __forceinline__ void cluster_stage(const BlockParams &p, int64_t u, uint32_t rank, unsigned char *stg,
                                              uint64_t *bar, bool allow_tma, bool &used_tma, int &offA,
                                              int &offB) {
    using C_ = ClusterCfg<LOGN, REAL>;
    constexpr int SB = C_::SB, C = C_::C, P = C_::P, Q = C_::Q;
    const int64_t s = u * (int64_t)p.L * (REAL ? 2 : 1) - (p.M - 1) + (int64_t)rank * Q;  // run 0 start
    const int nb = REAL ? 2 : 1;
    if (allow_tma && s >= 0) {
        const uintptr_t xb = reinterpret_cast<uintptr_t>(p.x);
        const uintptr_t xe = xb + (uintptr_t)p.n * SB;
        const uintptr_t a0A = xb + (uintptr_t)s * SB;
        const uintptr_t a0B = a0A + (uintptr_t)p.L * SB;
        const uintptr_t b0A = a0A & ~uintptr_t(15);
        const uintptr_t b0B = a0B & ~uintptr_t(15);
        const uint32_t bytesA = (uint32_t)(((a0A + Q * SB + 15) & ~uintptr_t(15)) - b0A);
        const uint32_t bytesB = (uint32_t)(((a0B + Q * SB + 15) & ~uintptr_t(15)) - b0B);
        const uintptr_t lastEnd = (nb == 2 ? b0B + bytesB : b0A + bytesA) + (uintptr_t)(C - 1) * P * SB;
        if (b0A >= xb && lastEnd <= xe) {
            if (threadIdx.x == 0) {
                fence_proxy_async_smem();
                mbar_arrive_expect_tx(bar, (uint32_t)C * (bytesA + (nb == 2 ? bytesB : 0u)));
#pragma unroll 1
                for (int a = 0; a < C; ++a) {
                    bulk_g2s(stg + a * C_::SEG_BYTES, reinterpret_cast<const void *>(b0A + (uintptr_t)a * P * SB),
                             bytesA, bar);
                    if (nb == 2)
                        bulk_g2s(stg + (C + a) * C_::SEG_BYTES,
                                 reinterpret_cast<const void *>(b0B + (uintptr_t)a * P * SB), bytesB, bar);
                }
            }
            used_tma = true;
            offA = (int)((a0A - b0A) / SB);
            offB = (int)((a0B - b0B) / SB);
            return;
        }
    }
    used_tma = false;
    offA = 0;
    offB = 0;
    const int64_t hist = p.M - 1;
    using T_ = typename std::conditional<REAL, float, float2>::type;
    const T_ *x = static_cast<const T_ *>(p.x);
    const T_ *s0 = static_cast<const T_ *>(p.state);
    // batches of independent loads, so their latencies overlap instead of adding up
    constexpr int U = 8;
    for (int i0 = threadIdx.x; i0 < nb * C * Q; i0 += U * C_::T) {
        T_ v[U];
#pragma unroll
        for (int q = 0; q < U; ++q) {
            const int i = i0 + q * C_::T;
            const int run = i / Q, k = i % Q;  // run = blockhalf * C + a
            const int a = run % C, half = run / C;
            const int64_t t = s + (int64_t)half * p.L + (int64_t)a * P + k;
            v[q] = T_{};
            if (i < nb * C * Q) {
                if (t >= 0) {
                    if (t < p.n) v[q] = x[t];
                } else if (t >= -hist) {
                    v[q] = s0[hist + t];
                }
            }
        }
#pragma unroll
        for (int q = 0; q < U; ++q) {
            const int i = i0 + q * C_::T;
            if (i < nb * C * Q) reinterpret_cast<T_ *>(stg + (i / Q) * C_::SEG_BYTES)[i % Q] = v[q];
        }
    }
    __syncthreads();
}

template <int LOGN, bool REAL>
__global__ void __launch_bounds__(256, 2) fos_cluster_kernel(const BlockParams p) {
    using C_ = ClusterCfg<LOGN, REAL>;
    constexpr int C = C_::C, P = C_::P, T = C_::T, Q = C_::Q, QT = C_::QT;
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem);
    float2 *recv1 = reinterpret_cast<float2 *>(smem + 128);
    float2 *recv2 = reinterpret_cast<float2 *>(smem + 128 + C_::RECV1_BYTES);
    unsigned char *stg = smem + 128 + C_::RECV1_BYTES + C_::RECV2_BYTES;

    const int j = threadIdx.x;
    const uint32_t rank = cluster_ctarank();
    const int64_t cid = cluster_id_x();
    const int64_t ncl = nclusters_x();

    if (j == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    // H[rank + C (j + e T)] / N: the bins this CTA multiplies in phase B
    float2 hreg[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) hreg[e] = __ldg(p.H + rank + C * (j + e * T));
    const uint32_t recv1_base = smem_addr(recv1);
    const uint32_t recv2_base = smem_addr(recv2);
    cluster_sync();  // every CTA of the cluster is running before any remote store

    uint32_t parity = 0u;
    bool used = false, allow_tma = !p.no_bulk;  // bulk copies read device memory only
    int offA = 0, offB = 0;
    int64_t u = cid;
    if (u < p.nunits) cluster_stage<LOGN, REAL>(p, u, rank, stg, bar, allow_tma, used, offA, offB);

    for (; u < p.nunits; u += ncl) {
        if (used) {
            const bool ok = mbar_wait_bounded(bar, parity);
            parity ^= 1u;
            if (__syncthreads_or(!ok)) {
                if (j == 0) atomicExch(p.err, 1);
                allow_tma = false;
                cluster_stage<LOGN, REAL>(p, u, rank, stg, bar, false, used, offA, offB);
            }
        }
        // ---- phase A: runs -> registers, C-point DFTs over a, twiddle, scatter to CTA c
        float2 v[16];
#pragma unroll
        for (int q = 0; q < QT; ++q) {
#pragma unroll
            for (int a = 0; a < C; ++a) {
                const int k = j + q * T;
                if constexpr (REAL) {
                    const float *ra = reinterpret_cast<const float *>(stg + a * C_::SEG_BYTES) + offA;
                    const float *rb = reinterpret_cast<const float *>(stg + (C + a) * C_::SEG_BYTES) + offB;
                    v[q * C + a] = make_float2(ra[k], rb[k]);
                } else {
                    v[q * C + a] = reinterpret_cast<const float2 *>(stg + a * C_::SEG_BYTES)[offA + k];
                }
            }
        }
#pragma unroll
        for (int q = 0; q < QT; ++q) {
            dft<C, -1>(&v[q * C]);
            const int b = (int)rank * Q + j + q * T;
#pragma unroll
            for (int c = 1; c < C; ++c) v[q * C + c] = cmul(v[q * C + c], __ldg(p.twa + c * P + b));
#pragma unroll
            for (int c = 0; c < C; ++c) st_cluster(map_rank(recv1_base, c) + 8u * xpad(b), v[q * C + c]);
        }
        cluster_sync();  // phase A data has landed everywhere; the staging runs are consumed
        // the staging runs are consumed: fetch the next block's runs now, by bulk copy during
        // phases B and C, or (blocks that touch S0 or the end of x) with plain loads here
        if (u + ncl < p.nunits) cluster_stage<LOGN, REAL>(p, u + ncl, rank, stg, bar, allow_tma, used, offA, offB);
        if (p.fuse_state && u == 0 && rank == 0) {
            // every read of S0 (block 0's gather, all CTAs of this cluster) happened before
            // the barrier above; S0' = the last M-1 input samples (n >= M-1 here)
            using T_ = typename std::conditional<REAL, float, float2>::type;
            const T_ *x = static_cast<const T_ *>(p.x);
            T_ *st = static_cast<T_ *>(p.state);
            for (int t = j; t < p.M - 1; t += T) st[t] = x[p.n - (p.M - 1) + t];
        }

        // ---- phase B: P-point FFT over b, multiply by H, inverse FFT, twiddle, scatter back
#pragma unroll
        for (int e = 0; e < 16; ++e) v[e] = recv1[xpad(j + e * T)];
        fft_regs<C_::LOGP, -1>(v, recv1, p.tw, j, true);
#pragma unroll
        for (int e = 0; e < 16; ++e) v[e] = cmul(v[e], hreg[e]);
        fft_regs<C_::LOGP, +1>(v, recv1, p.tw, j, true);
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            const int b = j + e * T;
            v[e] = cmulc(v[e], __ldg(p.twa + (int)rank * P + b));
            const uint32_t owner = (uint32_t)(b / Q);
            st_cluster(map_rank(recv2_base, owner) + 8u * (uint32_t)(rank * Q + (b - (int)owner * Q)), v[e]);
        }
        cluster_sync();  // phase B data has landed

        // ---- phase C: C-point inverse DFTs over c, discard, store
#pragma unroll
        for (int q = 0; q < QT; ++q) {
#pragma unroll
            for (int c = 0; c < C; ++c) v[q * C + c] = recv2[c * Q + j + q * T];
            dft<C, +1>(&v[q * C]);
        }
        const int64_t blk = REAL ? 2 * u : u;
        const int64_t obase = blk * p.L - (p.M - 1);
#pragma unroll
        for (int q = 0; q < QT; ++q) {
#pragma unroll
            for (int a = 0; a < C; ++a) {
                const int t = a * P + (int)rank * Q + j + q * T;
                if (t >= p.M - 1) {
                    const int64_t o = obase + t;
                    if constexpr (REAL) {
                        float *y = static_cast<float *>(p.y);
                        if (o < p.n) st_cs(y + o, v[q * C + a].x);
                        if (o + p.L < p.n) st_cs(y + o + p.L, v[q * C + a].y);
                    } else {
                        float2 *y = static_cast<float2 *>(p.y);
                        if (o < p.n) st_cs(y + o, v[q * C + a]);
                    }
                }
            }
        }
    }
}

template <int LOGN, bool REAL>
KernelEntry cluster_entry() {
    using C_ = ClusterCfg<LOGN, REAL>;
    KernelEntry k;
    k.func = reinterpret_cast<const void *>(&fos_cluster_kernel<LOGN, REAL>);
    k.threads = C_::T;
    k.smem = C_::SMEM_BYTES;
    k.cluster = C_::C;
    k.units_per_cta = 1;
    k.fft_logn = C_::LOGP;
    return k;
}

KernelEntry cluster_kernel(int logn, bool real) {
    switch (logn) {
        case 14: return real ? cluster_entry<14, true>() : cluster_entry<14, false>();
        case 15: return real ? cluster_entry<15, true>() : cluster_entry<15, false>();
        case 16: return real ? cluster_entry<16, true>() : cluster_entry<16, false>();
        default: return KernelEntry{};
    }
}

}  // namespace fos
