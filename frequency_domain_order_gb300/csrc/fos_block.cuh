// fos_block.cuh -- the fused overlap-save block kernel for N <= 8192 (one CTA per block group).
//
// One launch performs steps 3, 4 and 5 of the claim in "一种基于GPU的高阶数字FIR滤波器
// 频域并行处理实现方法" (zl.czvv.com/42398539.html, 主权项) for every block of one call, and
// the state carry of step 3:
//   gather   E_i = xt[i L - (M-1) .. i L - (M-1) + N) into shared memory.  Interior
//            groups of blocks arrive by one bulk (TMA) copy issued while the previous group
//            is being transformed (double-buffered); for groups that touch the state S0 or run
//            past the input, the part inside x comes by bulk copy and the rest (S0 in front,
//            the ragged ends, zeros behind) by plain loads.  The wait for a copy is bounded
//            (BlockParams::wait_ns); a copy that misses it sets the error word, the group waits
//            (bounded again) for that copy to land and then gathers with plain loads only.
//   FFT      F_i = FFT_N(E_i) in registers and two alternating exchange buffers
//   multiply I_i = F_i * H
//   IFFT     R_i = IFFT_N(I_i), natural order in registers
//   discard  Y_i = R_i[M-1 .. M-1+L) stored straight from registers, masked to n outputs
//   state    the CTA holding block 0 writes S0' = last M-1 samples of concat(S0, x)
//            after it has read S0 (no other CTA reads S0 when fuse_state is set)
// Real input packs two consecutive blocks into one complex transform (E_{2p} as real part,
// E_{2p+1} as imaginary part); with a real h the two outputs come back as the real and
// imaginary parts of R.
//
// Per-thread constants -- the 16 bins of H / N a thread multiplies and the twiddles of its
// passes -- are written once into Tensor Memory (this thread's lane) and read back with
// tcgen05.ld for every block, keeping them off the shared-memory / L1 path that carries the
// exchanges.  A call of less than one wave (each group one unit at most) runs the SMC variant
// instead (N <= 1024): the tables sit in shared memory beside the buffers, one coalesced copy
// per CTA, which takes the Tensor Memory set-up off the call's critical path.  Each group's
// shared memory holds three buffers: two staging windows (the one being filtered and the one
// being fetched) and one exchange buffer; the window being filtered doubles as the second
// exchange buffer once it has been read.
//
// A CTA that allocates Tensor Memory runs alone on its SM, so a CTA has 512 threads split
// into independent groups of max(64, N/16) threads (eight groups for N <= 1024, two for
// N = 4096, one for N = 8192), each with its own three buffers, mbarriers and hardware barrier,
// sharing only the Tensor Memory allocation.  Grid: persistent, one CTA per SM; a call of
// fewer units than groups deals them across CTAs first, a longer one gives each CTA a
// contiguous range of units that its groups take in turn.  A work unit is F consecutive blocks
// (complex) or F consecutive block pairs (real), F = max(1, 64 / (N/16)), each handled by N/16
// threads: small transforms spread over as many groups as possible, so that a call of few
// blocks finishes in the time of one unit.
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
    static constexpr int F = T >= 64 ? 1 : 64 / T;
    static constexpr int GT = F * T;              // threads of one group: max(64, N / 16)
    static constexpr int GROUPS = 512 / GT;       // independent groups per CTA (8 .. 1)
    static_assert(GT % 32 == 0, "whole warps per group");
    static constexpr int THREADS = 512;
    static constexpr int SB = REAL ? 4 : 8;  // bytes per sample
    // F blocks' gather windows (complex: (F-1)L + N samples; real: (2F-1)L + N floats) fit in
    // 8 F N bytes; +32 covers rounding the bulk copy out to 16-byte boundaries at both ends.
    // The same buffer then serves as the F padded exchange buffers (8 F xpad_len(N) bytes).
    static constexpr int EX_BYTES = 8 * F * xpad_len(N);
    static constexpr int BUF_BYTES = (((8 * F * N + 32) > EX_BYTES ? (8 * F * N + 32) : EX_BYTES) + 127) / 128 * 128;
    static constexpr int HDR_BYTES = 256;  // Tensor Memory address at 0, group g's mbarriers at 16 + 16 g
    static constexpr int SMEM_BYTES = HDR_BYTES + GROUPS * 3 * BUF_BYTES;
    static_assert(16 + 16 * GROUPS <= HDR_BYTES, "header");
    static_assert(GROUPS <= 15, "one hardware barrier id per group");
    static constexpr int MIN_BLOCKS = 1;  // a CTA that allocates Tensor Memory runs alone on its SM
    // Tensor Memory: per thread 32 columns of H bins + 32 per twiddled pass; warps w, w+4, ...
    // share a lane range and take consecutive column ranges.
    static constexpr int TM_COLS_THREAD = TwLayout<LOGN, 0>::TMEM_COLS;  // = 32 NPASS
    static constexpr int TM_SLOTS = THREADS / 128;
    static constexpr int TM_NEED = TM_COLS_THREAD * TM_SLOTS;
    static constexpr int TM_COLS =
        TM_NEED <= 32 ? 32 : TM_NEED <= 64 ? 64 : TM_NEED <= 128 ? 128 : TM_NEED <= 256 ? 256 : 512;
    static_assert(TM_NEED <= 512, "tensor memory columns");
    static_assert(THREADS % 128 == 0, "whole warp quarters");
    // the variant for calls of less than one wave keeps H / N and the pass twiddles in shared
    // memory after the buffers (no Tensor Memory): for N <= 1024 they fit beside them
    static constexpr int SMC_BYTES = 8 * (N + S::TW_ENTRIES);
    static constexpr bool HAS_SMC = SMEM_BYTES + SMC_BYTES <= 227 * 1024;
    // the tensor-core variant (N = 4096): the four 4 KB DFT-matrix tiles after the header, then
    // per group [staging 0][exchange][staging 1], so that the exchange buffer and whichever
    // staging window is being filtered are adjacent: the group's 64 KB of A tiles span the two
    static constexpr bool HAS_TC = (LOGN == 12);
    static constexpr int TC_B_OFF = HDR_BYTES;
    static constexpr int TC_GROUP_OFF = HDR_BYTES + 4 * (int)kTcBTileBytes;
    static constexpr int SMEM_TC = TC_GROUP_OFF + GROUPS * 3 * BUF_BYTES;
    static_assert(!HAS_TC || (2 * BUF_BYTES >= 4 * (int)kTcTileBytes && T == 256 && F == 1 &&
                              TM_NEED <= 384 && TM_COLS == 512 && SMEM_TC <= 227 * 1024 &&
                              16 + 24 * GROUPS <= HDR_BYTES),
                  "tensor-core variant layout");
    using Bar = GroupBarrier<GT>;
};

// dst[0 .. n) = src[0 .. n) by the `threads` threads of the CTA, 16 bytes per load (plan tables
// are 16-byte aligned), every load of a thread issued before its stores.
__device__ __forceinline__ void copy_table(const float2 *src, float2 *dst, int n, int tid, int threads) {
    const int n4 = n / 2;
    const float4 *s4 = reinterpret_cast<const float4 *>(src);
    float4 *d4 = reinterpret_cast<float4 *>(dst);
    for (int i0 = tid; i0 < n4; i0 += 4 * threads) {
        float4 t[4];
#pragma unroll
        for (int q = 0; q < 4; ++q)
            if (i0 + q * threads < n4) t[q] = __ldg(s4 + i0 + q * threads);
#pragma unroll
        for (int q = 0; q < 4; ++q)
            if (i0 + q * threads < n4) d4[i0 + q * threads] = t[q];
    }
    if ((n & 1) && tid == 0) dst[n - 1] = __ldg(src + n - 1);
}

// Gather the input window of work unit u into `buf`.  Returns the element offset of
// xt[start] inside the buffer.  A bulk copy is used (issued by thread 0, completing on
// `bar`; used_tma = true) when the 16-byte-rounded byte range lies inside x; otherwise every
// thread gathers with plain loads and the CTA synchronises (used_tma = false).
template <int LOGN, bool REAL>
__device__ __forceinline__ int stage_unit(const BlockParams &p, const Chan &ch, int64_t u, unsigned char *buf,
                                          uint64_t *bar,
                                          bool allow_tma, bool &used_tma, int tid,
                                          const typename BlockCfg<LOGN, REAL>::Bar &gbar) {
    using C = BlockCfg<LOGN, REAL>;
    constexpr int SB = C::SB;
    const int64_t span = (int64_t)C::F * p.L * (REAL ? 2 : 1);
    const int64_t start = u * span - (p.M - 1);
    const int64_t len = (int64_t)(REAL ? 2 * C::F - 1 : C::F - 1) * p.L + C::N;
    const uintptr_t xb = reinterpret_cast<uintptr_t>(ch.x);
    if (allow_tma && start >= 0) {
        const uintptr_t a0 = xb + (uintptr_t)start * SB, a1 = a0 + (uintptr_t)len * SB;
        const uintptr_t b0 = a0 & ~uintptr_t(15), b1 = (a1 + 15) & ~uintptr_t(15);
        if (b0 >= xb && b1 <= xb + (uintptr_t)p.n * SB) {
            if (tid == 0) {
                fence_proxy_async_smem();
                mbar_arrive_expect_tx(bar, (uint32_t)(b1 - b0));
                bulk_g2s(buf, reinterpret_cast<const void *>(b0), (uint32_t)(b1 - b0), bar);
            }
            used_tma = true;
            return (int)((a0 - b0) / SB);
        }
    }
    using T_ = typename std::conditional<REAL, float, float2>::type;
    const T_ *x = static_cast<const T_ *>(ch.x);
    const T_ *s0 = static_cast<const T_ *>(ch.state);
    const int64_t hist = p.M - 1;
    if (allow_tma) {
        // a window that reaches the state or the end of x: the part inside x, rounded inwards to
        // 16 bytes, by one bulk copy, placed so that its buffer address is 16-byte aligned;
        // the rest (state samples, at most three samples at either end of that part, zeros
        // past x) by plain loads of the group
        const int64_t xs = start > 0 ? start : 0, xe = start + len < p.n ? start + len : p.n;
        const uintptr_t c0 = (xb + (uintptr_t)xs * SB + 15) & ~uintptr_t(15);
        const uintptr_t c1 = (xb + (uintptr_t)xe * SB) & ~uintptr_t(15);
        if (xe > xs && c1 > c0) {
            const int64_t i0 = (int64_t)((c0 - xb) / SB) - start;  // window index of the copy's first sample
            const int64_t i1 = (int64_t)((c1 - xb) / SB) - start;
            const int off = (int)((16 - (i0 * SB) % 16) % 16) / SB;  // buffer index of window index 0
            if (tid == 0) {
                fence_proxy_async_smem();
                mbar_arrive_expect_tx(bar, (uint32_t)(c1 - c0));
                bulk_g2s(buf + (off + i0) * SB, reinterpret_cast<const void *>(c0), (uint32_t)(c1 - c0), bar);
            }
            T_ *dst = reinterpret_cast<T_ *>(buf) + off;
            for (int h = 0; h < 2; ++h) {  // window indices [0, i0), then [i1, len)
                for (int64_t i = (h ? i1 : 0) + tid; i < (h ? len : i0); i += C::GT) {
                    const int64_t t = start + i;
                    T_ v{};
                    if (t >= 0) {
                        if (t < p.n) v = x[t];
                    } else if (t >= -hist) {
                        v = s0[hist + t];
                    }
                    dst[i] = v;
                }
            }
            gbar.sync();
            used_tma = true;
            return off;
        }
    }
    used_tma = false;
    T_ *dst = reinterpret_cast<T_ *>(buf);
    // batches of independent loads, so their latencies overlap instead of adding up
    constexpr int U = 8;
    for (int64_t i0 = tid; i0 < len; i0 += (int64_t)U * C::GT) {
        T_ v[U];
#pragma unroll
        for (int q = 0; q < U; ++q) {
            const int64_t t = start + i0 + (int64_t)q * C::GT;
            v[q] = T_{};
            if (t >= 0) {
                if (t < p.n) v[q] = x[t];
            } else if (t >= -hist) {
                v[q] = s0[hist + t];
            }
        }
#pragma unroll
        for (int q = 0; q < U; ++q) {
            const int64_t i = i0 + (int64_t)q * C::GT;
            if (i < len) dst[i] = v[q];
        }
    }
    gbar.sync();
    return 0;
}

// Prefetch into L2 the part of unit u's window that lies in x (rounded inwards to 16 bytes),
// one instruction issued by thread 0 of the group (issuing costs time; the window is small).
// A prefetch makes nothing visible to this kernel, so it may run before the wait for the
// kernel before it: the later gather still reads whatever that kernel wrote.
template <int LOGN, bool REAL>
__device__ __forceinline__ void prefetch_unit(const BlockParams &p, const Chan &ch, int64_t u, int tid) {
    using C = BlockCfg<LOGN, REAL>;
    constexpr int SB = C::SB;
    if (tid != 0) return;
    const int64_t span = (int64_t)C::F * p.L * (REAL ? 2 : 1);
    int64_t lo = u * span - (p.M - 1);
    int64_t hi = lo + (int64_t)(REAL ? 2 * C::F - 1 : C::F - 1) * p.L + C::N;
    if (lo < 0) lo = 0;
    if (hi > p.n) hi = p.n;
    if (hi <= lo) return;
    const uintptr_t xb = reinterpret_cast<uintptr_t>(ch.x);
    const uintptr_t a0 = (xb + (uintptr_t)lo * SB + 15) & ~uintptr_t(15);
    const uintptr_t a1 = (xb + (uintptr_t)hi * SB) & ~uintptr_t(15);
    if (a1 <= a0) return;
    prefetch_l2_bulk(reinterpret_cast<const void *>(a0), (uint32_t)(a1 - a0));
}

// S0' = xt[n-(M-1) .. n): samples of x, or (when n < M-1) of S0, which the gather of unit 0
// left at buffer index off + (t + M - 1) for xt[t], t < 0.
template <int LOGN, bool REAL>
__device__ __forceinline__ void write_state(const BlockParams &p, const Chan &ch, const unsigned char *buf,
                                            int off, int tid) {
    using C = BlockCfg<LOGN, REAL>;
    using T_ = typename std::conditional<REAL, float, float2>::type;
    const T_ *x = static_cast<const T_ *>(ch.x);
    const T_ *stg = reinterpret_cast<const T_ *>(buf) + off;
    T_ *st = static_cast<T_ *>(ch.state);
    const int hist = p.M - 1;
    constexpr int U = 8;  // independent loads in flight per thread
    for (int t0 = tid; t0 < hist; t0 += U * C::GT) {
        T_ v[U];
#pragma unroll
        for (int q = 0; q < U; ++q) {
            const int t = t0 + q * C::GT;
            const int64_t src = p.n - hist + t;
            v[q] = T_{};
            if (t < hist) v[q] = src >= 0 ? x[src] : stg[src + hist];
        }
#pragma unroll
        for (int q = 0; q < U; ++q)
            if (t0 + q * C::GT < hist) st[t0 + q * C::GT] = v[q];
    }
}

// SMC: H / N and the twiddles in shared memory instead of Tensor Memory (calls of less than one
// wave, where the per-thread Tensor Memory set-up is on every call's critical path)
// TC: the 16-point DFTs of every pass on the tensor cores (N = 4096 only; fos_tc.cuh)
template <int LOGN, bool REAL, bool SMC, bool TC = false>
__global__ void __launch_bounds__(BlockCfg<LOGN, REAL>::THREADS, BlockCfg<LOGN, REAL>::MIN_BLOCKS)
    fos_block_kernel(const BlockParams p) {
    using C = BlockCfg<LOGN, REAL>;
    using S = typename C::S;
    constexpr int T = C::T;
    extern __shared__ __align__(128) unsigned char smem[];
    const int tid = threadIdx.x;
    // the warp index broadcast from lane 0, so that the compiler knows it (and the group, the
    // Tensor Memory addresses derived from it) to be the same in every lane of a warp
    const int warp = __shfl_sync(0xffffffffu, tid >> 5, 0);
    const int g = warp / (C::GT / 32);  // group within the CTA (GT is a multiple of 64)
    const int tg = tid % C::GT;     // thread within the group
    const int f = tg / T;           // transform slot within the group
    const int j = tg % T;           // thread within the transform
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + 16) + 2 * g;
    uint32_t *tm_base_slot = reinterpret_cast<uint32_t *>(smem);
    unsigned char *gbase = smem + (TC ? C::TC_GROUP_OFF : C::HDR_BYTES) + g * 3 * C::BUF_BYTES;
    // exchange buffer and the two staging windows (the tensor-core variant puts the exchange
    // buffer between the windows)
    float2 *xbuf = reinterpret_cast<float2 *>(gbase + (TC ? C::BUF_BYTES : 0));
    unsigned char *stg0 = gbase + (TC ? 0 : C::BUF_BYTES);
    unsigned char *stg1 = gbase + 2 * C::BUF_BYTES;
    uint64_t *tcbar = reinterpret_cast<uint64_t *>(smem + 16 + 16 * C::GROUPS) + g;  // TC: MMA completion
    const typename C::Bar gbar{1 + g};

    griddep_launch_dependents();  // the next call's kernel may start its own set-up
    if (!SMC && warp == 0) {
        tmem_alloc(tm_base_slot, C::TM_COLS);
        tmem_relinquish();
    }
    if (tg == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        if (TC) mbar_init(tcbar, 1);
        fence_mbar_init();
    }
    if constexpr (TC) {  // the split DFT matrices, read by the tensor cores (async proxy)
        copy_table(p.btc, reinterpret_cast<float2 *>(smem + C::TC_B_OFF), 4 * (int)kTcBTileBytes / 8, tid,
                   C::THREADS);
        fence_proxy_async_smem();
    }
    tmem_fence_before_sync();
    __syncthreads();
    tmem_fence_after_sync();
    // double buffering: `cur` holds the unit being filtered, `nxt` the one being fetched
    unsigned char *cur = stg0, *nxt = stg1;
    uint64_t *bcur = &bars[0], *bnxt = &bars[1];
    uint32_t pcur = 0u, pnxt = 0u;  // mbarrier phase parity to wait for
    bool ucur = false, unxt = false;  // filled by a bulk copy (else by plain loads)
    int ocur = 0, onxt = 0;           // element offset of the window in the buffer
    bool allow_tma = !p.no_bulk;  // bulk copies read device memory only

    // the groups of all CTAs take work units round-robin; a call of fewer units than groups
    // deals them across CTAs first, so that they spread over every CTA the launch has
    const int64_t stride = (int64_t)gridDim.x * C::GROUPS;
    int64_t u, ustep, uend;
    if (p.nunits < stride) {  // at most one unit per group, dealt across CTAs first
        u = (int64_t)g * gridDim.x + blockIdx.x;
        ustep = stride;
        uend = p.nunits;
    } else {  // a contiguous range of units per CTA, its groups taking them in turn
        u = blockIdx.x * p.nunits / gridDim.x + g;
        ustep = C::GROUPS;
        uend = (blockIdx.x + 1) * p.nunits / gridDim.x;
    }

    // this thread's TMEM columns: lane 32 (warp % 4) + (tid % 32), columns from slot * 32 NPASS
    const uint32_t tm0 = SMC ? 0u : __shfl_sync(0xffffffffu, *tm_base_slot, 0);
    const uint32_t tma = SMC ? 0u : tm0 + ((uint32_t)(32 * (warp & 3)) << 16) + (uint32_t)((warp >> 2) * C::TM_COLS_THREAD);
    // TC: the group's two 128-row accumulators in columns 384 + 64 g (+ 32); thread j's row is
    // j mod 128 of tile j / 128, which is its own lane
    TcCtx tc{};
    uint32_t tcpar = 0u;
    if constexpr (TC) {
        tc.b_base = smem_addr(smem + C::TC_B_OFF);
        tc.d_tile = tm0 + 384u + 64u * (uint32_t)g;
        tc.d_row = tm0 + ((uint32_t)(32 * (warp & 3)) << 16) + 384u + 64u * (uint32_t)g + 32u * (uint32_t)(j >> 7);
        tc.row_off = (uint32_t)(j >> 7) * 2u * kTcTileBytes + tc_offset(j & 127, 0);
        tc.mbar = tcbar;
        tc.err = p.err;
        tc.leader = tg == 0;
    }
    float2 *cH = reinterpret_cast<float2 *>(smem + C::SMEM_BYTES);  // SMC: H / N, then the twiddles
    float2 *cT = cH + C::N;
    if constexpr (SMC) {
        copy_table(p.H, cH, C::N, tid, C::THREADS);
        copy_table(p.tw, cT, S::TW_ENTRIES, tid, C::THREADS);
        __syncthreads();
    } else {
        // H[j + e T] / N for e = 0..15, then the twiddles W_{16 Ns}^{(j mod Ns) r} of each pass;
        // every load is issued before the first store into TMEM
        float w[S::NPASS][32];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            const float2 z = __ldg(p.H + j + e * T);
            w[0][2 * e] = z.x;
            w[0][2 * e + 1] = z.y;
        }
#pragma unroll
        for (int q = 1; q < S::NPASS; ++q) {
            const int Ns = S::ns(q);
            const float2 *tw = p.tw + S::twoff(q) + (j & (Ns - 1));
#pragma unroll
            for (int r = 1; r < 16; ++r) {
                const float2 z = __ldg(tw + (r - 1) * Ns);
                w[q][2 * r - 2] = z.x;
                w[q][2 * r - 1] = z.y;
            }
            w[q][30] = 0.f;
            w[q][31] = 0.f;
        }
#pragma unroll
        for (int q = 0; q < S::NPASS; ++q)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                float c[16];
#pragma unroll
                for (int k = 0; k < 16; ++k) c[k] = w[q][16 * h + k];
                tmem_st16(tma + 32u * q + 16u * h, c);
            }
        tmem_wait_st();
    }

    int64_t lu = 0, lun = 0;
    if (u < uend && allow_tma) {
        const int c0 = channel_of(p, u, lu);
        prefetch_unit<LOGN, REAL>(p, chan<REAL>(p, c0), lu, tg);
    }
    // everything above reads plan memory only; x, y and the state may belong to the kernel
    // before this one in the stream, which has to be complete from here on
    griddep_wait();
    if (u < uend) {
        const int c0 = channel_of(p, u, lu);
        ocur = stage_unit<LOGN, REAL>(p, chan<REAL>(p, c0), lu, cur, bcur, allow_tma, ucur, tg, gbar);
    }

    // outputs t = j + e T with t >= M - 1 are kept: e >= e_keep
    const int e_keep = (p.M - 1 - j + T - 1) < 0 ? 0 : (p.M - 1 - j + T - 1) / T;

    for (; u < uend; u += ustep) {
        const int chu = channel_of(p, u, lu);  // this unit's channel
        const int64_t un = u + ustep;
        if (un < uend) {
            const int chn = channel_of(p, un, lun);
            onxt = stage_unit<LOGN, REAL>(p, chan<REAL>(p, chn), lun, nxt, bnxt, allow_tma, unxt, tg, gbar);
        }
        if (ucur) {
            const bool ok = mbar_wait_bounded(bcur, pcur, p.wait_ns);
            if (gbar.sync_or(!ok)) {
                // the copy did not arrive within the limit: report it and stop issuing bulk
                // copies.  The copy still targets `cur` and completes on its mbarrier, so before
                // `cur` is written again the group waits (bounded by the fixed second limit)
                // for that phase; then it gathers this unit with plain loads.  A copy that
                // misses the second limit too leaves `cur` unusable: the group stops (its
                // remaining units are not filtered) with the error word set.
                if (tg == 0) atomicExch(p.err, 1);
                allow_tma = false;
                const bool landed = mbar_wait_bounded(bcur, pcur, kWaitLimitNs);
                if (gbar.sync_or(!landed)) break;
                ocur = stage_unit<LOGN, REAL>(p, chan<REAL>(p, chu), lu, cur, bcur, false, ucur, tg, gbar);
            }
            pcur ^= 1u;  // that phase has completed
        }

        // gather E_i (step 3) from the staged window into registers: v[e] = E[j + e T]
        float2 v[16];
        if constexpr (REAL) {
            const float *sr = reinterpret_cast<const float *>(cur) + ocur + 2 * f * p.L + j;
            const float *sr2 = sr + p.L;
#pragma unroll
            for (int e = 0; e < 16; ++e) v[e] = make_float2(sr[e * T], sr2[e * T]);
        } else {
            const float2 *sc = reinterpret_cast<const float2 *>(cur) + ocur + f * p.L + j;
#pragma unroll
            for (int e = 0; e < 16; ++e) v[e] = sc[e * T];
        }
        if (p.fuse_state && lu == 0) write_state<LOGN, REAL>(p, chan<REAL>(p, chu), cur, ocur, tg);

        // step 4: FFT, multiply by H, IFFT.  Exchange buffers: xbuf and (once read) cur.
        float2 *b0 = xbuf + f * xpad_len(C::N);
        float2 *b1 = reinterpret_cast<float2 *>(cur) + f * xpad_len(C::N);
        if constexpr (TC)  // the A tiles span the exchange buffer and `cur`, whichever comes first
            tc.a_base = smem_addr(cur < reinterpret_cast<unsigned char *>(xbuf) ? cur
                                                                               : reinterpret_cast<unsigned char *>(xbuf));
        fft_tm<LOGN, SMC ? (1 << 30) : 0, false, false, TC>(v, b0, b1, cT, tma, j, gbar, &tc, &tcpar);
        if constexpr (SMC) {
#pragma unroll
            for (int e = 0; e < 16; ++e) v[e] = cmul(v[e], cH[j + e * T]);
        } else {
            float h[16];
            tmem_ld16(tma, h);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 8; ++e) v[e] = cmul(v[e], make_float2(h[2 * e], h[2 * e + 1]));
            tmem_ld16(tma + 16u, h);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 8; ++e) v[8 + e] = cmul(v[8 + e], make_float2(h[2 * e], h[2 * e + 1]));
        }
        fft_tm<LOGN, SMC ? (1 << 30) : 0, true, false, TC>(v, b0, b1, cT, tma, j, gbar, &tc, &tcpar);

        // step 5: drop R[0 .. M-2], store R[M-1 .. N) as Y_i
        const int64_t blk = REAL ? 2 * (lu * C::F + f) : (lu * C::F + f);
        const int64_t o0 = blk * p.L - (p.M - 1) + j;  // output index of element e = 0
        const bool whole = o0 + (int64_t)(15 * T) + (REAL ? p.L : 0) < p.n;
        if constexpr (REAL) {
            float *y = static_cast<float *>(chan<REAL>(p, chu).y) + o0;
            float *y2 = y + p.L;
            if (whole) {
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    if (e >= e_keep) {
                        st_cs(y + e * T, v[e].x);
                        st_cs(y2 + e * T, v[e].y);
                    }
            } else {
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    if (e >= e_keep) {
                        if (o0 + e * T < p.n) st_cs(y + e * T, v[e].x);
                        if (o0 + e * T + p.L < p.n) st_cs(y2 + e * T, v[e].y);
                    }
            }
        } else {
            float2 *y = static_cast<float2 *>(chan<REAL>(p, chu).y) + o0;
            if (whole) {
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    if (e >= e_keep) st_cs(y + e * T, v[e]);
            } else {
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    if (e >= e_keep && o0 + e * T < p.n) st_cs(y + e * T, v[e]);
            }
        }
        gbar.sync();  // `cur` and the exchange buffer are free for the next unit
        unsigned char *tb = cur;
        cur = nxt;
        nxt = tb;
        uint64_t *tm = bcur;
        bcur = bnxt;
        bnxt = tm;
        uint32_t tp = pcur;
        pcur = pnxt;
        pnxt = tp;
        bool tu = ucur;
        ucur = unxt;
        unxt = tu;
        int to = ocur;
        ocur = onxt;
        onxt = to;
    }

    tmem_fence_before_sync();
    __syncthreads();
    tmem_fence_after_sync();
    if (!SMC && warp == 0) tmem_dealloc(*tm_base_slot, C::TM_COLS);
}

template <int LOGN, bool REAL>
KernelEntry block_entry() {
    using C = BlockCfg<LOGN, REAL>;
    KernelEntry k;
    k.func = reinterpret_cast<const void *>(&fos_block_kernel<LOGN, REAL, false>);
    if constexpr (C::HAS_SMC) {
        k.func_short = reinterpret_cast<const void *>(&fos_block_kernel<LOGN, REAL, true>);
        k.smem_short = C::SMEM_BYTES + C::SMC_BYTES;
    }
    if constexpr (C::HAS_TC) {
        k.func_tc = reinterpret_cast<const void *>(&fos_block_kernel<LOGN, REAL, false, true>);
        k.smem_tc = C::SMEM_TC;
    }
    k.threads = C::THREADS;
    k.smem = C::SMEM_BYTES;
    k.cluster = 1;
    k.units_per_cta = C::F;
    k.groups = C::GROUPS;
    k.fft_logn = LOGN;
    return k;
}

}  // namespace fos
