// fos_device.cuh -- device building blocks for the overlap-save block kernels (sm_103a).
//
// Complex float32 arithmetic, small in-register DFTs (radix 2, 4, 8, 16), the shared-memory
// swizzle used by the Stockham exchange passes, and thin inline-PTX wrappers for mbarrier,
// bulk (TMA) copies, cluster barriers and distributed shared memory.
//
// The transform convention follows the reading of "一种基于GPU的高阶数字FIR滤波器频域并行处理
// 实现方法" (zl.czvv.com/42398539.html) 主权项 step 4 used throughout this library: forward
// e^{-2 pi i nk/N}, inverse e^{+2 pi i nk/N}; DIR = -1 selects the forward sign, +1 the
// inverse (its 1/N is folded into the stored response H).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

// Pure arithmetic helpers are usable from host code too (host-side checks of the DFTs).
#define FOS_HD __host__ __device__ __forceinline__

namespace fos {

// --------------------------------------------------------------------------- complex ops

#if defined(__CUDA_ARCH__) && __CUDA_ARCH__ >= 1000
// one packed f32x2 instruction per complex add / subtract / component-wise multiply-add
__device__ __forceinline__ float2 cadd(float2 a, float2 b) { return __fadd2_rn(a, b); }
__device__ __forceinline__ float2 csub(float2 a, float2 b) { return __ffma2_rn(b, make_float2(-1.f, -1.f), a); }
__device__ __forceinline__ float2 cfma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
#else
FOS_HD float2 cadd(float2 a, float2 b) { return make_float2(a.x + b.x, a.y + b.y); }
FOS_HD float2 csub(float2 a, float2 b) { return make_float2(a.x - b.x, a.y - b.y); }
FOS_HD float2 cfma2(float2 a, float2 b, float2 c) { return make_float2(fmaf(a.x, b.x, c.x), fmaf(a.y, b.y, c.y)); }
#endif
FOS_HD float2 cneg(float2 a) { return make_float2(-a.x, -a.y); }

// a * w
FOS_HD float2 cmul(float2 a, float2 w) {
    return make_float2(fmaf(a.x, w.x, -a.y * w.y), fmaf(a.x, w.y, a.y * w.x));
}
// a * conj(w)
FOS_HD float2 cmulc(float2 a, float2 w) {
    return make_float2(fmaf(a.x, w.x, a.y * w.y), fmaf(a.y, w.x, -a.x * w.y));
}
// a * w for DIR = -1, a * conj(w) for DIR = +1 (w holds a forward-sign twiddle)
template <int DIR>
FOS_HD float2 ctw(float2 a, float2 w) {
    if constexpr (DIR < 0) return cmul(a, w);
    else return cmulc(a, w);
}
// a * (DIR * i): a rotation by a quarter turn in the transform's direction
template <int DIR>
FOS_HD float2 crot(float2 a) {
    if constexpr (DIR < 0) return make_float2(a.y, -a.x);  // * (-i)
    else return make_float2(-a.y, a.x);                    // * (+i)
}

// --------------------------------------------------------------------------- constant twiddles

// cos and sin of 2 pi m / 16, m = 0..15 (exact decimal expansions of cos(pi/8), sin(pi/8),
// sqrt(1/2), rounded by the compiler to float32).
__host__ __device__ constexpr float cos16(int m) {
    constexpr float c1 = 0.92387953251128675613f, s1 = 0.38268343236508977173f,
                    h = 0.70710678118654752440f;
    constexpr float t[16] = {1.f, c1, h, s1, 0.f, -s1, -h, -c1, -1.f, -c1, -h, -s1, 0.f, s1, h, c1};
    return t[m & 15];
}
__host__ __device__ constexpr float sin16(int m) { return cos16(m - 4); }

// a * e^{DIR * 2 pi i * m / R} for compile-time R (a power of two <= 16) and m,
// with the trivial angles done by swaps and sign changes.
template <int R, int M, int DIR>
FOS_HD float2 ctw_const(float2 a) {
    constexpr int m16 = ((M * (16 / R)) % 16 + 16) % 16;
    if constexpr (m16 == 0) return a;
    else if constexpr (m16 == 8) return cneg(a);
    else if constexpr (m16 == 4) return crot<DIR>(a);
    else if constexpr (m16 == 12) return crot<-DIR>(a);
    else if constexpr (m16 % 2 == 0) {
        // (+-1 +- i) / sqrt 2
        constexpr float h = 0.70710678118654752440f;
        constexpr float c = cos16(m16), s = (DIR < 0 ? -1.f : 1.f) * sin16(m16);
        // c, s are each +-h
        if constexpr (c > 0 && s > 0) return make_float2((a.x - a.y) * h, (a.x + a.y) * h);
        else if constexpr (c > 0 && s < 0) return make_float2((a.x + a.y) * h, (a.y - a.x) * h);
        else if constexpr (c < 0 && s > 0) return make_float2(-(a.x + a.y) * h, (a.x - a.y) * h);
        else return make_float2((a.y - a.x) * h, -(a.x + a.y) * h);
    } else {
        constexpr float c = cos16(m16), s = (DIR < 0 ? -1.f : 1.f) * sin16(m16);
        return cmul(a, make_float2(c, s));
    }
}

// a * e^{DIR 2 pi i m / R} for an m that is a compile-time constant after unrolling.
template <int R, int DIR>
FOS_HD float2 ctw_dyn(float2 a, int m) {
    switch (((m * (16 / R)) % 16 + 16) % 16) {
        case 0: return a;
        case 1: return ctw_const<16, 1, DIR>(a);
        case 2: return ctw_const<16, 2, DIR>(a);
        case 3: return ctw_const<16, 3, DIR>(a);
        case 4: return ctw_const<16, 4, DIR>(a);
        case 5: return ctw_const<16, 5, DIR>(a);
        case 6: return ctw_const<16, 6, DIR>(a);
        case 7: return ctw_const<16, 7, DIR>(a);
        case 8: return ctw_const<16, 8, DIR>(a);
        case 9: return ctw_const<16, 9, DIR>(a);
        case 10: return ctw_const<16, 10, DIR>(a);
        case 11: return ctw_const<16, 11, DIR>(a);
        case 12: return ctw_const<16, 12, DIR>(a);
        case 13: return ctw_const<16, 13, DIR>(a);
        case 14: return ctw_const<16, 14, DIR>(a);
        default: return ctw_const<16, 15, DIR>(a);
    }
}

// --------------------------------------------------------------------------- small DFTs
// In place, natural order in and out: a[k] <- sum_n a[n] e^{DIR 2 pi i nk/R}.

template <int DIR>
FOS_HD void dft2(float2 &a0, float2 &a1) {
    float2 t = a0;
    a0 = cadd(t, a1);
    a1 = csub(t, a1);
}

// PQ selects how the quarter turn of t3 = a1 - a3 is formed: false as scalar adds on t3's
// components; true with t3 formed component-swapped, so that a1, a3 = t1 +- (DIR i) t3 are one
// packed multiply-add each.  Both give identical results; which issues faster depends on the
// kernel around it (measured per kernel).
template <int DIR, bool PQ = false>
FOS_HD void dft4(float2 &a0, float2 &a1, float2 &a2, float2 &a3) {
    const float2 t0 = cadd(a0, a2), t1 = csub(a0, a2), t2 = cadd(a1, a3);
    if constexpr (PQ) {
        const float2 s = make_float2(a1.y - a3.y, a1.x - a3.x);  // (t3.y, t3.x)
        a0 = cadd(t0, t2);
        a2 = csub(t0, t2);
        if constexpr (DIR < 0) {  // t1 - i t3 = (t1.x + t3.y, t1.y - t3.x)
            a1 = cfma2(s, make_float2(1.f, -1.f), t1);
            a3 = cfma2(s, make_float2(-1.f, 1.f), t1);
        } else {
            a1 = cfma2(s, make_float2(-1.f, 1.f), t1);
            a3 = cfma2(s, make_float2(1.f, -1.f), t1);
        }
    } else {
        const float2 t3 = csub(a1, a3);
        a0 = cadd(t0, t2);
        a2 = csub(t0, t2);
        // t1 +- (DIR i) t3, component by component (a quarter turn swaps re and im)
        if constexpr (DIR < 0) {
            a1 = make_float2(t1.x + t3.y, t1.y - t3.x);
            a3 = make_float2(t1.x - t3.y, t1.y + t3.x);
        } else {
            a1 = make_float2(t1.x - t3.y, t1.y + t3.x);
            a3 = make_float2(t1.x + t3.y, t1.y - t3.x);
        }
    }
}

// R = R1 * 4 with n = 4 a + b, k = c + R1 d:
//   X[c + R1 d] = sum_b W4^{bd} W_R^{bc} sum_a x[4a + b] W_R1^{ac}
// The second radix-4 stage of a 16-point DFT with its twiddles W^{bc} (W = e^{DIR 2 pi i / 16})
// applied on the way in: y[b][c] -> a[c + 4 d].  The twiddles W^2 and W^6 are sqrt(1/2) times a
// sum or difference of components; that factor is folded into the stage's additions as fused
// multiply-adds (8 fewer float32 operations per 16 points than twiddling first).  Measured per
// kernel: the two-CTA kernel 2.4% faster with it, the block kernel at N = 4096 2% slower.
template <int DIR, bool PQ>
FOS_HD void dft16_stage2(float2 (&y)[4][4], float2 *a) {
    constexpr float h = 0.70710678118654752440f;
    constexpr float D = DIR < 0 ? -1.f : 1.f;
    // v W^2 = h (v.x - D v.y, v.y + D v.x);  v W^6 = h (-v.x - D v.y, D v.x - v.y)
    auto s2 = [](float2 v) { return make_float2(v.x - D * v.y, v.y + D * v.x); };
    auto s6 = [](float2 v) { return make_float2(-v.x - D * v.y, D * v.x - v.y); };
    const float2 hh = make_float2(h, h), nh = make_float2(-h, -h);
    // column c = 0: no twiddles
    dft4<DIR, PQ>(y[0][0], y[1][0], y[2][0], y[3][0]);
    // columns c = 1, 3: z2 = h S(y2) folded into t0, t1; z1, z3 general twiddles
#pragma unroll
    for (int c = 1; c < 4; c += 2) {
        const float2 s = c == 1 ? s2(y[2][c]) : s6(y[2][c]);
        const float2 t0 = cfma2(s, hh, y[0][c]), t1 = cfma2(s, nh, y[0][c]);
        const float2 z1 = ctw_dyn<16, DIR>(y[1][c], c), z3 = ctw_dyn<16, DIR>(y[3][c], 3 * c);
        const float2 t2 = cadd(z1, z3), t3 = csub(z1, z3);
        y[0][c] = cadd(t0, t2);
        y[2][c] = csub(t0, t2);
        // t1 +- (DIR i) t3
        y[1][c] = make_float2(t1.x - D * t3.y, t1.y + D * t3.x);
        y[3][c] = make_float2(t1.x + D * t3.y, t1.y - D * t3.x);
    }
    // column c = 2: z2 = (D i) y2 is a swap; z1 = h S2(y1), z3 = h S6(y3): t2, t3 = h (S2 +- S6)
    {
        const float2 y0 = y[0][2], y2 = y[2][2];
        const float2 t0 = make_float2(y0.x - D * y2.y, y0.y + D * y2.x);
        const float2 t1 = make_float2(y0.x + D * y2.y, y0.y - D * y2.x);
        const float2 p = s2(y[1][2]), q = s6(y[3][2]);
        const float2 u = cadd(p, q), w = csub(p, q);  // t2 = h u, t3 = h w
        y[0][2] = cfma2(u, hh, t0);
        y[2][2] = cfma2(u, nh, t0);
        // t1 +- (D i) h w
        y[1][2] = make_float2(fmaf(-D * h, w.y, t1.x), fmaf(D * h, w.x, t1.y));
        y[3][2] = make_float2(fmaf(D * h, w.y, t1.x), fmaf(-D * h, w.x, t1.y));
    }
#pragma unroll
    for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int d = 0; d < 4; ++d) a[c + 4 * d] = y[d][c];
}

// FS: for R = 16, the second stage with the sqrt(1/2) twiddle factors folded into its additions
// (dft16_stage2): fewer float32 operations, a different schedule; chosen per kernel by measurement.
template <int R, int DIR, bool PQ = false, bool FS = false>
FOS_HD void dft(float2 *a) {
    if constexpr (R == 1) {
    } else if constexpr (R == 2) {
        dft2<DIR>(a[0], a[1]);
    } else if constexpr (R == 4) {
        dft4<DIR, PQ>(a[0], a[1], a[2], a[3]);
    } else {
        constexpr int R1 = R / 4;
        float2 y[4][R1];
#pragma unroll
        for (int b = 0; b < 4; ++b) {
#pragma unroll
            for (int q = 0; q < R1; ++q) y[b][q] = a[4 * q + b];
            dft<R1, DIR, PQ>(y[b]);
        }
        if constexpr (R == 16 && FS) {
            dft16_stage2<DIR, PQ>(y, a);
        } else {
            // twiddles W_R^{bc}
#pragma unroll
            for (int c = 1; c < R1; ++c) {
                y[1][c] = ctw_dyn<R, DIR>(y[1][c], c);
                y[2][c] = ctw_dyn<R, DIR>(y[2][c], 2 * c);
                y[3][c] = ctw_dyn<R, DIR>(y[3][c], 3 * c);
            }
#pragma unroll
            for (int c = 0; c < R1; ++c) {
                dft4<DIR, PQ>(y[0][c], y[1][c], y[2][c], y[3][c]);
#pragma unroll
                for (int d = 0; d < 4; ++d) a[c + R1 * d] = y[d][c];
            }
        }
    }
}

// --------------------------------------------------------------------------- exchange layout
// Shared-memory index of logical element A of an exchange buffer: one padding element after
// every 16, so a buffer of N elements occupies N + N/16.  With 8-byte elements this makes the
// Stockham writes (stride Ns, or R0 for the first pass) and the reads (stride N/16) free of
// bank conflicts, and keeps every per-thread address an affine function of the element index
// (base + compile-time offset) whenever N/16 is a multiple of 16.
FOS_HD int xpad(int A) { return A + (A >> 4); }
__host__ __device__ constexpr int xpad_len(int n) { return n + n / 16; }

// --------------------------------------------------------------------------- PTX wrappers

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// Default limit of a kernel's wait for one bulk copy before it reports FIR_OS_E_DEVICE (1 s; a
// plan may set another, fir_os_plan_set_wait_limit), and the fixed limit of the second wait
// that lets a copy which missed the first one land before its buffer is reused.
constexpr uint64_t kWaitLimitNs = 1000000000ull;

// Bounded wait for the phase with the given parity to complete; false if it ran out.  A limit
// of 0 runs out before the first poll (every such wait fails: the setting that tests the
// fallback).  The poll count is bounded too, in case the timer stops.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, uint64_t limit_ns) {
    if (limit_ns == 0) return false;
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 0; it < (1u << 30); ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer_ns() - t0 > limit_ns) return false;
    }
    return false;
}

// Bulk copy global -> this CTA's shared memory, completing `bytes` on the mbarrier.
// dst and src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}
// Orders this thread's earlier generic-proxy shared-memory accesses before later
// async-proxy (bulk copy) accesses.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Hint: bring [src, src + bytes) of global memory into L2 (no completion to wait for).
// src 16-byte aligned, bytes a multiple of 16; the range must lie inside one allocation.
__device__ __forceinline__ void prefetch_l2_bulk(const void *src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Programmatic dependent launch.  launch_dependents lets the next kernel of the stream (when
// it was launched with programmatic serialization) start on free SMs; wait returns once the
// kernel before this one has completed and its memory operations are visible.  A kernel
// touches nothing that an earlier kernel of the stream may write before it has waited.
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// streaming (evict-first) global stores
__device__ __forceinline__ void st_cs(float2 *p, float2 v) { __stcs(p, v); }
__device__ __forceinline__ void st_cs(float *p, float v) { __stcs(p, v); }

// --------------------------------------------------------------------------- clusters

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t nclusters_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}
// All threads of all CTAs of the cluster; release/acquire orders shared-memory writes
// (local and distributed) made before it with reads made after it.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                     : "memory");
}
// Address of the same shared-memory location in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t map_rank(uint32_t local_smem_addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local_smem_addr), "r"(rank));
    return r;
}
__device__ __forceinline__ void st_cluster(uint32_t addr, float2 v) {
    asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(addr), "f"(v.x), "f"(v.y) : "memory");
}

// --------------------------------------------------------------------------- tensor memory
// Tensor Memory (TMEM) used as per-thread storage: 128 lanes x 512 32-bit columns per SM; warp w
// of a CTA reaches lanes 32 (w % 4) .. 32 (w % 4) + 31, and with the 32x32b shape thread t of
// the warp reads its own lane, so the threads t, t + 128, t + 256, ... of a CTA share a lane.
// The block kernels keep constants there (the response H and the pass twiddles), the resident
// kernel a whole block.  Allocation is by one whole warp; the CTA frees it before exit.

__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(dst_smem)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tmem_fence_before_sync() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tmem_fence_after_sync() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 16 consecutive columns of this thread's lane <-> 16 registers
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=f"(r[0]), "=f"(r[1]), "=f"(r[2]), "=f"(r[3]), "=f"(r[4]), "=f"(r[5]), "=f"(r[6]), "=f"(r[7]),
          "=f"(r[8]), "=f"(r[9]), "=f"(r[10]), "=f"(r[11]), "=f"(r[12]), "=f"(r[13]), "=f"(r[14]), "=f"(r[15])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
            taddr),
        "f"(r[0]), "f"(r[1]), "f"(r[2]), "f"(r[3]), "f"(r[4]), "f"(r[5]), "f"(r[6]), "f"(r[7]), "f"(r[8]), "f"(r[9]),
        "f"(r[10]), "f"(r[11]), "f"(r[12]), "f"(r[13]), "f"(r[14]), "f"(r[15])
        : "memory");
}

// Two complex values (four columns) of this thread's lane.  No memory clobber: Tensor Memory is
// not addressable by ordinary loads and stores, so these may move across them (ordering
// against tcgen05.wait / fences, which are volatile too, is kept).
__device__ __forceinline__ void tmem_ld4(uint32_t taddr, float2 &a, float2 &b) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(a.x), "=f"(a.y), "=f"(b.x), "=f"(b.y)
                 : "r"(taddr));
}
__device__ __forceinline__ void tmem_st4(uint32_t taddr, float2 a, float2 b) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1,%2,%3,%4};" ::"r"(taddr), "f"(a.x), "f"(a.y),
                 "f"(b.x), "f"(b.y));
}

// One complex value (two columns) of this thread's lane.
__device__ __forceinline__ void tmem_ld2(uint32_t taddr, float2 &a) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x2.b32 {%0,%1}, [%2];" : "=f"(a.x), "=f"(a.y) : "r"(taddr));
}
__device__ __forceinline__ void tmem_st2(uint32_t taddr, float2 a) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x2.b32 [%0], {%1,%2};" ::"r"(taddr), "f"(a.x), "f"(a.y));
}

// --------------------------------------------------------------------------- group barriers
// A CTA may run several independent thread groups; each synchronises on its own hardware
// barrier (id >= 1; id 0 is __syncthreads).  NT = threads in the group (a multiple of 32).
template <int NT>
struct GroupBarrier {
    int id;
    __device__ __forceinline__ void sync() const {
        asm volatile("bar.sync %0, %1;" ::"r"(id), "n"(NT) : "memory");
    }
    // barrier that also returns whether `pred` was true in any thread of the group
    __device__ __forceinline__ bool sync_or(bool pred) const {
        uint32_t r;
        asm volatile(
            "{\n\t.reg .pred p, q;\n\t"
            "setp.ne.u32 p, %1, 0;\n\t"
            "bar.red.or.pred q, %2, %3, p;\n\t"
            "selp.u32 %0, 1, 0, q;\n\t}"
            : "=r"(r)
            : "r"((uint32_t)pred), "r"(id), "n"(NT)
            : "memory");
        return r != 0;
    }
};

}  // namespace fos
