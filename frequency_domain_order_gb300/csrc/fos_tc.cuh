// fos_tc.cuh -- 16-point DFTs on the tensor cores (tcgen05.mma, kind::tf32) for the radix-16
// passes of the block kernel's optional tensor-core variant.
//
// Step 4 of the claim in "一种基于GPU的高阶数字FIR滤波器频域并行处理实现方法"
// (zl.czvv.com/42398539.html, 主权项) transforms each block; every radix-16 pass of that
// transform applies the 16-point DFT matrix to one 16-value vector per thread.  Here 128 such
// vectors are one GEMM row tile: D[row][c] = sum_k A[row][k] B[c][k] with A the vectors as 32
// reals (re, im interleaved), B the 32 x 32 real form of the DFT matrix (for forward or inverse
// sign) and D (128 lanes x 32 fp32 columns of Tensor Memory) the transformed vectors, which
// thread `row` reads back from its own lane.
//
// TF32 keeps 10 mantissa bits, far from the float32 the parity bar needs, so the operands are
// split: A = A_hi + A_lo with A_hi the value with its 13 low mantissa bits cleared (exactly a
// TF32 number) and A_lo = A - A_hi (exact); B likewise from float64.  D accumulates
// A_hi B_hi + A_hi B_lo + A_lo B_hi in float32 (the dropped A_lo B_lo is ~2^-22 relative).
//
// Shared-memory operand layout (K-major, no swizzle): 8-row x 16-byte core matrices; element
// (row, k) of a 128-row tile at (row / 8) * 1024 + (k / 4) * 128 + (row % 8) * 16 + (k % 4) * 4,
// i.e. a leading-dimension (K) stride of 128 bytes and a stride-dimension (row) stride of 1024.
// A group's two row tiles (its 256 vectors) take 2 x 32 KB: tile t's A_hi at t * 32768, its
// A_lo 16 KB after it.  Each B (hi or lo) is a 32-row tile of 4 KB.
#pragma once

#include "fos_device.cuh"

namespace fos {

constexpr uint32_t kTcTileBytes = 16384;   // one 128 x 32 TF32 operand tile
constexpr uint32_t kTcBTileBytes = 4096;   // one 32 x 32 TF32 operand tile (a B matrix part)

// byte offset of element (row, k) in a K-major no-swizzle TF32 tile with 32 K columns
FOS_HD uint32_t tc_offset(int row, int k) {
    return (uint32_t)((row >> 3) * 1024 + (k >> 2) * 128 + (row & 7) * 16 + (k & 3) * 4);
}

// Shared-memory matrix descriptor: start address, leading (K) and stride (row) byte offsets,
// the descriptor version bit, no swizzle.
__device__ __forceinline__ uint64_t tc_desc(uint32_t saddr) {
    uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)(128u >> 4) << 16;
    d |= (uint64_t)(1024u >> 4) << 32;
    d |= (uint64_t)1 << 46;
    return d;
}

// Instruction descriptor: float32 accumulator, TF32 A and B, both K-major, N = 32, M = 128.
constexpr uint32_t kTcIdesc = (1u << 4) | (2u << 7) | (2u << 10) | ((32u >> 3) << 17) | ((128u >> 4) << 24);

__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, bool accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(kTcIdesc), "r"((uint32_t)accumulate)
        : "memory");
}
__device__ __forceinline__ void tc_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
                 : "memory");
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, float a, float b, float c, float d) {
    asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(a), "f"(b), "f"(c), "f"(d) : "memory");
}
__device__ __forceinline__ float tf32_hi(float x) { return __uint_as_float(__float_as_uint(x) & 0xFFFFE000u); }

// 32 consecutive columns of this thread's lane
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=f"(r[0]), "=f"(r[1]), "=f"(r[2]), "=f"(r[3]), "=f"(r[4]), "=f"(r[5]), "=f"(r[6]), "=f"(r[7]),
          "=f"(r[8]), "=f"(r[9]), "=f"(r[10]), "=f"(r[11]), "=f"(r[12]), "=f"(r[13]), "=f"(r[14]), "=f"(r[15]),
          "=f"(r[16]), "=f"(r[17]), "=f"(r[18]), "=f"(r[19]), "=f"(r[20]), "=f"(r[21]), "=f"(r[22]), "=f"(r[23]),
          "=f"(r[24]), "=f"(r[25]), "=f"(r[26]), "=f"(r[27]), "=f"(r[28]), "=f"(r[29]), "=f"(r[30]), "=f"(r[31])
        : "r"(taddr)
        : "memory");
}

// What one thread group needs for its tensor-core DFTs.
struct TcCtx {
    uint32_t a_base;     // shared address of the group's two A tiles (64 KB, 16-byte aligned)
    uint32_t b_base;     // shared address of B: forward hi, forward lo, inverse hi, inverse lo
    uint32_t d_tile;     // Tensor Memory address (lane 0) of the group's tile-0 accumulator; tile 1 at +32
    uint32_t d_row;      // this thread's accumulator: its lane, its tile's 32 columns
    uint32_t row_off;    // byte offset of this thread's row in its A tile pair
    uint64_t *mbar;      // the group's MMA-completion mbarrier
    int *err;            // set when the wait for the MMAs ran out (1 s)
    bool leader;         // issues the group's MMAs
};

// v <- DFT16(v) (sign DIR) for the group's 256 vectors at once, by the tensor cores.  Called by
// every thread of the group at the same point; `bar` is the group's barrier and `parity` the
// group's MMA-mbarrier phase (flipped here).  The A tiles may overlap buffers that the group has
// read before the call: the first barrier makes those reads complete before any row is written.
template <int DIR, class Bar>
__device__ __forceinline__ void tc_dft16(float2 (&v)[16], const TcCtx &c, const Bar &bar, uint32_t &parity) {
    tmem_fence_before_sync();
    bar.sync();  // every thread is done with what the tiles overwrite, and with the last D read
    const uint32_t hi = c.a_base + c.row_off;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const float2 x0 = v[2 * q], x1 = v[2 * q + 1];
        const float h0 = tf32_hi(x0.x), h1 = tf32_hi(x0.y), h2 = tf32_hi(x1.x), h3 = tf32_hi(x1.y);
        st_shared_v4(hi + 128u * q, h0, h1, h2, h3);
        st_shared_v4(hi + kTcTileBytes + 128u * q, x0.x - h0, x0.y - h1, x1.x - h2, x1.y - h3);
    }
    fence_proxy_async_smem();
    tmem_fence_before_sync();
    bar.sync();  // every row is written and visible to the tensor cores
    tmem_fence_after_sync();
    if (c.leader) {
        const uint32_t bhi = c.b_base + (DIR < 0 ? 0u : 2u * kTcBTileBytes), blo = bhi + kTcBTileBytes;
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            const uint32_t ahi = c.a_base + (uint32_t)t * 2u * kTcTileBytes, alo = ahi + kTcTileBytes;
            const uint32_t d = c.d_tile + 32u * (uint32_t)t;
            // each instruction covers K = 8 (two core matrices, 256 bytes along K)
#pragma unroll
            for (int s = 0; s < 4; ++s) tc_mma(d, tc_desc(ahi + 256u * s), tc_desc(bhi + 256u * s), s > 0);
#pragma unroll
            for (int s = 0; s < 4; ++s) tc_mma(d, tc_desc(ahi + 256u * s), tc_desc(blo + 256u * s), true);
#pragma unroll
            for (int s = 0; s < 4; ++s) tc_mma(d, tc_desc(alo + 256u * s), tc_desc(bhi + 256u * s), true);
        }
        tc_commit(c.mbar);
    }
    if (!mbar_wait_bounded(c.mbar, parity, kWaitLimitNs))
        atomicExch(c.err, 1);  // the results are not valid; the error word reports it
    parity ^= 1u;
    tmem_fence_after_sync();
    float r[32];
    tmem_ld32(c.d_row, r);
    tmem_wait_ld();
#pragma unroll
    for (int m = 0; m < 16; ++m) v[m] = make_float2(r[2 * m], r[2 * m + 1]);
}

}  // namespace fos
