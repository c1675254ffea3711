// Device helpers shared by the A16 products (decode GEMV kernels): the x'
// layout that puts each lane's MMA operands side by side, the exact widening
// of int8/int4 codes to bf16 pairs, the bf16 MMA, and bounded mbarrier waits.
#pragma once

#include "tq_internal.cuh"

namespace tq {

// Bounded waits, in clock cycles (about 2 s each).  A build of the library
// made for its own tests may shorten the wait for operands
// (TQ_TEST_WAIT_CYCLES) so that an expiry can be provoked on purpose; the
// wait that lets a CTA's copies in flight land before it exits keeps the full
// limit in every build.
#ifdef TQ_TEST_WAIT_CYCLES
constexpr long long kA16WaitLimit = TQ_TEST_WAIT_CYCLES;
#else
constexpr long long kA16WaitLimit = 4000000000ll;
#endif
constexpr long long kA16DrainLimit = 4000000000ll;

// x' layout inside each K block so that the 4 values one lane needs for one
// mma (its k-slots 2t, 2t+1, 2t+8, 2t+9) are contiguous at jj*16 + 4t.
//   int8 (64 k per block):  lane t holds k = 16t..16t+15; word q -> mma q,
//     pairs (k0, k2) and (k1, k3) of the word.
//   int4 (128 k per block): lane t holds k = 32t..32t+31; word q -> mmas 2q
//     and 2q+1, pairs (k0,k4),(k1,k5) and (k2,k6),(k3,k7) of the word.
template <int BITS>
__device__ __forceinline__ int xpos(int kl) {
    if constexpr (BITS == 8) {
        const int t = kl >> 4, q = (kl >> 2) & 3, r = kl & 3;
        return q * 16 + 4 * t + (((r & 1) << 1) | (r >> 1));
    } else {
        const int t = kl >> 5, q = (kl >> 3) & 3, r = kl & 7;
        const int jj = 2 * q + ((r >> 1) & 1);
        return jj * 16 + 4 * t + ((r >> 2) | ((r & 1) << 1));
    }
}

__device__ __forceinline__ uint32_t bf16x2_sub(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// int8 codes (k0..k3 in bytes 0..3) -> bf16 pairs (k0,k2) and (k1,k3).
// 0x43xx is 128 + (low 7 bits); subtracting 128 or 256 by the sign bit gives
// the two's-complement value exactly.
__device__ __forceinline__ void widen_i8(uint32_t x, uint32_t &p02, uint32_t &p13) {
    p02 = bf16x2_sub((x & 0x007F007Fu) | 0x43004300u, (x & 0x00800080u) ^ 0x43004300u);
    const uint32_t y = x >> 8;
    p13 = bf16x2_sub((y & 0x007F007Fu) | 0x43004300u, (y & 0x00800080u) ^ 0x43004300u);
}

// int4 codes (k0..k7, low nibble first) -> bf16 pairs (k0,k4), (k1,k5),
// (k2,k6), (k3,k7): 0x4300 | (n ^ 8) is 136 + n, minus 136.
__device__ __forceinline__ void widen_i4(uint32_t w, uint32_t (&p)[4]) {
    const uint32_t c = 0x43084308u;
    p[0] = bf16x2_sub((w & 0x000F000Fu) ^ c, c);
    p[1] = bf16x2_sub(((w >> 4) & 0x000F000Fu) ^ c, c);
    p[2] = bf16x2_sub(((w >> 8) & 0x000F000Fu) ^ c, c);
    p[3] = bf16x2_sub(((w >> 12) & 0x000F000Fu) ^ c, c);
}

// fp16 form of the int8 widening, for products whose x' is fp16: codes
// (k0..k3) -> fp16 pairs (k0,k2), (k1,k3); the byte u = b ^ 0x80 under
// exponent 0x64 is 1024 + u exactly, minus 1152 is b.
__device__ __forceinline__ uint32_t f16x2_sub(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ void widen_i8_f16(uint32_t x, uint32_t &p02, uint32_t &p13) {
    const uint32_t u = x ^ 0x80808080u;
    uint32_t lo, hi;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(lo) : "r"(u), "r"(0x64646464u), "r"(0x4240u));
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(hi) : "r"(u), "r"(0x64646464u), "r"(0x4341u));
    p02 = f16x2_sub(lo, 0x64806480u);
    p13 = f16x2_sub(hi, 0x64806480u);
}

// int4 codes (k0..k7) -> fp16 pairs (k0,k4), (16 k1, 16 k5), (k2,k6),
// (16 k3, 16 k7): the odd codes are read in place (bits 4..7 of each half)
// under exponent 0x64, which makes them 16 times their value, so only the
// even/odd split needs a shift.  The operand they meet must hold x'/16 at odd k.
__device__ __forceinline__ void widen_i4_f16_odd16(uint32_t w, uint32_t (&p)[4]) {
    const uint32_t ce = 0x64086408u, co = 0x64806480u;   // 1024 + 8, 1024 + 128
    const uint32_t w8 = w >> 8;
    p[0] = f16x2_sub((w & 0x000F000Fu) ^ ce, ce);
    p[1] = f16x2_sub((w & 0x00F000F0u) ^ co, co);
    p[2] = f16x2_sub((w8 & 0x000F000Fu) ^ ce, ce);
    p[3] = f16x2_sub((w8 & 0x00F000F0u) ^ co, co);
}

// Biased widenings without the subtraction: a 16-bit pattern u < 2^10 is the
// fp16 subnormal u * 2^-24 exactly, so the code c plus its bias B (128 for
// int8, 8 for int4: c + B >= 0) is an fp16 value by a mask or a byte permute
// alone.  A product of these with x' holds 2^-24 (sum_k c_k x'_k + B sum_k
// x'_k); whoever consumes it takes off B times the token's sum of x'.
// int8: pairs (k0, k2), (k1, k3) of (c + 128) 2^-24.
__device__ __forceinline__ void widen_i8_f16_biased(uint32_t x, uint32_t &p02, uint32_t &p13) {
    const uint32_t u = x ^ 0x80808080u;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(p02) : "r"(u), "r"(0u), "r"(0x4240u));
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(p13) : "r"(u), "r"(0u), "r"(0x4341u));
}

// int4: pairs (k0, k4), (16 k1, 16 k5), (k2, k6), (16 k3, 16 k7) of
// (c + 8) 2^-24, the odd codes in place as in widen_i4_f16_odd16.
__device__ __forceinline__ void widen_i4_f16_biased(uint32_t w, uint32_t (&p)[4]) {
    const uint32_t w8 = w >> 8;
    p[0] = (w & 0x000F000Fu) ^ 0x00080008u;
    p[1] = (w & 0x00F000F0u) ^ 0x00800080u;
    p[2] = (w8 & 0x000F000Fu) ^ 0x00080008u;
    p[3] = (w8 & 0x00F000F0u) ^ 0x00800080u;
}

__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1,
                                         uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        "selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase of `parity` to complete, for at most `limit` clock
// cycles; false on expiry.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  long long limit = kA16WaitLimit) {
    const long long t0 = clock64();
    while (!mbar_try(bar, parity))
        if (clock64() - t0 > limit) return false;
    return true;
}

}  // namespace tq
