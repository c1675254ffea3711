// Device helpers of the tcgen05 products (the A8 product and the batched A16
// product): shared-memory addresses and matrix descriptors of the K-major
// 8x8 core-matrix operand layout, bounded mbarrier polling, 2-D tensor copies,
// TMEM loads and stores, and the exact widening of int8 / packed int4 codes to
// fp16 in that layout.
#pragma once

#include <cuda.h>

#include "tq_internal.cuh"

namespace tq {
namespace {

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// byte offset of (row r, k) in a [rows x 64] fp16 tile of 8x8 core matrices:
// core matrix (r/8, k/8) is 128 contiguous bytes, K-adjacent ones 128 bytes
// apart (leading offset), row groups 1024 bytes apart (stride offset)
__device__ __forceinline__ int cm_off(int r, int k) {
    return ((r >> 3) * 8 + (k >> 3)) * 128 + (r & 7) * 16 + (k & 7) * 2;
}

__device__ __forceinline__ uint64_t smem_desc(uint32_t addr) {
    constexpr uint64_t lbo = 128, sbo = 1024;
    return static_cast<uint64_t>((addr & 0x3FFFF) >> 4) | ((lbo >> 4) << 16) | ((sbo >> 4) << 32) |
           (1ull << 46);
}

__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n.reg .pred p;\nmbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
        "selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

__device__ __forceinline__ uint32_t hsub2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ uint32_t hfma2(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// four int8 codes -> fp16 pairs (k0,k1), (k2,k3): 0x64xx is 1024 + xx, and
// xx = code + 128 after flipping the sign bit; subtract 1152.
__device__ __forceinline__ void widen8(uint32_t w, uint32_t &p01, uint32_t &p23) {
    const uint32_t u = w ^ 0x80808080u;
    p01 = hsub2(prmt(u, 0x64646464u, 0x4140u), 0x64806480u);
    p23 = hsub2(prmt(u, 0x64646464u, 0x4342u), 0x64806480u);
}

// eight int4 codes (low nibble first) -> fp16 pairs (k0,k1) .. (k6,k7).  With
// u = code + 8: the low half is 0x6400 | u = 1024 + u, the high half
// 0x6400 | (u << 4) = 1024 + 16u; one fma with (1, 1/16) and (-1032, -72).
__device__ __forceinline__ void widen4(uint32_t w, uint32_t (&p)[4]) {
    const uint32_t u = w ^ 0x88888888u;
    const uint32_t scale = 0x2C003C00u;   // (1/16, 1.0)
    const uint32_t bias = 0xD480E408u;    // (-72, -1032)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t t = prmt(u, 0u, 0x4040u + 0x0101u * i);  // byte i in both halves
        p[i] = hfma2((t & 0x00F0000Fu) | 0x64006400u, scale, bias);
    }
}

__device__ __forceinline__ void store_i8x16(unsigned char *tile, int r, int seg, const uint4 &w) {
    uint4 lo, hi;
    widen8(w.x, lo.x, lo.y);
    widen8(w.y, lo.z, lo.w);
    widen8(w.z, hi.x, hi.y);
    widen8(w.w, hi.z, hi.w);
    *reinterpret_cast<uint4 *>(tile + cm_off(r, seg * 16)) = lo;
    *reinterpret_cast<uint4 *>(tile + cm_off(r, seg * 16 + 8)) = hi;
}

__device__ __forceinline__ void store_i4x32(unsigned char *tile, int r, int seg, const uint4 &w) {
    const uint32_t v[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint32_t pr[4];
        widen4(v[q], pr);
        *reinterpret_cast<uint4 *>(tile + cm_off(r, seg * 32 + q * 8)) = make_uint4(pr[0], pr[1], pr[2], pr[3]);
    }
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
          "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
          "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]),
          "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]),
          "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
        ::"r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]),
          "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]),
          "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]),
          "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]),
          "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
        : "memory");
}


// byte offset of the 16-byte chunk c of row r in a TMA tile with 64-byte rows
// and 64-byte swizzle (chunk index XOR address bits 7-8), or with 32-byte rows
// and 32-byte swizzle (chunk bit XOR address bit 7)
__device__ __forceinline__ int swz64(int r, int c) { return r * 64 + ((c ^ ((r >> 1) & 3)) << 4); }
__device__ __forceinline__ int swz32(int r, int c) { return r * 32 + ((c ^ ((r >> 2) & 1)) << 4); }
// the same for 128-byte rows and the 128-byte swizzle (chunk XOR address bits 7-9)
__device__ __forceinline__ int swz128(int r, int c) { return r * 128 + ((c ^ (r & 7)) << 4); }

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int c0, int c1,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3}], [%4];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void mbar_arrive_local(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

}  // namespace
}  // namespace tq
