// Skinny A16 product for M <= 64 (decode and batched decode):
//   Y[m][n] = sw[n] * sum_k q_w[n][k] * x'_bf16[m][k],  fp32 sums,
// where x' is the group-256 Hadamard rotation of the token row rounded to bf16
// (tensai docs, "画像生成" / Image generation, section "幅とメモリ": the input of
// the product gets the same rotation as the weights).  Decode is bound by the
// weight stream (kvad-gpu internals, "Numbers": decode is memory-bound).
//
// Design (one launch, no workspace):
//   - A CTA owns RT = 16*WR weight rows and a K range of whole 256-groups;
//     C CTAs of a thread-block cluster split K, and their partial sums are
//     added in a fixed order through distributed shared memory (no float
//     atomics, so repeated calls give identical bytes).
//   - Prologue: the CTA rotates its K range of every token row in fp32 (warp
//     butterfly), rounds to bf16 and keeps it in shared memory, laid out so
//     that each mma B fragment is one conflict-free 8-byte load.
//   - Main loop: each lane streams 16-byte chunks of two weight rows with
//     non-allocating loads, PF blocks ahead, widens int8/int4 codes to bf16
//     pairs in registers (exact integers), and feeds mma.sync m16n8k16.
//   - Programmatic dependent launch: the CTA lets the next kernel launch at
//     once, prefetches its weight rows into L2 (L2 is coherent, so this is
//     safe before the dependency is met), then waits for the previous kernel
//     before it reads X or writes Y.

#include <cooperative_groups.h>

#include "tq_internal.cuh"

namespace cg = cooperative_groups;

namespace tq {
namespace {

struct GemvParams {
    const uint16_t *X;
    int64_t ldx;
    int M;
    int64_t K;
    int G;          // groups of 256 (last may be a tail)
    const uint8_t *W;
    int64_t wld;    // bytes per weight row
    const float *sw;
    int64_t N;
    void *Y;
    int64_t ldy;
    int ytype;      // 0 fp32, 1 bf16
    int WR, WK, C;  // warps along rows, warps along K, cluster size
    int SX;         // shared-memory row stride of x' (bf16 elements)
};

// Each lane's 16-byte chunk of a block covers the block's k in a fixed way;
// x' is stored so that the 4 values one lane needs for one mma (its k-slots
// 2t, 2t+1, 2t+8, 2t+9) are contiguous at jj*16 + 4t.
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

__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1,
                                         uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

template <int BITS, int NT, int PF>
__global__ void __launch_bounds__(kThreads)
k_gemv_a16(const GemvParams p) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    uint16_t *xs = reinterpret_cast<uint16_t *>(smem_raw);
    constexpr int KB = BITS == 8 ? 64 : 128;  // k per block
    constexpr int BB = 64;                    // bytes per row per block

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int C = p.C;
    const int crank = C > 1 ? static_cast<int>(cg::this_cluster().block_rank()) : 0;
    const int RT = 16 * p.WR;
    const int64_t n0 = static_cast<int64_t>(blockIdx.x / C) * RT;
    const int gb = static_cast<int>(static_cast<int64_t>(p.G) * crank / C);
    const int ge = static_cast<int>(static_cast<int64_t>(p.G) * (crank + 1) / C);
    const int64_t kbeg = static_cast<int64_t>(gb) * kGroup;
    const int64_t kend = min(static_cast<int64_t>(ge) * kGroup, p.K);
    const int nk = static_cast<int>(kend - kbeg);
    const int nblk = (nk + KB - 1) / KB;
    const int64_t wbyte0 = kbeg * BITS / 8;
    const int rbytes = nk * BITS / 8;  // this CTA's bytes of one weight row

    pdl_launch_dependents();
    for (int r = threadIdx.x; r < RT; r += kThreads) {
        const int64_t n = n0 + r;
        if (n < p.N && rbytes > 0) prefetch_l2(p.W + n * p.wld + wbyte0, static_cast<uint32_t>(rbytes));
    }
    pdl_wait();

    // ---- prologue: rotated, bf16-rounded x' of this K range in shared memory
    const int M = p.M, SX = p.SX;
    if (nblk > 0) {
        const int z0 = (nblk - 1) * KB;  // the last block may be partial: zero it
        for (int i = threadIdx.x; i < M * KB; i += kThreads) xs[(i / KB) * SX + z0 + (i % KB)] = 0;
    }
    __syncthreads();
    const int ngrp = ge - gb;
    for (int w = warp; w < M * ngrp; w += kThreads / 32) {
        const int m = w / ngrp, gi = w % ngrp;
        const int64_t g0 = kbeg + static_cast<int64_t>(gi) * kGroup;
        float v[8] = {};
        const int E = rotate_group32_any(p.X + m * p.ldx + g0, group_width(p.K, g0), v);
        uint16_t *xrow = xs + m * SX;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            if (e < E) {
                const int kl = gi * kGroup + lane * E + e;
                xrow[(kl / KB) * KB + xpos<BITS>(kl % KB)] = f32_to_bf16_bits(v[e]);
            }
        }
    }
    __syncthreads();

    // ---- main loop
    const int WR = p.WR, WK = p.WK;
    const int wr = warp % WR, wk = warp / WR;
    const int g = lane >> 2, t = lane & 3;
    const int64_t rA = n0 + wr * 16 + g, rB = rA + 8;
    const bool okA = rA < p.N, okB = rB < p.N;
    const uint8_t *pA = p.W + (okA ? rA : 0) * p.wld + wbyte0 + t * 16;
    const uint8_t *pB = p.W + (okB ? rB : 0) * p.wld + wbyte0 + t * 16;
    const int nbw = nblk > wk ? (nblk - wk + WK - 1) / WK : 0;

    float acc[NT][4];
#pragma unroll
    for (int i = 0; i < NT; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.0f;

    // B fragment base for each n-tile (token nt*8 + g); tokens >= M read zeros
    const uint16_t *xb[NT];
    bool xin[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int tok = nt * 8 + g;
        xin[nt] = tok < M;
        xb[nt] = xs + (xin[nt] ? tok : 0) * SX + 4 * t;
    }

    auto load = [&](int i, uint4 &a, uint4 &b) {
        const int off = (wk + i * WK) * BB;
        const bool in = (i < nbw) && (off + t * 16 < rbytes);
        a = (in && okA) ? ldg_stream(pA + off) : make_uint4(0, 0, 0, 0);
        b = (in && okB) ? ldg_stream(pB + off) : make_uint4(0, 0, 0, 0);
    };
    auto mma_all = [&](int blk, int jj, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            uint2 bv = make_uint2(0, 0);
            if (xin[nt]) bv = *reinterpret_cast<const uint2 *>(xb[nt] + blk * KB + jj * 16);
            mma_bf16(acc[nt], a0, a1, a2, a3, bv.x, bv.y);
        }
    };

    uint4 ra[PF], rb[PF];
#pragma unroll
    for (int s = 0; s < PF; ++s) load(s, ra[s], rb[s]);
    for (int i0 = 0; i0 < nbw; i0 += PF) {
#pragma unroll
        for (int s = 0; s < PF; ++s) {
            const int i = i0 + s;
            if (i < nbw) {
                const int blk = wk + i * WK;
                const uint32_t A[4] = {ra[s].x, ra[s].y, ra[s].z, ra[s].w};
                const uint32_t B[4] = {rb[s].x, rb[s].y, rb[s].z, rb[s].w};
                if constexpr (BITS == 8) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        uint32_t a0, a1, a2, a3;
                        widen_i8(A[q], a0, a2);
                        widen_i8(B[q], a1, a3);
                        mma_all(blk, q, a0, a1, a2, a3);
                    }
                } else {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        uint32_t pa[4], pb[4];
                        widen_i4(A[q], pa);
                        widen_i4(B[q], pb);
                        mma_all(blk, 2 * q, pa[0], pb[0], pa[1], pb[1]);
                        mma_all(blk, 2 * q + 1, pa[2], pb[2], pa[3], pb[3]);
                    }
                }
            }
            load(i + PF, ra[s], rb[s]);
        }
    }

    // ---- reduction: warps along K, then CTAs of the cluster, fixed order
    __syncthreads();
    float *red = reinterpret_cast<float *>(smem_raw);  // [WK][RT][M]
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int row = wr * 16 + g + 8 * h;
            const int m0 = nt * 8 + 2 * t;
            if (m0 < M) red[(wk * RT + row) * M + m0] = acc[nt][2 * h];
            if (m0 + 1 < M) red[(wk * RT + row) * M + m0 + 1] = acc[nt][2 * h + 1];
        }
    }
    __syncthreads();
    const int RM = RT * M;
    for (int idx = threadIdx.x; idx < RM; idx += kThreads) {
        float s = red[idx];
        for (int k = 1; k < WK; ++k) s += red[k * RM + idx];
        red[idx] = s;
    }
    if (C > 1) cg::this_cluster().sync();
    else __syncthreads();
    if (crank == 0) {
        for (int idx = threadIdx.x; idx < RM; idx += kThreads) {
            const int m = idx / RT, r = idx % RT;
            const int li = r * M + m;
            float s = red[li];
            for (int q = 1; q < C; ++q) s += cg::this_cluster().map_shared_rank(red, q)[li];
            const int64_t n = n0 + r;
            if (n < p.N) {
                const float y = p.sw[n] * s;
                if (p.ytype == 0)
                    static_cast<float *>(p.Y)[m * p.ldy + n] = y;
                else
                    static_cast<uint16_t *>(p.Y)[m * p.ldy + n] = f32_to_bf16_bits(y);
            }
        }
    }
    if (C > 1) cg::this_cluster().sync();
}

struct Plan {
    int WR, WK, C, SX;
    size_t smem;
};

constexpr size_t kGemvSmemMax = 200 * 1024;

size_t smem_for(int64_t M, int SX, int WR, int WK) {
    const size_t xs = static_cast<size_t>(M) * SX * 2;
    const size_t red = static_cast<size_t>(WK) * 16 * WR * M * 4;
    return xs > red ? xs : red;
}

int sx_for(int64_t G, int C) {
    const int64_t gmax = (G + C - 1) / C;   // most groups any CTA of the cluster gets
    return static_cast<int>(gmax * kGroup + 16);  // 2*SX = 32 mod 128: conflict-free B loads
}

Plan plan_gemv(int64_t M, int64_t N, int64_t K, const DeviceInfo &dev) {
    const int64_t G = (K + kGroup - 1) / kGroup;
    Plan pl{};
    pl.WR = M <= 4 ? 1 : (M <= 16 ? 2 : 8);
    pl.WK = 8 / pl.WR;
    const int64_t tiles = (N + 16 * pl.WR - 1) / (16 * pl.WR);
    int C = 1;
    while (C < 8 && 2 * C <= G &&
           (tiles * C < 2 * dev.sms || smem_for(M, sx_for(G, C), pl.WR, pl.WK) > kGemvSmemMax))
        C *= 2;
    pl.C = C;
    pl.SX = sx_for(G, C);
    pl.smem = smem_for(M, pl.SX, pl.WR, pl.WK);
    return pl;
}

template <int BITS, int NT>
tq_status launch_typed(const GemvParams &p, const Plan &pl, int64_t tiles,
                       const DeviceInfo &dev, cudaStream_t s) {
    auto kern = k_gemv_a16<BITS, NT, 4>;
    static int configured_for[64] = {0};  // per device: max dynamic smem set
    if (dev.id >= 0 && dev.id < 64 && !configured_for[dev.id]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(kGemvSmemMax));
        if (e != cudaSuccess) return cuda_fail(e);
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        (void)e;
        cudaGetLastError();
        configured_for[dev.id] = 1;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(tiles * pl.C), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = pl.smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    int na = 0;
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
    if (pl.C > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = pl.C;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, p);
    return e == cudaSuccess ? TQ_OK : cuda_fail(e);
}

}  // namespace

bool gemv_fits(int64_t M, int64_t K, const DeviceInfo &dev) {
    if (M < 1 || M > TQ_MAX_M_A16) return false;
    const Plan pl = plan_gemv(M, 1 << 20, K, dev);
    return pl.smem <= kGemvSmemMax;
}

tq_status launch_gemv_a16(const uint16_t *X, int64_t M, int64_t K, int64_t ldx,
                          const uint8_t *Wq, const float *sw, int64_t N,
                          int bits, void *Y, int ytype, int64_t ldy,
                          const DeviceInfo &dev, cudaStream_t s) {
    const Plan pl = plan_gemv(M, N, K, dev);
    if (pl.smem > kGemvSmemMax) return TQ_ERR_SHAPE;
    GemvParams p{};
    p.X = X;
    p.ldx = ldx;
    p.M = static_cast<int>(M);
    p.K = K;
    p.G = static_cast<int>((K + kGroup - 1) / kGroup);
    p.W = Wq;
    p.wld = bits == 8 ? K : K / 2;
    p.sw = sw;
    p.N = N;
    p.Y = Y;
    p.ldy = ldy;
    p.ytype = ytype;
    p.WR = pl.WR;
    p.WK = pl.WK;
    p.C = pl.C;
    p.SX = pl.SX;
    const int64_t tiles = (N + 16 * pl.WR - 1) / (16 * pl.WR);
    const int nt = M <= 8 ? 1 : M <= 16 ? 2 : M <= 32 ? 4 : 8;
    if (bits == 8) {
        switch (nt) {
            case 1: return launch_typed<8, 1>(p, pl, tiles, dev, s);
            case 2: return launch_typed<8, 2>(p, pl, tiles, dev, s);
            case 4: return launch_typed<8, 4>(p, pl, tiles, dev, s);
            default: return launch_typed<8, 8>(p, pl, tiles, dev, s);
        }
    }
    switch (nt) {
        case 1: return launch_typed<4, 1>(p, pl, tiles, dev, s);
        case 2: return launch_typed<4, 2>(p, pl, tiles, dev, s);
        case 4: return launch_typed<4, 4>(p, pl, tiles, dev, s);
        default: return launch_typed<4, 8>(p, pl, tiles, dev, s);
    }
}

}  // namespace tq
