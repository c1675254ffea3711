// Skinny A16 product for M <= 64 (decode and batched decode):
//   Y[m][n] = sw[n] * sum_k q_w[n][k] * x'_bf16[m][k],  fp32 sums,
// where x' is the group-256 Hadamard rotation of the token row rounded to bf16
// (tensai docs, "画像生成" / Image generation, section "幅とメモリ": the input of
// the product gets the same rotation as the weights).  Decode is bound by the
// weight stream (kvad-gpu internals, "Numbers": decode is memory-bound).
//
// One call moves a few MB, so latency, not bandwidth, decides its time.  The
// kernel is laid out so that the weight stream never waits for anything:
//   1. Each CTA owns RT = 16*WR weight rows and a K range of whole 256-groups
//      (C CTAs of a thread-block cluster split K).  Its first thread issues
//      bulk copies (cp.async.bulk, through L2) of the CTA's whole weight slice
//      into shared memory, then lets the next kernel on the stream launch
//      (programmatic dependent launch), so the next calls' weight streams
//      start while this call still computes.
//   2. Only then does it wait for the previous kernel (griddepcontrol.wait),
//      rotate its K range of every token row in fp32 (warp butterfly), round
//      to bf16 and keep it in shared memory.
//   3. Warps widen int8/int4 codes to exact bf16 pairs in registers and feed
//      mma.sync m16n8k16 from shared memory.
//   4. Partial sums are added in a fixed order: warps along K through shared
//      memory, then the CTAs of the cluster through distributed shared memory
//      (no atomics: repeated calls give identical bytes).
// Weights are read before the wait, so Wq/sw must not be written by a kernel
// that may still be running when this one starts (only this library's product
// kernels trigger early, and they write Y alone).
// Every wait is bounded: on expiry the kernel sets the library status word and
// skips its arithmetic (tq_device_status reports it), never hangs.

#include <cooperative_groups.h>

#include "tq_a16.cuh"

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
    int WS;         // shared row stride of the weight slice (bytes, = 64 mod 128)
    int SX;         // shared row stride of x' (bf16 elements, 2*SX = 32 mod 128)
    int w_off, x_off;  // byte offsets of the weight slice and of x' in shared memory
    unsigned int *status;
};

constexpr unsigned int kStatusGemvTimeout = 1u;

template <int BITS, int NT>
__global__ void __launch_bounds__(kThreads)
k_gemv_a16(const GemvParams p) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem_raw);
    unsigned char *ws = smem_raw + p.w_off;
    uint16_t *xs = reinterpret_cast<uint16_t *>(smem_raw + p.x_off);
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
    const int rows = static_cast<int>(min(static_cast<int64_t>(RT), p.N - n0));
    const uint32_t wbar = smem_addr(bar);

    // ---- 1. weight slice -> shared memory, before anything else
    if (warp == 0) {
        if (lane == 0) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(wbar));
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
            asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(wbar),
                         "r"(static_cast<uint32_t>(rows * rbytes))
                         : "memory");
        }
        __syncwarp();
        for (int r = lane; r < rows; r += 32) {
            const unsigned char *src = p.W + (n0 + r) * p.wld + wbyte0;
            asm volatile(
                "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                ::"r"(smem_addr(ws + r * p.WS)), "l"(src), "r"(static_cast<uint32_t>(rbytes)), "r"(wbar)
                : "memory");
        }
    } else if (warp == 1) {
        // the token rows this CTA rotates: warm L2 (coherent, so safe before the wait)
        for (int m = lane; m < p.M; m += 32)
            prefetch_l2(p.X + m * p.ldx + kbeg, static_cast<uint32_t>(nk * 2));
    }
    // the row scales of this tile, read under the same rule as the weights
    float *sws = reinterpret_cast<float *>(smem_raw + 128);  // [RT], before the weight slice
    if (threadIdx.x < rows) sws[threadIdx.x] = __ldg(p.sw + n0 + threadIdx.x);
    pdl_launch_dependents();
    pdl_wait();

    // ---- 2. rotated, bf16-rounded x' of this K range in shared memory.  The
    // warp that writes a token's last group also zeroes the padding of the
    // last (partial) K block, so one barrier covers both.
    const int M = p.M, SX = p.SX;
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
        if (gi == ngrp - 1) {
            for (int kl = nk + lane; kl < nblk * KB; kl += 32)
                xrow[(kl / KB) * KB + xpos<BITS>(kl % KB)] = 0;
        }
    }
    __syncthreads();

    // ---- 3. products from shared memory
    const bool have_w = mbar_wait_bounded(wbar, 0);
    if (!have_w && threadIdx.x == 0) atomicOr(p.status, kStatusGemvTimeout);
    const int WR = p.WR, WK = p.WK;
    const int wr = warp % WR, wk = warp / WR;
    const int g = lane >> 2, t = lane & 3;
    const int rA = wr * 16 + g, rB = rA + 8;
    const bool okA = rA < rows, okB = rB < rows;
    const unsigned char *pA = ws + rA * p.WS + t * 16;
    const unsigned char *pB = ws + rB * p.WS + t * 16;
    const int nbw = (have_w && nblk > wk) ? (nblk - wk + WK - 1) / WK : 0;

    // two accumulator sets, alternating by mma index, halve the dependent chain
    float acc[NT][4], acc2[NT][4];
#pragma unroll
    for (int i = 0; i < NT; ++i) {
        acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.0f;
        acc2[i][0] = acc2[i][1] = acc2[i][2] = acc2[i][3] = 0.0f;
    }
    const uint16_t *xb[NT];
    bool xin[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int tok = nt * 8 + g;
        xin[nt] = tok < M;
        xb[nt] = xs + (xin[nt] ? tok : 0) * SX + 4 * t;
    }
    auto mma_all = [&](int blk, int jj, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            uint2 bv = make_uint2(0, 0);
            if (xin[nt]) bv = *reinterpret_cast<const uint2 *>(xb[nt] + blk * KB + jj * 16);
            mma_bf16((jj & 1) ? acc2[nt] : acc[nt], a0, a1, a2, a3, bv.x, bv.y);
        }
    };
    for (int i = 0; i < nbw; ++i) {
        const int blk = wk + i * WK;
        const int off = blk * BB;
        const bool in = off + t * 16 < rbytes;
        const uint4 wa = (in && okA) ? *reinterpret_cast<const uint4 *>(pA + off) : make_uint4(0, 0, 0, 0);
        const uint4 wb = (in && okB) ? *reinterpret_cast<const uint4 *>(pB + off) : make_uint4(0, 0, 0, 0);
        const uint32_t A[4] = {wa.x, wa.y, wa.z, wa.w};
        const uint32_t B[4] = {wb.x, wb.y, wb.z, wb.w};
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

    // ---- 4. reduction: warps along K, then CTAs of the cluster, fixed order
    __syncthreads();
    float *red = reinterpret_cast<float *>(smem_raw + p.x_off);  // [WK][RT][M], over x'
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int row = wr * 16 + g + 8 * h;
            const int m0 = nt * 8 + 2 * t;
            if (m0 < M) red[(wk * RT + row) * M + m0] = acc[nt][2 * h] + acc2[nt][2 * h];
            if (m0 + 1 < M) red[(wk * RT + row) * M + m0 + 1] = acc[nt][2 * h + 1] + acc2[nt][2 * h + 1];
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
    if (crank == 0 && have_w) {
        for (int idx = threadIdx.x; idx < RM; idx += kThreads) {
            const int m = idx / RT, r = idx % RT;
            const int li = r * M + m;
            float s = red[li];
            for (int q = 1; q < C; ++q) s += cg::this_cluster().map_shared_rank(red, q)[li];
            const int64_t n = n0 + r;
            if (n < p.N) {
                const float y = sws[r] * s;
                if (p.ytype == 0)
                    static_cast<float *>(p.Y)[m * p.ldy + n] = y;
                else
                    static_cast<uint16_t *>(p.Y)[m * p.ldy + n] = f32_to_bf16_bits(y);
            }
        }
    }
    if (C > 1) cg::this_cluster().sync();
    // never leave with bulk copies still landing in this CTA's shared memory
    if (!have_w) mbar_wait_bounded(wbar, 0, kA16DrainLimit);
}

struct Plan {
    int WR, WK, C, WS, SX, w_off, x_off;
    size_t smem;
};

constexpr size_t kGemvSmemMax = 200 * 1024;

Plan make_plan(int64_t M, int64_t K, int bits, int WR, int C) {
    const int64_t G = (K + kGroup - 1) / kGroup;
    const int64_t gmax = (G + C - 1) / C;       // most groups any CTA of the cluster gets
    Plan pl{};
    pl.WR = WR;
    pl.WK = 8 / WR;
    pl.C = C;
    const int64_t kr = gmax * kGroup;
    const int64_t rb = kr * bits / 8;
    pl.WS = static_cast<int>((rb + 127) / 128 * 128 + 64);  // 64 mod 128: conflict-free A loads
    pl.SX = static_cast<int>(kr + 16);                     // 2*SX = 32 mod 128: B loads
    const int RT = 16 * WR;
    pl.w_off = 128 + (4 * RT + 127) / 128 * 128;  // barrier, then the row scales
    pl.x_off = pl.w_off + RT * pl.WS;
    const size_t xs = static_cast<size_t>(M) * pl.SX * 2;
    const size_t red = static_cast<size_t>(pl.WK) * RT * M * 4;
    pl.smem = static_cast<size_t>(pl.x_off) + (xs > red ? xs : red);
    return pl;
}

Plan plan_gemv(int64_t M, int64_t N, int64_t K, int bits, const DeviceInfo &dev) {
    const int64_t G = (K + kGroup - 1) / kGroup;
    Plan pl{};
    // prefer more rows per CTA for more tokens (x' is shared by the rows);
    // fall back to fewer rows when the slices do not fit in shared memory
    for (int WR = M <= 4 ? 1 : (M <= 16 ? 2 : 8); WR >= 1; WR /= 2) {
        const int64_t tiles = (N + 16 * WR - 1) / (16 * WR);
        int C = 1;
        pl = make_plan(M, K, bits, WR, C);
        // split K over a cluster until the slices fit and the grid covers the GPU
        while (2 * C <= G &&
               ((C < 8 && tiles * C < dev.sms) || (C < 16 && pl.smem > 96 * 1024))) {
            C *= 2;
            pl = make_plan(M, K, bits, WR, C);
        }
        if (pl.smem <= kGemvSmemMax) return pl;
    }
    return pl;
}

template <int BITS, int NT>
tq_status launch_typed(const GemvParams &p, const Plan &pl, int64_t tiles,
                       const DeviceInfo &dev, cudaStream_t s) {
    auto kern = k_gemv_a16<BITS, NT>;
    static int configured_for[64] = {0};  // per device: max dynamic smem set
    if (dev.id >= 0 && dev.id < 64 && !configured_for[dev.id]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(kGemvSmemMax));
        if (e != cudaSuccess) return cuda_fail(e);
        // clusters of 16 CTAs (the largest split of K, used for M up to 64)
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return cuda_fail(e);
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

bool gemv_fits(int64_t M, int64_t K, int bits, const DeviceInfo &dev) {
    if (M < 1 || M > TQ_MAX_M_A16) return false;
    return plan_gemv(M, 1 << 20, K, bits, dev).smem <= kGemvSmemMax;
}

tq_status launch_gemv_a16(const uint16_t *X, int64_t M, int64_t K, int64_t ldx,
                          const uint8_t *Wq, const float *sw, int64_t N,
                          int bits, void *Y, int ytype, int64_t ldy,
                          const DeviceInfo &dev, cudaStream_t s) {
    const Plan pl = plan_gemv(M, N, K, bits, dev);
    if (pl.smem > kGemvSmemMax) return TQ_ERR_SHAPE;
    unsigned int *status = status_word();
    if (!status) return TQ_ERR_DEVICE;
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
    p.WS = pl.WS;
    p.SX = pl.SX;
    p.w_off = pl.w_off;
    p.x_off = pl.x_off;
    p.status = status;
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
