// Decode product on block-scaled weights, M <= 8 tokens:
//   Y[m][n] = sum_b s[n][b] * sum_{k in block b} q[n][k] * x[m][k],  fp32 sums,
// one fp32 scale per block of G weight columns (G = 32, 64, 128, 256; G = 0,
// one scale per row, serves the per-row format's large single-token calls): the
// blocks with a shared scale of the GGML formats and kvad's own q8 (kvad-gpu
// internals, "Quantised weights on the GPU").  With rotate = 1 the weights
// were rotated before quantisation and x is the token row's group-256
// Hadamard rotation rounded to bf16, as in the per-row A16 product (tensai
// docs, "画像生成" / Image generation, section "幅とメモリ"); with rotate = 0 both
// are used as they are (the unrotated format).
//
// Decode is bound by the weight stream (kvad-gpu internals, "Numbers"), so the
// kernel is built to keep HBM busy:
//   - Each CTA first stages the token rows in shared memory as fp32 (rotating
//     them itself when asked), in 16-byte units swizzled so that the warp's
//     vector reads below hit distinct banks.
//   - A warp then takes two adjacent weight rows at a time when the matrix
//     has rows enough to fill every SM that way and there are at most two
//     tokens (else one), so that each x value read from shared memory serves
//     both;
//     each lane streams 16-byte chunks of codes (16 int8 or 32 int4 codes,
//     inside one block) with L1-bypassing loads, and the block scale of each
//     chunk; the next chunk of each row is loaded before this one is used.
//   - Codes are widened to fp32 exactly (the biased byte, or nibble masked
//     into a byte, is placed in the mantissa of 2^23 and the bias
//     subtracted: one byte permute and one add a code), multiplied with x into a
//     per-chunk partial sum, and the partial is added into the row sum times
//     the chunk's block scale.
//   - A shuffle tree sums the lanes; lane 0 stores the M outputs.
// The CTA count is a whole number of waves over the SMs; rows are taken in a
// grid-stride loop, so any grid is correct.

#include "tq_internal.cuh"

namespace tq {
namespace {

struct BlockedParams {
    const uint16_t *X;
    int64_t ldx;
    int M;
    int64_t K;
    const uint8_t *W;
    const float *sw;
    int G;
    int64_t N;
    void *Y;
    int64_t ldy;
    int ytype;
    int rotate;
};

constexpr int kBlkThreads = 256;
// Chunks of each row a lane loads per batch: two while the sums are few (at
// most two token-row pairs), else one.
__host__ __device__ constexpr int blk_unr(int MT, int RW) { return MT * RW <= 2 ? 2 : 1; }
// Resident CTAs per SM the register budget is set for: four (64 registers a
// thread), three (80) for four and eight tokens, whose sums need the room and
// whose staged rows allow few CTAs an SM anyway, and for two-chunk batches.
__host__ __device__ constexpr int blk_min_ctas(int BITS, int MT, int RW) {
    return MT >= 4 || blk_unr(MT, RW) == 2 ? 3 : 4;
}

// Swizzled position of 16-byte unit u of a staged token row: bits 3..5 of u
// are folded into bits 0..2, so the eight lanes of a vector-load phase, which
// read units 4l + j (int8) or 8l + j (int4), land in eight distinct bank groups.
__device__ __forceinline__ int xunit(int u) { return u ^ ((u >> 3) & 7); }

__device__ __forceinline__ void stage_x(float *xs, int k, float v) { xs[xunit(k >> 2) * 4 + (k & 3)] = v; }

// Exact fp32 value of the signed byte i of w: the biased byte b ^ 0x80 placed
// in the low mantissa bits of 2^23, minus 2^23 + 128.
__device__ __forceinline__ float i8_to_f32(uint32_t wb, int i) {
    return __int_as_float(static_cast<int>(__byte_perm(wb, 0x4B000000u, 0x7650u + i))) - 8388736.0f;
}

// Exact fp32 value of an int4 code held biased (code + 8, 0..15) in byte i of
// t: placed in the low mantissa bits of 2^23, minus 2^23 + 8.
__device__ __forceinline__ float i4b_to_f32(uint32_t t, int i) {
    return __int_as_float(static_cast<int>(__byte_perm(t, 0x4B000000u, 0x7650u + i))) - 8388616.0f;
}

template <int BITS, int MT, int RW>
__global__ void __launch_bounds__(kBlkThreads, blk_min_ctas(BITS, MT, RW))
k_gemv_blocked(const BlockedParams p) {
    extern __shared__ __align__(16) float xs[];   // [MT][K] fp32, swizzled 16-byte units
    constexpr int UNR = blk_unr(MT, RW);    // RW: weight rows a warp takes at once
    constexpr int KPC = 128 / BITS;               // codes per 16-byte chunk
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t K = p.K;

    // ---- stage the token rows (rows M..MT-1 are zero)
    if (p.rotate) {
        const int64_t NG = (K + kGroup - 1) / kGroup;
        for (int64_t it = warp; it < static_cast<int64_t>(p.M) * NG; it += kBlkThreads / 32) {
            const int m = static_cast<int>(it / NG);
            const int64_t g0 = (it % NG) * kGroup;
            float v[8] = {};
            const int E = rotate_group32_any(p.X + m * p.ldx + g0, group_width(K, g0), v);
#pragma unroll
            for (int e = 0; e < 8; ++e)
                if (e < E)
                    stage_x(xs + m * K, static_cast<int>(g0) + lane * E + e,
                            bf16_bits_to_f32(f32_to_bf16_bits(v[e])));
        }
    } else {
        const int K2 = static_cast<int>(K >> 1);   // two bf16 a word (K even, rows 16-byte aligned)
        for (int m = 0; m < p.M; ++m) {
            const uint32_t *row = reinterpret_cast<const uint32_t *>(p.X + m * p.ldx);
            for (int k2 = threadIdx.x; k2 < K2; k2 += kBlkThreads) {
                const uint32_t w = __ldg(row + k2);
                stage_x(xs + m * K, 2 * k2, __uint_as_float(w << 16));
                stage_x(xs + m * K, 2 * k2 + 1, __uint_as_float(w & 0xFFFF0000u));
            }
        }
    }
    for (int i = p.M * static_cast<int>(K) + threadIdx.x; i < MT * static_cast<int>(K); i += kBlkThreads)
        xs[i] = 0.0f;
    __syncthreads();

    const float4 *xs4 = reinterpret_cast<const float4 *>(xs);
    // K <= 65536: unit and chunk indices fit 32 bits
    const int U = static_cast<int>(K >> 2);        // 16-byte units of a staged row
    const int64_t rb = K * BITS / 8;               // code bytes of a weight row
    const int C = static_cast<int>(rb >> 4);       // 16-byte chunks of a weight row
    // G == 0: one scale per row (the per-row format of tq_quantize_weights)
    const int64_t nb = p.G ? K / p.G : 1;
    const int cshift = p.G ? __ffs(p.G / KPC) - 1 : 31;   // chunk -> block: c >> cshift
    const int64_t nsets = (p.N + RW - 1) / RW;

    for (int64_t set = static_cast<int64_t>(blockIdx.x) * (kBlkThreads / 32) + warp; set < nsets;
         set += static_cast<int64_t>(gridDim.x) * (kBlkThreads / 32)) {
        const int64_t n0 = set * RW;
        const uint8_t *wrow[RW];
        const float *srow[RW];
        bool valid[RW];
#pragma unroll
        for (int r = 0; r < RW; ++r) {
            valid[r] = n0 + r < p.N;
            const int64_t n = valid[r] ? n0 + r : n0;
            wrow[r] = p.W + n * rb;
            srow[r] = p.sw + n * nb;
        }
        float acc[RW][MT];
#pragma unroll
        for (int r = 0; r < RW; ++r)
#pragma unroll
            for (int m = 0; m < MT; ++m) acc[r][m] = 0.0f;
        // chunks c0 + 32 u of each row (zeros past the row's end or for a row past N)
        auto load_batch = [&](int c0, uint4 (&q)[RW][UNR], float (&sc)[RW][UNR]) {
#pragma unroll
            for (int u = 0; u < UNR; ++u) {
                const int c = c0 + 32 * u;
#pragma unroll
                for (int r = 0; r < RW; ++r) {
                    if (c < C && valid[r]) {
                        q[r][u] = ldg_stream(wrow[r] + (static_cast<int64_t>(c) << 4));
                        sc[r][u] = __ldg(srow[r] + (c >> cshift));
                    } else {
                        q[r][u] = make_uint4(0, 0, 0, 0);
                        sc[r][u] = 0.0f;
                    }
                }
            }
        };
        // two batches in flight: the next is loaded before this one is used
        uint4 qn[RW][UNR];
        float sn[RW][UNR];
        load_batch(lane, qn, sn);
        for (int c0 = lane; c0 < C; c0 += 32 * UNR) {
            uint4 qb[RW][UNR];
            float sb[RW][UNR];
#pragma unroll
            for (int r = 0; r < RW; ++r)
#pragma unroll
                for (int u = 0; u < UNR; ++u) {
                    qb[r][u] = qn[r][u];
                    sb[r][u] = sn[r][u];
                }
            if (c0 + 32 * UNR < C) load_batch(c0 + 32 * UNR, qn, sn);
#pragma unroll
            for (int u = 0; u < UNR; ++u) {
            const int c = c0 + 32 * u;
            if (c >= C) break;
            uint4 q[RW];
            float sc[RW];
#pragma unroll
            for (int r = 0; r < RW; ++r) {
                q[r] = qb[r][u];
                sc[r] = sb[r][u];
            }
            float part[RW][MT];
#pragma unroll
            for (int r = 0; r < RW; ++r)
#pragma unroll
                for (int m = 0; m < MT; ++m) part[r][m] = 0.0f;
            // the chunk's x units are xunit(first) ^ o for o = 0 .. units - 1: the
            // first unit is a multiple of the unit count (4 or 8), so the fold of
            // bits 3..5 is the same for all of them
            if constexpr (BITS == 8) {
                const int base = xunit(c * 4);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    float f[RW][4];
#pragma unroll
                    for (int r = 0; r < RW; ++r) {
                        const uint32_t wj = j == 0 ? q[r].x : (j == 1 ? q[r].y : (j == 2 ? q[r].z : q[r].w));
                        const uint32_t wb = wj ^ 0x80808080u;
#pragma unroll
                        for (int i = 0; i < 4; ++i) f[r][i] = i8_to_f32(wb, i);
                    }
#pragma unroll
                    for (int m = 0; m < MT; ++m) {
                        const float4 xv = xs4[m * U + (base ^ j)];
#pragma unroll
                        for (int r = 0; r < RW; ++r) {
                            part[r][m] = fmaf(f[r][0], xv.x, part[r][m]);
                            part[r][m] = fmaf(f[r][1], xv.y, part[r][m]);
                            part[r][m] = fmaf(f[r][2], xv.z, part[r][m]);
                            part[r][m] = fmaf(f[r][3], xv.w, part[r][m]);
                        }
                    }
                }
            } else {
                const int base = xunit(c * 8);
#pragma unroll
                for (int i = 0; i < 4; ++i) {           // word i: codes 8i .. 8i + 7, x units 2i, 2i + 1
                    uint32_t lo[RW], hi[RW];
#pragma unroll
                    for (int r = 0; r < RW; ++r) {
                        const uint32_t wi = i == 0 ? q[r].x : (i == 1 ? q[r].y : (i == 2 ? q[r].z : q[r].w));
                        const uint32_t wb = wi ^ 0x88888888u;
                        lo[r] = wb & 0x0F0F0F0Fu;               // byte b: code 8i + 2b, plus 8
                        hi[r] = (wb >> 4) & 0x0F0F0F0Fu;        // byte b: code 8i + 2b + 1, plus 8
                    }
#pragma unroll
                    for (int h = 0; h < 2; ++h) {               // x unit 2i + h: bytes 2h, 2h + 1
                        float f[RW][4];
#pragma unroll
                        for (int r = 0; r < RW; ++r) {
                            f[r][0] = i4b_to_f32(lo[r], 2 * h);
                            f[r][1] = i4b_to_f32(hi[r], 2 * h);
                            f[r][2] = i4b_to_f32(lo[r], 2 * h + 1);
                            f[r][3] = i4b_to_f32(hi[r], 2 * h + 1);
                        }
#pragma unroll
                        for (int m = 0; m < MT; ++m) {
                            const float4 xv = xs4[m * U + (base ^ (2 * i + h))];
#pragma unroll
                            for (int r = 0; r < RW; ++r) {
                                part[r][m] = fmaf(f[r][0], xv.x, part[r][m]);
                                part[r][m] = fmaf(f[r][1], xv.y, part[r][m]);
                                part[r][m] = fmaf(f[r][2], xv.z, part[r][m]);
                                part[r][m] = fmaf(f[r][3], xv.w, part[r][m]);
                            }
                        }
                    }
                }
            }
#pragma unroll
            for (int r = 0; r < RW; ++r)
#pragma unroll
                for (int m = 0; m < MT; ++m) acc[r][m] = fmaf(sc[r], part[r][m], acc[r][m]);
            }
        }
#pragma unroll
        for (int r = 0; r < RW; ++r)
#pragma unroll
            for (int m = 0; m < MT; ++m)
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) acc[r][m] += __shfl_xor_sync(0xffffffffu, acc[r][m], off);
        if (lane == 0) {
#pragma unroll
            for (int r = 0; r < RW; ++r) {
                if (!valid[r]) break;
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    if (m >= p.M) break;
                    if (p.ytype == 0)
                        static_cast<float *>(p.Y)[m * p.ldy + n0 + r] = acc[r][m];
                    else
                        static_cast<uint16_t *>(p.Y)[m * p.ldy + n0 + r] = f32_to_bf16_bits(acc[r][m]);
                }
            }
        }
    }
}

template <int BITS, int MT, int RW>
tq_status launch_rw(const BlockedParams &p, const DeviceInfo &dev, cudaStream_t s) {
    const size_t smem = static_cast<size_t>(MT) * p.K * 4;
    static bool attr_set[64] = {};
    if (smem > 48 * 1024 && dev.id < 64 && !attr_set[dev.id]) {
        const cudaError_t e = cudaFuncSetAttribute(k_gemv_blocked<BITS, MT, RW>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   dev.smem_optin);
        if (e != cudaSuccess) return cuda_fail(e);
        attr_set[dev.id] = true;
    }
    // resident CTAs per SM: as the kernel's registers allow (64K a SM, taken in
    // steps of 8 a thread), fewer when the staged rows (plus the 1 KB each CTA
    // reserves) do not fit the SM's 228 KB
    static int regs[64] = {};
    if (dev.id < 64 && regs[dev.id] == 0) {
        cudaFuncAttributes fa;
        const cudaError_t e = cudaFuncGetAttributes(&fa, k_gemv_blocked<BITS, MT, RW>);
        if (e != cudaSuccess) return cuda_fail(e);
        regs[dev.id] = fa.numRegs > 0 ? fa.numRegs : 64;
    }
    const int r8 = ((dev.id < 64 ? regs[dev.id] : 80) + 7) / 8 * 8;
    const int occ_regs = 65536 / (r8 * kBlkThreads);
    int occ = static_cast<int>((228 * 1024) / (smem + 1024));
    occ = occ > occ_regs ? occ_regs : occ;
    occ = occ < 1 ? 1 : (occ > 8 ? 8 : occ);
    const int64_t need = ((p.N + RW - 1) / RW + kBlkThreads / 32 - 1) / (kBlkThreads / 32);
    const int64_t wave = static_cast<int64_t>(dev.sms) * occ;
    const unsigned grid = static_cast<unsigned>(need < wave ? need : wave);
    k_gemv_blocked<BITS, MT, RW><<<grid, kBlkThreads, smem, s>>>(p);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? TQ_OK : cuda_fail(e);
}

// Two rows a warp only when they still fill every SM with three CTAs (up to
// two tokens): fewer, longer warps stream better, but a short matrix would
// leave SMs idle.
template <int BITS, int MT>
tq_status launch_mt(const BlockedParams &p, const DeviceInfo &dev, cudaStream_t s) {
    if (MT <= 2 && p.N >= static_cast<int64_t>(2) * (kBlkThreads / 32) * 3 * dev.sms)
        return launch_rw<BITS, MT, (MT <= 2 ? 2 : 1)>(p, dev, s);
    return launch_rw<BITS, MT, 1>(p, dev, s);
}

template <int BITS>
tq_status launch_bits(const BlockedParams &p, const DeviceInfo &dev, cudaStream_t s) {
    if (p.M <= 1) return launch_mt<BITS, 1>(p, dev, s);
    if (p.M <= 2) return launch_mt<BITS, 2>(p, dev, s);
    if (p.M <= 4) return launch_mt<BITS, 4>(p, dev, s);
    return launch_mt<BITS, 8>(p, dev, s);
}

}  // namespace

int gemv_blocked_mt(int M) { return M <= 1 ? 1 : (M <= 2 ? 2 : (M <= 4 ? 4 : 8)); }

tq_status launch_gemv_blocked(const uint16_t *X, int M, int64_t K, int64_t ldx, const uint8_t *Wq,
                              const float *sw, int G, int64_t N, int bits, int rotate, void *Y, int ytype,
                              int64_t ldy, const DeviceInfo &dev, cudaStream_t s) {
    if (M == 0 || N == 0) return TQ_OK;
    const BlockedParams p{X, ldx, M, K, Wq, sw, G, N, Y, ldy, ytype, rotate};
    return bits == 8 ? launch_bits<8>(p, dev, s) : launch_bits<4>(p, dev, s);
}

}  // namespace tq
