// Decode product on block-scaled weights, M <= 8 tokens:
//   Y[m][n] = sum_b s[n][b] * sum_{k in block b} q[n][k] * x[m][k],  fp32 sums,
// one fp32 scale per block of G weight columns (G = 32, 64, 128, 256): the
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
//   - A warp then takes one weight row at a time; each lane streams 16-byte
//     chunks of codes (16 int8 or 32 int4 codes, inside one block) with
//     L1-bypassing loads, and the block scale of each chunk; the loads of the
//     next batch of chunks are issued before the current batch is used.
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
// Resident CTAs per SM the register budget is set for: four (64 registers a
// thread), three (80) for four and eight tokens, whose sums need the room and
// whose staged rows allow few CTAs an SM anyway.
__host__ __device__ constexpr int blk_min_ctas(int MT) { return MT >= 4 ? 3 : 4; }

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

template <int BITS, int MT>
__global__ void __launch_bounds__(kBlkThreads, blk_min_ctas(MT))
k_gemv_blocked(const BlockedParams p) {
    extern __shared__ __align__(16) float xs[];   // [MT][K] fp32, swizzled 16-byte units
    constexpr int UNR = MT <= 2 ? 2 : 1;          // chunks a batch per lane (two batches in flight)
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
    const int64_t nb = K / p.G;
    const int cshift = __ffs(p.G / KPC) - 1;       // chunk -> block: c >> cshift

    for (int64_t n = static_cast<int64_t>(blockIdx.x) * (kBlkThreads / 32) + warp; n < p.N;
         n += static_cast<int64_t>(gridDim.x) * (kBlkThreads / 32)) {
        const uint8_t *wrow = p.W + n * rb;
        const float *srow = p.sw + n * nb;
        float acc[MT];
#pragma unroll
        for (int m = 0; m < MT; ++m) acc[m] = 0.0f;
        // chunks c0 .. c0 + 32 (UNR - 1) of this lane, zeros past the row's end
        auto load_batch = [&](int c0, uint4 (&q)[UNR], float (&s)[UNR]) {
#pragma unroll
            for (int u = 0; u < UNR; ++u) {
                const int c = c0 + 32 * u;
                if (c < C) {
                    q[u] = ldg_stream(wrow + (static_cast<int64_t>(c) << 4));
                    s[u] = __ldg(srow + (c >> cshift));
                } else {
                    q[u] = make_uint4(0, 0, 0, 0);
                    s[u] = 0.0f;
                }
            }
        };
        // two batches in flight: the next one is loaded before this one is used
        uint4 qn[UNR];
        float sn[UNR];
        load_batch(lane, qn, sn);
        for (int c0 = lane; c0 < C; c0 += 32 * UNR) {
            uint4 q[UNR];
            float s[UNR];
#pragma unroll
            for (int u = 0; u < UNR; ++u) {
                q[u] = qn[u];
                s[u] = sn[u];
            }
            if (c0 + 32 * UNR < C) load_batch(c0 + 32 * UNR, qn, sn);
#pragma unroll
            for (int u = 0; u < UNR; ++u) {
                const int c = c0 + 32 * u;
                if (c >= C) break;
                const uint32_t w[4] = {q[u].x, q[u].y, q[u].z, q[u].w};
                float part[MT];
#pragma unroll
                for (int m = 0; m < MT; ++m) part[m] = 0.0f;
                if constexpr (BITS == 8) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const uint32_t wb = w[j] ^ 0x80808080u;
                        const float f0 = i8_to_f32(wb, 0), f1 = i8_to_f32(wb, 1);
                        const float f2 = i8_to_f32(wb, 2), f3 = i8_to_f32(wb, 3);
                        const int ph = xunit(c * 4 + j);
#pragma unroll
                        for (int m = 0; m < MT; ++m) {
                            const float4 xv = xs4[m * U + ph];
                            part[m] = fmaf(f0, xv.x, part[m]);
                            part[m] = fmaf(f1, xv.y, part[m]);
                            part[m] = fmaf(f2, xv.z, part[m]);
                            part[m] = fmaf(f3, xv.w, part[m]);
                        }
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 4; ++i) {          // word i: codes 8i .. 8i + 7, x units 2i, 2i + 1
                        const uint32_t wb = w[i] ^ 0x88888888u;
                        const uint32_t lo = wb & 0x0F0F0F0Fu;          // byte b: code 8i + 2b, plus 8
                        const uint32_t hi = (wb >> 4) & 0x0F0F0F0Fu;   // byte b: code 8i + 2b + 1, plus 8
#pragma unroll
                        for (int h = 0; h < 2; ++h) {                  // x unit 2i + h: bytes 2h, 2h + 1
                            const float f0 = i4b_to_f32(lo, 2 * h), f1 = i4b_to_f32(hi, 2 * h);
                            const float f2 = i4b_to_f32(lo, 2 * h + 1), f3 = i4b_to_f32(hi, 2 * h + 1);
                            const int ph = xunit(c * 8 + 2 * i + h);
#pragma unroll
                            for (int m = 0; m < MT; ++m) {
                                const float4 xv = xs4[m * U + ph];
                                part[m] = fmaf(f0, xv.x, part[m]);
                                part[m] = fmaf(f1, xv.y, part[m]);
                                part[m] = fmaf(f2, xv.z, part[m]);
                                part[m] = fmaf(f3, xv.w, part[m]);
                            }
                        }
                    }
                }
#pragma unroll
                for (int m = 0; m < MT; ++m) acc[m] = fmaf(s[u], part[m], acc[m]);
            }
        }
#pragma unroll
        for (int m = 0; m < MT; ++m) {
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) acc[m] += __shfl_xor_sync(0xffffffffu, acc[m], off);
        }
        if (lane == 0) {
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                if (m >= p.M) break;
                if (p.ytype == 0)
                    static_cast<float *>(p.Y)[m * p.ldy + n] = acc[m];
                else
                    static_cast<uint16_t *>(p.Y)[m * p.ldy + n] = f32_to_bf16_bits(acc[m]);
            }
        }
    }
}

template <int BITS, int MT>
tq_status launch_mt(const BlockedParams &p, const DeviceInfo &dev, cudaStream_t s) {
    const size_t smem = static_cast<size_t>(MT) * p.K * 4;
    static bool attr_set[64] = {};
    if (smem > 48 * 1024 && dev.id < 64 && !attr_set[dev.id]) {
        const cudaError_t e = cudaFuncSetAttribute(k_gemv_blocked<BITS, MT>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   dev.smem_optin);
        if (e != cudaSuccess) return cuda_fail(e);
        attr_set[dev.id] = true;
    }
    // resident CTAs per SM: as the register bound allows, fewer when the staged
    // rows (plus the 1 KB each CTA reserves) do not fit the SM's 228 KB
    int occ = static_cast<int>((228 * 1024) / (smem + 1024));
    occ = occ < 1 ? 1 : (occ > blk_min_ctas(MT) ? blk_min_ctas(MT) : occ);
    const int64_t need = (p.N + kBlkThreads / 32 - 1) / (kBlkThreads / 32);
    const int64_t wave = static_cast<int64_t>(dev.sms) * occ;
    const unsigned grid = static_cast<unsigned>(need < wave ? need : wave);
    k_gemv_blocked<BITS, MT><<<grid, kBlkThreads, smem, s>>>(p);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? TQ_OK : cuda_fail(e);
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
