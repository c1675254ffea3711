// Activation rotation: a 256-wide fast Walsh-Hadamard transform per group of
// each token row, fused with the per-token symmetric int8 quantisation (A8),
// or rounded to bf16 (A16 operand).  The input rows of a product get the same
// rotation as the weights, "viewing a row as groups of 256 and taking one
// product with H" (tensai docs, "画像生成" / Image generation, section
// "幅とメモリ"); the device quantises each product's activations finely
// (section "GPU"), here with one scale per token over all of K.
//
// Memory-bound: read 2 B and write 1 B (A8) or 2 B (A16) per element.  Each
// lane moves 16-byte vectors; one warp holds one 256-group (8 values a lane)
// through the whole butterfly in registers and shuffles.

#include "tq_internal.cuh"

namespace tq {
namespace {

__device__ __forceinline__ uint32_t quant4(const float *v, float s) {
    uint32_t w = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        int q = 0;
        if (s != 0.0f) q = min(max(__float2int_rn(__fdiv_rn(v[e], s)), -127), 127);
        w |= (static_cast<uint32_t>(q) & 0xFFu) << (8 * e);
    }
    return w;
}

// One CTA (8 warps) per token row.  Warp w owns groups w, w+8, ...; the first
// GPW of them stay in registers between the amax pass and the quantise pass,
// any further ones are recomputed (rows longer than 8*GPW*256).
template <int GPW>
__global__ void __launch_bounds__(kThreads)
k_rotate_quant_act(const uint16_t *__restrict__ X, int64_t M, int64_t K,
                   int64_t ldx, int8_t *__restrict__ Xq, float *__restrict__ sx) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr int W = kThreads / 32;
    const int64_t G = (K + kGroup - 1) / kGroup;
    __shared__ float red[W];

    for (int64_t m = blockIdx.x; m < M; m += gridDim.x) {
        const uint16_t *row = X + m * ldx;
        float v[GPW][8];
        int E[GPW];
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < GPW; ++i) {
            const int64_t g = warp + static_cast<int64_t>(i) * W;
#pragma unroll
            for (int e = 0; e < 8; ++e) v[i][e] = 0.0f;
            E[i] = 0;
            if (g < G) E[i] = rotate_group32_any(row + g * kGroup, group_width(K, g * kGroup), v[i]);
#pragma unroll
            for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(v[i][e]));
        }
        for (int64_t g = warp + static_cast<int64_t>(GPW) * W; g < G; g += W) {
            float t[8] = {};
            rotate_group32_any(row + g * kGroup, group_width(K, g * kGroup), t);
#pragma unroll
            for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(t[e]));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        if (lane == 0) red[warp] = amax;
        __syncthreads();
        amax = red[0];
#pragma unroll
        for (int w = 1; w < W; ++w) amax = fmaxf(amax, red[w]);
        __syncthreads();

        const float s = __fdiv_rn(amax, 127.0f);
        if (threadIdx.x == 0) sx[m] = s;
        int8_t *qrow = Xq + m * K;

        auto store = [&](int64_t g, int e_per_lane, const float *vals) {
            int8_t *dst = qrow + g * kGroup + static_cast<int64_t>(lane) * e_per_lane;
            const uint32_t lo = quant4(vals, s);
            if (e_per_lane == 8) {
                const uint32_t hi = quant4(vals + 4, s);
                *reinterpret_cast<uint2 *>(dst) = make_uint2(lo, hi);
            } else if (e_per_lane == 4) {
                *reinterpret_cast<uint32_t *>(dst) = lo;
            } else if (e_per_lane == 2) {
                *reinterpret_cast<uint16_t *>(dst) = static_cast<uint16_t>(lo);
            } else {
                *reinterpret_cast<uint8_t *>(dst) = static_cast<uint8_t>(lo);
            }
        };
#pragma unroll
        for (int i = 0; i < GPW; ++i) {
            const int64_t g = warp + static_cast<int64_t>(i) * W;
            if (g < G) store(g, E[i], v[i]);
        }
        for (int64_t g = warp + static_cast<int64_t>(GPW) * W; g < G; g += W) {
            float t[8] = {};
            const int e = rotate_group32_any(row + g * kGroup, group_width(K, g * kGroup), t);
            store(g, e, t);
        }
    }
}

// One warp per (token row, group): the rotated row rounded to bf16.
__global__ void __launch_bounds__(kThreads)
k_rotate_bf16(const uint16_t *__restrict__ X, int64_t M, int64_t K, int64_t ldx,
              uint16_t *__restrict__ Xr) {
    const int lane = threadIdx.x & 31;
    const int64_t G = (K + kGroup - 1) / kGroup;
    const int64_t total = M * G;
    const int64_t wpb = kThreads / 32;
    for (int64_t w = blockIdx.x * wpb + (threadIdx.x >> 5); w < total;
         w += static_cast<int64_t>(gridDim.x) * wpb) {
        const int64_t m = w / G, g = w % G;
        float v[8] = {};
        const int E = rotate_group32_any(X + m * ldx + g * kGroup, group_width(K, g * kGroup), v);
        uint32_t p[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
            p[i] = static_cast<uint32_t>(f32_to_bf16_bits(v[2 * i])) |
                   (static_cast<uint32_t>(f32_to_bf16_bits(v[2 * i + 1])) << 16);
        uint16_t *dst = Xr + m * K + g * kGroup + static_cast<int64_t>(lane) * E;
        if (E == 8) *reinterpret_cast<uint4 *>(dst) = make_uint4(p[0], p[1], p[2], p[3]);
        else if (E == 4) *reinterpret_cast<uint2 *>(dst) = make_uint2(p[0], p[1]);
        else if (E == 2) *reinterpret_cast<uint32_t *>(dst) = p[0];
        else *dst = static_cast<uint16_t>(p[0]);
    }
}

}  // namespace

tq_status launch_rotate_quant_act(const uint16_t *X, int64_t M, int64_t K,
                                  int64_t ldx, int8_t *Xq, float *sx,
                                  cudaStream_t s) {
    const int64_t G = (K + kGroup - 1) / kGroup;
    const int64_t gpw = (G + 7) / 8;
    const unsigned grid = static_cast<unsigned>(M < (1ll << 30) ? M : (1ll << 30));
    if (gpw <= 1) k_rotate_quant_act<1><<<grid, kThreads, 0, s>>>(X, M, K, ldx, Xq, sx);
    else if (gpw <= 2) k_rotate_quant_act<2><<<grid, kThreads, 0, s>>>(X, M, K, ldx, Xq, sx);
    else if (gpw <= 4) k_rotate_quant_act<4><<<grid, kThreads, 0, s>>>(X, M, K, ldx, Xq, sx);
    else k_rotate_quant_act<6><<<grid, kThreads, 0, s>>>(X, M, K, ldx, Xq, sx);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? TQ_OK : cuda_fail(e);
}

tq_status launch_rotate_bf16(const uint16_t *X, int64_t M, int64_t K,
                             int64_t ldx, uint16_t *Xr, cudaStream_t s) {
    const int64_t G = (K + kGroup - 1) / kGroup;
    const int64_t warps = M * G;
    int64_t blocks = (warps + 7) / 8;
    if (blocks > (1ll << 30)) blocks = 1ll << 30;
    k_rotate_bf16<<<static_cast<unsigned>(blocks), kThreads, 0, s>>>(X, M, K, ldx, Xr);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? TQ_OK : cuda_fail(e);
}

}  // namespace tq
