// Weight rotate + quantise + pack (one-time).
//
// Each weight row is cut into groups of 256 input columns (the last group may
// be a power-of-two tail of 32..128); every group is multiplied by the
// normalised Sylvester-Hadamard matrix, then the whole row is quantised with
// one fp32 scale (tensai docs, "画像生成" / Image generation, section
// "チェックポイントの入手": rotated by a Hadamard matrix every 256 input columns,
// then per-row-scaled int8; 4-bit with -q4, section "幅とメモリ").
//
// The transform runs in fp64 by a warp butterfly.  The sums of at most 256
// bf16 values are exact in fp64 whenever a group's nonzero magnitudes span
// fewer than about 37 binades, so every partial sum, whatever its order, is
// the exact value; the scale c_n = sqrt(1/n), the ratio amax/qmax, its fp32
// rounding and the quotient v'/s are single IEEE operations.  The codes and
// scales are then bit-identical to an fp64 explicit-product evaluation.
//
// One CTA (8 warps) per row; warp w takes groups w, w+8, ...  Pass 1 finds the
// row's amax, pass 2 recomputes the transform and writes codes (recomputing is
// cheaper than holding up to 64K fp64 values per row).

#include "tq_internal.cuh"

namespace tq {
namespace {

template <int E>
__device__ __forceinline__ void rotate_group64(const uint16_t *src, double (&v)[8]) {
    const int lane = threadIdx.x & 31;
    load_bf16<E, double>(src + lane * E, v);
    warp_fwht<E, double>(v);
    const double c = sqrt(1.0 / (32.0 * E));  // correctly rounded 1/sqrt(n)
#pragma unroll
    for (int e = 0; e < E; ++e) v[e] = c * v[e];
}

// Dispatch on the group width 32*E.
__device__ __forceinline__ int rotate_group64_any(const uint16_t *src, int n,
                                                  double (&v)[8]) {
    switch (n) {
        case 256: rotate_group64<8>(src, v); return 8;
        case 128: rotate_group64<4>(src, v); return 4;
        case 64: rotate_group64<2>(src, v); return 2;
        default: rotate_group64<1>(src, v); return 1;
    }
}

template <int BITS>
__global__ void __launch_bounds__(kThreads)
k_quantize_weights(const uint16_t *__restrict__ W, int64_t N, int64_t K,
                   int64_t ldw, uint8_t *__restrict__ codes,
                   float *__restrict__ scales) {
    constexpr double qmax = BITS == 8 ? 127.0 : 7.0;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t G = (K + kGroup - 1) / kGroup;
    __shared__ double red[kThreads / 32];

    for (int64_t n = blockIdx.x; n < N; n += gridDim.x) {
        const uint16_t *row = W + n * ldw;
        // pass 1: row amax of the rotated values
        double amax = 0.0;
        for (int64_t g = warp; g < G; g += kThreads / 32) {
            double v[8] = {};
            const int E = rotate_group64_any(row + g * kGroup, group_width(K, g * kGroup), v);
#pragma unroll
            for (int e = 0; e < 8; ++e)
                if (e < E) amax = fmax(amax, fabs(v[e]));
        }
#pragma unroll
        for (int m = 16; m > 0; m >>= 1) amax = fmax(amax, __shfl_xor_sync(0xffffffffu, amax, m));
        if (lane == 0) red[warp] = amax;
        __syncthreads();
        amax = red[0];
#pragma unroll
        for (int w = 1; w < kThreads / 32; ++w) amax = fmax(amax, red[w]);
        __syncthreads();  // red is reused by the next row

        const float s = static_cast<float>(amax / qmax);
        if (threadIdx.x == 0) scales[n] = s;
        const double sd = static_cast<double>(s);

        // pass 2: codes
        for (int64_t g = warp; g < G; g += kThreads / 32) {
            const int64_t g0 = g * kGroup;
            double v[8] = {};
            const int E = rotate_group64_any(row + g0, group_width(K, g0), v);
            int q[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                double r = 0.0;
                if (s != 0.0f) r = fmin(fmax(rint(v[e] / sd), -qmax), qmax);
                q[e] = static_cast<int>(r);
            }
            const int64_t k0 = g0 + static_cast<int64_t>(lane) * E;  // first column of this lane
            if constexpr (BITS == 8) {
                uint8_t *dst = codes + n * K + k0;
                uint32_t lo = 0, hi = 0;
#pragma unroll
                for (int e = 0; e < 4; ++e) lo |= (static_cast<uint32_t>(q[e]) & 0xFFu) << (8 * e);
#pragma unroll
                for (int e = 0; e < 4; ++e) hi |= (static_cast<uint32_t>(q[4 + e]) & 0xFFu) << (8 * e);
                if (E == 8) *reinterpret_cast<uint2 *>(dst) = make_uint2(lo, hi);
                else if (E == 4) *reinterpret_cast<uint32_t *>(dst) = lo;
                else if (E == 2) *reinterpret_cast<uint16_t *>(dst) = static_cast<uint16_t>(lo);
                else *dst = static_cast<uint8_t>(lo);
            } else {
                // two codes per byte, low nibble = even column
                uint32_t packed = 0;
#pragma unroll
                for (int e = 0; e < 8; ++e) packed |= (static_cast<uint32_t>(q[e]) & 0xFu) << (4 * e);
                uint8_t *dst = codes + n * (K / 2) + k0 / 2;
                if (E == 8) *reinterpret_cast<uint32_t *>(dst) = packed;
                else if (E == 4) *reinterpret_cast<uint16_t *>(dst) = static_cast<uint16_t>(packed);
                else if (E == 2) *dst = static_cast<uint8_t>(packed);
                else {
                    // one code per lane: even lanes pair with their odd neighbour
                    const uint32_t other = __shfl_down_sync(0xffffffffu, packed, 1);
                    if (!(lane & 1)) *dst = static_cast<uint8_t>((packed & 0xFu) | ((other & 0xFu) << 4));
                }
            }
        }
    }
}

}  // namespace

tq_status launch_quantize_weights(const uint16_t *W, int64_t N, int64_t K,
                                  int64_t ldw, int bits, void *codes,
                                  float *scales, cudaStream_t s) {
    const int64_t grid = N < (1ll << 30) ? N : (1ll << 30);
    if (bits == 8)
        k_quantize_weights<8><<<static_cast<unsigned>(grid), kThreads, 0, s>>>(
            W, N, K, ldw, static_cast<uint8_t *>(codes), scales);
    else
        k_quantize_weights<4><<<static_cast<unsigned>(grid), kThreads, 0, s>>>(
            W, N, K, ldw, static_cast<uint8_t *>(codes), scales);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? TQ_OK : cuda_fail(e);
}

}  // namespace tq
