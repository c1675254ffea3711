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

#include <cuda_fp16.h>

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

// Store the E codes of this lane (columns k0 .. k0 + E - 1 of row n):
// int8 as bytes, int4 two per byte with the low nibble the even column.
template <int BITS>
__device__ __forceinline__ void store_codes(uint8_t *codes, int64_t n, int64_t K, int64_t k0, int E,
                                            const int (&q)[8]) {
    const int lane = threadIdx.x & 31;
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
            store_codes<BITS>(codes, n, K, g0 + static_cast<int64_t>(lane) * E, E, q);
        }
    }
}

// Block-scaled variant: one scale per block of G columns (G = 32, 64, 128 or
// 256, dividing K) instead of one per row; the blocks with a shared scale of
// the GGML formats and kvad's own q8 (kvad-gpu internals, "Quantised weights
// on the GPU"), taken of the rotated row (rotate = 1) or of the bf16 weights
// as they are (rotate = 0).  Every group width is a multiple of G, so a block
// lies inside one group: the warp that transforms a group also finds each of
// its blocks' amax (a shuffle reduction over the G/E lanes holding it), the
// scale and the codes, in one pass.  Exactness as above: the fp64 values, the
// ratio, its fp32 rounding and the quotients match the fp64 reference bit for
// bit.  One warp per (row, group) item.
template <int BITS>
__global__ void __launch_bounds__(kThreads)
k_quantize_weights_blocked(const uint16_t *__restrict__ W, int64_t N, int64_t K, int64_t ldw, int G,
                           int rotate, uint8_t *__restrict__ codes, float *__restrict__ scales) {
    constexpr double qmax = BITS == 8 ? 127.0 : 7.0;
    const int lane = threadIdx.x & 31;
    const int64_t NG = (K + kGroup - 1) / kGroup, nb = K / G;
    const int64_t items = N * NG;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * (kThreads / 32);
    for (int64_t it = static_cast<int64_t>(blockIdx.x) * (kThreads / 32) + (threadIdx.x >> 5); it < items;
         it += stride) {
        const int64_t n = it / NG, g0 = (it % NG) * kGroup;
        const int w = group_width(K, g0);
        const uint16_t *src = W + n * ldw + g0;
        double v[8] = {};
        int E;
        if (rotate) {
            E = rotate_group64_any(src, w, v);
        } else {
            E = w >> 5;
            switch (E) {
                case 8: load_bf16<8, double>(src + lane * 8, v); break;
                case 4: load_bf16<4, double>(src + lane * 4, v); break;
                case 2: load_bf16<2, double>(src + lane * 2, v); break;
                default: load_bf16<1, double>(src + lane, v); break;
            }
        }
        double amax = 0.0;
#pragma unroll
        for (int e = 0; e < 8; ++e)
            if (e < E) amax = fmax(amax, fabs(v[e]));
        const int L = G / E;                       // lanes per block: 4..32, a power of two
        for (int m = L >> 1; m > 0; m >>= 1) amax = fmax(amax, __shfl_xor_sync(0xffffffffu, amax, m));
        const float s = static_cast<float>(amax / qmax);
        const int64_t k0 = g0 + static_cast<int64_t>(lane) * E;
        if ((lane & (L - 1)) == 0) scales[n * nb + k0 / G] = s;
        const double sd = static_cast<double>(s);
        int q[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            double r = 0.0;
            if (s != 0.0f) r = fmin(fmax(rint(v[e] / sd), -qmax), qmax);
            q[e] = static_cast<int>(r);
        }
        store_codes<BITS>(codes, n, K, k0, E, q);
    }
}

// Weight codes widened once into the A8 product's own operand form: fp16 (the
// codes are small integers, so exactly), in 128-row x 64-column tiles of 8x8
// core matrices, the image the tensor core reads from shared memory.  Tile
// (nt, kt) sits at byte (nt * KT + kt) * 16384; inside it core matrix
// (r / 8, k / 8) is 128 contiguous bytes, K-adjacent ones 128 bytes apart and
// row groups 1024 bytes apart.  Rows are padded to whole 256-row tile pairs and
// columns past K to the tile edge, with zeros.  One thread writes one 16-byte
// core-matrix row: 8 codes of one weight row.
template <int BITS>
__global__ void __launch_bounds__(256)
k_tile_weights(const uint8_t *Wq, int64_t N, int64_t K, int64_t KT, int64_t Npad, uint16_t *Wt) {
    const int64_t segs = KT * 8;                       // 8-column segments per row
    const int64_t total = Npad * segs;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t n = i / segs, k0 = (i % segs) * 8;
        uint32_t h[4] = {0, 0, 0, 0};
        if (n < N && k0 < K) {                         // K is a multiple of 32: whole segments
            int c[8];
            if (BITS == 8) {
                const uint2 w = *reinterpret_cast<const uint2 *>(Wq + n * K + k0);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    c[j] = static_cast<int8_t>((w.x >> (8 * j)) & 0xFF);
                    c[4 + j] = static_cast<int8_t>((w.y >> (8 * j)) & 0xFF);
                }
            } else {
                const uint32_t w = *reinterpret_cast<const uint32_t *>(Wq + n * (K / 2) + k0 / 2);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int v = static_cast<int>((w >> (4 * j)) & 0xF);
                    c[j] = v >= 8 ? v - 16 : v;        // two's complement nibble, code k0 + j
                }
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const __half2 pr = __halves2half2(__int2half_rn(c[2 * j]), __int2half_rn(c[2 * j + 1]));
                h[j] = *reinterpret_cast<const uint32_t *>(&pr);
            }
        }
        const int64_t nt = n >> 7, kt = k0 >> 6;
        const int r = static_cast<int>(n & 127), kk = static_cast<int>(k0 & 63);
        uint16_t *dst = Wt + ((nt * KT + kt) << 13) + ((((r >> 3) << 3) + (kk >> 3)) << 6) + ((r & 7) << 3);
        *reinterpret_cast<uint4 *>(dst) = make_uint4(h[0], h[1], h[2], h[3]);
    }
}

// The largest row sums of codes squared, for the product's exactness bound:
// word 0 of the tiled weights' trailer over whole rows, word 1 + j over
// aligned runs of 2^j windows of 1024 columns (at most 127^2 * 16384 < 2^32).
// One warp per row: window w's sum is reduced over the lanes into lane w,
// then runs of windows are summed by butterfly within aligned lane groups.
template <int BITS>
__global__ void __launch_bounds__(256)
k_weight_sq(const uint8_t *Wq, int64_t N, int64_t K, unsigned int *out) {
    const int lane = threadIdx.x & 31;
    const int64_t rb = K * BITS / 8;                   // a multiple of 16
    const int64_t wb = 1024 * BITS / 8;                // bytes of a 1024-column window
    for (int64_t n = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; n < N;
         n += (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5) {
        const uint8_t *row = Wq + n * rb;
        unsigned int mine = 0;                         // lane w: window w (zero past K)
        for (int w = 0; w * wb < rb; ++w) {
            unsigned int sq = 0;
            const int64_t end = (w + 1) * wb < rb ? (w + 1) * wb : rb;
            for (int64_t b = w * wb + static_cast<int64_t>(lane) * 16; b < end; b += 32 * 16) {
                const uint4 u = __ldg(reinterpret_cast<const uint4 *>(row + b));
                const uint32_t q[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    if constexpr (BITS == 8) {
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const int c = static_cast<int8_t>((q[i] >> (8 * j)) & 0xFFu);
                            sq += static_cast<unsigned int>(c * c);
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const int v = static_cast<int>((q[i] >> (4 * j)) & 0xFu);
                            const int c = v >= 8 ? v - 16 : v;
                            sq += static_cast<unsigned int>(c * c);
                        }
                    }
                }
            }
            sq = __reduce_add_sync(0xffffffffu, sq);
            if (lane == w) mine = sq;
        }
#pragma unroll
        for (int j = 0; j < 5; ++j) {
            if (j > 0) mine += __shfl_xor_sync(0xffffffffu, mine, 1 << (j - 1));
            unsigned int mx = mine;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            if (lane == 0) {
                atomicMax(out + 1 + j, mx);
                if (j == 4) atomicMax(out, mx);
            }
        }
    }
}

}  // namespace

tq_status launch_quantize_weights_blocked(const uint16_t *W, int64_t N, int64_t K, int64_t ldw, int bits,
                                          int G, int rotate, void *codes, float *scales, cudaStream_t s) {
    const int64_t items = N * ((K + kGroup - 1) / kGroup);
    const int64_t want = (items + kThreads / 32 - 1) / (kThreads / 32);
    const unsigned grid = static_cast<unsigned>(want < (1ll << 20) ? want : (1ll << 20));
    if (grid == 0) return TQ_OK;
    if (bits == 8)
        k_quantize_weights_blocked<8><<<grid, kThreads, 0, s>>>(W, N, K, ldw, G, rotate,
                                                                 static_cast<uint8_t *>(codes), scales);
    else
        k_quantize_weights_blocked<4><<<grid, kThreads, 0, s>>>(W, N, K, ldw, G, rotate,
                                                                 static_cast<uint8_t *>(codes), scales);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? TQ_OK : cuda_fail(e);
}

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

// The tiles, then a 256-byte trailer of the largest row sums of codes squared
// (k_weight_sq).
int64_t weights_tiled_bytes(int64_t N, int64_t K) {
    return ((N + 255) / 256) * 2 * ((K + 63) / 64) * 16384 + 256;
}

tq_status launch_tile_weights(const uint8_t *Wq, int64_t N, int64_t K, int bits, void *Wt, cudaStream_t s) {
    const int64_t KT = (K + 63) / 64, Npad = (N + 255) / 256 * 256;
    const int64_t total = Npad * KT * 8;
    if (total == 0) return TQ_OK;
    const int64_t blocks = (total + 255) / 256 < 152 * 64 ? (total + 255) / 256 : 152 * 64;
    auto kern = bits == 8 ? k_tile_weights<8> : k_tile_weights<4>;
    kern<<<static_cast<unsigned>(blocks), 256, 0, s>>>(Wq, N, K, KT, Npad, static_cast<uint16_t *>(Wt));
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e);
    unsigned int *trailer = reinterpret_cast<unsigned int *>(static_cast<unsigned char *>(Wt) +
                                                             weights_tiled_bytes(N, K) - 256);
    if ((e = cudaMemsetAsync(trailer, 0, 256, s)) != cudaSuccess) return cuda_fail(e);
    const int64_t wblocks = (N + 7) / 8 < 152 * 64 ? (N + 7) / 8 : 152 * 64;   // 8 rows a block
    auto sq = bits == 8 ? k_weight_sq<8> : k_weight_sq<4>;
    sq<<<static_cast<unsigned>(wblocks), 256, 0, s>>>(Wq, N, K, trailer);
    e = cudaGetLastError();
    return e == cudaSuccess ? TQ_OK : cuda_fail(e);
}

}  // namespace tq
