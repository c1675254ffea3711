// Activation rotation: a 256-wide fast Walsh-Hadamard transform per group of
// each token row, fused with the per-token symmetric int8 quantisation (A8),
// or rounded to bf16 (A16 operand).  The input rows of a product get the same
// rotation as the weights: each row is cut into 256-wide groups and each group
// is multiplied by H (tensai docs, "画像生成" / Image generation, section
// "幅とメモリ"); on the device the activations of each product are quantised
// at a finer grain than the weights (section "GPU"), here one scale per token
// over all of K.
//
// Memory-bound: read 2 B and write 1 B (A8) or 2 B (A16) per element.  One
// warp holds one 256-group (8 values a lane) through the whole butterfly in
// registers and shuffles.  For the A8 path, rows of up to 16384 values are
// streamed through a ring of shared-memory row buffers filled by bulk copies
// several rows ahead (persistent CTAs), so the HBM reads of the next rows
// overlap the transform, amax and stores of the current one; longer rows use
// a plain one-CTA-per-row kernel that loads each group straight from global.

#include <cfloat>
#include <type_traits>

#include "tq_internal.cuh"

namespace tq {
namespace {

// Code of one value: clamp(rint(v / s)) with the quotient correctly rounded
// (IEEE division), as the scale formula reads.  r = 1/s when that is finite,
// else 0.  The product t = v * r is within a few ulps of v / s (|v / s| <= 127
// here, an ulp at most 2^-17), so rint(t) equals rint of the rounded quotient
// unless t lies near a half-integer; only there is the division taken.
__device__ __forceinline__ int quant_code(float v, float s, float r) {
    if (s == 0.0f) return 0;
    float t = v * r;
    if (r == 0.0f || fabsf((t - floorf(t)) - 0.5f) < 1e-3f) t = __fdiv_rn(v, s);
    return min(max(__float2int_rn(t), -127), 127);
}

__device__ __forceinline__ float recip_or_zero(float s) {
    const float r = __frcp_rn(s);
    return (s != 0.0f && isfinite(r)) ? r : 0.0f;
}

__device__ __forceinline__ uint32_t quant4(const float *v, float s, float r) {
    uint32_t w = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e)
        w |= (static_cast<uint32_t>(quant_code(v[e], s, r)) & 0xFFu) << (8 * e);
    return w;
}

constexpr long long kWaitLimit = 4000000000ll;  // clock cycles (about 2 s)
constexpr unsigned int kStatusActTimeout = 8u;
constexpr int64_t kRingMaxK = TQ_MAX_K_TILED;    // longest row the ring path takes

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

// SwiGLU of one gate value g and up value u, h = silu(g) * u with
// silu(g) = g / (1 + e^-g) (Shazeer, "GLU Variants Improve Transformer"), in
// fp32; the caller rounds h to bf16, as an unfused SwiGLU kernel would store it.
// The exponential and the division are the hardware's approximate ones
// (__expf, __fdividef): a relative error of a few parts in 10^6 at most for
// |g| < 16, so h's bf16 rounding (a step of 2^-8) differs from that of the
// exact value only for the rare h within that distance of a rounding tie, and
// it cuts this pass's arithmetic to about a third.  For g <= -87 the quotient
// is 0 (|h| < 1e-36 |u|), as the exact fp32 form gives -0 below -88.7.
__device__ __forceinline__ float silu_mul(float g, float u) {
    return __fdividef(g, 1.0f + __expf(-g)) * u;
}

// Two bf16 values a word: h = bf16(silu(g) * u) of the gate word and up word.
__device__ __forceinline__ uint32_t swiglu_word(uint32_t gw, uint32_t uw) {
    const float h0 = silu_mul(__uint_as_float(gw << 16), __uint_as_float(uw << 16));
    const float h1 = silu_mul(__uint_as_float(gw & 0xFFFF0000u), __uint_as_float(uw & 0xFFFF0000u));
    return f32_to_bf16_bits(h0) | (static_cast<uint32_t>(f32_to_bf16_bits(h1)) << 16);
}

// The lane's E bf16 values (E = 8, 4, 2, 1) at src as packed words; with
// SWIGLU, those of h = bf16(silu(g) * u), g at src and u at src + up_off.
template <bool SWIGLU>
__device__ __forceinline__ void lane_words(const unsigned char *src, int up_off, int E, uint32_t (&w)[4]) {
    auto load = [&](const unsigned char *a, uint32_t (&o)[4]) {
        o[0] = o[1] = o[2] = o[3] = 0u;
        if (E == 8) {
            const uint4 u = *reinterpret_cast<const uint4 *>(a);
            o[0] = u.x; o[1] = u.y; o[2] = u.z; o[3] = u.w;
        } else if (E == 4) {
            const uint2 u = *reinterpret_cast<const uint2 *>(a);
            o[0] = u.x; o[1] = u.y;
        } else if (E == 2) {
            o[0] = *reinterpret_cast<const uint32_t *>(a);
        } else {
            o[0] = *reinterpret_cast<const uint16_t *>(a);
        }
    };
    load(src, w);
    if constexpr (SWIGLU) {
        uint32_t u[4];
        load(src + up_off, u);
#pragma unroll
        for (int i = 0; i < 4; ++i) w[i] = swiglu_word(w[i], u[i]);
    }
}

// Rotate one group (width n = 32*E) read from a shared-memory row buffer:
// v = c_n * Hs_n * x in fp32, the same butterfly and scale as the global path.
template <bool SWIGLU>
__device__ __forceinline__ int rotate_group_shared(const unsigned char *grp, int up_off, int n, float (&v)[8]) {
    const int lane = threadIdx.x & 31;
    uint32_t w[4];
    const int E = n >> 5;
    lane_words<SWIGLU>(grp + lane * E * 2, up_off, E, w);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        v[2 * i] = __uint_as_float(w[i] << 16);
        v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
    switch (E) {
        case 8: warp_fwht<8, float>(v); break;
        case 4: warp_fwht<4, float>(v); break;
        case 2: warp_fwht<2, float>(v); break;
        default: warp_fwht<1, float>(v); break;
    }
    const float c = sqrtf(1.0f / static_cast<float>(n));
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] = e < E ? c * v[e] : 0.0f;
    return E;
}

__device__ __forceinline__ void store_codes(int8_t *dst, int e_per_lane, const float *vals, float s,
                                            float r) {
    const uint32_t lo = quant4(vals, s, r);
    if (e_per_lane == 8) {
        const uint32_t hi = quant4(vals + 4, s, r);
        *reinterpret_cast<uint2 *>(dst) = make_uint2(lo, hi);
    } else if (e_per_lane == 4) {
        *reinterpret_cast<uint32_t *>(dst) = lo;
    } else if (e_per_lane == 2) {
        *reinterpret_cast<uint16_t *>(dst) = static_cast<uint16_t>(lo);
    } else {
        *reinterpret_cast<uint8_t *>(dst) = static_cast<uint8_t>(lo);
    }
}

// Unnormalised transform (Hs x, Sylvester order) of one full 256-group read
// from a shared-memory row buffer: 8 values a lane.
template <bool SWIGLU>
__device__ __forceinline__ void fwht256_shared(const unsigned char *grp, int up_off, float (&v)[8]) {
    const int lane = threadIdx.x & 31;
    uint32_t w[4];
    lane_words<SWIGLU>(grp + lane * 16, up_off, 8, w);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        v[2 * i] = __uint_as_float(w[i] << 16);
        v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
    warp_fwht<8, float>(v);
}

// Code of one rotated value x = k * v (k a power of two, so x is exact):
// rint(x / s) with the quotient correctly rounded, as a float (|code| <= 127;
// no clamp is needed, as |x| <= amax and s = amax / 127 rounded give
// |x / s| <= 127 (1 + 2^-23) < 127.5).  rk = k / s when that is a normal
// number, else 0.  v * rk is within a few ulps of x / s (an ulp at most
// 2^-17 here), so its rounding matches that of the exact quotient unless it
// lies near a half-integer; only there, or without rk, is the division taken.
__device__ __forceinline__ float code_of(float v, float k, float rk, float s) {
    const float t = v * rk;
    float q = rintf(t);
    if (rk == 0.0f || fabsf(t - q) > 0.499f) q = s == 0.0f ? 0.0f : rintf(__fdiv_rn(v * k, s));
    return q;
}

__device__ __forceinline__ void put_int8(int8_t *dst, int e_per_lane, const float (&q)[8]) {
    uint32_t w[2] = {0u, 0u};
#pragma unroll
    for (int e = 0; e < 8; ++e)
        if (e < e_per_lane) w[e >> 2] |= (static_cast<uint32_t>(__float2int_rz(q[e])) & 0xFFu) << (8 * (e & 3));
    if (e_per_lane == 8) *reinterpret_cast<uint2 *>(dst) = make_uint2(w[0], w[1]);
    else if (e_per_lane == 4) *reinterpret_cast<uint32_t *>(dst) = w[0];
    else if (e_per_lane == 2) *reinterpret_cast<uint16_t *>(dst) = static_cast<uint16_t>(w[0]);
    else *reinterpret_cast<uint8_t *>(dst) = static_cast<uint8_t>(w[0]);
}

// The codes as fp16 in the tensor core's operand layout: tile (m / 128,
// k / 64) is the 8192 values at ((m / 128) * KT + k / 64) * 8192; inside it,
// 8x8 core matrices of 128 contiguous bytes, K-adjacent ones 128 bytes apart,
// row groups 1024 bytes apart.  A lane's E values (columns k0 .. k0 + E - 1,
// k0 a multiple of E) are contiguous there.  Where K % 64 == 32 the tail
// group's lanes also write the zeros that pad the last tile.
__device__ __forceinline__ void put_tiled(uint16_t *At, int64_t KT, int64_t K, int64_t m, int64_t k0,
                                          int E, const float (&q)[8]) {
    const int64_t mt = m >> 7;
    const int rr = static_cast<int>(m & 127);
    auto at = [&](int64_t k) {
        const int kk = static_cast<int>(k & 63);
        return At + ((mt * KT + (k >> 6)) << 13) + ((((rr >> 3) << 3) + (kk >> 3)) << 6) + ((rr & 7) << 3) +
               (kk & 7);
    };
    uint32_t h[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __half2 p = __floats2half2_rn(q[2 * i], q[2 * i + 1]);   // exact: small integers
        h[i] = *reinterpret_cast<const uint32_t *>(&p);
    }
    uint16_t *dst = at(k0);
    if (E == 8) {
        *reinterpret_cast<uint4 *>(dst) = make_uint4(h[0], h[1], h[2], h[3]);
    } else if (E == 4) {
        *reinterpret_cast<uint2 *>(dst) = make_uint2(h[0], h[1]);
    } else if (E == 2) {
        *reinterpret_cast<uint32_t *>(dst) = h[0];
    } else {
        *dst = static_cast<uint16_t>(h[0]);
        if ((K & 63) == 32) *at(k0 + 32) = 0;
    }
}

// Persistent CTAs (8 warps); CTA b takes rows b, b + gridDim.x, ...  Thread 0
// keeps S rows in flight: row i of this CTA goes to buffer i % S, copied by
// one bulk copy that completes on that buffer's barrier.  Warp w owns groups
// w, w + 8, ...; the first GPW stay in registers between the amax pass and
// the quantise pass, further ones are recomputed from the buffer.
// SWIGLU: the row is h = bf16(silu(g) * u), gate rows from X (ldx) and up
// rows from U (ldu); a buffer then holds a gate row and an up row.
template <int GPW, bool TILED, int NT, bool SWIGLU = false>
__global__ void __launch_bounds__(NT, NT == 128 ? 5 : 2)   // 5 CTAs of 4 warps, or 2 of 8, an SM
k_rotate_quant_ring(const uint16_t *__restrict__ X, int64_t M, int64_t K, int64_t ldx,
                    void *__restrict__ out, float *__restrict__ sx, int S,
                    unsigned int *status, unsigned int *max_l1, const uint16_t *__restrict__ U,
                    int64_t ldu) {
    extern __shared__ __align__(128) unsigned char ring[];   // [S][2K or 4K] then S barriers
    __shared__ float red[NT / 32];
    __shared__ unsigned int win[16];   // a row's sum of |codes| per 1024-column window
    __shared__ unsigned int winq[16];  // a row's sum of codes squared per 1024-column window
    __shared__ unsigned int run_sh[2][5][32];   // warp 0's largest run sums over the rows
    __shared__ int abort_sh;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr int W = NT / 32;
    const int64_t Gf = K / kGroup;                        // full 256-groups
    const int tail = static_cast<int>(K % kGroup);        // 0, 32, 64 or 128
    const int tail_warp = static_cast<int>(Gf % W);
    const uint32_t row_bytes = static_cast<uint32_t>(K * 2);
    const uint32_t slot_bytes = SWIGLU ? 2 * row_bytes : row_bytes;
    const int up_off = static_cast<int>(row_bytes);   // the up row, after the gate row (SWIGLU)
    const uint32_t ring0 = static_cast<uint32_t>(__cvta_generic_to_shared(ring));
    const uint32_t bar0 = ring0 + static_cast<uint32_t>(S) * slot_bytes;
    const int64_t nrows = blockIdx.x < M ? (M - 1 - blockIdx.x) / gridDim.x + 1 : 0;

    auto issue = [&](int64_t i) {   // thread 0: row i of this CTA into buffer i % S
        const int slot = static_cast<int>(i % S);
        const uint32_t bar = bar0 + 8u * slot;
        const int64_t m = blockIdx.x + i * gridDim.x;
        const uint16_t *src = X + m * ldx;
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(slot_bytes)
                     : "memory");
        asm volatile(
            "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
            ::"r"(ring0 + static_cast<uint32_t>(slot) * slot_bytes), "l"(src), "r"(row_bytes), "r"(bar)
            : "memory");
        if constexpr (SWIGLU) {
            asm volatile(
                "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                ::"r"(ring0 + static_cast<uint32_t>(slot) * slot_bytes + row_bytes), "l"(U + m * ldu),
                  "r"(row_bytes), "r"(bar)
                : "memory");
        }
    };

    if (threadIdx.x < 16) win[threadIdx.x] = winq[threadIdx.x] = 0;
    if (TILED && threadIdx.x < 32)
        for (int j = 0; j < 5; ++j) run_sh[0][j][threadIdx.x] = run_sh[1][j][threadIdx.x] = 0u;
    if (threadIdx.x == 0) {
        abort_sh = 0;
        for (int i = 0; i < S; ++i)
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar0 + 8u * i));
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        for (int64_t i = 0; i < nrows && i < S; ++i) issue(i);
    }
    __syncthreads();

    int64_t i = 0;
    for (; i < nrows; ++i) {
        const int slot = static_cast<int>(i % S);
        const uint32_t parity = static_cast<uint32_t>((i / S) & 1);
        const long long t0 = clock64();
        bool ok = true;
        while (!mbar_try(bar0 + 8u * slot, parity)) {
            if (abort_sh || clock64() - t0 > kWaitLimit) { ok = false; break; }
        }
        if (!ok) {
            abort_sh = 1;
            if (lane == 0) atomicOr(status, kStatusActTimeout);
        }
        __syncthreads();
        if (abort_sh) break;
        const unsigned char *buf = ring + static_cast<size_t>(slot) * slot_bytes;
        const int64_t m = blockIdx.x + i * gridDim.x;

        // Pass 1: the full 256-groups unscaled (Hs x; their factor 1/16 is a
        // power of two, applied exactly later), the tail group scaled.
        float v[GPW][8];
        float amax_full = 0.0f, amax_tail = 0.0f;
#pragma unroll
        for (int j = 0; j < GPW; ++j) {
            const int64_t g = warp + static_cast<int64_t>(j) * W;
            if (g < Gf) {
                fwht256_shared<SWIGLU>(buf + g * kGroup * 2, up_off, v[j]);
#pragma unroll
                for (int e = 0; e < 8; ++e) amax_full = fmaxf(amax_full, fabsf(v[j][e]));
            }
        }
        for (int64_t g = warp + static_cast<int64_t>(GPW) * W; g < Gf; g += W) {
            float t[8];
            fwht256_shared<SWIGLU>(buf + g * kGroup * 2, up_off, t);
#pragma unroll
            for (int e = 0; e < 8; ++e) amax_full = fmaxf(amax_full, fabsf(t[e]));
        }
        float vt[8];
        int Et = 0;
        if (tail && warp == tail_warp) {
            Et = rotate_group_shared<SWIGLU>(buf + Gf * kGroup * 2, up_off, tail, vt);
#pragma unroll
            for (int e = 0; e < 8; ++e) amax_tail = fmaxf(amax_tail, fabsf(vt[e]));
        }
        // max |c x| over the row: fl(c v) is monotone in |v|, so the largest
        // scaled value of the full groups is (largest unscaled) / 16 exactly
        float amax = fmaxf(amax_full * 0.0625f, amax_tail);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        if (lane == 0) red[warp] = amax;
        __syncthreads();
        amax = red[0];
#pragma unroll
        for (int w = 1; w < W; ++w) amax = fmaxf(amax, red[w]);

        const float s = __fdiv_rn(amax, 127.0f);
        const float r = recip_or_zero(s);
        const float r16 = r * 0.0625f >= FLT_MIN ? r * 0.0625f : 0.0f;   // exact: a power of two
        if (threadIdx.x == 0) sx[m] = s;
        const int64_t KT = (K + 63) >> 6;
        // with the tiled operand, also the row's sum of |codes| per 1024-column
        // window (each at most 127 * 1024) and its sum of codes squared per
        // window (a whole row at most 127^2 * 16384 < 2^32)
        auto put = [&](int64_t g, int e, const float (&q)[8]) {
            const int64_t k0 = g * kGroup + static_cast<int64_t>(lane) * e;
            if constexpr (TILED) {
                put_tiled(static_cast<uint16_t *>(out), KT, K, m, k0, e, q);
                float fs = 0.0f, fq = 0.0f;      // exact: at most 8 x 127 and 8 x 127^2
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    if (j < e) {
                        fs += fabsf(q[j]);
                        fq = fmaf(q[j], q[j], fq);
                    }
                const unsigned int gs = __reduce_add_sync(0xffffffffu, static_cast<unsigned int>(fs));
                const unsigned int gq = __reduce_add_sync(0xffffffffu, static_cast<unsigned int>(fq));
                if (lane == 0) {
                    atomicAdd(&win[g >> 2], gs);
                    atomicAdd(&winq[g >> 2], gq);
                }
            } else
                put_int8(static_cast<int8_t *>(out) + m * K + k0, e, q);
        };
        // Pass 2: codes.  Full groups: x = v / 16.  Tail: x = v.
#pragma unroll
        for (int j = 0; j < GPW; ++j) {
            const int64_t g = warp + static_cast<int64_t>(j) * W;
            if (g < Gf) {
                float q[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) q[e] = code_of(v[j][e], 0.0625f, r16, s);
                put(g, 8, q);
            }
        }
        for (int64_t g = warp + static_cast<int64_t>(GPW) * W; g < Gf; g += W) {
            float t[8], q[8];
            fwht256_shared<SWIGLU>(buf + g * kGroup * 2, up_off, t);
#pragma unroll
            for (int e = 0; e < 8; ++e) q[e] = code_of(t[e], 0.0625f, r16, s);
            put(g, 8, q);
        }
        if (Et) {
            float q[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) q[e] = code_of(vt[e], 1.0f, r, s);
            put(Gf, Et, q);
        }
        // This thread's reads of the buffer are ordered before the bulk copy
        // (async proxy) that will refill it; the barrier then makes every
        // thread's reads, and the reads of red[], precede the refill.
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncthreads();
        if (TILED && warp == 0) {
            // lane l holds window l (1024 columns; zero past K).  Sums over
            // aligned runs of 2^j windows by butterfly within aligned lane
            // groups; each lane keeps its largest over the rows in run_sh (the
            // maximum over the lanes and CTAs is taken once, after the last row).
            unsigned int ws = lane < 16 ? win[lane] : 0u;
            unsigned int wq = lane < 16 ? winq[lane] : 0u;
            if (lane < 16) win[lane] = winq[lane] = 0;
#pragma unroll
            for (int j = 0; j < 5; ++j) {
                if (j > 0) {
                    ws += __shfl_xor_sync(0xffffffffu, ws, 1 << (j - 1));
                    wq += __shfl_xor_sync(0xffffffffu, wq, 1 << (j - 1));
                }
                run_sh[0][j][lane] = max(run_sh[0][j][lane], ws);
                run_sh[1][j][lane] = max(run_sh[1][j][lane], wq);
            }
        }
        if (threadIdx.x == 0 && i + S < nrows) issue(i + S);
    }
    // Trailer: word 1 + j the largest sum of |codes| over an aligned run of
    // 2^j windows, word 0 over a whole row (16 windows hold the longest row);
    // words 7 + j and 6 the same for codes squared.
    if (TILED && warp == 0) {
#pragma unroll
        for (int j = 0; j < 5; ++j) {
            unsigned int mx = run_sh[0][j][lane], mq = run_sh[1][j][lane];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                mq = max(mq, __shfl_xor_sync(0xffffffffu, mq, o));
            }
            if (lane == 0 && nrows > 0) {
                atomicMax(max_l1 + 1 + j, mx);
                atomicMax(max_l1 + 7 + j, mq);
                if (j == 4) {
                    atomicMax(max_l1, mx);
                    atomicMax(max_l1 + 6, mq);
                }
            }
        }
    }
    // After an expired wait, let the copies still in flight land (bounded)
    // before the CTA's shared memory is released.
    if (threadIdx.x == 0 && i < nrows) {
        const long long t0 = clock64();
        for (int64_t j = i; j < nrows && j < i + S; ++j) {
            while (!mbar_try(bar0 + 8u * static_cast<uint32_t>(j % S), static_cast<uint32_t>((j / S) & 1)) &&
                   clock64() - t0 < kWaitLimit) {
            }
        }
    }
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
        const float r = recip_or_zero(s);
        if (threadIdx.x == 0) sx[m] = s;
        int8_t *qrow = Xq + m * K;

        auto store = [&](int64_t g, int e_per_lane, const float *vals) {
            store_codes(qrow + g * kGroup + static_cast<int64_t>(lane) * e_per_lane, e_per_lane, vals, s, r);
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

template <bool TILED, bool SWIGLU = false>
tq_status launch_ring(const uint16_t *X, int64_t M, int64_t K, int64_t ldx, void *out, float *sx,
                      unsigned int *max_l1, cudaStream_t s, const uint16_t *U = nullptr, int64_t ldu = 0) {
    const int64_t G = (K + kGroup - 1) / kGroup;
    // rows of up to 16 groups: CTAs of 4 warps, more of them, so that more
    // rows are in flight per SM; longer rows: 8 warps
    const bool small = G <= 16;
    const int NT = small ? 128 : 256;
    const int64_t gpw = (G + NT / 32 - 1) / (NT / 32);
    DeviceInfo dev;
    const tq_status ds = current_device(&dev);
    if (ds != TQ_OK) return ds;
    unsigned int *status = status_word();
    if (!status) return TQ_ERR_DEVICE;
    // rows in flight per CTA: about 48 KB of them (24 KB with 4 warps), 2 to 8 rows
    // (a gate and an up row per buffer with SWIGLU)
    const int64_t rb = (SWIGLU ? 4 : 2) * K;
    int S = static_cast<int>(((small ? 24 : 48) * 1024) / rb);
    S = S < 2 ? 2 : (S > 8 ? 8 : S);
    const size_t smem = static_cast<size_t>(S) * rb + 8 * S;
    auto pick = [&](auto nt) {
        constexpr int N = decltype(nt)::value;
        return gpw <= 1 ? k_rotate_quant_ring<1, TILED, N, SWIGLU>
             : gpw <= 2 ? k_rotate_quant_ring<2, TILED, N, SWIGLU>
             : gpw <= 4 ? k_rotate_quant_ring<4, TILED, N, SWIGLU>
                        : k_rotate_quant_ring<8, TILED, N, SWIGLU>;
    };
    auto kern = small ? pick(std::integral_constant<int, 128>{}) : pick(std::integral_constant<int, 256>{});
    const int ki = (gpw <= 1 ? 0 : gpw <= 2 ? 1 : gpw <= 4 ? 2 : 3) + (small ? 4 : 0);
    static bool configured[64][8] = {{false}};
    if (dev.id < 0 || dev.id >= 64) return TQ_ERR_DEVICE;
    if (!configured[dev.id][ki]) {
        // the largest ring: two of the longest rows (gate and up rows with SWIGLU)
        const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   static_cast<int>(kRingMaxK * (SWIGLU ? 4 : 2) * 2 + 64));
        if (e != cudaSuccess) return cuda_fail(e);
        configured[dev.id][ki] = true;
    }
    // persistent: as many CTAs as are resident at once, at most 4 (8 with 4 warps) per SM
    int per_sm = 0;
    const cudaError_t oe = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, NT, smem);
    if (oe != cudaSuccess) return cuda_fail(oe);
    const int cap = small ? 8 : 4;
    per_sm = per_sm < 1 ? 1 : (per_sm > cap ? cap : per_sm);
    const int64_t want = static_cast<int64_t>(dev.sms) * per_sm;
    const unsigned grid = static_cast<unsigned>(M < want ? M : want);
    kern<<<grid, NT, smem, s>>>(X, M, K, ldx, out, sx, S, status, max_l1, U, ldu);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? TQ_OK : cuda_fail(e);
}

}  // namespace

int64_t tiled_act_tiles_bytes(int64_t M, int64_t K) {
    return ((M + 255) / 256) * 2 * ((K + 63) / 64) * 16384;
}

int64_t tiled_act_bytes(int64_t M, int64_t K) { return tiled_act_tiles_bytes(M, K) + 256; }

tq_status launch_rotate_quant_tiled(const uint16_t *X, int64_t M, int64_t K, int64_t ldx,
                                    void *At, float *sx, cudaStream_t s) {
    if (M == 0) return TQ_OK;
    if (K > kRingMaxK) return TQ_ERR_SHAPE;
    unsigned int *max_l1 = reinterpret_cast<unsigned int *>(static_cast<unsigned char *>(At) +
                                                            tiled_act_tiles_bytes(M, K));
    const cudaError_t e = cudaMemsetAsync(max_l1, 0, 12 * sizeof(unsigned int), s);
    if (e != cudaSuccess) return cuda_fail(e);
    return launch_ring<true>(X, M, K, ldx, At, sx, max_l1, s);
}

tq_status launch_swiglu_quant_tiled(const uint16_t *G, int64_t ldg, const uint16_t *U, int64_t ldu,
                                    int64_t M, int64_t K, void *At, float *sx, cudaStream_t s) {
    if (M == 0) return TQ_OK;
    if (K > kRingMaxK) return TQ_ERR_SHAPE;
    unsigned int *max_l1 = reinterpret_cast<unsigned int *>(static_cast<unsigned char *>(At) +
                                                            tiled_act_tiles_bytes(M, K));
    const cudaError_t e = cudaMemsetAsync(max_l1, 0, 12 * sizeof(unsigned int), s);
    if (e != cudaSuccess) return cuda_fail(e);
    return launch_ring<true, true>(G, M, K, ldg, At, sx, max_l1, s, U, ldu);
}

tq_status launch_rotate_quant_act(const uint16_t *X, int64_t M, int64_t K,
                                  int64_t ldx, int8_t *Xq, float *sx,
                                  cudaStream_t s) {
    const int64_t G = (K + kGroup - 1) / kGroup;
    const int64_t gpw = (G + 7) / 8;
    if (M == 0) return TQ_OK;
    if (K <= kRingMaxK) return launch_ring<false>(X, M, K, ldx, Xq, sx, nullptr, s);
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
