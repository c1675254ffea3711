// Activation rotation: a 256-wide fast Walsh-Hadamard transform per group of
// each token row, fused with the per-token symmetric int8 quantisation (A8),
// or rounded to bf16 (A16 operand).  The input rows of a product get the same
// rotation as the weights: each row is cut into 256-wide groups and each group
// is multiplied by H (tensai docs, "画像生成" / Image generation, section
// "幅とメモリ"); on the device the activations of each product are quantised
// at a finer grain than the weights (section "GPU"), here one scale per token
// over all of K.
//
// Memory-bound in principle: read 2 B and write 1 B (int8 codes) or 2 B (fp16
// codes of the tiled operand, or the A16 bf16 operand) per element.  Rows of
// up to 16384 values go through k_rotq: one CTA per row at a time, a warp per
// 1024-column window, each 256-group held by 8 lanes x 32 values in registers
// (five butterfly stages inside a lane, three across lanes), the row's amax
// after one CTA barrier, then the codes.  Longer rows (int8 codes only) use a
// plain one-CTA-per-row kernel with a warp per group.
//
// Two row kernels that sit in front of a product are fused into k_rotq's
// prologue, so their bf16 output is never written: SwiGLU (the down
// projection's input) and the modulated layer norm (the input of a DiT
// block's QKV and gate/up products).  The pages list both among the row
// kernels next to the projections, candidates for fusion, with fp32 norms
// (TensorFold PR #948, "What comes next").

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

constexpr int64_t kRingMaxK = TQ_MAX_K_TILED;    // longest row k_rotq takes

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

// ---------------------------------------------------------------- row kernel
// A 256-group as 8 lanes x 32 values: lane j of the group holds the four runs
// of 8 columns 8 j + 64 i .. 8 j + 64 i + 7 (i = 0 .. 3), value 8 i + e being
// column 8 j + 64 i + e.  Column bits 0-2 and 6-7 are then inside a lane and
// bits 3-5 are the lane's, so five butterfly stages run inside the lane (four
// of them on two values per instruction, f32x2) and three across the group's
// 8 lanes: 3 shuffles a value instead of 5 with 8 values a lane, and the 8
// lanes of a group read 128 contiguous bytes per load.  (The transform does
// not depend on the order of its stages, only on each stage pairing the
// columns that differ in one bit, lower one first.)

__device__ __forceinline__ unsigned long long f2pack(float a, float b) {
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}

__device__ __forceinline__ void f2unpack(unsigned long long r, float &a, float &b) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}

// (a, b) <- (a + b, a - b) for two pairs at once, each sum rounded once
__device__ __forceinline__ void bfly_x2(float &a0, float &a1, float &b0, float &b1) {
    const unsigned long long a = f2pack(a0, a1), b = f2pack(b0, b1);
    unsigned long long s, d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(s) : "l"(a), "l"(b));
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    f2unpack(s, a0, a1);
    f2unpack(d, b0, b1);
}

// modnorm_value on two values at once, each operation rounded as there (the
// pair's sums and products on f32x2, one conversion to a bf16 pair).
__device__ __forceinline__ void modnorm_pair(float &x0, float &x1, unsigned long long mu2, unsigned long long r2,
                                             float sc0, float sc1, float sh0, float sh1) {
    unsigned long long d, n, k, h;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(f2pack(x0, x1)), "l"(mu2));
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(n) : "l"(d), "l"(r2));
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(k) : "l"(f2pack(sc0, sc1)), "l"(f2pack(1.0f, 1.0f)));
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(h) : "l"(n), "l"(k), "l"(f2pack(sh0, sh1)));
    float h0, h1;
    f2unpack(h, h0, h1);
    uint32_t w;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(w) : "f"(h1), "f"(h0));   // h0 in the low half
    x0 = __uint_as_float(w << 16);
    x1 = __uint_as_float(w & 0xFFFF0000u);
}

// Unnormalised transform (Hs_256 x, Sylvester order) of the group this lane's
// 8-lane slice holds; in-lane value index bits are column bits 0-2 and 6-7.
__device__ __forceinline__ void fwht_8x32(float (&v)[32]) {
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
        const float a = v[i], b = v[i + 1];
        v[i] = a + b;
        v[i + 1] = a - b;
    }
#pragma unroll
    for (int h = 2; h < 32; h <<= 1) {
#pragma unroll
        for (int i = 0; i < 32; i += 2)
            if (!(i & h)) {
                bfly_x2(v[i], v[i + 1], v[i + h], v[i + h + 1]);
            }
    }
    // across the 8 lanes: the lane whose bit m is set keeps o - v, its
    // partner v + o (one fused multiply-add by +-1: one rounding, like the add)
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int m = 1; m < 8; m <<= 1) {
        const float sg = (lane & m) ? -1.0f : 1.0f;
        const unsigned long long sg2 = f2pack(sg, sg);
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
            const float o0 = __shfl_xor_sync(0xffffffffu, v[i], m);
            const float o1 = __shfl_xor_sync(0xffffffffu, v[i + 1], m);
            unsigned long long r;
            asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(sg2), "l"(f2pack(v[i], v[i + 1])), "l"(f2pack(o0, o1)));
            f2unpack(r, v[i], v[i + 1]);
        }
    }
}

// 32 bf16 values from 4 raw 16-byte words (two a word, low half first); with
// SWIGLU, h = bf16(silu(g) * u) of gate words g and up words u.
template <bool SWIGLU>
__device__ __forceinline__ void unpack32(const uint4 (&g)[4], const uint4 (&u)[4], float (&v)[32]) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint32_t w[4] = {g[i].x, g[i].y, g[i].z, g[i].w};
        if constexpr (SWIGLU) {
            const uint32_t uw[4] = {u[i].x, u[i].y, u[i].z, u[i].w};
#pragma unroll
            for (int k = 0; k < 4; ++k) w[k] = swiglu_word(w[k], uw[k]);
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            v[8 * i + 2 * k] = __uint_as_float(w[k] << 16);
            v[8 * i + 2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
        }
    }
}

__device__ __forceinline__ uint4 ld_stream(const void *p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// The tail group (width n = 32, 64 or 128; E = n / 32 values a lane) of a
// row, read from global memory: lane l holds columns l E .. l E + E - 1 as
// values 0 .. E - 1 (with SWIGLU, h of the gate and up rows).
template <bool SWIGLU>
__device__ __forceinline__ int load_tail_global(const uint16_t *x, const uint16_t *u, int n, float (&v)[8]) {
    const int lane = threadIdx.x & 31;
    const int E = n >> 5;
    uint32_t w[4] = {0u, 0u, 0u, 0u}, uw[4] = {0u, 0u, 0u, 0u};
    auto load = [&](const uint16_t *p, uint32_t (&o)[4]) {
        const uint16_t *a = p + lane * E;
        if (E == 4) {
            const uint2 t = *reinterpret_cast<const uint2 *>(a);
            o[0] = t.x; o[1] = t.y;
        } else if (E == 2) {
            o[0] = *reinterpret_cast<const uint32_t *>(a);
        } else {
            o[0] = *a;
        }
    };
    load(x, w);
    if constexpr (SWIGLU) {
        load(u, uw);
#pragma unroll
        for (int i = 0; i < 4; ++i) w[i] = swiglu_word(w[i], uw[i]);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        v[2 * i] = __uint_as_float(w[i] << 16);
        v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
    return E;
}

// The tail group's rotation by c_n * Hs_n, as the 32-lane butterfly of the
// other rotation kernels; values past E come out 0.
__device__ __forceinline__ void rotate_tail(int n, float (&v)[8]) {
    const int E = n >> 5;
    switch (E) {
        case 4: warp_fwht<4, float>(v); break;
        case 2: warp_fwht<2, float>(v); break;
        default: warp_fwht<1, float>(v); break;
    }
    const float c = sqrtf(1.0f / static_cast<float>(n));
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] = e < E ? c * v[e] : 0.0f;
}

// Row prologues of k_rotq: the row as given, SwiGLU of a gate and an up row,
// or the modulated layer norm of the row.
constexpr int kPrePlain = 0, kPreSwiglu = 1, kPreNorm = 2;

// The modulated layer norm's fp32 arithmetic on one value, rounded to bf16
// as an unfused norm kernel would store it: h = (x - mu) rstd (1 + sc) + sh.
__device__ __forceinline__ float modnorm_value(float x, float mu, float rstd, float sc, float sh) {
    return __uint_as_float(static_cast<uint32_t>(f32_to_bf16_bits(fmaf((x - mu) * rstd, 1.0f + sc, sh))) << 16);
}

constexpr int kRotqMaxWarps = 17;   // 64 full groups (4 a warp) and a tail warp

// Rotation + per-token int8 quantisation, one token row per CTA at a time
// (persistent over rows m = blockIdx.x, blockIdx.x + gridDim.x, ...).  Warp
// w < WF owns the full groups 4w .. 4w + 3, which are the 1024-column window
// w; its lanes 8s .. 8s + 7 hold group 4w + s.  A tail group (width 32, 64 or
// 128) has a warp of its own.  Per row: the transform in registers, the
// row's amax (one CTA barrier), the codes.  Rows in flight come from the
// several CTAs an SM holds (measured on M = 4032, K = 12288: two CTAs an SM
// with the loads of each row issued at its start, 79 us, against 92 us with
// one CTA an SM that loaded the next row during the current one).
// TILED writes the codes as fp16 in the product's operand layout and records
// the |code| and code-squared window sums for the product's exactness bound;
// else int8 rows.  PRE = kPreSwiglu: the row is h = bf16(silu(g) * u), gate
// rows from X and up rows from U.  PRE = kPreNorm: the row is the modulated
// layer norm h = bf16((x - mu) rstd (1 + scale) + shift), mu and the biased
// variance var over the row in fp32 (one more CTA barrier: two passes inside
// each warp, then the warps' moments merged), rstd = rsqrtf(var + eps), the
// modulation read per column through the read-only cache.

// CTAs an SM should hold, by warps a CTA: a thread keeps about 80 registers
constexpr int rotq_min_blocks(int maxw) {
    return maxw <= 4 ? 6 : maxw <= 8 ? 3 : maxw <= 12 ? 2 : 1;
}
template <bool TILED, int PRE, int MAXW>
__global__ void __launch_bounds__(MAXW * 32, rotq_min_blocks(MAXW))
k_rotq(const uint16_t *__restrict__ X, int64_t M, int64_t K, int64_t ldx, void *__restrict__ out,
       float *__restrict__ sx, unsigned int *trl, const uint16_t *__restrict__ U, int64_t ldu,
       const float *__restrict__ shift, const float *__restrict__ scale, float eps) {
    constexpr bool SWIGLU = PRE == kPreSwiglu;
    __shared__ float red[2][kRotqMaxWarps];
    __shared__ float red_n[2][PRE == kPreNorm ? kRotqMaxWarps : 1];   // the warps' means and M2
    __shared__ unsigned int win[2][16], winq[2][16];   // a row's window sums of |codes|, codes squared
    __shared__ unsigned int run_sh[2][5][32];           // warp 0's largest run sums over the rows
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int W = blockDim.x >> 5;
    const int64_t Gf = K / kGroup;                   // full 256-groups
    const int tail = static_cast<int>(K % kGroup);   // 0, 32, 64 or 128
    const int WF = static_cast<int>((Gf + 3) / 4);   // warps of full groups
    const bool tail_warp = tail != 0 && warp == WF;
    const int64_t g = static_cast<int64_t>(warp) * 4 + (lane >> 3);   // this lane's group
    const bool active = !tail_warp && g < Gf;
    const int64_t col0 = g * kGroup + (lane & 7) * 8;    // first of this lane's 4 runs of 8 columns
    constexpr int kRun = 64;                              // column step between the runs
    const int64_t KT = (K + 63) >> 6;

    if (threadIdx.x < 32) {
        for (int p = 0; p < 2; ++p) {
            if (lane < 16) win[p][lane] = winq[p][lane] = 0u;
            for (int j = 0; j < 5; ++j) run_sh[p][j][lane] = 0u;
        }
    }
    __syncthreads();

    uint4 raw[4], rawu[4];
    auto load_row = [&](int64_t m) {
        if (!active) return;
        const uint16_t *src = X + m * ldx + col0;
#pragma unroll
        for (int i = 0; i < 4; ++i) raw[i] = ld_stream(src + kRun * i);
        if constexpr (SWIGLU) {
            const uint16_t *us = U + m * ldu + col0;
#pragma unroll
            for (int i = 0; i < 4; ++i) rawu[i] = ld_stream(us + kRun * i);
        }
    };
    // warp 0: fold a finished row's window sums into its running maxima over
    // aligned runs of 2^j windows (lane l holds window l; zero past K)
    auto fold_windows = [&](int p) {
        unsigned int ws = lane < 16 ? win[p][lane] : 0u;
        unsigned int wq = lane < 16 ? winq[p][lane] : 0u;
        if (lane < 16) win[p][lane] = winq[p][lane] = 0u;
#pragma unroll
        for (int j = 0; j < 5; ++j) {
            if (j > 0) {
                ws += __shfl_xor_sync(0xffffffffu, ws, 1 << (j - 1));
                wq += __shfl_xor_sync(0xffffffffu, wq, 1 << (j - 1));
            }
            run_sh[0][j][lane] = max(run_sh[0][j][lane], ws);
            run_sh[1][j][lane] = max(run_sh[1][j][lane], wq);
        }
    };

    int64_t m = blockIdx.x;
    int par = 0;
    bool pending = false;   // a row's window sums wait to be folded
    for (; m < M; m += gridDim.x, par ^= 1) {
        float v[32];
        load_row(m);
        if (active) {
            unpack32<SWIGLU>(raw, rawu, v);
        } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) v[e] = 0.0f;
        }

        // transform; the full groups stay unscaled (their factor 1/16 is a
        // power of two, applied exactly with the codes), the tail is scaled
        float vt[8];
        int Et = 0;
        float amax = 0.0f;
        const int64_t t0 = Gf * kGroup;
        if (tail_warp) Et = load_tail_global<SWIGLU>(X + m * ldx + t0, SWIGLU ? U + m * ldu + t0 : nullptr, tail, vt);
        if constexpr (PRE == kPreNorm) {
            // each warp's mean and sum of squared deviations over its own
            // values (two passes inside the warp), merged after one barrier
            // by the parallel formula of Chan, Golub and LeVeque (1979):
            // mean = sum_w n_w m_w / K, M2 = sum_w (M2_w + n_w (m_w - mean)^2)
            auto warp_n = [&](int w) {   // values warp w holds
                const int64_t ng = Gf - 4 * static_cast<int64_t>(w);
                return w < WF ? static_cast<float>((ng < 4 ? ng : 4) * kGroup) : static_cast<float>(tail);
            };
            float s1 = 0.0f;
            if (tail_warp) {
#pragma unroll
                for (int e = 0; e < 8; ++e) s1 += e < Et ? vt[e] : 0.0f;
            } else {
                unsigned long long acc = f2pack(v[0], v[1]);
#pragma unroll
                for (int e = 2; e < 32; e += 2)
                    asm("add.rn.f32x2 %0, %0, %1;" : "+l"(acc) : "l"(f2pack(v[e], v[e + 1])));
                float a0, a1;
                f2unpack(acc, a0, a1);
                s1 = a0 + a1;
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) s1 += __shfl_xor_sync(0xffffffffu, s1, o);
            const float mw = s1 / warp_n(warp);
            float s2 = 0.0f;
            if (tail_warp) {
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float d = vt[e] - mw;
                    s2 = e < Et ? fmaf(d, d, s2) : s2;
                }
            } else if (active) {
                const unsigned long long m2w = f2pack(mw, mw);
                unsigned long long acc = f2pack(0.0f, 0.0f);
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                    unsigned long long d;
                    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(f2pack(v[e], v[e + 1])), "l"(m2w));
                    asm("fma.rn.f32x2 %0, %1, %1, %0;" : "+l"(acc) : "l"(d));
                }
                float a0, a1;
                f2unpack(acc, a0, a1);
                s2 = a0 + a1;
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) s2 += __shfl_xor_sync(0xffffffffu, s2, o);
            if (lane == 0) {
                red_n[0][warp] = mw;
                red_n[1][warp] = s2;
            }
            __syncthreads();
            float msum = 0.0f;
            for (int w = 0; w < W; ++w) msum = fmaf(warp_n(w), red_n[0][w], msum);
            const float mu = msum / static_cast<float>(K);
            float m2 = 0.0f;
            for (int w = 0; w < W; ++w) {
                const float d = red_n[0][w] - mu;
                m2 += fmaf(warp_n(w) * d, d, red_n[1][w]);
            }
            const float var = m2 / static_cast<float>(K);
            const float rstd = rsqrtf(var + eps);
            if (tail_warp) {
                const int64_t c0 = t0 + static_cast<int64_t>(lane) * Et;
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    if (e < Et) vt[e] = modnorm_value(vt[e], mu, rstd, __ldg(scale + c0 + e), __ldg(shift + c0 + e));
            } else if (active) {
                const unsigned long long mu2 = f2pack(mu, mu), r2 = f2pack(rstd, rstd);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float4 *sc4 = reinterpret_cast<const float4 *>(scale + col0 + kRun * i);
                    const float4 *sh4 = reinterpret_cast<const float4 *>(shift + col0 + kRun * i);
                    const float4 a = __ldg(sc4), b = __ldg(sc4 + 1), c = __ldg(sh4), d = __ldg(sh4 + 1);
                    const float sc[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
                    const float sh[8] = {c.x, c.y, c.z, c.w, d.x, d.y, d.z, d.w};
#pragma unroll
                    for (int e = 0; e < 8; e += 2)
                        modnorm_pair(v[8 * i + e], v[8 * i + e + 1], mu2, r2, sc[e], sc[e + 1], sh[e], sh[e + 1]);
                }
            }
        }
        if (tail_warp) {
            rotate_tail(tail, vt);
#pragma unroll
            for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(vt[e]));
        } else {
            fwht_8x32(v);
#pragma unroll
            for (int e = 0; e < 32; ++e) amax = fmaxf(amax, fabsf(v[e]));
            amax *= 0.0625f;   // exact; fl(c v) is monotone in |v|
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        if (lane == 0) red[par][warp] = amax;
        __syncthreads();
        amax = red[par][0];
        for (int w = 1; w < W; ++w) amax = fmaxf(amax, red[par][w]);
        if (TILED && warp == 0 && pending) fold_windows(par ^ 1);
        pending = true;

        const float s = __fdiv_rn(amax, 127.0f);
        const float r = recip_or_zero(s);
        const float r16 = r * 0.0625f >= FLT_MIN ? r * 0.0625f : 0.0f;   // exact: a power of two
        if (threadIdx.x == 0) sx[m] = s;

        if (!tail_warp) {
            // codes eight at a time: 16 bytes of fp16 codes (one core-matrix
            // row of the tiled operand) or 8 bytes of int8 codes
            float fs = 0.0f;                                   // exact: at most 32 x 127
            unsigned long long fq2 = f2pack(0.0f, 0.0f);       // exact: at most 16 x 127^2 a half
            const unsigned long long r2 = f2pack(r16, r16);
            uint16_t *tdst = nullptr;
            if constexpr (TILED) {
                const int64_t mt = m >> 7;
                const int rr = static_cast<int>(m & 127);
                tdst = static_cast<uint16_t *>(out) + ((mt * KT + (col0 >> 6)) << 13) +
                       ((((rr >> 3) << 3) + static_cast<int>((col0 & 63) >> 3)) << 6) + ((rr & 7) << 3);
            }
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                float q[8];
                // rint of the product; where it may differ from rint of the
                // correctly rounded quotient (near a half-integer, or no
                // reciprocal), the warp takes the division for those values
                // (products and differences on pairs, each rounded as a
                // single one; the largest distance decides for the eight)
                float dmax = 0.0f;
#pragma unroll
                for (int e = 0; e < 8; e += 2) {
                    unsigned long long t2, d2;
                    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(t2) : "l"(f2pack(v[8 * c + e], v[8 * c + e + 1])), "l"(r2));
                    float t0, t1, d0, d1;
                    f2unpack(t2, t0, t1);
                    q[e] = rintf(t0);
                    q[e + 1] = rintf(t1);
                    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d2) : "l"(t2), "l"(f2pack(q[e], q[e + 1])));
                    f2unpack(d2, d0, d1);
                    dmax = fmaxf(dmax, fmaxf(fabsf(d0), fabsf(d1)));
                }
                const bool amb = r16 == 0.0f || dmax > 0.499f;
                if (__any_sync(0xffffffffu, amb) && amb) {
#pragma unroll
                    for (int e = 0; e < 8; ++e) q[e] = code_of(v[8 * c + e], 0.0625f, r16, s);
                }
#pragma unroll
                for (int e = 0; e < 8; e += 2) {
                    fs += fabsf(q[e]) + fabsf(q[e + 1]);
                    const unsigned long long q2 = f2pack(q[e], q[e + 1]);
                    asm("fma.rn.f32x2 %0, %1, %1, %0;" : "+l"(fq2) : "l"(q2));
                }
                if (!active) continue;
                if constexpr (TILED) {
                    uint32_t h[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const __half2 p2 = __floats2half2_rn(q[2 * i], q[2 * i + 1]);
                        h[i] = *reinterpret_cast<const uint32_t *>(&p2);
                    }
                    *reinterpret_cast<uint4 *>(tdst + (c << 13)) = make_uint4(h[0], h[1], h[2], h[3]);
                } else {
                    uint32_t wv[2] = {0u, 0u};
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        wv[e >> 2] |= (static_cast<uint32_t>(__float2int_rz(q[e])) & 0xFFu) << (8 * (e & 3));
                    *reinterpret_cast<uint2 *>(static_cast<int8_t *>(out) + m * K + col0 + kRun * c) =
                        make_uint2(wv[0], wv[1]);
                }
            }
            if constexpr (TILED) {
                float fq0, fq1;
                f2unpack(fq2, fq0, fq1);
                const unsigned int gs = __reduce_add_sync(0xffffffffu, static_cast<unsigned int>(fs));
                const unsigned int gq = __reduce_add_sync(0xffffffffu, static_cast<unsigned int>(fq0 + fq1));
                if (lane == 0 && warp < WF) {
                    atomicAdd(&win[par][warp], gs);
                    atomicAdd(&winq[par][warp], gq);
                }
            }
        } else {
            float q[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) q[e] = code_of(vt[e], 1.0f, r, s);
            const int64_t k0 = Gf * kGroup + static_cast<int64_t>(lane) * Et;
            if constexpr (TILED) {
                put_tiled(static_cast<uint16_t *>(out), KT, K, m, k0, Et, q);
                float fs = 0.0f, fq = 0.0f;
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    if (e < Et) {
                        fs += fabsf(q[e]);
                        fq = fmaf(q[e], q[e], fq);
                    }
                const unsigned int gs = __reduce_add_sync(0xffffffffu, static_cast<unsigned int>(fs));
                const unsigned int gq = __reduce_add_sync(0xffffffffu, static_cast<unsigned int>(fq));
                if (lane == 0) {
                    atomicAdd(&win[par][Gf >> 2], gs);
                    atomicAdd(&winq[par][Gf >> 2], gq);
                }
            } else {
                put_int8(static_cast<int8_t *>(out) + m * K + k0, Et, q);
            }
        }
    }
    if constexpr (TILED) {
        __syncthreads();
        if (warp == 0) {
            if (pending) fold_windows(par ^ 1);
            // Trailer: word 1 + j the largest sum of |codes| over an aligned
            // run of 2^j windows, word 0 over a whole row (16 windows hold the
            // longest row); words 7 + j and 6 the same for codes squared.
            // This CTA's maxima go into copy blockIdx % 16, once the kernel
            // that zeroes the copies has finished (this launch's primary).
            unsigned int *cp = trl + (blockIdx.x % kTrailerCopies) * kTrailerStride;
            asm volatile("griddepcontrol.wait;" ::: "memory");
#pragma unroll
            for (int j = 0; j < 5; ++j) {
                unsigned int mx = run_sh[0][j][lane], mq = run_sh[1][j][lane];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                    mq = max(mq, __shfl_xor_sync(0xffffffffu, mq, o));
                }
                if (pending && lane == j) {
                    atomicMax(cp + 1 + j, mx);
                    atomicMax(cp + 7 + j, mq);
                }
                if (pending && j == 4 && lane == 5) {
                    atomicMax(cp, mx);
                    atomicMax(cp + 6, mq);
                }
            }
        }
    }
}

// Zeroes a tiled operand's trailer copies; the rotation launched next is its
// programmatic dependent, released at once.
__global__ void __launch_bounds__(32) k_zero_trailer(unsigned int *trl) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    for (int i = threadIdx.x; i < kTrailerCopies * kTrailerStride; i += 32) trl[i] = 0u;
}

template <bool TILED, int PRE = kPrePlain>
tq_status launch_rotq(const uint16_t *X, int64_t M, int64_t K, int64_t ldx, void *out, float *sx,
                      unsigned int *trl, cudaStream_t s, const uint16_t *U = nullptr, int64_t ldu = 0,
                      const float *shift = nullptr, const float *scale = nullptr, float eps = 0.0f) {
    const int64_t Gf = K / kGroup;
    const int warps = static_cast<int>((Gf + 3) / 4) + (K % kGroup ? 1 : 0);
    if (warps < 1 || warps > kRotqMaxWarps) return TQ_ERR_SHAPE;
    const int NT = warps * 32;
    DeviceInfo dev;
    const tq_status ds = current_device(&dev);
    if (ds != TQ_OK) return ds;
    // up to 16 warps (every row of at most 16384 columns but those of 63 full
    // groups and a tail) with the register budget of 512 threads
    auto kern = warps <= 4    ? k_rotq<TILED, PRE, 4>
                : warps <= 8  ? k_rotq<TILED, PRE, 8>
                : warps <= 12 ? k_rotq<TILED, PRE, 12>
                : warps <= 16 ? k_rotq<TILED, PRE, 16>
                              : k_rotq<TILED, PRE, kRotqMaxWarps>;
    // persistent: as many CTAs as are resident at once
    int per_sm = 0;
    const cudaError_t oe = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, NT, 0);
    if (oe != cudaSuccess) return cuda_fail(oe);
    per_sm = per_sm < 1 ? 1 : per_sm;
    const int64_t want = static_cast<int64_t>(dev.sms) * per_sm;
    const unsigned grid = static_cast<unsigned>(M < want ? M : want);
    if constexpr (TILED) {
        k_zero_trailer<<<1, 32, 0, s>>>(trl);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return cuda_fail(e);
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(grid);
        cfg.blockDim = dim3(NT);
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, kern, X, M, K, ldx, out, sx, trl, U, ldu, shift, scale, eps);
        return e == cudaSuccess ? TQ_OK : cuda_fail(e);
    } else {
        kern<<<grid, NT, 0, s>>>(X, M, K, ldx, out, sx, trl, U, ldu, shift, scale, eps);
        const cudaError_t e = cudaGetLastError();
        return e == cudaSuccess ? TQ_OK : cuda_fail(e);
    }
}

}  // namespace

int64_t tiled_act_tiles_bytes(int64_t M, int64_t K) {
    return ((M + 255) / 256) * 2 * ((K + 63) / 64) * 16384;
}

int64_t tiled_act_bytes(int64_t M, int64_t K) { return tiled_act_tiles_bytes(M, K) + kTrailerBytes; }

unsigned int *tiled_act_trailer(void *At, int64_t M, int64_t K) {
    return reinterpret_cast<unsigned int *>(static_cast<unsigned char *>(At) + tiled_act_tiles_bytes(M, K));
}

tq_status launch_rotate_quant_tiled(const uint16_t *X, int64_t M, int64_t K, int64_t ldx,
                                    void *At, float *sx, cudaStream_t s) {
    if (M == 0) return TQ_OK;
    if (K > kRingMaxK) return TQ_ERR_SHAPE;
    return launch_rotq<true>(X, M, K, ldx, At, sx, tiled_act_trailer(At, M, K), s);
}

tq_status launch_swiglu_quant_tiled(const uint16_t *G, int64_t ldg, const uint16_t *U, int64_t ldu,
                                    int64_t M, int64_t K, void *At, float *sx, cudaStream_t s) {
    if (M == 0) return TQ_OK;
    if (K > kRingMaxK) return TQ_ERR_SHAPE;
    return launch_rotq<true, kPreSwiglu>(G, M, K, ldg, At, sx, tiled_act_trailer(At, M, K), s, U, ldu);
}

tq_status launch_modnorm_quant_tiled(const uint16_t *X, int64_t M, int64_t K, int64_t ldx, const float *shift,
                                     const float *scale, float eps, void *At, float *sx, cudaStream_t s) {
    if (M == 0) return TQ_OK;
    if (K > kRingMaxK) return TQ_ERR_SHAPE;
    return launch_rotq<true, kPreNorm>(X, M, K, ldx, At, sx, tiled_act_trailer(At, M, K), s, nullptr, 0, shift,
                                       scale, eps);
}

tq_status launch_rotate_quant_act(const uint16_t *X, int64_t M, int64_t K,
                                  int64_t ldx, int8_t *Xq, float *sx,
                                  cudaStream_t s) {
    const int64_t G = (K + kGroup - 1) / kGroup;
    const int64_t gpw = (G + 7) / 8;
    if (M == 0) return TQ_OK;
    if (K <= kRingMaxK) return launch_rotq<false>(X, M, K, ldx, Xq, sx, nullptr, s);
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
