// Internal declarations shared by the CUDA translation units of libtq.
// Everything here runs on the device path; nothing is shared with the CPU
// oracle that checks it.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "tq.h"

namespace tq {

constexpr int kGroup = 256;       // rotation group width
constexpr int kThreads = 256;     // threads of the row kernels

// ---------------------------------------------------------------- host side

struct DeviceInfo {
    int id = -1;
    int sms = 0;
    int smem_optin = 0;      // max dynamic shared memory per block (bytes)
    bool ok = false;         // compute capability 10.3
};

// Cached properties of the current device (TQ_ERR_DEVICE if none usable).
tq_status current_device(DeviceInfo *out);
// Records a CUDA error code for tq_last_cuda_error and returns TQ_ERR_CUDA.
tq_status cuda_fail(cudaError_t e);
// Device address of the library's status word on the current device.
unsigned int *status_word();

// Launchers (one per kernel family).  Arguments are validated by the caller.
tq_status launch_quantize_weights(const uint16_t *W, int64_t N, int64_t K,
                                  int64_t ldw, int bits, void *codes,
                                  float *scales, cudaStream_t s);
tq_status launch_rotate_quant_act(const uint16_t *X, int64_t M, int64_t K,
                                  int64_t ldx, int8_t *Xq, float *sx,
                                  cudaStream_t s);
tq_status launch_rotate_bf16(const uint16_t *X, int64_t M, int64_t K,
                             int64_t ldx, uint16_t *Xr, cudaStream_t s);

// Skinny A16 product (M <= 64): rotation fused into the prologue.
bool gemv_fits(int64_t M, int64_t K, int bits, const DeviceInfo &dev);
tq_status launch_quantize_weights_blocked(const uint16_t *W, int64_t N, int64_t K, int64_t ldw, int bits,
                                          int G, int rotate, void *codes, float *scales, cudaStream_t s);
int gemv_blocked_mt(int M);
bool a16_streams(int64_t M, int64_t N, int64_t K, int bits);
tq_status launch_gemv_blocked(const uint16_t *X, int M, int64_t K, int64_t ldx, const uint8_t *Wq,
                              const float *sw, int G, int64_t N, int bits, int rotate, void *Y, int ytype,
                              int64_t ldy, const DeviceInfo &dev, cudaStream_t s);
tq_status launch_gemv_a16(const uint16_t *X, int64_t M, int64_t K, int64_t ldx,
                          const uint8_t *Wq, const float *sw, int64_t N,
                          int bits, void *Y, int ytype, int64_t ldy,
                          const DeviceInfo &dev, cudaStream_t s);

// Batched A16 product on tcgen05 (M <= 64; large matrices or more than 8
// tokens): a pre-pass writes x' as fp16 tiles into the workspace.
bool splitk_fits(int64_t M, int64_t N, int64_t K, int bits, const DeviceInfo &dev);
tq_status launch_splitk(const uint16_t *X, int64_t M, int64_t K, int64_t ldx, const uint8_t *Wq, const float *sw,
                        int64_t N, int bits, void *Y, int ytype, int64_t ldy, const DeviceInfo &dev,
                        cudaStream_t s);
bool skinny_tc_applies(int64_t M, int64_t N, int64_t K);
int64_t skinny_tc_workspace(int64_t M, int64_t K);
bool skinny_tc_fits_device(int64_t N, const DeviceInfo &dev);
tq_status launch_skinny_tc(const uint16_t *X, int64_t M, int64_t K, int64_t ldx, const uint8_t *Wq,
                           const float *sw, int64_t N, int bits, void *Y, int ytype, int64_t ldy, void *ws,
                           const DeviceInfo &dev, cudaStream_t s);

// Decode product for M <= 8: whole rows per CTA, no cluster reduction.
bool gemv_small_fits(int64_t M, int64_t N, int64_t K, int bits, const DeviceInfo &dev);
// U non-null: the input row is h = bf16(silu(x) * u) of X's and U's rows (SwiGLU)
tq_status launch_gemv_small(const uint16_t *X, int64_t M, int64_t K, int64_t ldx,
                            const uint8_t *Wq, const float *sw, int64_t N, int bits,
                            void *Y, int ytype, int64_t ldy, const DeviceInfo &dev,
                            cudaStream_t s, const uint16_t *U = nullptr, int64_t ldu = 0);
// the small kernel or the eight-row kernel takes this decode shape
bool gemv_decode_fits(int64_t M, int64_t N, int64_t K, int bits, const DeviceInfo &dev);

// A8 product on quantised activations: tcgen05 / TMEM, exact int32 sums.
tq_status launch_gemm_a8(const int8_t *Xq, const float *sx, int64_t M,
                         int64_t K, const uint8_t *Wq, const float *sw,
                         int64_t N, int bits, void *Y, int ytype, int64_t ldy,
                         const DeviceInfo &dev, cudaStream_t s);

// The activation codes as fp16 in the tensor core's operand layout ("tiled"):
// 128-row x 64-column tiles, tile (mt, kt) the 16 KB at byte
// (mt * ceil(K/64) + kt) * 16384, inside a tile the K-major 8x8 core-matrix
// order (core matrix (r/8, k/8) is 128 contiguous bytes, K-adjacent ones 128
// bytes apart, row groups 1024 bytes apart).  Rows are padded to a whole
// number of 256-row tile pairs; columns past K inside the last tile are zero.
// After the tiles (at byte tiled_act_tiles_bytes), a 2048-byte trailer of 12
// bounds: word 0 the largest sum of |codes| over the rows, word 1 + j the
// largest such sum over an aligned window of 1024 << j columns (j < 5), words
// 6 and 7 + j the same for codes squared.  It holds 16 copies of the 12 words,
// 128 bytes apart: each CTA of the rotation takes the atomic maximum into copy
// blockIdx % 16 (so that the CTAs' atomics spread over 16 lines), and a reader
// takes the maximum over the copies.  The copies are zeroed by a one-warp
// kernel launched just before the rotation, which the rotation follows as a
// programmatic dependent: its rows run while the zeroing does, and it waits
// for it (griddepcontrol.wait) only before its atomics.
constexpr int kTrailerCopies = 16;
constexpr int kTrailerStride = 32;       // 32-bit words between copies
constexpr int kTrailerBytes = kTrailerCopies * kTrailerStride * 4;
unsigned int *tiled_act_trailer(void *At, int64_t M, int64_t K);

// Bound j of a tiled operand's trailer: the maximum over its copies.
__device__ __forceinline__ unsigned int trailer_bound(const unsigned int *trl, int j) {
    unsigned int best = 0u;
#pragma unroll
    for (int c = 0; c < kTrailerCopies; ++c) best = max(best, trl[c * kTrailerStride + j]);
    return best;
}
bool make_map_u8(CUtensorMap *map, const void *base, int64_t rows, int64_t cols, int box_cols,
                 int box_rows, CUtensorMapSwizzle swz);

int grouped_item_rows(int64_t M, int64_t K, int bits);
tq_status grouped_bytes(const tq_a16_call *calls, int64_t n, int bits, size_t *bytes);
tq_status grouped_create(const tq_a16_call *calls, int64_t n, int bits, int ytype, void *dmem,
                         size_t dbytes, const DeviceInfo &dev, tq_grouped *out);
tq_status chain_bytes(const tq_chain_call *calls, int64_t n, int bits, size_t *bytes);
tq_status chain_create(const tq_chain_call *calls, int64_t n, int bits, int ytype, void *dmem,
                       size_t dbytes, const DeviceInfo &dev, tq_grouped *out);
int chain_item_rows(int64_t M, int64_t K, int64_t N, int bits, int grid);
tq_status grouped_run(tq_grouped plan, const DeviceInfo &dev, int phase, cudaStream_t s);
void grouped_destroy(tq_grouped plan);
int64_t grouped_weight_bytes(tq_grouped plan);

int64_t weights_tiled_bytes(int64_t N, int64_t K);
tq_status launch_tile_weights(const uint8_t *Wq, int64_t N, int64_t K, int bits, void *Wt, cudaStream_t s);
// Optional epilogue of the A8 product: Y = R + gate[n] * (sx sw acc + bias[n]).
struct EpilogueArgs {
    const float *bias = nullptr;
    const float *gate = nullptr;
    const void *R = nullptr;
    int64_t ldr = 0;
    int rtype = 0;      // 0 fp32, 1 bf16
};
tq_status launch_gemm_a8_tt(const void *At, const float *sx, int64_t M, int64_t K, const void *Wt,
                            const float *sw, int64_t N, int bits, void *Y, int ytype, int64_t ldy,
                            const DeviceInfo &dev, cudaStream_t s, const EpilogueArgs *ea = nullptr,
                            void *split_ws = nullptr);
// Bytes of the split workspace of the both-tiled product on this device, and
// of its flag area at the start (the rest holds one partial tile per CTA).
size_t split_workspace_bytes(const DeviceInfo &dev);
size_t split_flag_bytes(const DeviceInfo &dev);

int64_t tiled_act_tiles_bytes(int64_t M, int64_t K);
int64_t tiled_act_bytes(int64_t M, int64_t K);
tq_status launch_rotate_quant_tiled(const uint16_t *X, int64_t M, int64_t K,
                                    int64_t ldx, void *At, float *sx, cudaStream_t s);
tq_status launch_swiglu_quant_tiled(const uint16_t *G, int64_t ldg, const uint16_t *U, int64_t ldu,
                                    int64_t M, int64_t K, void *At, float *sx, cudaStream_t s);
tq_status launch_modnorm_quant_tiled(const uint16_t *X, int64_t M, int64_t K, int64_t ldx, const float *shift,
                                     const float *scale, float eps, void *At, float *sx, cudaStream_t s);
tq_status launch_gemm_a8_tiled(const void *At, const float *sx, int64_t M, int64_t K,
                               const uint8_t *Wq, const float *sw, int64_t N, int bits,
                               void *Y, int ytype, int64_t ldy, const DeviceInfo &dev,
                               cudaStream_t s);

// ---------------------------------------------------------------- device side

__device__ __forceinline__ float bf16_bits_to_f32(uint16_t b) {
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

__device__ __forceinline__ uint16_t f32_to_bf16_bits(float f) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// Widen E consecutive bf16 values (E in {1,2,4,8}) from an aligned pointer.
template <int E, typename T>
__device__ __forceinline__ void load_bf16(const uint16_t *p, T (&v)[8]) {
    if constexpr (E == 8) {
        const uint4 u = __ldg(reinterpret_cast<const uint4 *>(p));
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            v[2 * i] = static_cast<T>(__uint_as_float(w[i] << 16));
            v[2 * i + 1] = static_cast<T>(__uint_as_float(w[i] & 0xFFFF0000u));
        }
    } else if constexpr (E == 4) {
        const uint2 u = __ldg(reinterpret_cast<const uint2 *>(p));
        v[0] = static_cast<T>(__uint_as_float(u.x << 16));
        v[1] = static_cast<T>(__uint_as_float(u.x & 0xFFFF0000u));
        v[2] = static_cast<T>(__uint_as_float(u.y << 16));
        v[3] = static_cast<T>(__uint_as_float(u.y & 0xFFFF0000u));
    } else if constexpr (E == 2) {
        const uint32_t u = __ldg(reinterpret_cast<const unsigned int *>(p));
        v[0] = static_cast<T>(__uint_as_float(u << 16));
        v[1] = static_cast<T>(__uint_as_float(u & 0xFFFF0000u));
    } else {
        v[0] = static_cast<T>(bf16_bits_to_f32(__ldg(reinterpret_cast<const unsigned short *>(p))));
    }
}

// Fused multiply-add in the type of the operands (one rounding).
__device__ __forceinline__ float fused_madd(float a, float b, float c) { return fmaf(a, b, c); }
__device__ __forceinline__ double fused_madd(double a, double b, double c) { return fma(a, b, c); }

// Unnormalised Walsh-Hadamard transform, natural (Sylvester) order, of one
// group of 32*E values held E per lane (element index = lane*E + e): the
// in-place butterfly (a, b) -> (a + b, a - b) over every bit of the index,
// first the bits inside a lane, then the lane bits through shuffles.
template <int E, typename T>
__device__ __forceinline__ void warp_fwht(T (&v)[8]) {
#pragma unroll
    for (int h = 1; h < E; h <<= 1) {
#pragma unroll
        for (int i = 0; i < E; ++i) {
            if (!(i & h)) {
                const T a = v[i], b = v[i + h];
                v[i] = a + b;
                v[i + h] = a - b;
            }
        }
    }
    // Across lanes: the lane with bit m set keeps o - v, its partner v + o.
    // Both are one fused multiply-add with a +-1 factor, which rounds the
    // exact sum or difference once, like the plain add or subtract.
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
        const T sg = (lane & m) ? T(-1) : T(1);
#pragma unroll
        for (int i = 0; i < E; ++i) {
            const T o = __shfl_xor_sync(0xffffffffu, v[i], m);
            v[i] = fused_madd(sg, v[i], o);
        }
    }
}

// Width of the group starting at column g0 of a K-wide row (256 or the tail).
__device__ __forceinline__ int group_width(int64_t K, int64_t g0) {
    const int64_t rest = K - g0;
    return rest >= kGroup ? kGroup : static_cast<int>(rest);
}

// Rotate one group (width n = 32*E: 256, 128, 64 or 32) of a bf16 row in
// fp32: v = c_n * Hs_n * x with c_n = sqrt(1/n) correctly rounded in fp32.
template <int E>
__device__ __forceinline__ void rotate_group32(const uint16_t *src, float (&v)[8]) {
    const int lane = threadIdx.x & 31;
    load_bf16<E, float>(src + lane * E, v);
    warp_fwht<E, float>(v);
    const float c = sqrtf(1.0f / (32.0f * E));
#pragma unroll
    for (int e = 0; e < E; ++e) v[e] = c * v[e];
}

// Returns E, the number of values each lane holds.
__device__ __forceinline__ int rotate_group32_any(const uint16_t *src, int n, float (&v)[8]) {
    switch (n) {
        case 256: rotate_group32<8>(src, v); return 8;
        case 128: rotate_group32<4>(src, v); return 4;
        case 64: rotate_group32<2>(src, v); return 2;
        default: rotate_group32<1>(src, v); return 1;
    }
}

// The same rotation split in two, so that a warp can issue the loads of several
// groups before transforming any: the raw bits of this lane's E = n/32 values...
__device__ __forceinline__ uint4 load_group_raw(const uint16_t *p, int E) {
    if (E == 8) return __ldg(reinterpret_cast<const uint4 *>(p));
    if (E == 4) {
        const uint2 u = __ldg(reinterpret_cast<const uint2 *>(p));
        return make_uint4(u.x, u.y, 0, 0);
    }
    if (E == 2) return make_uint4(__ldg(reinterpret_cast<const unsigned int *>(p)), 0, 0, 0);
    return make_uint4(__ldg(reinterpret_cast<const unsigned short *>(p)), 0, 0, 0);
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

// The SwiGLU of a gate group's raw words and an up group's (E bf16 values a
// lane each, as load_group_raw returns them), packed the same way.
__device__ __forceinline__ uint4 swiglu_raw(const uint4 &g, const uint4 &u) {
    return make_uint4(swiglu_word(g.x, u.x), swiglu_word(g.y, u.y), swiglu_word(g.z, u.z), swiglu_word(g.w, u.w));
}

// ...and their transform: widen, butterfly, scale by sqrt(1/n).  Returns E.
__device__ __forceinline__ int fwht_group_raw(const uint4 &r, int n, float (&v)[8]) {
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        v[2 * i] = __uint_as_float(w[i] << 16);
        v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
    int E;
    switch (n) {
        case 256: warp_fwht<8, float>(v); E = 8; break;
        case 128: warp_fwht<4, float>(v); E = 4; break;
        case 64: warp_fwht<2, float>(v); E = 2; break;
        default: warp_fwht<1, float>(v); E = 1; break;
    }
    const float c = sqrtf(1.0f / static_cast<float>(n));
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] = e < E ? c * v[e] : 0.0f;
    return E;
}

// ---- PTX wrappers

__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void pdl_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Asynchronous prefetch of [p, p + bytes) into L2 (p and bytes 16-aligned).
__device__ __forceinline__ void prefetch_l2(const void *p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ uint4 ldg_stream(const void *p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

}  // namespace tq
