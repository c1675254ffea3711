// C-ABI entry points of libtq: host-side validation, then dispatch to the
// kernels.  Every check runs before any launch, and a refusal names its reason.
// The pages do the same: a format the sizes do not allow is rejected with a
// message before any work starts (kvad-gpu internals, "Quantised weights on
// the GPU"), and size products are checked for overflow (TensorFold PR #948,
// review follow-up).

#include <limits.h>

#include <cmath>

#include "tq_internal.cuh"

namespace tq {

static thread_local int g_last_cuda_error = 0;

// Status word written by kernels whose bounded waits expire.
__device__ unsigned int g_status_word = 0;

tq_status cuda_fail(cudaError_t e) {
    g_last_cuda_error = static_cast<int>(e);
    return TQ_ERR_CUDA;
}

unsigned int *status_word() {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
    return static_cast<unsigned int *>(p);
}

tq_status current_device(DeviceInfo *out) {
    static DeviceInfo cache[64];
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) {
        cudaGetLastError();
        return TQ_ERR_DEVICE;
    }
    if (dev < 64 && cache[dev].id == dev) {
        *out = cache[dev];
        return cache[dev].ok ? TQ_OK : TQ_ERR_DEVICE;
    }
    DeviceInfo d;
    d.id = dev;
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) {
        cudaGetLastError();
        return TQ_ERR_DEVICE;
    }
    d.ok = (major == 10 && minor == 3);
    if (dev < 64) cache[dev] = d;
    *out = d;
    return d.ok ? TQ_OK : TQ_ERR_DEVICE;
}

namespace {

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool valid_k(int64_t K) {
    if (K <= 0 || K > TQ_MAX_K) return false;
    const int64_t t = K % kGroup;
    return t == 0 || t == 32 || t == 64 || t == 128;
}

// A block width of the block-scaled format: 32, 64, 128 or 256, dividing K.
bool valid_block(int G, int64_t K) {
    return (G == 32 || G == 64 || G == 128 || G == 256) && K % G == 0;
}

// a * b without int64 overflow, and within `limit`
bool mul_ok(int64_t a, int64_t b, int64_t limit = INT64_MAX / 4) {
    if (a < 0 || b < 0) return false;
    if (a == 0 || b == 0) return true;
    return a <= limit / b;
}

// Shared checks of a bf16 [rows, K] input with row stride ld.
tq_status check_bf16_rows(const void *p, int64_t rows, int64_t K, int64_t ld) {
    if (!p) return TQ_ERR_NULL;
    if (ld < K) return TQ_ERR_SHAPE;
    if (!mul_ok(rows, ld) || !mul_ok(rows * ld, 2)) return TQ_ERR_OVERFLOW;
    if (!aligned(p, 16) || ld % 8) return TQ_ERR_ALIGN;
    return TQ_OK;
}

tq_status check_output(const void *Y, int64_t M, int64_t N, int64_t ldy, int esize) {
    if (!Y) return TQ_ERR_NULL;
    if (ldy < N) return TQ_ERR_SHAPE;
    if (!mul_ok(M, ldy) || !mul_ok(M * ldy, esize)) return TQ_ERR_OVERFLOW;
    if (!aligned(Y, static_cast<uintptr_t>(esize))) return TQ_ERR_ALIGN;
    return TQ_OK;
}

tq_status check_weights(const void *Wq, const float *sw, int64_t N, int64_t K, int bits) {
    if (bits != 8 && bits != 4) return TQ_ERR_BITS;
    if (!Wq || !sw) return TQ_ERR_NULL;
    if (!mul_ok(N, K)) return TQ_ERR_OVERFLOW;
    if (!aligned(Wq, 16) || !aligned(sw, 4)) return TQ_ERR_ALIGN;
    return TQ_OK;
}

int out_size(tq_out y) { return y == TQ_OUT_BF16 ? 2 : 4; }

// The checks of tq_linear (A16 modes) for every call of a grouped plan.
tq_status check_grouped(const tq_a16_call *calls, int64_t n, int bits, tq_out ytype) {
    if (bits != 8 && bits != 4) return TQ_ERR_BITS;
    if (ytype != TQ_OUT_F32 && ytype != TQ_OUT_BF16) return TQ_ERR_MODE;
    if (n < 0) return TQ_ERR_SHAPE;
    if (n > 0 && !calls) return TQ_ERR_NULL;
    for (int64_t c = 0; c < n; ++c) {
        const tq_a16_call &a = calls[c];
        if (a.M < 0 || a.M > TQ_MAX_M_GROUPED || a.N < 0 || !valid_k(a.K)) return TQ_ERR_SHAPE;
        if (a.M == 0 || a.N == 0) continue;
        tq_status st = check_bf16_rows(a.X, a.M, a.K, a.ldx);
        if (st != TQ_OK) return st;
        if ((st = check_weights(a.Wq, a.sw, a.N, a.K, bits)) != TQ_OK) return st;
        if ((st = check_output(a.Y, a.M, a.N, a.ldy, out_size(ytype))) != TQ_OK) return st;
        if (grouped_item_rows(a.M, a.K, bits) == 0) return TQ_ERR_SHAPE;
    }
    return TQ_OK;
}

// The checks of a chained plan: each call as a grouped call, plus its up rows.
tq_status check_chain(const tq_chain_call *calls, int64_t n, int bits, tq_out ytype) {
    if (bits != 8 && bits != 4) return TQ_ERR_BITS;
    if (ytype != TQ_OUT_F32 && ytype != TQ_OUT_BF16) return TQ_ERR_MODE;
    if (n < 0) return TQ_ERR_SHAPE;
    if (n > 0 && !calls) return TQ_ERR_NULL;
    for (int64_t c = 0; c < n; ++c) {
        const tq_a16_call &a = calls[c].call;
        if (a.M < 0 || a.M > TQ_MAX_M_GROUPED || a.N < 0 || !valid_k(a.K)) return TQ_ERR_SHAPE;
        if (a.M == 0 || a.N == 0) continue;
        tq_status st = check_bf16_rows(a.X, a.M, a.K, a.ldx);
        if (st != TQ_OK) return st;
        if (calls[c].U && (st = check_bf16_rows(calls[c].U, a.M, a.K, calls[c].ldu)) != TQ_OK) return st;
        if ((st = check_weights(a.Wq, a.sw, a.N, a.K, bits)) != TQ_OK) return st;
        if ((st = check_output(a.Y, a.M, a.N, a.ldy, out_size(ytype))) != TQ_OK) return st;
        if (chain_item_rows(a.M, a.K, a.N, bits, 0) == 0) return TQ_ERR_SHAPE;
    }
    return TQ_OK;
}

}  // namespace
}  // namespace tq

using namespace tq;

extern "C" {

const char *tq_status_str(tq_status s) {
    switch (s) {
        case TQ_OK: return "TQ_OK";
        case TQ_ERR_NULL: return "TQ_ERR_NULL: a required pointer is NULL";
        case TQ_ERR_SHAPE: return "TQ_ERR_SHAPE: a size, stride or group width is not allowed";
        case TQ_ERR_BITS: return "TQ_ERR_BITS: bits must be 8 or 4";
        case TQ_ERR_MODE: return "TQ_ERR_MODE: unknown mode or output type, or bits disagree with the mode";
        case TQ_ERR_OVERFLOW: return "TQ_ERR_OVERFLOW: a size product overflows";
        case TQ_ERR_ALIGN: return "TQ_ERR_ALIGN: a pointer or stride breaks the 16-byte rule";
        case TQ_ERR_WORKSPACE: return "TQ_ERR_WORKSPACE: workspace missing or too small";
        case TQ_ERR_CUDA: return "TQ_ERR_CUDA: a CUDA call failed";
        case TQ_ERR_DEVICE_TIMEOUT: return "TQ_ERR_DEVICE_TIMEOUT: a bounded device wait expired";
        case TQ_ERR_DEVICE: return "TQ_ERR_DEVICE: no usable sm_103 device is current";
    }
    return "TQ_ERR_UNKNOWN";
}

int tq_last_cuda_error(void) { return g_last_cuda_error; }

int tq_version(void) { return 100; }

tq_status tq_quantize_weights(const void *W, int64_t N, int64_t K, int64_t ldw,
                              int bits, int group, void *codes, float *scales,
                              cudaStream_t stream) {
    if (bits != 8 && bits != 4) return TQ_ERR_BITS;
    if (group != kGroup || N < 0 || !valid_k(K)) return TQ_ERR_SHAPE;
    if (N == 0) return TQ_OK;
    tq_status st = check_bf16_rows(W, N, K, ldw);
    if (st != TQ_OK) return st;
    if (!codes || !scales) return TQ_ERR_NULL;
    if (!mul_ok(N, K)) return TQ_ERR_OVERFLOW;
    if (!aligned(codes, 16) || !aligned(scales, 4)) return TQ_ERR_ALIGN;
    DeviceInfo dev;
    if ((st = current_device(&dev)) != TQ_OK) return st;
    return launch_quantize_weights(static_cast<const uint16_t *>(W), N, K, ldw, bits,
                                   codes, scales, stream);
}

tq_status tq_quantize_weights_blocked(const void *W, int64_t N, int64_t K, int64_t ldw, int bits, int G,
                                      int rotate, void *codes, float *scales, cudaStream_t stream) {
    if (bits != 8 && bits != 4) return TQ_ERR_BITS;
    if (rotate != 0 && rotate != 1) return TQ_ERR_MODE;
    if (N < 0 || !valid_k(K) || !valid_block(G, K)) return TQ_ERR_SHAPE;
    if (N == 0) return TQ_OK;
    tq_status st = check_bf16_rows(W, N, K, ldw);
    if (st != TQ_OK) return st;
    if (!codes || !scales) return TQ_ERR_NULL;
    if (!mul_ok(N, K)) return TQ_ERR_OVERFLOW;
    if (!aligned(codes, 16) || !aligned(scales, 4)) return TQ_ERR_ALIGN;
    DeviceInfo dev;
    if ((st = current_device(&dev)) != TQ_OK) return st;
    return launch_quantize_weights_blocked(static_cast<const uint16_t *>(W), N, K, ldw, bits, G, rotate, codes,
                                           scales, stream);
}

tq_status tq_linear_blocked(const void *X, int64_t M, int64_t K, int64_t ldx, const void *Wq, const float *sw,
                            int G, int64_t N, int bits, int rotate, void *Y, tq_out ytype, int64_t ldy,
                            cudaStream_t stream) {
    if (bits != 8 && bits != 4) return TQ_ERR_BITS;
    if (rotate != 0 && rotate != 1) return TQ_ERR_MODE;
    if (ytype != TQ_OUT_F32 && ytype != TQ_OUT_BF16) return TQ_ERR_MODE;
    if (M < 0 || M > TQ_MAX_M_BLOCKED || N < 0 || !valid_k(K) || !valid_block(G, K)) return TQ_ERR_SHAPE;
    if (M == 0 || N == 0) return TQ_OK;
    tq_status st = check_bf16_rows(X, M, K, ldx);
    if (st != TQ_OK) return st;
    if ((st = check_weights(Wq, sw, N, K, bits)) != TQ_OK) return st;
    if ((st = check_output(Y, M, N, ldy, out_size(ytype))) != TQ_OK) return st;
    DeviceInfo dev;
    if ((st = current_device(&dev)) != TQ_OK) return st;
    // the token rows are staged in shared memory as fp32
    if (static_cast<int64_t>(gemv_blocked_mt(static_cast<int>(M))) * K * 4 > dev.smem_optin) return TQ_ERR_SHAPE;
    return launch_gemv_blocked(static_cast<const uint16_t *>(X), static_cast<int>(M), K, ldx,
                               static_cast<const uint8_t *>(Wq), sw, G, N, bits, rotate, Y,
                               ytype == TQ_OUT_BF16 ? 1 : 0, ldy, dev, stream);
}

tq_status tq_linear_swiglu(const void *G, int64_t ldg, const void *U, int64_t ldu, int64_t M, int64_t K,
                           const void *Wq, const float *sw, int64_t N, int bits, tq_mode mode, void *Y,
                           tq_out ytype, int64_t ldy, cudaStream_t stream) {
    if (bits != 8 && bits != 4) return TQ_ERR_BITS;
    if (mode != TQ_W8A16 && mode != TQ_W4A16) return TQ_ERR_MODE;
    if ((mode == TQ_W8A16 && bits != 8) || (mode == TQ_W4A16 && bits != 4)) return TQ_ERR_MODE;
    if (ytype != TQ_OUT_F32 && ytype != TQ_OUT_BF16) return TQ_ERR_MODE;
    if (M < 0 || M > 8 || N < 0 || !valid_k(K)) return TQ_ERR_SHAPE;
    if (M == 0 || N == 0) return TQ_OK;
    tq_status st = check_bf16_rows(G, M, K, ldg);
    if (st != TQ_OK) return st;
    if ((st = check_bf16_rows(U, M, K, ldu)) != TQ_OK) return st;
    if ((st = check_weights(Wq, sw, N, K, bits)) != TQ_OK) return st;
    if ((st = check_output(Y, M, N, ldy, out_size(ytype))) != TQ_OK) return st;
    DeviceInfo dev;
    if ((st = current_device(&dev)) != TQ_OK) return st;
    if (!gemv_decode_fits(M, N, K, bits, dev)) return TQ_ERR_SHAPE;
    return launch_gemv_small(static_cast<const uint16_t *>(G), M, K, ldg, static_cast<const uint8_t *>(Wq), sw, N,
                             bits, Y, ytype == TQ_OUT_BF16 ? 1 : 0, ldy, dev, stream,
                             static_cast<const uint16_t *>(U), ldu);
}

tq_status tq_rotate_quant_act(const void *X, int64_t M, int64_t K, int64_t ldx,
                              int8_t *Xq, float *sx, cudaStream_t stream) {
    if (M < 0 || !valid_k(K)) return TQ_ERR_SHAPE;
    if (M == 0) return TQ_OK;
    tq_status st = check_bf16_rows(X, M, K, ldx);
    if (st != TQ_OK) return st;
    if (!Xq || !sx) return TQ_ERR_NULL;
    if (!mul_ok(M, K)) return TQ_ERR_OVERFLOW;
    if (!aligned(Xq, 16) || !aligned(sx, 4)) return TQ_ERR_ALIGN;
    DeviceInfo dev;
    if ((st = current_device(&dev)) != TQ_OK) return st;
    return launch_rotate_quant_act(static_cast<const uint16_t *>(X), M, K, ldx, Xq, sx, stream);
}

tq_status tq_rotate_act_bf16(const void *X, int64_t M, int64_t K, int64_t ldx,
                             void *Xr, cudaStream_t stream) {
    if (M < 0 || !valid_k(K)) return TQ_ERR_SHAPE;
    if (M == 0) return TQ_OK;
    tq_status st = check_bf16_rows(X, M, K, ldx);
    if (st != TQ_OK) return st;
    if (!Xr) return TQ_ERR_NULL;
    if (!mul_ok(M, K) || !mul_ok(M * K, 2)) return TQ_ERR_OVERFLOW;
    if (!aligned(Xr, 16)) return TQ_ERR_ALIGN;
    DeviceInfo dev;
    if ((st = current_device(&dev)) != TQ_OK) return st;
    return launch_rotate_bf16(static_cast<const uint16_t *>(X), M, K, ldx,
                              static_cast<uint16_t *>(Xr), stream);
}

size_t tq_act_tiled_bytes(int64_t M, int64_t K) {
    if (M <= 0 || !valid_k(K) || K > TQ_MAX_K_TILED) return 0;
    if (!mul_ok(M + 256, K + 64, INT64_MAX / 8)) return 0;
    return static_cast<size_t>(tiled_act_bytes(M, K));
}

size_t tq_linear_workspace_bytes(int64_t M, int64_t K, int64_t N, int bits, tq_mode mode) {
    (void)bits;
    if (M <= 0 || K <= 0) return 0;
    if (mode == TQ_W8A16 || mode == TQ_W4A16) {
        // optional: the tensor-core product's x' tiles (see tq.h)
        if (M > TQ_MAX_M_A16 || N <= 0 || !valid_k(K) || !mul_ok(N, K)) return 0;
        return skinny_tc_applies(M, N, K) ? static_cast<size_t>(skinny_tc_workspace(M, K)) : 0;
    }
    if (mode != TQ_W8A8) return 0;
    if (!mul_ok(M, K)) return 0;
    const size_t scales = (static_cast<size_t>(M) * 4 + 255) / 256 * 256;
    // K <= TQ_MAX_K_TILED: tiled fp16 codes, then fp32 token scales;
    // longer rows: int8 codes [M, K], then the scales; each 256-byte aligned
    const size_t tiled = tq_act_tiled_bytes(M, K);
    if (tiled > 0) return tiled + scales;
    return (static_cast<size_t>(M) * K + 255) / 256 * 256 + scales;
}

tq_status tq_linear(const void *X, int64_t M, int64_t K, int64_t ldx,
                    const void *Wq, const float *sw, int64_t N, int bits,
                    tq_mode mode, void *Y, tq_out ytype, int64_t ldy,
                    void *workspace, size_t ws_bytes, cudaStream_t stream) {
    if (mode != TQ_W8A16 && mode != TQ_W4A16 && mode != TQ_W8A8) return TQ_ERR_MODE;
    if (ytype != TQ_OUT_F32 && ytype != TQ_OUT_BF16) return TQ_ERR_MODE;
    if (bits != 8 && bits != 4) return TQ_ERR_BITS;
    if ((mode == TQ_W8A16 && bits != 8) || (mode == TQ_W4A16 && bits != 4)) return TQ_ERR_MODE;
    if (M < 0 || N < 0 || !valid_k(K)) return TQ_ERR_SHAPE;
    if (mode != TQ_W8A8 && M > TQ_MAX_M_A16) return TQ_ERR_SHAPE;
    if (M == 0 || N == 0) return TQ_OK;
    tq_status st = check_bf16_rows(X, M, K, ldx);
    if (st != TQ_OK) return st;
    if ((st = check_weights(Wq, sw, N, K, bits)) != TQ_OK) return st;
    if ((st = check_output(Y, M, N, ldy, out_size(ytype))) != TQ_OK) return st;
    const size_t need = tq_linear_workspace_bytes(M, K, N, bits, mode);
    const bool a16 = mode != TQ_W8A8;
    // A16: the workspace is optional (the tensor-core product uses it when
    // given and large enough); W8A8: required
    if (!a16 && need > 0 && (!workspace || ws_bytes < need)) return TQ_ERR_WORKSPACE;
    const bool use_ws = need > 0 && workspace && ws_bytes >= need;
    if (use_ws && !aligned(workspace, 256)) return TQ_ERR_ALIGN;
    DeviceInfo dev;
    if ((st = current_device(&dev)) != TQ_OK) return st;
    if (a16) {
        if (splitk_fits(M, N, K, bits, dev))
            return launch_splitk(static_cast<const uint16_t *>(X), M, K, ldx, static_cast<const uint8_t *>(Wq), sw,
                                 N, bits, Y, ytype == TQ_OUT_BF16 ? 1 : 0, ldy, dev, stream);
        if (use_ws && skinny_tc_fits_device(N, dev))
            return launch_skinny_tc(static_cast<const uint16_t *>(X), M, K, ldx, static_cast<const uint8_t *>(Wq),
                                    sw, N, bits, Y, ytype == TQ_OUT_BF16 ? 1 : 0, ldy, workspace, dev, stream);
        if (a16_streams(M, N, K, bits) &&
            static_cast<int64_t>(gemv_blocked_mt(static_cast<int>(M))) * K * 4 <= dev.smem_optin)
            return launch_gemv_blocked(static_cast<const uint16_t *>(X), static_cast<int>(M), K, ldx,
                                       static_cast<const uint8_t *>(Wq), sw, 0, N, bits, 1, Y,
                                       ytype == TQ_OUT_BF16 ? 1 : 0, ldy, dev, stream);
        if (gemv_small_fits(M, N, K, bits, dev))
            return launch_gemv_small(static_cast<const uint16_t *>(X), M, K, ldx,
                                     static_cast<const uint8_t *>(Wq), sw, N, bits, Y,
                                     ytype == TQ_OUT_BF16 ? 1 : 0, ldy, dev, stream);
        if (!gemv_fits(M, K, bits, dev)) return TQ_ERR_SHAPE;
        return launch_gemv_a16(static_cast<const uint16_t *>(X), M, K, ldx,
                               static_cast<const uint8_t *>(Wq), sw, N, bits, Y,
                               ytype == TQ_OUT_BF16 ? 1 : 0, ldy, dev, stream);
    }
    const size_t tiled = tq_act_tiled_bytes(M, K);
    if (tiled > 0) {
        float *sx = reinterpret_cast<float *>(static_cast<char *>(workspace) + tiled);
        st = launch_rotate_quant_tiled(static_cast<const uint16_t *>(X), M, K, ldx, workspace, sx, stream);
        if (st != TQ_OK) return st;
        return launch_gemm_a8_tiled(workspace, sx, M, K, static_cast<const uint8_t *>(Wq), sw, N, bits,
                                    Y, ytype == TQ_OUT_BF16 ? 1 : 0, ldy, dev, stream);
    }
    int8_t *Xq = static_cast<int8_t *>(workspace);
    float *sx = reinterpret_cast<float *>(static_cast<char *>(workspace) +
                                          (static_cast<size_t>(M) * K + 255) / 256 * 256);
    st = launch_rotate_quant_act(static_cast<const uint16_t *>(X), M, K, ldx, Xq, sx, stream);
    if (st != TQ_OK) return st;
    return launch_gemm_a8(Xq, sx, M, K, static_cast<const uint8_t *>(Wq), sw, N, bits,
                          Y, ytype == TQ_OUT_BF16 ? 1 : 0, ldy, dev, stream);
}

tq_status tq_linear_q8(const int8_t *Xq, const float *sx, int64_t M, int64_t K,
                       const void *Wq, const float *sw, int64_t N, int bits,
                       void *Y, tq_out ytype, int64_t ldy, cudaStream_t stream) {
    if (ytype != TQ_OUT_F32 && ytype != TQ_OUT_BF16 && ytype != TQ_OUT_I32) return TQ_ERR_MODE;
    if (bits != 8 && bits != 4) return TQ_ERR_BITS;
    if (M < 0 || N < 0 || !valid_k(K)) return TQ_ERR_SHAPE;
    if (M == 0 || N == 0) return TQ_OK;
    if (!Xq || (ytype != TQ_OUT_I32 && !sx)) return TQ_ERR_NULL;
    if (!mul_ok(M, K)) return TQ_ERR_OVERFLOW;
    if (!aligned(Xq, 16) || (sx && !aligned(sx, 4))) return TQ_ERR_ALIGN;
    tq_status st = check_weights(Wq, sw, N, K, bits);
    if (st != TQ_OK) return st;
    if ((st = check_output(Y, M, N, ldy, out_size(ytype))) != TQ_OK) return st;
    DeviceInfo dev;
    if ((st = current_device(&dev)) != TQ_OK) return st;
    return launch_gemm_a8(Xq, sx, M, K, static_cast<const uint8_t *>(Wq), sw, N, bits, Y,
                          static_cast<int>(ytype), ldy, dev, stream);
}

tq_status tq_rotate_quant_act_tiled(const void *X, int64_t M, int64_t K, int64_t ldx, void *At,
                                    size_t at_bytes, float *sx, cudaStream_t stream) {
    if (M < 0 || !valid_k(K) || K > TQ_MAX_K_TILED) return TQ_ERR_SHAPE;
    if (M == 0) return TQ_OK;
    tq_status st = check_bf16_rows(X, M, K, ldx);
    if (st != TQ_OK) return st;
    if (!At || !sx) return TQ_ERR_NULL;
    const size_t need = tq_act_tiled_bytes(M, K);
    if (need == 0) return TQ_ERR_OVERFLOW;
    if (at_bytes < need) return TQ_ERR_WORKSPACE;
    if (!aligned(At, 256) || !aligned(sx, 4)) return TQ_ERR_ALIGN;
    DeviceInfo dev;
    if ((st = current_device(&dev)) != TQ_OK) return st;
    return launch_rotate_quant_tiled(static_cast<const uint16_t *>(X), M, K, ldx, At, sx, stream);
}

tq_status tq_swiglu_quant_act_tiled(const void *G, int64_t ldg, const void *U, int64_t ldu, int64_t M,
                                    int64_t K, void *At, size_t at_bytes, float *sx, cudaStream_t stream) {
    if (M < 0 || !valid_k(K) || K > TQ_MAX_K_TILED) return TQ_ERR_SHAPE;
    if (M == 0) return TQ_OK;
    tq_status st = check_bf16_rows(G, M, K, ldg);
    if (st != TQ_OK) return st;
    if ((st = check_bf16_rows(U, M, K, ldu)) != TQ_OK) return st;
    if (!At || !sx) return TQ_ERR_NULL;
    const size_t need = tq_act_tiled_bytes(M, K);
    if (need == 0) return TQ_ERR_OVERFLOW;
    if (at_bytes < need) return TQ_ERR_WORKSPACE;
    if (!aligned(At, 256) || !aligned(sx, 4)) return TQ_ERR_ALIGN;
    DeviceInfo dev;
    if ((st = current_device(&dev)) != TQ_OK) return st;
    return launch_swiglu_quant_tiled(static_cast<const uint16_t *>(G), ldg, static_cast<const uint16_t *>(U),
                                     ldu, M, K, At, sx, stream);
}

tq_status tq_modnorm_quant_act_tiled(const void *X, int64_t M, int64_t K, int64_t ldx, const float *shift,
                                     const float *scale, float eps, void *At, size_t at_bytes, float *sx,
                                     cudaStream_t stream) {
    if (M < 0 || !valid_k(K) || K > TQ_MAX_K_TILED) return TQ_ERR_SHAPE;
    if (!(eps >= 0.0f) || !std::isfinite(eps)) return TQ_ERR_MODE;   // NaN, negative or infinite
    if (M == 0) return TQ_OK;
    tq_status st = check_bf16_rows(X, M, K, ldx);
    if (st != TQ_OK) return st;
    if (!shift || !scale || !At || !sx) return TQ_ERR_NULL;
    const size_t need = tq_act_tiled_bytes(M, K);
    if (need == 0) return TQ_ERR_OVERFLOW;
    if (at_bytes < need) return TQ_ERR_WORKSPACE;
    if (!aligned(At, 256) || !aligned(sx, 4) || !aligned(shift, 16) || !aligned(scale, 16)) return TQ_ERR_ALIGN;
    DeviceInfo dev;
    if ((st = current_device(&dev)) != TQ_OK) return st;
    return launch_modnorm_quant_tiled(static_cast<const uint16_t *>(X), M, K, ldx, shift, scale, eps, At, sx,
                                      stream);
}

tq_status tq_linear_tiled(const void *At, const float *sx, int64_t M, int64_t K, const void *Wq,
                          const float *sw, int64_t N, int bits, void *Y, tq_out ytype, int64_t ldy,
                          cudaStream_t stream) {
    if (ytype != TQ_OUT_F32 && ytype != TQ_OUT_BF16 && ytype != TQ_OUT_I32) return TQ_ERR_MODE;
    if (bits != 8 && bits != 4) return TQ_ERR_BITS;
    if (M < 0 || N < 0 || !valid_k(K) || K > TQ_MAX_K_TILED) return TQ_ERR_SHAPE;
    if (M == 0 || N == 0) return TQ_OK;
    if (!At || (ytype != TQ_OUT_I32 && !sx)) return TQ_ERR_NULL;
    if (tq_act_tiled_bytes(M, K) == 0) return TQ_ERR_OVERFLOW;
    if (!aligned(At, 256) || (sx && !aligned(sx, 4))) return TQ_ERR_ALIGN;
    tq_status st = check_weights(Wq, sw, N, K, bits);
    if (st != TQ_OK) return st;
    if ((st = check_output(Y, M, N, ldy, out_size(ytype))) != TQ_OK) return st;
    DeviceInfo dev;
    if ((st = current_device(&dev)) != TQ_OK) return st;
    return launch_gemm_a8_tiled(At, sx, M, K, static_cast<const uint8_t *>(Wq), sw, N, bits, Y,
                                static_cast<int>(ytype), ldy, dev, stream);
}

size_t tq_weights_tiled_bytes(int64_t N, int64_t K) {
    if (N <= 0 || !valid_k(K) || K > TQ_MAX_K_TILED) return 0;
    if (!mul_ok(N + 256, K + 64, INT64_MAX / 8)) return 0;
    return static_cast<size_t>(weights_tiled_bytes(N, K));
}

tq_status tq_tile_weights(const void *Wq, int64_t N, int64_t K, int bits, void *Wt, size_t wt_bytes,
                          cudaStream_t stream) {
    if (bits != 8 && bits != 4) return TQ_ERR_BITS;
    if (N < 0 || !valid_k(K) || K > TQ_MAX_K_TILED) return TQ_ERR_SHAPE;
    if (N == 0) return TQ_OK;
    if (!Wq || !Wt) return TQ_ERR_NULL;
    const size_t need = tq_weights_tiled_bytes(N, K);
    if (need == 0) return TQ_ERR_OVERFLOW;
    if (wt_bytes < need) return TQ_ERR_WORKSPACE;
    if (!aligned(Wq, 16) || !aligned(Wt, 256)) return TQ_ERR_ALIGN;
    DeviceInfo dev;
    const tq_status st = current_device(&dev);
    if (st != TQ_OK) return st;
    return launch_tile_weights(static_cast<const uint8_t *>(Wq), N, K, bits, Wt, stream);
}

tq_status tq_linear_tt(const void *At, const float *sx, int64_t M, int64_t K, const void *Wt,
                       const float *sw, int64_t N, int bits, void *Y, tq_out ytype, int64_t ldy,
                       cudaStream_t stream) {
    return tq_linear_tt_ex(At, sx, M, K, Wt, sw, N, bits, nullptr, Y, ytype, ldy, stream);
}

static tq_status linear_tt_impl(const void *At, const float *sx, int64_t M, int64_t K, const void *Wt,
                                const float *sw, int64_t N, int bits, const tq_epilogue *epi, void *Y,
                                tq_out ytype, int64_t ldy, void *split_ws, size_t split_bytes,
                                cudaStream_t stream);

tq_status tq_linear_tt_ex(const void *At, const float *sx, int64_t M, int64_t K, const void *Wt,
                          const float *sw, int64_t N, int bits, const tq_epilogue *epi, void *Y,
                          tq_out ytype, int64_t ldy, cudaStream_t stream) {
    return linear_tt_impl(At, sx, M, K, Wt, sw, N, bits, epi, Y, ytype, ldy, nullptr, 0, stream);
}

size_t tq_split_workspace_bytes(void) {
    DeviceInfo dev;
    if (current_device(&dev) != TQ_OK) return 0;
    return split_workspace_bytes(dev);
}

tq_status tq_linear_tt_split(const void *At, const float *sx, int64_t M, int64_t K, const void *Wt,
                             const float *sw, int64_t N, int bits, const tq_epilogue *epi, void *Y,
                             tq_out ytype, int64_t ldy, void *workspace, size_t ws_bytes, cudaStream_t stream) {
    return linear_tt_impl(At, sx, M, K, Wt, sw, N, bits, epi, Y, ytype, ldy, workspace, ws_bytes, stream);
}

static tq_status linear_tt_impl(const void *At, const float *sx, int64_t M, int64_t K, const void *Wt,
                                const float *sw, int64_t N, int bits, const tq_epilogue *epi, void *Y,
                                tq_out ytype, int64_t ldy, void *split_ws, size_t split_bytes,
                                cudaStream_t stream) {
    if (ytype != TQ_OUT_F32 && ytype != TQ_OUT_BF16 && ytype != TQ_OUT_I32) return TQ_ERR_MODE;
    if (bits != 8 && bits != 4) return TQ_ERR_BITS;
    if (M < 0 || N < 0 || !valid_k(K) || K > TQ_MAX_K_TILED) return TQ_ERR_SHAPE;
    if (M == 0 || N == 0) return TQ_OK;
    if (!At || !Wt || !sw || (ytype != TQ_OUT_I32 && !sx)) return TQ_ERR_NULL;
    if (tq_act_tiled_bytes(M, K) == 0 || tq_weights_tiled_bytes(N, K) == 0) return TQ_ERR_OVERFLOW;
    if (!aligned(At, 256) || !aligned(Wt, 256) || !aligned(sw, 4) || (sx && !aligned(sx, 4)))
        return TQ_ERR_ALIGN;
    tq_status st = check_output(Y, M, N, ldy, out_size(ytype));
    if (st != TQ_OK) return st;
    EpilogueArgs ea;
    if (epi) {
        if (ytype == TQ_OUT_I32) return TQ_ERR_MODE;
        if (epi->rtype != TQ_OUT_F32 && epi->rtype != TQ_OUT_BF16) return TQ_ERR_MODE;
        if ((epi->bias && !aligned(epi->bias, 4)) || (epi->gate && !aligned(epi->gate, 4))) return TQ_ERR_ALIGN;
        if (epi->residual) {
            const int rs = out_size(epi->rtype);
            if ((st = check_output(epi->residual, M, N, epi->ldr, rs)) != TQ_OK) return st;
            // the same buffer is an in-place update; any other overlap is refused
            const uintptr_t r0 = reinterpret_cast<uintptr_t>(epi->residual);
            const uintptr_t r1 = r0 + static_cast<uintptr_t>(((M - 1) * epi->ldr + N) * rs);
            const uintptr_t y0 = reinterpret_cast<uintptr_t>(Y);
            const uintptr_t y1 = y0 + static_cast<uintptr_t>(((M - 1) * ldy + N) * out_size(ytype));
            if (r0 == y0) {
                if (epi->ldr != ldy || epi->rtype != ytype) return TQ_ERR_SHAPE;
            } else if (r0 < y1 && y0 < r1) {
                return TQ_ERR_SHAPE;
            }
        }
        ea.bias = epi->bias;
        ea.gate = epi->gate;
        ea.R = epi->residual;
        ea.ldr = epi->ldr;
        ea.rtype = epi->rtype == TQ_OUT_BF16 ? 1 : 0;
    }
    DeviceInfo dev;
    if ((st = current_device(&dev)) != TQ_OK) return st;
    if (split_ws) {
        if (split_bytes < split_workspace_bytes(dev)) return TQ_ERR_WORKSPACE;
        if (!aligned(split_ws, 256)) return TQ_ERR_ALIGN;
    }
    return launch_gemm_a8_tt(At, sx, M, K, Wt, sw, N, bits, Y, static_cast<int>(ytype), ldy, dev, stream,
                             epi ? &ea : nullptr, split_ws);
}

tq_status tq_device_status(cudaStream_t stream) {
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_fail(e);
    unsigned int v = 0;
    e = cudaMemcpyFromSymbol(&v, g_status_word, sizeof(v));
    if (e != cudaSuccess) return cuda_fail(e);
    if (v != 0) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(g_status_word, &zero, sizeof(zero));
        if (e != cudaSuccess) return cuda_fail(e);
        return TQ_ERR_DEVICE_TIMEOUT;
    }
    return TQ_OK;
}

tq_status tq_grouped_bytes(const tq_a16_call *calls, int64_t ncalls, int bits, size_t *bytes) {
    if (!bytes) return TQ_ERR_NULL;
    const tq_status st = check_grouped(calls, ncalls, bits, TQ_OUT_F32);
    if (st != TQ_OK) return st;
    return grouped_bytes(calls, ncalls, bits, bytes);
}

tq_status tq_grouped_create(const tq_a16_call *calls, int64_t ncalls, int bits, tq_out ytype,
                            void *dmem, size_t dbytes, tq_grouped *plan) {
    if (!plan) return TQ_ERR_NULL;
    tq_status st = check_grouped(calls, ncalls, bits, ytype);
    if (st != TQ_OK) return st;
    size_t need = 0;
    if ((st = grouped_bytes(calls, ncalls, bits, &need)) != TQ_OK) return st;
    if (need > 0 && (!dmem || dbytes < need)) return TQ_ERR_WORKSPACE;
    if (dmem && !aligned(dmem, 256)) return TQ_ERR_ALIGN;
    DeviceInfo dev;
    if ((st = current_device(&dev)) != TQ_OK) return st;
    return grouped_create(calls, ncalls, bits, ytype == TQ_OUT_BF16 ? 1 : 0, dmem, dbytes, dev, plan);
}

static tq_status grouped_phase(tq_grouped plan, int phase, cudaStream_t stream) {
    if (!plan) return TQ_ERR_NULL;
    DeviceInfo dev;
    const tq_status st = current_device(&dev);
    if (st != TQ_OK) return st;
    return grouped_run(plan, dev, phase, stream);
}

tq_status tq_grouped_run(tq_grouped plan, cudaStream_t stream) { return grouped_phase(plan, 3, stream); }

tq_status tq_grouped_rotate(tq_grouped plan, cudaStream_t stream) { return grouped_phase(plan, 1, stream); }

tq_status tq_grouped_product(tq_grouped plan, cudaStream_t stream) { return grouped_phase(plan, 2, stream); }

tq_status tq_chain_bytes(const tq_chain_call *calls, int64_t ncalls, int bits, size_t *bytes) {
    if (!bytes) return TQ_ERR_NULL;
    const tq_status st = check_chain(calls, ncalls, bits, TQ_OUT_F32);
    if (st != TQ_OK) return st;
    return chain_bytes(calls, ncalls, bits, bytes);
}

tq_status tq_chain_create(const tq_chain_call *calls, int64_t ncalls, int bits, tq_out ytype,
                          void *dmem, size_t dbytes, tq_grouped *plan) {
    if (!plan) return TQ_ERR_NULL;
    tq_status st = check_chain(calls, ncalls, bits, ytype);
    if (st != TQ_OK) return st;
    size_t need = 0;
    if ((st = chain_bytes(calls, ncalls, bits, &need)) != TQ_OK) return st;
    if (need > 0 && (!dmem || dbytes < need)) return TQ_ERR_WORKSPACE;
    if (dmem && !aligned(dmem, 256)) return TQ_ERR_ALIGN;
    DeviceInfo dev;
    if ((st = current_device(&dev)) != TQ_OK) return st;
    return chain_create(calls, ncalls, bits, ytype == TQ_OUT_BF16 ? 1 : 0, dmem, dbytes, dev, plan);
}

int64_t tq_grouped_weight_bytes(tq_grouped plan) { return plan ? grouped_weight_bytes(plan) : 0; }

void tq_grouped_destroy(tq_grouped plan) {
    if (plan) grouped_destroy(plan);
}

}  // extern "C"
