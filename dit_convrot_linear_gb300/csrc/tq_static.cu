// tq_linear_a8_static: the W8A8 / W4A8 product without any caller-provided
// workspace and without any allocation.
//
// tq_linear needs device scratch for the quantised activations (int8 codes
// [M, K] and fp32 token scales [M]) and expects the caller to provide it.  Some
// callers cannot: a plugin whose host application owns every device
// allocation and does not hand one out, or a service that reserves all device
// memory at start-up and forbids allocating afterwards, has no workspace to
// give and may not call cudaMalloc itself.  This entry point keeps that scratch
// in one fixed array compiled into the library instead.
//
// The array below is a file-scope __device__ variable: each GPU that loads the
// library holds TQ_STATIC_SCRATCH_BYTES for it until the process exits.  In host
// code its name is only a host-side stand-in, so its device address is looked
// up with cudaGetSymbolAddress, once per device, on the first call made with
// that device current, and then passed to the kernels.  The lookup is tied to
// the CUDA context it was made in: if that context is destroyed and another
// one created for the device (cudaDeviceReset, for example), the module is
// loaded anew at another address, so the next call repeats the lookup.
// Nothing here calls cudaMalloc, cudaFree or any allocating routine.

#include <cuda.h>

#include <mutex>

#include "tq_internal.cuh"

namespace tq {
namespace {

static __device__ __align__(256) unsigned char g_static_scratch[TQ_STATIC_SCRATCH_BYTES];

typedef CUresult (*CtxGetCurrentFn)(CUcontext *);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long *);

// Process-unique identity of the context current on this thread (context ids
// are never reused), or 0 when there is none or it cannot be read.
unsigned long long current_context_id() {
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *a = nullptr, *b = nullptr;
        cudaDriverEntryPointQueryResult qa{}, qb{};
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &a, 12000, cudaEnableDefault, &qa) ==
                    cudaSuccess && qa == cudaDriverEntryPointSuccess &&
            cudaGetDriverEntryPointByVersion("cuCtxGetId", &b, 12000, cudaEnableDefault, &qb) == cudaSuccess &&
            qb == cudaDriverEntryPointSuccess) {
            get_current = reinterpret_cast<CtxGetCurrentFn>(a);
            get_id = reinterpret_cast<CtxGetIdFn>(b);
        }
        cudaGetLastError();
    });
    if (!get_current || !get_id) return 0;
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

struct ScratchSlot {
    void *ptr = nullptr;          // device address of g_static_scratch
    unsigned long long ctx = 0;   // context it was looked up in
};

std::mutex g_static_mu;
ScratchSlot g_static_slot[64];   // per device

tq_status static_scratch(int dev, void **out) {
    if (dev < 0 || dev >= 64) return TQ_ERR_DEVICE;
    std::lock_guard<std::mutex> lock(g_static_mu);
    ScratchSlot &s = g_static_slot[dev];
    const unsigned long long ctx = current_context_id();
    if (!s.ptr || ctx == 0 || s.ctx != ctx) {
        void *p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
        if (e != cudaSuccess || !p) return cuda_fail(e != cudaSuccess ? e : cudaErrorInvalidSymbol);
        s.ptr = p;
        // read again: the lookup may itself have made the context current
        s.ctx = current_context_id();
    }
    *out = s.ptr;
    return TQ_OK;
}

bool is_aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool k_ok(int64_t K) {
    if (K <= 0 || K > TQ_MAX_K) return false;
    const int64_t t = K % kGroup;
    return t == 0 || t == 32 || t == 64 || t == 128;
}

}  // namespace
}  // namespace tq

using namespace tq;

extern "C" tq_status tq_linear_a8_static(const void *X, int64_t M, int64_t K, int64_t ldx,
                                         const void *Wq, const float *sw, int64_t N, int bits,
                                         void *Y, tq_out ytype, int64_t ldy,
                                         cudaStream_t stream) {
    if (ytype != TQ_OUT_F32 && ytype != TQ_OUT_BF16) return TQ_ERR_MODE;
    if (bits != 8 && bits != 4) return TQ_ERR_BITS;
    if (M < 0 || N < 0 || !k_ok(K)) return TQ_ERR_SHAPE;
    if (M == 0 || N == 0) return TQ_OK;
    if (!X || !Wq || !sw || !Y) return TQ_ERR_NULL;
    if (ldx < K || ldy < N) return TQ_ERR_SHAPE;
    const int esize = ytype == TQ_OUT_BF16 ? 2 : 4;
    if (M > (INT64_MAX / 4) / ldx || N > (INT64_MAX / 4) / K || M > (INT64_MAX / 4) / ldy)
        return TQ_ERR_OVERFLOW;
    if (!is_aligned(X, 16) || ldx % 8 || !is_aligned(Wq, 16) || !is_aligned(sw, 4) ||
        !is_aligned(Y, static_cast<uintptr_t>(esize)))
        return TQ_ERR_ALIGN;
    // int8 codes [M, K], then fp32 token scales [M], each 256-byte aligned
    if (M > static_cast<int64_t>(TQ_STATIC_SCRATCH_BYTES) / K) return TQ_ERR_WORKSPACE;
    const size_t codes = (static_cast<size_t>(M) * K + 255) / 256 * 256;
    const size_t need = codes + (static_cast<size_t>(M) * 4 + 255) / 256 * 256;
    if (need > TQ_STATIC_SCRATCH_BYTES) return TQ_ERR_WORKSPACE;

    DeviceInfo dev;
    tq_status st = current_device(&dev);
    if (st != TQ_OK) return st;
    void *scratch = nullptr;
    if ((st = static_scratch(dev.id, &scratch)) != TQ_OK) return st;
    // every byte the product reads from the scratch is written first by the
    // quantiser, so nothing has to be cleared between calls
    int8_t *Xq = static_cast<int8_t *>(scratch);
    float *sx = reinterpret_cast<float *>(static_cast<char *>(scratch) + codes);
    st = launch_rotate_quant_act(static_cast<const uint16_t *>(X), M, K, ldx, Xq, sx, stream);
    if (st != TQ_OK) return st;
    return launch_gemm_a8(Xq, sx, M, K, static_cast<const uint8_t *>(Wq), sw, N, bits, Y,
                          ytype == TQ_OUT_BF16 ? 1 : 0, ldy, dev, stream);
}
