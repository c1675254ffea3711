// A8 product, legacy tensor-core path: int8 activation codes x int8 (or
// int4, widened to int8 in registers) weight codes, exact int32 sums by
// mma.sync m16n8k32 s8.s8.s32, then Y = sx[m] * sw[n] * acc (DiT projections,
// compute-bound at large M; kvad-gpu internals, "Quantised weights on the
// GPU": past the crossover the batch makes every matmul real work).
//
// CTA tile 128 x 128, K step 64, 3-stage cp.async pipeline; 8 warps as 2 x 4,
// each 64 x 32.  Shared rows are padded to 80 bytes so the 4-byte fragment
// reads of 8 rows x 4 lanes hit 32 distinct banks.

#include "tq_internal.cuh"

namespace tq {
namespace {

constexpr int BM = 128, BN = 128, BK = 64, STAGES = 3;
constexpr int LDA = 80;            // bytes per shared row of A (and int8 B)
constexpr int LDB4 = 48;           // bytes per shared row of packed int4 B

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem, bool valid) {
    const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
    const int n = valid ? 16 : 0;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(s), "l"(gmem), "r"(n)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__device__ __forceinline__ void mma_s8(int (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                       uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+r"(d[0]), "+r"(d[1]), "+r"(d[2]), "+r"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// four packed int4 codes (16 bits) -> four sign-extended int8 bytes
__device__ __forceinline__ uint32_t widen4_i8(uint32_t x) {
    const uint32_t u = (x & 0xFu) | ((x & 0xF0u) << 4) | ((x & 0xF00u) << 8) | ((x & 0xF000u) << 12);
    return __vsub4(u ^ 0x08080808u, 0x08080808u);
}

template <int BITS>
__global__ void __launch_bounds__(256)
k_gemm_a8_mma(const int8_t *__restrict__ Xq, const float *__restrict__ sx, int64_t M,
              int64_t K, const uint8_t *__restrict__ Wq, const float *__restrict__ sw,
              int64_t N, void *__restrict__ Y, int ytype, int64_t ldy) {
    constexpr int LDB = BITS == 8 ? LDA : LDB4;
    constexpr int BKB = BITS == 8 ? BK : BK / 2;   // weight bytes per row per step
    extern __shared__ __align__(16) uint8_t smem_mma[];
    uint8_t (*sA)[BM * LDA] = reinterpret_cast<uint8_t (*)[BM * LDA]>(smem_mma);
    uint8_t (*sB)[BN * LDB] = reinterpret_cast<uint8_t (*)[BN * LDB]>(smem_mma + STAGES * BM * LDA);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int wm = warp >> 2, wn = warp & 3;         // 2 x 4 warps
    const int g = lane >> 2, t = lane & 3;
    const int64_t m0 = static_cast<int64_t>(blockIdx.y) * BM;
    const int64_t n0 = static_cast<int64_t>(blockIdx.x) * BN;
    const int64_t wld = BITS == 8 ? K : K / 2;
    const int nsteps = static_cast<int>((K + BK - 1) / BK);

    auto load_stage = [&](int st, int step) {
        const int64_t k0 = static_cast<int64_t>(step) * BK;
        // A: 128 rows x 64 bytes = 512 chunks of 16 B
        for (int c = tid; c < BM * 4; c += 256) {
            const int r = c >> 2, cc = c & 3;
            const int64_t gm = m0 + r, gk = k0 + cc * 16;
            const bool ok = gm < M && gk < K;
            cp_async16(&sA[st][r * LDA + cc * 16], Xq + (ok ? gm * K + gk : 0), ok);
        }
        // B: 128 rows x BKB bytes
        constexpr int CPR = BKB / 16;
        for (int c = tid; c < BN * CPR; c += 256) {
            const int r = c / CPR, cc = c % CPR;
            const int64_t gn = n0 + r;
            const int64_t gb = static_cast<int64_t>(step) * BKB + cc * 16;
            const bool ok = gn < N && gb < wld;
            cp_async16(&sB[st][r * LDB + cc * 16], Wq + (ok ? gn * wld + gb : 0), ok);
        }
    };

    int acc[4][4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j][0] = acc[i][j][1] = acc[i][j][2] = acc[i][j][3] = 0;

#pragma unroll
    for (int s = 0; s < STAGES - 1; ++s) {
        if (s < nsteps) load_stage(s, s);
        cp_async_commit();
    }
    for (int step = 0; step < nsteps; ++step) {
        cp_async_wait<STAGES - 2>();
        __syncthreads();
        {
            const int nxt = step + STAGES - 1;
            if (nxt < nsteps) load_stage(nxt % STAGES, nxt);
            cp_async_commit();
        }
        const uint8_t *a = sA[step % STAGES];
        const uint8_t *b = sB[step % STAGES];
#pragma unroll
        for (int kk = 0; kk < BK; kk += 32) {
            uint32_t af[4][4], bf[4][2];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int r = wm * 64 + i * 16 + g;
                af[i][0] = *reinterpret_cast<const uint32_t *>(a + r * LDA + kk + 4 * t);
                af[i][1] = *reinterpret_cast<const uint32_t *>(a + (r + 8) * LDA + kk + 4 * t);
                af[i][2] = *reinterpret_cast<const uint32_t *>(a + r * LDA + kk + 16 + 4 * t);
                af[i][3] = *reinterpret_cast<const uint32_t *>(a + (r + 8) * LDA + kk + 16 + 4 * t);
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int r = wn * 32 + j * 8 + g;
                if constexpr (BITS == 8) {
                    bf[j][0] = *reinterpret_cast<const uint32_t *>(b + r * LDB + kk + 4 * t);
                    bf[j][1] = *reinterpret_cast<const uint32_t *>(b + r * LDB + kk + 16 + 4 * t);
                } else {
                    const uint8_t *br = b + r * LDB + kk / 2;
                    bf[j][0] = widen4_i8(*reinterpret_cast<const uint16_t *>(br + 2 * t));
                    bf[j][1] = widen4_i8(*reinterpret_cast<const uint16_t *>(br + 8 + 2 * t));
                }
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    mma_s8(acc[i][j], af[i][0], af[i][1], af[i][2], af[i][3], bf[j][0], bf[j][1]);
        }
    }
    cp_async_wait<0>();

    // epilogue
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int64_t m = m0 + wm * 64 + i * 16 + g + 8 * h;
            if (m >= M) continue;
            const float xs = ytype == 2 ? 1.0f : sx[m];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int64_t n = n0 + wn * 32 + j * 8 + 2 * t + e;
                    if (n >= N) continue;
                    const int a = acc[i][j][2 * h + e];
                    if (ytype == 2) {
                        static_cast<int32_t *>(Y)[m * ldy + n] = a;
                    } else {
                        const float y = (xs * sw[n]) * static_cast<float>(a);
                        if (ytype == 0) static_cast<float *>(Y)[m * ldy + n] = y;
                        else static_cast<uint16_t *>(Y)[m * ldy + n] = f32_to_bf16_bits(y);
                    }
                }
            }
        }
    }
}

}  // namespace

tq_status launch_gemm_a8_mma(const int8_t *Xq, const float *sx, int64_t M, int64_t K,
                             const uint8_t *Wq, const float *sw, int64_t N, int bits,
                             void *Y, int ytype, int64_t ldy, cudaStream_t s) {
    const dim3 grid(static_cast<unsigned>((N + BN - 1) / BN), static_cast<unsigned>((M + BM - 1) / BM));
    const size_t smem8 = STAGES * (BM * LDA + BN * LDA), smem4 = STAGES * (BM * LDA + BN * LDB4);
    static bool configured = false;  // attributes are per function, set once
    if (!configured) {
        cudaFuncSetAttribute(k_gemm_a8_mma<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem8));
        cudaFuncSetAttribute(k_gemm_a8_mma<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem4));
        configured = true;
    }
    if (bits == 8)
        k_gemm_a8_mma<8><<<grid, 256, smem8, s>>>(Xq, sx, M, K, Wq, sw, N, Y, ytype, ldy);
    else
        k_gemm_a8_mma<4><<<grid, 256, smem4, s>>>(Xq, sx, M, K, Wq, sw, N, Y, ytype, ldy);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? TQ_OK : cuda_fail(e);
}

}  // namespace tq
