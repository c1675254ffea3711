// Batched A16 product for a few token rows (M <= 16) over a weight matrix
// that fills the GPU, one call at a time:
//   Y[m][n] = sw[n] * sum_k q[n][k] * x'_bf16[m][k],  fp32 sums,
// x' the group-256 Hadamard rotation of token row m rounded to bf16 (tensai
// docs, "画像生成" / Image generation, section "幅とメモリ": the product's input
// gets the rotation of the weights).  With so few tokens the product is bound
// by the weight stream (kvad-gpu internals, "Numbers"), and the work per
// weight is a handful of multiply-adds: the legacy mma.sync with the tokens as
// its 8-wide N side covers it, so the codes never pass through tensor memory.
//
// One launch, clusters of C CTAs along K, one CTA an SM:
//   - CTA (tile, c) owns 256 weight rows and the c-th of C runs of whole
//     256-groups of K; consumer warp w owns rows 16w .. 16w + 15.  The
//     producer warp streams the run through two 64 KB stages by tensor
//     copies, a stage 256 contiguous bytes of every row (two 128-byte
//     chunks, each stored with the 128-byte swizzle); every consumer warp
//     takes every stage, in order (ring slots are never shared between
//     different warps' uses, which would make a barrier's phase parity
//     ambiguous).  256 bytes of a row a request rather than 128: each row's
//     bytes reach DRAM in longer bursts.  The weights do not depend on the
//     launch before, so the copies start at once.
//   - Its 16 consumer warps wait for the launch before (X may come from it),
//     rotate the tokens' groups of the run, round them to bf16 and keep them
//     in shared memory as fp16 times 2^e, e per token from the run's largest
//     |x| (for 4-bit weights the odd k hold a sixteenth of that), in the
//     lanes' MMA order.  Then warp w multiplies its rows of every stage: each
//     code plus its bias widened into an fp16 subnormal, mma.sync m16n8k16,
//     fp32 sums kept in registers over the whole run.
//   - At the end each CTA writes its partial sums (2^24 times the sum less
//     the bias times the token's sum of x', times 2^-e) to shared memory;
//     after a cluster barrier CTA c adds a 1/C share of the rows over the C
//     CTAs in rank order (distributed shared memory; the result does not
//     depend on timing), scales by sw and stores Y.
// Every wait is bounded: on expiry the status word is set, the cluster skips
// its stores (Y is left unwritten), copies in flight land before the CTA
// exits, and every thread still reaches both cluster barriers.

#include <cooperative_groups.h>
#include <cuda.h>

#include "tq_a16.cuh"

namespace cg = cooperative_groups;

namespace tq {
namespace {

constexpr int SP_R = 2;                       // stages
constexpr int SP_ST = 65536;                  // bytes a stage: 256 rows x two 128-byte chunks
constexpr int SP_RING = SP_R * SP_ST;
constexpr int SP_RB = 256;                    // weight rows a CTA
constexpr int SP_CONS = 16;                   // consumer warps (16 rows each)
constexpr int SP_THREADS = (SP_CONS + 1) * 32;
constexpr int SP_XOFF = SP_RING;              // x' rows
constexpr int SP_XBYTES = 88064;
constexpr int SP_PAMOFF = SP_XOFF + SP_XBYTES;   // per (token, group) maxima, then sums
constexpr int SP_PAMN = 512;                  // pairs' maxima, then (from SP_PAMN / 2) their sums
constexpr int SP_SWOFF = SP_PAMOFF + SP_PAMN * 4;    // the tile's row scales
constexpr int SP_TOKOFF = SP_SWOFF + SP_RB * 4;      // tokens' factors and sums
constexpr int SP_ABOFF = SP_TOKOFF + 3 * 16 * 4;     // abort flag
constexpr int SP_BAROFF = SP_ABOFF + 16;             // full[R], empty[R]
constexpr int SP_SMEM = SP_BAROFF + 2 * SP_R * 8 + 1024;   // + alignment of the ring
static_assert(SP_SMEM <= 232448, "within the opt-in shared memory of a CTA");
static_assert(SP_BAROFF % 8 == 0, "mbarriers 8-byte aligned");
constexpr unsigned int kStatusSplitTimeout = 64u;
constexpr int SP_PAIRS = 8;                   // (token, group) pairs a consumer warp rotates, at most
static_assert(SP_CONS * SP_PAIRS <= SP_PAMN / 2, "every pair has its maximum and its sum");

struct SplitParams {
    const uint16_t *X;
    int64_t ldx;
    int M;              // token rows, at most 8 NG
    int64_t K;
    int G;              // 256-groups of K (the last may be partial)
    int C;              // CTAs of a cluster (the split of K)
    int XS;             // x' row stride (fp16 values; 2 XS = 32 mod 128 bytes)
    const float *sw;
    int64_t N;
    void *Y;
    int64_t ldy;
    int ytype;          // 0 fp32, 1 bf16
    unsigned int *status;
};

__device__ __forceinline__ void consumers_sync() {
    asm volatile("bar.sync 1, %0;" ::"r"(SP_CONS * 32) : "memory");
}

// One poll of an mbarrier phase that may suspend the thread (up to about a
// microsecond, or until the phase completes) instead of returning at once: a
// tight loop of polls keeps the shared-memory pipe busy, which slows every
// other warp's shared loads and shuffles.
__device__ __forceinline__ bool mbar_try_suspend(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
        "selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(1000u)
        : "memory");
    return ok != 0;
}

// Wait for the phase of `parity`, for at most kA16WaitLimit cycles, giving up
// early when another warp has already stopped the CTA.
__device__ __forceinline__ bool sp_wait(uint32_t bar, uint32_t parity, volatile int *abort, unsigned int *status) {
    const long long t0 = clock64();
    while (!mbar_try_suspend(bar, parity)) {
        if (*abort) return false;
        if (clock64() - t0 > kA16WaitLimit) {
            *abort = 1;
            atomicOr(status, kStatusSplitTimeout);
            return false;
        }
    }
    return true;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// One K block (16 bytes of the lane's two rows) into the accumulators of NG
// groups of 8 tokens; x' of token group j is 8 XS values after group j - 1.
template <int BITS, int NG>
__device__ __forceinline__ void sp_block(float (&acc)[NG][4][4], const unsigned char *pa, const unsigned char *pb,
                                         const uint16_t *xblk, int xs8) {
    const uint4 wa = *reinterpret_cast<const uint4 *>(pa);
    const uint4 wb = *reinterpret_cast<const uint4 *>(pb);
    const uint32_t A[4] = {wa.x, wa.y, wa.z, wa.w};
    const uint32_t B[4] = {wb.x, wb.y, wb.z, wb.w};
    if constexpr (BITS == 8) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            uint32_t a0, a1, a2, a3;
            widen_i8_f16_biased(A[q], a0, a2);
            widen_i8_f16_biased(B[q], a1, a3);
#pragma unroll
            for (int j = 0; j < NG; ++j) {
                const uint2 bv = *reinterpret_cast<const uint2 *>(xblk + j * xs8 + q * 16);
                mma_f16(acc[j][q], a0, a1, a2, a3, bv.x, bv.y);
            }
        }
    } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            uint32_t pa4[4], pb4[4];
            widen_i4_f16_biased(A[q], pa4);
            widen_i4_f16_biased(B[q], pb4);
#pragma unroll
            for (int j = 0; j < NG; ++j) {
                const uint2 b0 = *reinterpret_cast<const uint2 *>(xblk + j * xs8 + (2 * q) * 16);
                const uint2 b1 = *reinterpret_cast<const uint2 *>(xblk + j * xs8 + (2 * q + 1) * 16);
                mma_f16(acc[j][(2 * q) % 4], pa4[0], pb4[0], pa4[1], pb4[1], b0.x, b0.y);
                mma_f16(acc[j][(2 * q + 1) % 4], pa4[2], pb4[2], pa4[3], pb4[3], b1.x, b1.y);
            }
        }
    }
}

// Shared-memory position, within a block of x', of value e of a lane that
// holds 8 consecutive columns starting at a multiple of 8: the lanes' MMA
// order of xpos is a fixed permutation of each run of eight.
template <int BITS>
__device__ __forceinline__ constexpr int xpos8(int e) {
    return BITS == 8 ? ((e >> 2) * 16 + (((e & 1) << 1) | ((e >> 1) & 1)))
                     : (((e >> 1) & 1) * 16 + ((e >> 2) | ((e & 1) << 1)));
}

// The last group of a row when K is not a multiple of 256 (width n = 32, 64
// or 128): its transform, scaled stores and sum of x', out of line so that
// the unrolled full-group code stays small (the kernel is otherwise bound by
// instruction fetch in its rotation phase).  Returns the warp's sum.
template <int BITS>
__device__ __noinline__ float sp_tail_group(uint4 r, int n, int gl, float up, uint16_t *row) {
    constexpr int KB = BITS == 8 ? 64 : 128;
    const int lane = threadIdx.x & 31;
    float v[8];
    const int E = fwht_group_raw(r, n, v);
    float ls = 0.0f;
    for (int e = 0; e < E; ++e) {
        const int kl = gl * kGroup + lane * E + e;
        const float xb = bf16_bits_to_f32(f32_to_bf16_bits(v[e]));
        const bool odd4 = BITS == 4 && (kl & 1);
        const __half h = __float2half_rn(xb * (odd4 ? up * 0.0625f : up));
        row[(kl / KB) * KB + xpos<BITS>(kl % KB)] = __half_as_ushort(h);
        ls += odd4 ? 16.0f * __half2float(h) : __half2float(h);
    }
    return warp_sum(ls);
}

template <int BITS, int NG>
__global__ void __launch_bounds__(SP_THREADS, 1)
k_gemv_splitk(const __grid_constant__ CUtensorMap tmW, const SplitParams p) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    // the stages on a 1024-byte boundary (the tensor copies' 128-byte swizzle)
    unsigned char *smem = smem_raw + ((1024 - (smem_addr(smem_raw) & 1023)) & 1023);
    constexpr int KB = BITS == 8 ? 64 : 128;          // k per block (64 bytes of a row)
    constexpr int KC = 2 * KB;                        // k per chunk (128 bytes of a row)
    constexpr int MT = 8 * NG;                        // token rows of x' (the MMAs' N)
    uint16_t *xs = reinterpret_cast<uint16_t *>(smem + SP_XOFF);
    unsigned int *pmx = reinterpret_cast<unsigned int *>(smem + SP_PAMOFF);   // pairs' largest |x| (bf16 bits)
    float *pss = reinterpret_cast<float *>(smem + SP_PAMOFF) + SP_PAMN / 2;   // pairs' sums of x'
    float *swv = reinterpret_cast<float *>(smem + SP_SWOFF);                  // the tile's row scales
    float *tok_f = reinterpret_cast<float *>(smem + SP_TOKOFF + 64);
    float *tok_s = reinterpret_cast<float *>(smem + SP_TOKOFF + 128);
    volatile int *abort_sh = reinterpret_cast<volatile int *>(smem + SP_ABOFF);
    const uint32_t full0 = smem_addr(smem + SP_BAROFF), empty0 = full0 + 8 * SP_R;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int C = p.C;
    const int crank = C > 1 ? static_cast<int>(cg::this_cluster().block_rank()) : 0;
    const int tile = static_cast<int>(blockIdx.x) / C;
    const int64_t n0 = static_cast<int64_t>(tile) * SP_RB;
    const int g0 = static_cast<int>(static_cast<int64_t>(p.G) * crank / C);
    const int g1 = static_cast<int>(static_cast<int64_t>(p.G) * (crank + 1) / C);
    const int ng = g1 - g0;
    const int64_t kc0 = static_cast<int64_t>(g0) * kGroup;
    const int64_t kc1 = min(static_cast<int64_t>(g1) * kGroup, p.K);
    // 128-byte chunks of the run; stage j holds chunks 2j and 2j + 1
    const int nch = static_cast<int>((kc1 - kc0 + KC - 1) / KC);
    const int nst = (nch + 1) / 2;
    const int XS = p.XS;

    if (threadIdx.x == 0) {
        for (int s = 0; s < SP_R; ++s) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(full0 + 8 * s));
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(empty0 + 8 * s), "r"(SP_CONS));
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        *abort_sh = 0;
    }
    // the tile's row scales (weights: not written by the launch before)
    if (threadIdx.x < SP_RB) swv[threadIdx.x] = n0 + threadIdx.x < p.N ? __ldg(p.sw + n0 + threadIdx.x) : 0.0f;
    __syncthreads();

    float acc[NG][4][4];
#pragma unroll
    for (int j = 0; j < NG; ++j)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[j][c][0] = acc[j][c][1] = acc[j][c][2] = acc[j][c][3] = 0.0f;
    const int g = lane >> 2, t = lane & 3;
    // fragment row g of the warp's 16 rows: the two rows a quarter-warp reads
    // are 4 apart, so their swizzled units fall in opposite halves of a line
    const int gr = (g >> 1) | ((g & 1) << 2);

    if (warp == SP_CONS) {
        // ------------------------------------------------ producer
        if (lane == 0) {
            int issued = 0;
            for (int it = 0; it < nst && !*abort_sh; ++it) {
                const int s = it % SP_R;
                if (it >= SP_R &&
                    !sp_wait(empty0 + 8 * s, static_cast<uint32_t>((it / SP_R - 1) & 1), abort_sh, p.status))
                    break;
                const uint32_t full = full0 + 8 * s;
                const int nc = min(2, nch - 2 * it);
                // A build for the library's own tests (TQ_TEST_UNSET_BYTES)
                // expects bytes that no copy brings, so no stage's phase
                // completes and the bounded waits expire, with every issued
                // copy landed; the drain below then runs to its full limit.
#ifdef TQ_TEST_UNSET_BYTES
                constexpr uint32_t kUnset = TQ_TEST_UNSET_BYTES;
#else
                constexpr uint32_t kUnset = 0;
#endif
                // a tensor copy counts its whole box, zero fill included
                asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(full),
                             "r"(static_cast<uint32_t>(nc * (SP_ST / 2)) + kUnset)
                             : "memory");
                for (int c = 0; c < nc; ++c) {
                    const int x = static_cast<int>((kc0 + static_cast<int64_t>(2 * it + c) * KC) * BITS / 8);
#pragma unroll
                    for (int h = 0; h < 2; ++h)
                        asm volatile(
                            "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
                            "[%0], [%1, {%2, %3}], [%4];"
                            ::"r"(smem_addr(smem + s * SP_ST + c * (SP_ST / 2) + h * (SP_ST / 4))),
                              "l"(reinterpret_cast<uint64_t>(&tmW)), "r"(x), "r"(static_cast<int>(n0) + 128 * h),
                              "r"(full)
                            : "memory");
                }
                ++issued;
            }
            // never leave with copies landing: the last use of every slot
            const long long t0 = clock64();
            for (int it = issued - SP_R > 0 ? issued - SP_R : 0; it < issued; ++it)
                while (!mbar_try_suspend(full0 + 8 * (it % SP_R), static_cast<uint32_t>((it / SP_R) & 1)) &&
                       clock64() - t0 < kA16DrainLimit) {
                }
        }
        __syncwarp();
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    } else {
        // ------------------------------------------------ consumers
        asm volatile("griddepcontrol.wait;" ::: "memory");     // X may come from the launch before
        const int pairs = p.M * ng;
        // x' rows start at zero: token rows past M and columns past K stay so
        {
            uint4 *z = reinterpret_cast<uint4 *>(xs);
            const int nz = MT * XS / 8;
            for (int i = threadIdx.x; i < nz; i += SP_CONS * 32) z[i] = make_uint4(0, 0, 0, 0);
        }
        // the warp's (token, group) pairs q = warp + 16 i: every load issued
        // first (one latency for all of them)
        uint4 raw[SP_PAIRS];
#pragma unroll
        for (int i = 0; i < SP_PAIRS; ++i) {
            const int q = warp + SP_CONS * i;
            raw[i] = make_uint4(0, 0, 0, 0);
            if (q < pairs) {
                const int m = q / ng, gl = q - m * ng;
                const int64_t gk = static_cast<int64_t>(g0 + gl) * kGroup;
                const int E = group_width(p.K, gk) / 32;
                raw[i] = load_group_raw(p.X + m * p.ldx + gk + lane * E, E);
            }
        }
        // each pair's largest |x| (bf16 magnitudes order as their bits)
#pragma unroll
        for (int i = 0; i < SP_PAIRS; ++i) {
            const int q = warp + SP_CONS * i;
            if (q >= pairs) break;
            const uint32_t w[4] = {raw[i].x, raw[i].y, raw[i].z, raw[i].w};
            uint32_t mx = 0;
#pragma unroll
            for (int k = 0; k < 4; ++k) mx = max(mx, max(w[k] & 0x7FFFu, (w[k] >> 16) & 0x7FFFu));
            mx = __reduce_max_sync(0xffffffffu, mx);
            if (lane == 0) pmx[q] = mx;
        }
        consumers_sync();
        // the transform, once: x' of a group is at most 16 times the group's
        // largest |x| (|H_n x|_inf <= sqrt(n) max|x|), so with e = 10 - E for
        // the run's largest |x| = f 2^E (1 <= f < 2) every x' 2^e lies below
        // 2^15 and keeps its bf16 value exactly in fp16 (down to 2^-28 of the
        // largest); for 4-bit weights the odd k hold a sixteenth of it
#pragma unroll
        for (int i = 0; i < SP_PAIRS; ++i) {
            const int q = warp + SP_CONS * i;
            if (q >= pairs) break;
            const int m = q / ng, gl = q - m * ng;
            uint32_t mx = 0;
            for (int g2 = 0; g2 < ng; ++g2) mx = max(mx, pmx[m * ng + g2]);
            const int ex = mx == 0 ? 0 : min(max(10 - (static_cast<int>((mx >> 7) & 0xFF) - 127), -100), 100);
            const float up = __uint_as_float(static_cast<uint32_t>(127 + ex) << 23);
            const int n = group_width(p.K, static_cast<int64_t>(g0 + gl) * kGroup);
            uint16_t *row = xs + m * XS;
            float ls;
            if (n == kGroup) {
                // a full group: eight consecutive columns a lane, at fixed
                // offsets from the first
                const uint32_t w[4] = {raw[i].x, raw[i].y, raw[i].z, raw[i].w};
                float v[8];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    v[2 * k] = __uint_as_float(w[k] << 16);
                    v[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
                }
                warp_fwht<8, float>(v);
                const int kl0 = gl * kGroup + lane * 8;
                uint16_t *base = row + (kl0 / KB) * KB + xpos<BITS>(kl0 % KB);
                ls = 0.0f;
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float xb = bf16_bits_to_f32(f32_to_bf16_bits(0.0625f * v[e]));   // exact: 1/sqrt(256)
                    const bool odd4 = BITS == 4 && (e & 1);
                    const __half h = __float2half_rn(xb * (odd4 ? up * 0.0625f : up));
                    base[xpos8<BITS>(e)] = __half_as_ushort(h);
                    ls += odd4 ? 16.0f * __half2float(h) : __half2float(h);
                }
                ls = warp_sum(ls);
            } else {
                ls = sp_tail_group<BITS>(raw[i], n, gl, up, row);
            }
            if (lane == 0) pss[q] = ls;
        }
        consumers_sync();

        // ---- the stream: rows 16 warp + (gr, gr + 8) of every stage
        const int rA = 16 * warp + gr, rB = rA + 8;
        const int sw7 = rA & 7;
        const int offE = (t ^ sw7) << 4, offO = ((4 | t) ^ sw7) << 4;
        const uint16_t *xb = xs + g * XS + 4 * t;
        for (int it = 0; it < nst; ++it) {
            const int s = it % SP_R;
            if (!sp_wait(full0 + 8 * s, static_cast<uint32_t>((it / SP_R) & 1), abort_sh, p.status)) break;
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                const int ch = 2 * it + c;
                if (ch >= nch) break;
                const unsigned char *st = smem + s * SP_ST + c * (SP_ST / 2);
                sp_block<BITS, NG>(acc, st + rA * 128 + offE, st + rB * 128 + offE, xb + (2 * ch) * KB, 8 * XS);
                sp_block<BITS, NG>(acc, st + rA * 128 + offO, st + rB * 128 + offO, xb + (2 * ch + 1) * KB, 8 * XS);
            }
            // the stage's shared reads end here; the next tensor copy into it
            // is ordered after them by the proxy fence and the release
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(empty0 + 8 * s) : "memory");
        }
        consumers_sync();          // every warp is done with the ring: partial sums over it
        if (warp < p.M) {
            // token `warp`: its sum of x' over the run and its factor 2^-e
            const int m = warp;
            float sum = 0.0f;
            uint32_t mx = 0;
            for (int g2 = lane; g2 < ng; g2 += 32) {
                sum += pss[m * ng + g2];
                mx = max(mx, pmx[m * ng + g2]);
            }
            sum = warp_sum(sum);
            mx = __reduce_max_sync(0xffffffffu, mx);
            const int ex = mx == 0 ? 0 : min(max(10 - (static_cast<int>((mx >> 7) & 0xFF) - 127), -100), 100);
            if (lane == 0) {
                tok_s[m] = sum;
                tok_f[m] = __uint_as_float(static_cast<uint32_t>(127 - ex) << 23);
            }
        }
        consumers_sync();
        if (!*abort_sh) {
            float *part = reinterpret_cast<float *>(smem);   // [token][256 rows]
            const float B = BITS == 8 ? 128.0f : 8.0f;
#pragma unroll
            for (int j = 0; j < NG; ++j) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int row = rA + 8 * h;
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        const int m = 8 * j + 2 * t + i;
                        if (m >= p.M) continue;
                        const float sacc = (acc[j][0][2 * h + i] + acc[j][1][2 * h + i]) +
                                           (acc[j][2][2 * h + i] + acc[j][3][2 * h + i]);
                        part[m * SP_RB + row] = fmaf(sacc, 16777216.0f, -B * tok_s[m]) * tok_f[m];
                    }
                }
            }
        }
    }

    // ---- sum over the cluster, scale, store
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");   // Y may still be read by the launch before
    // any CTA of the cluster that stopped: the cluster stores nothing
    int stopped = 0;
    for (int c = 0; c < C; ++c) {
        uint32_t ra;
        asm("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(smem_addr(smem + SP_ABOFF)), "r"(c));
        int v;
        asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(ra));
        stopped |= v;
    }
    if (!stopped) {
        // CTA c takes quads of rows [64 c / C, 64 (c + 1) / C): a thread adds
        // four rows of one token over the C CTAs in rank order, scales, stores
        const int q0 = (SP_RB / 4) * crank / C, q1 = (SP_RB / 4) * (crank + 1) / C;
        const int nq = q1 - q0;
        const bool y16 = p.ytype == 0 ? ((reinterpret_cast<uintptr_t>(p.Y) & 15) == 0 && (p.ldy & 3) == 0)
                                      : ((reinterpret_cast<uintptr_t>(p.Y) & 7) == 0 && (p.ldy & 3) == 0);
        const uint32_t part0 = smem_addr(smem);
        for (int idx = threadIdx.x; idx < nq * p.M; idx += SP_THREADS) {
            const int m = idx / nq, row = 4 * (q0 + idx % nq);
            const int64_t n = n0 + row;
            if (n >= p.N) continue;
            const uint32_t addr = part0 + static_cast<uint32_t>((m * SP_RB + row) * 4);
            float4 v[8];
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                if (c < C) {
                    uint32_t ra;
                    asm("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(addr), "r"(c));
                    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                                 : "=f"(v[c].x), "=f"(v[c].y), "=f"(v[c].z), "=f"(v[c].w) : "r"(ra));
                }
            }
            float4 sum = v[0];
#pragma unroll
            for (int c = 1; c < 8; ++c)
                if (c < C) {
                    sum.x += v[c].x;
                    sum.y += v[c].y;
                    sum.z += v[c].z;
                    sum.w += v[c].w;
                }
            const float s4[4] = {sum.x, sum.y, sum.z, sum.w};
            float y[4];
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) y[jj] = s4[jj] * swv[row + jj];
            if (p.ytype == 0) {
                float *yp = static_cast<float *>(p.Y) + m * p.ldy + n;
                if (y16 && n + 4 <= p.N) {
                    *reinterpret_cast<float4 *>(yp) = make_float4(y[0], y[1], y[2], y[3]);
                } else {
                    for (int jj = 0; jj < 4; ++jj)
                        if (n + jj < p.N) yp[jj] = y[jj];
                }
            } else {
                uint16_t *yp = static_cast<uint16_t *>(p.Y) + m * p.ldy + n;
                if (y16 && n + 4 <= p.N) {
                    *reinterpret_cast<uint2 *>(yp) =
                        make_uint2(f32_to_bf16_bits(y[0]) | (static_cast<uint32_t>(f32_to_bf16_bits(y[1])) << 16),
                                   f32_to_bf16_bits(y[2]) | (static_cast<uint32_t>(f32_to_bf16_bits(y[3])) << 16));
                } else {
                    for (int jj = 0; jj < 4; ++jj)
                        if (n + jj < p.N) yp[jj] = f32_to_bf16_bits(y[jj]);
                }
            }
        }
    }
    // nobody leaves while a peer may still read its shared memory
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Largest run of groups a CTA may hold: its x' rows (8 NG tokens of the run's
// columns and 16 more) fit SP_XBYTES.
int splitk_max_run(int NG) { return ((SP_XBYTES / (16 * NG)) - 16) / kGroup; }

struct SplitChoice {
    int C;
    int NG;
};

// clusters of C CTAs that can be resident at once, by (bits, NG, C), found
// once per device
int splitk_clusters(int bits, int NG, int C, const DeviceInfo &dev) {
    static int table[64][2][2][9] = {};
    static bool configured[64][2][2] = {};
    if (dev.id < 0 || dev.id >= 64) return 0;
    const int bi = bits == 8 ? 0 : 1, ni = NG == 1 ? 0 : 1;
    if (!configured[dev.id][bi][ni]) {
        const void *kern = bits == 8 ? (NG == 1 ? reinterpret_cast<const void *>(k_gemv_splitk<8, 1>)
                                                : reinterpret_cast<const void *>(k_gemv_splitk<8, 2>))
                                     : (NG == 1 ? reinterpret_cast<const void *>(k_gemv_splitk<4, 1>)
                                                : reinterpret_cast<const void *>(k_gemv_splitk<4, 2>));
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SP_SMEM) != cudaSuccess) return 0;
        for (int c = 1; c <= 8; ++c) {
            cudaLaunchConfig_t q = {};
            q.gridDim = dim3(static_cast<unsigned>(c), 1, 1);
            q.blockDim = dim3(SP_THREADS, 1, 1);
            q.dynamicSmemBytes = SP_SMEM;
            cudaLaunchAttribute qa[1];
            qa[0].id = cudaLaunchAttributeClusterDimension;
            qa[0].val.clusterDim.x = static_cast<unsigned>(c);
            qa[0].val.clusterDim.y = 1;
            qa[0].val.clusterDim.z = 1;
            q.attrs = qa;
            q.numAttrs = 1;
            int n = 0;
            if (cudaOccupancyMaxActiveClusters(&n, kern, &q) != cudaSuccess) n = 0;
            table[dev.id][bi][ni][c] = n;
        }
        configured[dev.id][bi][ni] = true;
    }
    return table[dev.id][bi][ni][C];
}

// The cluster size for a call, or C = 0 when the product does not take it:
// the most CTAs a cluster (at most 8, at least one group each) for which
// every cluster of the launch is resident at once and a CTA's run of groups
// fits its x' rows.
SplitChoice splitk_choice(int64_t M, int64_t N, int64_t K, int bits, const DeviceInfo &dev) {
    SplitChoice r{0, M <= 8 ? 1 : 2};
    if (M < 1 || M > 16 || N < 1 || K < 1 || (K * bits / 8) % 16 != 0) return r;
    if (N > (1ll << 31) - SP_RB || K * bits / 8 > (1ll << 31) - 256) return r;
    const int64_t G = (K + kGroup - 1) / kGroup;
    const int64_t tiles = (N + SP_RB - 1) / SP_RB;
    const int run = splitk_max_run(r.NG);
    for (int c = 8; c >= 1; --c) {
        if (G < c || (G + c - 1) / c > run || M * ((G + c - 1) / c) > SP_CONS * SP_PAIRS) continue;
        if (tiles <= splitk_clusters(bits, r.NG, c, dev)) {
            r.C = c;
            break;
        }
    }
    return r;
}

}  // namespace

// Which calls take the split-K product: up to 16 tokens over a matrix of at
// least 2^24 weights that fills the GPU in one wave of clusters.
bool splitk_fits(int64_t M, int64_t N, int64_t K, int bits, const DeviceInfo &dev) {
    if (M < 1 || M > 16 || N * K < (int64_t(1) << 24)) return false;
    return splitk_choice(M, N, K, bits, dev).C > 0;
}

tq_status launch_splitk(const uint16_t *X, int64_t M, int64_t K, int64_t ldx, const uint8_t *Wq, const float *sw,
                        int64_t N, int bits, void *Y, int ytype, int64_t ldy, const DeviceInfo &dev,
                        cudaStream_t s) {
    unsigned int *status = status_word();
    if (!status) return TQ_ERR_DEVICE;
    const SplitChoice ch = splitk_choice(M, N, K, bits, dev);
    if (ch.C == 0) return TQ_ERR_SHAPE;
    CUtensorMap tmW;
    if (!make_map_u8(&tmW, Wq, N, K * bits / 8, 128, 128, CU_TENSOR_MAP_SWIZZLE_128B)) return TQ_ERR_DEVICE;
    SplitParams p{};
    p.X = X;
    p.ldx = ldx;
    p.M = static_cast<int>(M);
    p.K = K;
    p.G = static_cast<int>((K + kGroup - 1) / kGroup);
    p.C = ch.C;
    // the longest run of a CTA, rounded to whole groups, and 16 more values
    const int run = (p.G + ch.C - 1) / ch.C;
    p.XS = run * kGroup + 16;

    p.sw = sw;
    p.N = N;
    p.Y = Y;
    p.ldy = ldy;
    p.ytype = ytype;
    p.status = status;
    const void *kern = bits == 8 ? (ch.NG == 1 ? reinterpret_cast<const void *>(k_gemv_splitk<8, 1>)
                                               : reinterpret_cast<const void *>(k_gemv_splitk<8, 2>))
                                 : (ch.NG == 1 ? reinterpret_cast<const void *>(k_gemv_splitk<4, 1>)
                                               : reinterpret_cast<const void *>(k_gemv_splitk<4, 2>));
    const int64_t tiles = (N + SP_RB - 1) / SP_RB;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(tiles * ch.C), 1, 1);
    cfg.blockDim = dim3(SP_THREADS, 1, 1);
    cfg.dynamicSmemBytes = SP_SMEM;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = static_cast<unsigned>(ch.C);
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    void *args[] = {&tmW, &p};
    const cudaError_t e = cudaLaunchKernelExC(&cfg, kern, args);
    return e == cudaSuccess ? TQ_OK : cuda_fail(e);
}

}  // namespace tq
