// Batched A16 product on the 5th-generation tensor cores, for M <= 64 token
// rows and weight matrices that fill the GPU:
//   Y[m][n] = sw[n] * sum_k q[n][k] * x'_bf16[m][k],  fp32 sums,
// x' the group-256 rotation of token row m rounded to bf16 (the A16 operand;
// tensai docs, "画像生成", section "幅とメモリ": the product's input gets the
// rotation of the weights).  Decode and small batches are bound by the weight
// stream (kvad-gpu internals, "Numbers"); at 64 tokens the fp32 FMA or legacy
// mma.sync work of the CUDA-core kernels exceeds the time the weights take to
// stream, so the multiply runs on tcgen05 instead, with the weights as the
// MMA's 128-row side and the tokens as its N side (16 to 64 columns).
//
// Two launches:
//   k_rotate_tiles16  one CTA per token row: rotates the row, rounds it to
//                     bf16 and stores x' * 2^e as fp16 in the tensor core's
//                     operand layout, one [Mp x 64] tile per K step (Mp = M
//                     rounded up to 16, pad rows zero).  2^e is a power of two
//                     chosen per token from the row's largest |x| so that
//                     16 max|x| 2^e < 2^15: every rotated value then fits fp16
//                     (|x'| <= 16 max|x| for a normalised 256-group), and the
//                     fp16 value is the bf16 x' times 2^e exactly (fp16 keeps
//                     every bf16 mantissa; only values below 2^-24 of the
//                     fp16 range, under 2^-28 of the row's largest, lose bits).
//                     fp16 lets an int8 code widen in 3 ALU operations per two
//                     codes instead of 5 for bf16.  The factor 2^-e goes to Y.
//   k_skinny_tc       a cluster of C CTAs (along K) per 256 weight rows.  Per
//                     CTA: a TMA warp streams the raw int8 / packed int4 codes
//                     of its 2 x 128 rows and its K slice into a raw ring, 128
//                     bytes of each row a copy (two K steps of int8 codes, four
//                     of int4: whole 128-byte lines, and 128 KB in flight); each
//                     of eight converter warps widens the codes of 32 rows to
//                     fp16 straight into tensor memory (TMEM lanes are rows,
//                     the MMA reads its A operand from there), so the widened
//                     weights never pass through shared memory;
//                     a bulk-copy warp brings the x' tile of each K step into
//                     a ring of its own, eight steps ahead (after the
//                     dependency wait: x' comes from the launch before);
//                     one thread a row block (two issuing warps) issues
//                     tcgen05.mma (M = 128, N = Mp, K = 16, A from TMEM).  The weights are read
//                     before the dependency wait, so the next call's weight
//                     stream starts in the shadow of this one (programmatic
//                     dependent launch).  At the end each CTA drains its fp32
//                     partial sums to shared memory, and after a cluster barrier
//                     CTA c adds a 1/C share of the rows over the C CTAs in a
//                     fixed order (distributed shared memory; the result does
//                     not depend on timing) and writes Y.
// Every wait is bounded: on expiry the kernel records it in the library
// status word, skips the rest, lets its copies and MMAs in flight finish
// (bounded), frees its TMEM and returns.

#include <cooperative_groups.h>

#include "tq_tc.cuh"

namespace cg = cooperative_groups;

namespace tq {
namespace {

constexpr int SK_RB = 2;                  // 128-row weight blocks per CTA
constexpr int SK_ROWS = 128 * SK_RB;      // weight rows per CTA
constexpr int SK_BK = 64;                 // K per step
constexpr int SK_MAXMP = 64;              // token columns of the MMA, at most
constexpr int SK_CONV = 8;                // converter warps 0..7: row block w / 4, TMEM lanes of quarter w % 4
constexpr int SK_W_TMA = 8, SK_W_X = 9, SK_W_MMA = 10;   // MMA issuers: warps 10 and 11, a row block each
constexpr int SK_THREADS = 12 * 32;
constexpr int SK_R = 4;                   // raw stages (128 bytes of every row each)
constexpr int SK_LINE = 128;              // raw bytes of a row per stage
constexpr int SK_XS = 8;                  // x' stages: its tiles come from L2, so
                                          // they are issued well ahead of the MMA
// TMEM: the accumulators of the two row blocks in columns [0, 2 Mp) (at most
// 128), then SK_AS stages of the widened weights, 64 columns each (32 fp16
// pairs of K a row and row block).  The converters take the K steps in order,
// so each waits only for its stage's previous use to be consumed.
constexpr int SK_AS = 6;
constexpr uint32_t SK_ACOL = 128;
constexpr uint32_t SK_TCOLS = 512;
constexpr int SK_B_ST = SK_MAXMP * SK_BK * 2;     // x' operand per stage (8 KB at most)
constexpr int SK_RAW_ST = SK_ROWS * SK_LINE;      // raw codes per stage (32 KB)
constexpr int SK_NBAR = 2 * SK_R + 2 * SK_AS + 2 * SK_XS + 2;   // mbarriers after the rings
constexpr int SK_BAR_BYTES = 512;
static_assert(SK_NBAR * 8 <= SK_BAR_BYTES, "mbarriers fit their reserved bytes");
static_assert(SK_W_MMA + SK_RB == SK_THREADS / 32, "one issuing warp per row block, the last warps");
constexpr int SK_SMEM = SK_XS * SK_B_ST + SK_R * SK_RAW_ST + SK_BAR_BYTES;
constexpr long long kSkWaitLimit = 4000000000ll;  // clock cycles, about 2 s
constexpr unsigned int kStatusSkinnyTimeout = 32u;

struct SkParams {
    const unsigned char *xt;   // x' tiles: K step ks at ks * Mp * 128 bytes
    const float *xf;           // per-token factors 2^-e [Mp]
    int M, Mp;
    int64_t K;
    int ksteps;
    int C;                     // CTAs of a cluster (split of K)
    const float *sw;
    int64_t N;
    void *Y;
    int64_t ldy;
    int ytype;                 // 0 fp32, 1 bf16
    unsigned int *status;
};

__device__ __forceinline__ bool sk_wait(uint32_t bar, uint32_t parity, volatile int *abort, unsigned int *status) {
    const long long t0 = clock64();
    while (!mbar_try(bar, parity)) {
        if (*abort) return false;
        if (clock64() - t0 > kSkWaitLimit) {
            *abort = 1;
            atomicOr(status, kStatusSkinnyTimeout);
            return false;
        }
    }
    return true;
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
          "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
          "=r"(v[14]), "=r"(v[15])
        : "r"(taddr));
}

template <int BITS>
__global__ void __launch_bounds__(SK_THREADS, 1)
k_skinny_tc(const __grid_constant__ CUtensorMap tmW, const SkParams p) {
    extern __shared__ __align__(1024) unsigned char smem[];
    unsigned char *raw = smem;                                        // [R][SK_RAW_ST]
    unsigned char *opB = smem + SK_R * SK_RAW_ST;                     // [XS][SK_B_ST]
    uint64_t *bars = reinterpret_cast<uint64_t *>(opB + SK_XS * SK_B_ST);
    // bars: raw_full[R], raw_empty[R], a_full[AS], a_empty[AS], x_full[XS],
    //       x_empty[XS], acc_full, done
    __shared__ uint32_t tmem_base_sh;
    __shared__ volatile int abort_sh;

    constexpr int RAWB = 128 * SK_LINE;               // raw bytes of one 128-row block (16 KB)
    constexpr int KSB = SK_BK * BITS / 8;             // bytes of a row per K step (64 or 32)
    constexpr int QK = SK_LINE / KSB;                 // K steps per raw stage (2 or 4)
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int C = p.C;
    const int crank = C > 1 ? static_cast<int>(cg::this_cluster().block_rank()) : 0;
    const int tile = static_cast<int>(blockIdx.x) / C;
    const int64_t n0 = static_cast<int64_t>(tile) * SK_ROWS;
    const int ks0 = static_cast<int>(static_cast<int64_t>(p.ksteps) * crank / C);
    const int ks1 = static_cast<int>(static_cast<int64_t>(p.ksteps) * (crank + 1) / C);
    const int nks = ks1 - ks0;
    const int nss = (nks + QK - 1) / QK;              // raw stages of this CTA
    const uint32_t raw_full0 = smem_u32(bars), raw_empty0 = raw_full0 + 8 * SK_R;
    const uint32_t a_full0 = raw_empty0 + 8 * SK_R, a_empty0 = a_full0 + 8 * SK_AS;
    const uint32_t x_full0 = a_empty0 + 8 * SK_AS, x_empty0 = x_full0 + 8 * SK_XS;
    const uint32_t acc_full = x_empty0 + 8 * SK_XS, done = acc_full + 8;
    const uint32_t b_bytes = static_cast<uint32_t>(p.Mp) * SK_BK * 2;
    // D f32, A/B f16, K-major; N = Mp, M = 128
    const uint32_t idesc = (1u << 4) | (static_cast<uint32_t>(p.Mp >> 3) << 17) | (static_cast<uint32_t>(128 >> 4) << 24);

    if (threadIdx.x == 0) {
        for (int s = 0; s < SK_R; ++s) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(raw_full0 + 8 * s));
            // every K step of a raw stage is converted by one group's warps
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(raw_empty0 + 8 * s), "r"(SK_CONV * QK));
        }
        for (int s = 0; s < SK_AS; ++s) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(a_full0 + 8 * s), "r"(SK_CONV));
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(a_empty0 + 8 * s), "r"(SK_RB));
        }
        for (int s = 0; s < SK_XS; ++s) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(x_full0 + 8 * s));
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(x_empty0 + 8 * s), "r"(SK_RB));
        }
        asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(acc_full), "r"(SK_RB));
        asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(done), "r"(SK_RB));
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        abort_sh = 0;
    }
    if (warp == SK_W_MMA) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(smem_u32(&tmem_base_sh)), "r"(SK_TCOLS));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = tmem_base_sh;

    if (warp == SK_W_TMA) {
        // ---------------------------------------------------- raw weight tiles
        if (lane == 0) {
            int issued = 0;
            for (int it = 0; it < nss && !abort_sh; ++it) {
                const int s = it % SK_R;
                if (!sk_wait(raw_empty0 + 8 * s, ((it / SK_R) & 1) ^ 1, &abort_sh, p.status)) break;
                asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                             ::"r"(raw_full0 + 8 * s), "r"(static_cast<uint32_t>(SK_RB * RAWB)) : "memory");
                // the line may run past this CTA's K slice (or past K: zeros);
                // only the slice's K steps are converted
                const int kx = ks0 * KSB + it * SK_LINE;
#pragma unroll
                for (int b = 0; b < SK_RB; ++b)
                    tma_load_2d(smem_u32(raw + s * SK_RAW_ST + b * RAWB), &tmW, kx,
                                static_cast<int>(n0) + 128 * b, raw_full0 + 8 * s);
                ++issued;
            }
            // never leave with copies landing: the last use of every slot
            const long long t0 = clock64();
            for (int it = issued - SK_R > 0 ? issued - SK_R : 0; it < issued; ++it)
                while (!mbar_try(raw_full0 + 8 * (it % SK_R), (it / SK_R) & 1) && clock64() - t0 < kSkWaitLimit) {
                }
        }
        __syncwarp();
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    } else if (warp == SK_W_X) {
        // ---------------------------------------------------- x' tiles (after the dependency wait)
        asm volatile("griddepcontrol.wait;" ::: "memory");
        if (lane == 0) {
            int issued = 0;
            for (int it = 0; it < nks && !abort_sh; ++it) {
                const int s = it % SK_XS;
                if (!sk_wait(x_empty0 + 8 * s, ((it / SK_XS) & 1) ^ 1, &abort_sh, p.status)) break;
                asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                             ::"r"(x_full0 + 8 * s), "r"(b_bytes) : "memory");
                asm volatile(
                    "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                    ::"r"(smem_u32(opB + s * SK_B_ST)),
                      "l"(p.xt + static_cast<int64_t>(ks0 + it) * b_bytes), "r"(b_bytes), "r"(x_full0 + 8 * s)
                    : "memory");
                ++issued;
            }
            const long long t0 = clock64();
            for (int it = issued - SK_XS > 0 ? issued - SK_XS : 0; it < issued; ++it)
                while (!mbar_try(x_full0 + 8 * (it % SK_XS), (it / SK_XS) & 1) && clock64() - t0 < kSkWaitLimit) {
                }
        }
        __syncwarp();
    } else if (warp < SK_CONV) {
        // ---------------------------------------------------- converters
        // warp w widens rows 32 (w % 4) .. + 31 of row block w / 4; a thread
        // owns one row (its TMEM lane) and writes the row's 64 fp16 values of
        // a K step as 32 columns (pair k = 2j, 2j + 1 in column j, low half
        // first).  Reading the raw line of 32 consecutive rows at one chunk
        // hits every bank once per 8 rows (the 128-byte swizzle).
        const int rb = warp >> 2, q = warp & 3;
        const int r = q * 32 + lane;
        const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
        for (int it = 0; it < nks && !abort_sh; ++it) {
            const int ss = it / QK, rs = ss % SK_R, as = it % SK_AS;
            const int c0 = (it % QK) * (KSB / 16);    // first 16-byte chunk of this K step in a line
            if (!sk_wait(a_empty0 + 8 * as, ((it / SK_AS) & 1) ^ 1, &abort_sh, p.status)) break;
            if (!sk_wait(raw_full0 + 8 * rs, (ss / SK_R) & 1, &abort_sh, p.status)) break;
            const unsigned char *line = raw + rs * SK_RAW_ST + rb * RAWB;
            uint32_t v[32];
            if constexpr (BITS == 8) {
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const uint4 w = *reinterpret_cast<const uint4 *>(line + swz128(r, c0 + c));
                    widen8(w.x, v[8 * c + 0], v[8 * c + 1]);
                    widen8(w.y, v[8 * c + 2], v[8 * c + 3]);
                    widen8(w.z, v[8 * c + 4], v[8 * c + 5]);
                    widen8(w.w, v[8 * c + 6], v[8 * c + 7]);
                }
            } else {
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    const uint4 w = *reinterpret_cast<const uint4 *>(line + swz128(r, c0 + c));
                    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        uint32_t pr[4];
                        widen4(ww[i], pr);
                        v[16 * c + 4 * i + 0] = pr[0];
                        v[16 * c + 4 * i + 1] = pr[1];
                        v[16 * c + 4 * i + 2] = pr[2];
                        v[16 * c + 4 * i + 3] = pr[3];
                    }
                }
            }
            tmem_st32(tmem + lane_base + SK_ACOL + static_cast<uint32_t>(as * 64 + rb * 32), v);
            asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
            __syncwarp();
            if (lane == 0) {
                asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(a_full0 + 8 * as) : "memory");
                asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(raw_empty0 + 8 * rs) : "memory");
            }
        }
    } else if (warp >= SK_W_MMA && warp < SK_W_MMA + SK_RB) {
        // ---------------------------------------------------- MMA issue (one thread a
        // row block: each issuer commits to the stage, accumulator and done
        // barriers, which count SK_RB arrivals; measured 7-8% faster than one
        // thread issuing both row blocks)
        const int rb = warp - SK_W_MMA;
        if (lane == 0) {
            bool issued = false;
            for (int it = 0; it < nks && !abort_sh; ++it) {
                const int as = it % SK_AS, xs = it % SK_XS;
                if (!sk_wait(a_full0 + 8 * as, (it / SK_AS) & 1, &abort_sh, p.status)) break;
                if (!sk_wait(x_full0 + 8 * xs, (it / SK_XS) & 1, &abort_sh, p.status)) break;
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                const uint32_t b = smem_u32(opB + xs * SK_B_ST);
                {
#pragma unroll
                    for (int kk = 0; kk < SK_BK / 16; ++kk) {
                        // A: 128 lanes x 8 columns (16 fp16 of K a row) in TMEM
                        const uint32_t at = tmem + SK_ACOL + static_cast<uint32_t>(as * 64 + rb * 32 + kk * 8);
                        const uint64_t bd = smem_desc(b + kk * 256);
                        const uint32_t accum = (it > 0 || kk > 0) ? 1u : 0u;
                        asm volatile(
                            "{\n.reg .pred q;\nsetp.ne.b32 q, %4, 0;\n"
                            "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, q;\n}\n"
                            ::"r"(tmem + static_cast<uint32_t>(rb * p.Mp)), "r"(at), "l"(bd), "r"(idesc), "r"(accum));
                    }
                }
                issued = true;
                asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                             ::"r"(a_empty0 + 8 * as) : "memory");
                asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                             ::"r"(x_empty0 + 8 * xs) : "memory");
            }
            if (!abort_sh && issued)
                asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                             ::"r"(acc_full) : "memory");
            // every issued MMA finishes before the TMEM is released
            if (issued) {
                asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                             ::"r"(done) : "memory");
                const long long t0 = clock64();
                while (!mbar_try(done, 0) && clock64() - t0 < kSkWaitLimit) {
                }
            }
        }
        __syncwarp();
    }

    // ---------------------------------------------------- drain to shared memory
    // warps 4..7 (TMEM lane quarter warp % 4): fp32 partial sums of this CTA's
    // rows, token-major: part[m][row], row < 256, over the raw ring (every
    // stage has been converted by then)
    float *part = reinterpret_cast<float *>(smem);
    const bool have = nks > 0;
    if (warp >= 4 && warp < 8) {
        const int q = warp & 3;
        bool ok = !have;
        if (have) ok = sk_wait(acc_full, 0, &abort_sh, p.status);
        if (ok && have) {
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
#pragma unroll
            for (int rb = 0; rb < SK_RB; ++rb) {
                const int row = rb * 128 + q * 32 + lane;
                for (int c0 = 0; c0 < p.Mp; c0 += 16) {
                    uint32_t v[16];
                    tmem_ld16(tmem + lane_base + static_cast<uint32_t>(rb * p.Mp + c0), v);
                    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
                    for (int j = 0; j < 16; ++j) part[(c0 + j) * SK_ROWS + row] = __uint_as_float(v[j]);
                }
            }
        } else if (!have) {
            for (int rb = 0; rb < SK_RB; ++rb)
                for (int m = 0; m < p.Mp; ++m) part[m * SK_ROWS + rb * 128 + q * 32 + lane] = 0.0f;
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    // every CTA's partials in place (and every CTA still resident)
    if (C > 1) {
        asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
        asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
    } else {
        __syncthreads();
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");   // x' factors: from the launch before

    // ---------------------------------------------------- sum over the cluster, scale, store
    // CTA c of the cluster takes quads of rows [64 c / C, 64 (c + 1) / C): a
    // thread adds four rows of one token over the C CTAs in rank order (16-byte
    // loads of distributed shared memory, issued together), scales and stores.
    if (!abort_sh) {
        const int q0 = (SK_ROWS / 4) * crank / C, q1 = (SK_ROWS / 4) * (crank + 1) / C;
        const int nq = q1 - q0;
        const bool y16 = p.ytype == 0 ? ((reinterpret_cast<uintptr_t>(p.Y) & 15) == 0 && (p.ldy & 3) == 0)
                                      : ((reinterpret_cast<uintptr_t>(p.Y) & 7) == 0 && (p.ldy & 3) == 0);
        for (int idx = threadIdx.x; idx < nq * p.M; idx += SK_THREADS) {
            const int m = idx / nq, row = 4 * (q0 + idx % nq);
            const int64_t n = n0 + row;
            if (n >= p.N) continue;
            const uint32_t addr = smem_u32(part + m * SK_ROWS + row);
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
                    sum.x += v[c].x; sum.y += v[c].y; sum.z += v[c].z; sum.w += v[c].w;
                }
            const float f = p.xf[m];
            float y[4] = {sum.x * f, sum.y * f, sum.z * f, sum.w * f};
#pragma unroll
            for (int j = 0; j < 4; ++j) y[j] *= n + j < p.N ? __ldg(p.sw + n + j) : 0.0f;
            if (p.ytype == 0) {
                float *yp = static_cast<float *>(p.Y) + m * p.ldy + n;
                if (y16 && n + 4 <= p.N) {
                    *reinterpret_cast<float4 *>(yp) = make_float4(y[0], y[1], y[2], y[3]);
                } else {
                    for (int j = 0; j < 4; ++j)
                        if (n + j < p.N) yp[j] = y[j];
                }
            } else {
                uint16_t *yp = static_cast<uint16_t *>(p.Y) + m * p.ldy + n;
                if (y16 && n + 4 <= p.N) {
                    *reinterpret_cast<uint2 *>(yp) =
                        make_uint2(f32_to_bf16_bits(y[0]) | (static_cast<uint32_t>(f32_to_bf16_bits(y[1])) << 16),
                                   f32_to_bf16_bits(y[2]) | (static_cast<uint32_t>(f32_to_bf16_bits(y[3])) << 16));
                } else {
                    for (int j = 0; j < 4; ++j)
                        if (n + j < p.N) yp[j] = f32_to_bf16_bits(y[j]);
                }
            }
        }
    }
    // nobody leaves while a peer may still read its shared memory
    if (C > 1) {
        asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
        asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
    }
    if (warp == SK_W_MMA) {
        __syncwarp();
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(SK_TCOLS));
    }
}

// x' of token row m (CTA m < Mp; rows m >= M are zero): rotate each group,
// round to bf16, times 2^e, fp16 into the tile of its K step.  Warp w takes
// groups w, w + 8, ...  All the row's loads are issued first; the largest |x|
// of the row (one CTA barrier) fixes e.
constexpr int RT_GPW = 8;   // groups a warp holds (rows of up to 64 groups)

__global__ void __launch_bounds__(256)
k_rotate_tiles16(const uint16_t *__restrict__ X, int M, int64_t K, int64_t ldx, unsigned char *__restrict__ xt,
                 float *__restrict__ xf, int Mp) {
    __shared__ uint32_t red[8];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m = blockIdx.x;
    const int64_t G = (K + kGroup - 1) / kGroup;
    const int64_t ks_bytes = static_cast<int64_t>(Mp) * SK_BK * 2;   // one K step's tile
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");   // X may come from the launch before
    uint4 rawv[RT_GPW];
    uint32_t mx = 0;
#pragma unroll
    for (int j = 0; j < RT_GPW; ++j) {
        rawv[j] = make_uint4(0, 0, 0, 0);
        const int64_t g = warp + static_cast<int64_t>(j) * 8;
        if (m < M && g < G) {
            const int64_t gk = g * kGroup;
            const int E = group_width(K, gk) / 32;
            rawv[j] = load_group_raw(X + static_cast<int64_t>(m) * ldx + gk + lane * E, E);
            const uint32_t w[4] = {rawv[j].x, rawv[j].y, rawv[j].z, rawv[j].w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                mx = max(mx, w[i] & 0x7FFFu);
                mx = max(mx, (w[i] >> 16) & 0x7FFFu);
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (lane == 0) red[warp] = mx;
    __syncthreads();
    mx = red[0];
#pragma unroll
    for (int w = 1; w < 8; ++w) mx = max(mx, red[w]);
    // largest |x| = 2^E * f (1 <= f < 2, bf16 bits mx); 16 max|x| 2^e < 2^(E + 5 + e) <= 2^15
    const int E = static_cast<int>((mx >> 7) & 0xFF) - 127;
    const int e = mx == 0 ? 0 : min(max(10 - E, -100), 100);
    const float scale = __uint_as_float(static_cast<uint32_t>(127 + e) << 23);
    if (threadIdx.x == 0) xf[m] = m < M ? __uint_as_float(static_cast<uint32_t>(127 - e) << 23) : 0.0f;
    const int rr = m;   // token row inside the tile
#pragma unroll
    for (int j = 0; j < RT_GPW; ++j) {
        const int64_t g = warp + static_cast<int64_t>(j) * 8;
        if (g >= G) continue;
        const int64_t gk = g * kGroup;
        const int n = group_width(K, gk);
        float v[8] = {};
        int E8 = n / 32;
        if (m < M) E8 = fwht_group_raw(rawv[j], n, v);
        // 8 values a lane at columns gk + lane * E8 ..: bf16, times 2^e, fp16
        uint32_t h[4] = {0u, 0u, 0u, 0u};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float a = bf16_bits_to_f32(f32_to_bf16_bits(v[2 * i])) * scale;
            const float b = bf16_bits_to_f32(f32_to_bf16_bits(v[2 * i + 1])) * scale;
            const __half2 p2 = __floats2half2_rn(a, b);
            h[i] = *reinterpret_cast<const uint32_t *>(&p2);
        }
        const int64_t k0 = gk + static_cast<int64_t>(lane) * E8;
        unsigned char *tile = xt + (k0 >> 6) * ks_bytes;
        const int kk = static_cast<int>(k0 & 63);
        unsigned char *dst = tile + (((rr >> 3) << 3) + (kk >> 3)) * 128 + (rr & 7) * 16 + (kk & 7) * 2;
        if (E8 == 8) {
            *reinterpret_cast<uint4 *>(dst) = make_uint4(h[0], h[1], h[2], h[3]);
        } else if (E8 == 4) {
            *reinterpret_cast<uint2 *>(dst) = make_uint2(h[0], h[1]);
        } else if (E8 == 2) {
            *reinterpret_cast<uint32_t *>(dst) = h[0];
        } else {
            *reinterpret_cast<uint16_t *>(dst) = static_cast<uint16_t>(h[0]);
            // K % 64 == 32: the last tile's columns 32 .. 63 are zero
            if ((K & 63) == 32) {
                const int kz = kk + 32;
                *reinterpret_cast<uint16_t *>(tile + (((rr >> 3) << 3) + (kz >> 3)) * 128 + (rr & 7) * 16 +
                                              (kz & 7) * 2) = 0;
            }
        }
    }
}

}  // namespace

// Workspace of the tensor-core A16 product: x' tiles, then the token factors.
int64_t skinny_tc_mp(int64_t M) { return (M + 15) / 16 * 16; }

int64_t skinny_tc_workspace(int64_t M, int64_t K) {
    const int64_t ks = (K + SK_BK - 1) / SK_BK;
    return (ks * skinny_tc_mp(M) * SK_BK * 2 + 255) / 256 * 256 + 256;
}

// Which A16 kernel a call takes when the split-K product (k_gemv_splitk.cu,
// up to 16 tokens over a matrix that fills the GPU in one wave of clusters:
// 10.9 / 11.5 us a call at one token, 15.0 / 15.6 at eight) does not,
// measured with 4-bit weights of 12288 x 4096 and 4096 x 12288, calls back
// to back (us a call):
//   tokens   tensor cores   streaming (a row a warp)   small kernel
//   1        27.4 / 30.5    13.4 / 20.5                24.5 / 19.8
//   2        25.4 / 30.5    20.0 / 26.2                34.9 / 27.5
//   3, 4     25.3 / 28.1    -                          27.0 / 35.5, 32.6 / 43.7
// So one token over a matrix of at least 2^24 weights streams when N >= K
// (the staged rotated row is short next to a CTA's rows), two tokens always;
// from three tokens on the tensor cores take it.  Below 2^24 weights the
// small kernel keeps M <= 8 (its weight copies start before the previous
// launch ends, which is what short decode calls need).
bool a16_streams(int64_t M, int64_t N, int64_t K, int bits) {
    if (M < 1 || M > 2 || N * K < (int64_t(1) << 24) || (K * bits / 8) % 16 != 0) return false;
    return M == 2 || N >= K;
}

bool skinny_tc_applies(int64_t M, int64_t N, int64_t K) {
    if (M < 1 || M > SK_MAXMP || K > TQ_MAX_K_TILED) return false;
    if (M > 8) return true;
    return M >= 3 && N * K >= (int64_t(1) << 24);
}

// One wave of CTAs (at most a tile of 256 rows per SM): a later wave could
// find its SMs taken by the next call's CTAs, launched early and waiting for
// this call to end.
bool skinny_tc_fits_device(int64_t N, const DeviceInfo &dev) {
    return (N + SK_ROWS - 1) / SK_ROWS <= dev.sms;
}

tq_status launch_skinny_tc(const uint16_t *X, int64_t M, int64_t K, int64_t ldx, const uint8_t *Wq,
                           const float *sw, int64_t N, int bits, void *Y, int ytype, int64_t ldy, void *ws,
                           const DeviceInfo &dev, cudaStream_t s) {
    unsigned int *status = status_word();
    if (!status) return TQ_ERR_DEVICE;
    if (N > (1ll << 31) - SK_ROWS) return TQ_ERR_OVERFLOW;
    const int Mp = static_cast<int>(skinny_tc_mp(M));
    const int ksteps = static_cast<int>((K + SK_BK - 1) / SK_BK);
    unsigned char *xt = static_cast<unsigned char *>(ws);
    float *xf = reinterpret_cast<float *>(xt + (static_cast<int64_t>(ksteps) * Mp * SK_BK * 2 + 255) / 256 * 256);
    // K steps past K: their x' columns must be zero (the pre-pass writes only
    // real columns, and those of a half tile)
    {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(Mp), 1, 1);
        cfg.blockDim = dim3(256, 1, 1);
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        const cudaError_t e = cudaLaunchKernelEx(&cfg, k_rotate_tiles16, X, static_cast<int>(M), K, ldx, xt, xf, Mp);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    CUtensorMap tmW;
    const bool mapped = make_map_u8(&tmW, Wq, N, bits == 8 ? K : K / 2, SK_LINE, 128, CU_TENSOR_MAP_SWIZZLE_128B);
    if (!mapped) return TQ_ERR_DEVICE;
    SkParams p{};
    p.xt = xt;
    p.xf = xf;
    p.M = static_cast<int>(M);
    p.Mp = Mp;
    p.K = K;
    p.ksteps = ksteps;
    p.sw = sw;
    p.N = N;
    p.Y = Y;
    p.ldy = ldy;
    p.ytype = ytype;
    p.status = status;
    auto kern = bits == 8 ? k_skinny_tc<8> : k_skinny_tc<4>;
    const int bi = bits == 8 ? 0 : 1;
    // clusters of C CTAs that can be resident at once, by C (1 .. 8), found
    // once per device: the SMs of a cluster must share a GPC, so not every SM
    // can take part in a cluster of C
    static bool configured_for[64][2] = {{false}};
    static int max_clusters[64][2][9] = {};
    if (dev.id < 0 || dev.id >= 64) return TQ_ERR_DEVICE;
    if (!configured_for[dev.id][bi]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SK_SMEM);
        if (e != cudaSuccess) return cuda_fail(e);
        for (int c = 1; c <= 8; ++c) {
            cudaLaunchConfig_t q = {};
            q.gridDim = dim3(static_cast<unsigned>(c), 1, 1);
            q.blockDim = dim3(SK_THREADS, 1, 1);
            q.dynamicSmemBytes = SK_SMEM;
            cudaLaunchAttribute qa[1];
            qa[0].id = cudaLaunchAttributeClusterDimension;
            qa[0].val.clusterDim.x = static_cast<unsigned>(c);
            qa[0].val.clusterDim.y = 1;
            qa[0].val.clusterDim.z = 1;
            q.attrs = qa;
            q.numAttrs = 1;
            int n = 0;
            e = cudaOccupancyMaxActiveClusters(&n, kern, &q);
            if (e != cudaSuccess) return cuda_fail(e);
            max_clusters[dev.id][bi][c] = n;
        }
        configured_for[dev.id][bi] = true;
    }
    // clusters along K: the most CTAs a cluster (at most 8, at least two K
    // steps a CTA) for which every cluster of the launch is resident at once
    const int64_t tiles = (N + SK_ROWS - 1) / SK_ROWS;
    int C = 1;
    for (int c = 8; c >= 1; --c) {
        if (c > 1 && ksteps / c < 2) continue;
        if (tiles <= max_clusters[dev.id][bi][c]) {
            C = c;
            break;
        }
    }
    p.C = C;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(tiles * C), 1, 1);
    cfg.blockDim = dim3(SK_THREADS, 1, 1);
    cfg.dynamicSmemBytes = SK_SMEM;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    int na = 0;
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = static_cast<unsigned>(C);
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
    cfg.attrs = attr;
    cfg.numAttrs = na;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, tmW, p);
    return e == cudaSuccess ? TQ_OK : cuda_fail(e);
}

}  // namespace tq
