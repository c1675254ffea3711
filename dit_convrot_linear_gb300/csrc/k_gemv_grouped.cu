// Grouped A16 product: many independent decode calls in one persistent pass,
//   Y_c[m][n] = sw_c[n] * sum_k q_c[n][k] * x'_c,bf16[m][k],  fp32 sums,
// x'_c the group-256 Hadamard rotation of call c's token rows rounded to bf16
// (tensai docs, "画像生成" / Image generation, section "幅とメモリ": the input of
// the product gets the same rotation as the weights).  Decode is bound by the
// weight stream (kvad-gpu internals, "Numbers"), but one call of a small model
// moves only a few MB: launched one by one, each call waits for the previous
// one to finish before it may read its input, and that chain of latencies,
// not the weight stream, sets the time.  Calls that do not depend on one
// another (gate and up of a layer, or the independent calls of a batch) can
// instead share one weight stream:
//   1. k_rotate_grouped rotates every call's token rows once (a CTA per
//      call), into a workspace of the plan, in the lane-contiguous x' order
//      of the MMAs.
//   2. k_gemv_grouped runs one CTA per SM.  Work items are (call, block of
//      weight rows, all of K), dealt round-robin, so the SMs sweep through the
//      calls together and a weight matrix is never read by two SMs at once.
//      A producer warp bulk-copies each item's weight rows and x' into two
//      96 KB shared-memory stages and stays an item ahead (two large items
//      amortise each item's fixed cost better than three smaller ones: 0.89
//      against 0.75 of the HBM copy rate on 1000 decode calls); sixteen
//      consumer warps multiply (each code plus its bias widened into an
//      exact fp16 subnormal in registers against the scaled fp16 x',
//      mma.sync m16n8k16, fp32), add the K blocks in a fixed order, take off
//      the bias times the token's sum of x' and store Y.  The stream never
//      waits for a call to finish.
// A chained plan runs calls that do depend on one another, in order, the way
// a decoder walks its layers: call c may read the output of any earlier call
// (kvad-gpu internals, "Numbers": one projection at a time, each input the
// previous output).  The same persistent kernel (a cooperative launch: every
// CTA resident) keeps streaming weights ahead, so call c's rows are in shared
// memory before call c - 1 ends; the consumers of a CTA's first item of call
// c wait until every item of call c - 1 has counted itself done (a counter per
// call in device memory), then rotate the call's input themselves (optionally
// the SwiGLU of two rows, as a gated FFN's down projection takes it) and
// multiply.  There is no launch and no rotation pre-pass between calls.
// Every wait is bounded: on expiry the status word is set, the CTA stops, and
// the outputs of the items it had not finished are left unwritten.

#include <cuda_fp16.h>

#include <new>
#include <vector>

#include "tq_a16.cuh"

namespace tq {
namespace {

// One work item, as the producer reads it and copies it into the stage header.
// Its weight rows reach shared memory in one of two forms:
//   rows:  one bulk copy per row, rows ws bytes apart (ws = 64 mod 128, so the
//          lanes of a quarter-warp read distinct banks);
//   tiles: one tensor copy per 128-byte column chunk of all rows (few copies
//          for short rows: a bulk copy has a fixed cost of tens of cycles),
//          chunk c at c * rb * 128, each 128-byte row line stored with the
//          128-byte swizzle (16-byte unit j of row r at unit j ^ (r & 7)).
struct GItem {
    const uint8_t *w;      // rows: first weight row of the item
    const void *tmap;      // tiles: the call's tensor map (rows x row bytes)
    const uint16_t *xq;    // the call's x' rows (bf16, M rows of xk)
    const float *sw;       // row scale of the first row
    void *y;               // Y of the first row, token 0
    int64_t ldy;           // Y row stride (elements)
    int32_t rows;          // valid weight rows
    int32_t rb;            // rows the stage holds (multiple of 8)
    int32_t rbytes;        // bytes of one weight row
    int32_t ws;            // rows: shared row stride (bytes)
    int32_t xk;            // x' row length: K rounded up to whole blocks
    int32_t n0;            // tiles: first row of the item in the call
    int32_t xoff;          // byte offset of x' in the stage
    int16_t M;             // token rows
    int16_t tiles;         // 1: tile form
    int32_t call;          // chained plans: index of the item's call
    uint32_t wait;         // chained plans: items of the previous call (0: none)
    // Set by the host so that the consumers divide by none of the item's
    // sizes (an integer division is about twenty instructions a thread):
    uint32_t nbm;          // ceil(2^20 / NB), NB = xk / (k per block): u / NB = (u nbm) >> 20
    uint32_t rowm;         // ceil(2^20 / rows): j / rows = (j rowm) >> 20 for j < rows M
    uint8_t wf[10], wl[10];  // per 16-row tile: the first and last consumer warp whose units touch it
    uint8_t pad[12];
};
static_assert(sizeof(GItem) == 128, "item record of 128 bytes, one stage header");

// The fields of an item its producer needs to issue the copies (the whole
// record reaches the stage header by a bulk copy of its own).
struct GIssue {
    const uint8_t *w;
    const void *tmap;
    const uint16_t *xq;
    int32_t rows, rb, rbytes, ws, xk, n0, xoff, M, tiles;
};

__device__ __forceinline__ GIssue issue_of(const GItem *ip) {
    GIssue r;
    r.w = ip->w;
    r.tmap = ip->tmap;
    r.xq = ip->xq;
    r.rows = ip->rows;
    r.rb = ip->rb;
    r.rbytes = ip->rbytes;
    r.ws = ip->ws;
    r.xk = ip->xk;
    r.n0 = ip->n0;
    r.xoff = ip->xoff;
    r.M = ip->M;
    r.tiles = ip->tiles;
    return r;
}

struct GCall {
    const uint16_t *X;
    int64_t ldx;
    uint16_t *xq;
    int32_t M, K, xk, pad;
};

// A build for the library's own tests (TQ_TEST_CHAIN_WAIT_EXTRA) waits for
// that many items more than the previous call of a chained plan has, so the
// wait between calls cannot end and its bounded expiry is taken.
#ifdef TQ_TEST_CHAIN_WAIT_EXTRA
constexpr unsigned int kChainWaitExtra = TQ_TEST_CHAIN_WAIT_EXTRA;
#else
constexpr unsigned int kChainWaitExtra = 0;
#endif

constexpr int kGStages = 2;
constexpr int kGStageBytes = 96 * 1024;
constexpr int kGConsWarps = 16;
constexpr int kGThreads = (kGConsWarps + 1) * 32;     // + the producer warp
// Rows x tokens of one item at most (the partial sums' area): independent
// plans take 160 (a 96 KB stage holds 160 rows of 896 4-bit codes); chained
// plans 128, which leaves their own x' buffer room.
constexpr int kGRedInd = 160, kGRedChain = 128;
constexpr int kGRed = kGRedChain;                      // the chained plans' layout below
static_assert(kGRedInd / 16 <= 10 && kGRedChain / 16 <= 10, "an item's tiles fit the record's warp ranges");
constexpr int kGRedOff = kGStages * kGStageBytes;
constexpr int kGHdrOff = kGRedOff + 2 * kGConsWarps * kGRed * 4;
constexpr int kGBarOff = kGHdrOff + kGStages * 128;
// independent plans: the same layout with the larger partial-sum area
constexpr int kGHdrOffInd = kGRedOff + 2 * kGConsWarps * kGRedInd * 4;
constexpr int kGBarOffInd = kGHdrOffInd + kGStages * 128;
constexpr int kGSmem = kGBarOffInd + 2 * kGStages * 8 + 16 + 1024;   // + alignment of the stages
static_assert(kGSmem <= 232448, "within the opt-in shared memory of a CTA");
constexpr unsigned int kStatusGroupedTimeout = 16u;
// bytes after a call's x' rows: a float 2^-e per token, then the token's sum
// of x' (the fp16 values as the product multiplies them)
constexpr int kXTail = 64;

// One call of a chained plan, as its consumers read it.
struct CCall {
    const uint16_t *X;
    const uint16_t *U;     // NULL, or the up rows: the input is bf16(silu(X) * U)
    int64_t ldx, ldu;
    int32_t M, K, xk, pad;
};

// Chained plans: the consumers build each call's x' in shared memory of
// their own, after the stages (no x' travels with the items).  It is the
// bf16 operand itself (the rotated rows rounded to bf16, in the lanes' MMA
// order): no scaling into fp16, so no pass over the row for its largest value.
constexpr int kCPairs = 3;                                 // (token, group) pairs a warp rotates
constexpr int kCXOff = kGBarOff + 2 * kGStages * 8 + 16;
constexpr int kCXBytes = 17984;                            // x' rows
constexpr int kCSmem = kCXOff + kCXBytes + 1024;
static_assert(kCXOff % 16 == 0, "x' rows 16-byte aligned");
static_assert(kCSmem <= 232448, "within the opt-in shared memory of a CTA");

struct GroupedParams {
    const GItem *items;
    int64_t nitems;
    int ytype;
    unsigned int *status;
    const CCall *chain;    // chained plans: the calls
    unsigned int *done;    // chained plans: finished items per call (zero at launch)
};

// Barrier 1 among the consumer threads, returning whether any of them
// passed `pred`: every consumer reaches it on every item, so the decision to
// stop is the same in all of them.
__device__ __forceinline__ bool consumers_sync_any(bool pred) {
    uint32_t r;
    asm volatile(
        "{\n.reg .pred p, q;\nsetp.ne.u32 p, %1, 0;\n"
        "bar.red.or.pred q, 1, %2, p;\nselp.u32 %0, 1, 0, q;\n}\n"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(pred)), "r"(kGConsWarps * 32)
        : "memory");
    return r != 0;
}

// Barrier 2 among the consumer threads (chained plans).
__device__ __forceinline__ void chain_sync() {
    asm volatile("bar.sync 2, %0;" ::"r"(kGConsWarps * 32) : "memory");
}

// Chained plans: wait until *done reaches `target` (every item of the
// previous call has stored its outputs), for at most kA16WaitLimit cycles.
// The acquire load orders this thread's later reads after the count; the
// consumer barrier that follows orders the other threads' reads after it.
__device__ __forceinline__ bool chain_wait(const unsigned int *done, unsigned int target) {
    const long long t0 = clock64();
    while (true) {
        unsigned int v;
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(done) : "memory");
        if (v >= target) return true;
        if (clock64() - t0 > kA16WaitLimit) return false;
        __nanosleep(32);
    }
}

// A lane's E bf16 values of a group through L2 (ld.global.cg): rows that
// other CTAs wrote during this launch are never read through the
// non-coherent path or a stale L1 line.
__device__ __forceinline__ uint4 load_group_raw_cg(const uint16_t *p, int E) {
    if (E == 8) return __ldcg(reinterpret_cast<const uint4 *>(p));
    if (E == 4) {
        const uint2 u = __ldcg(reinterpret_cast<const uint2 *>(p));
        return make_uint4(u.x, u.y, 0, 0);
    }
    if (E == 2) return make_uint4(__ldcg(reinterpret_cast<const unsigned int *>(p)), 0, 0, 0);
    return make_uint4(__ldcg(reinterpret_cast<const unsigned short *>(p)), 0, 0, 0);
}

// Two floats rounded to bf16 (nearest, ties to even) and packed, a low.
__device__ __forceinline__ uint32_t bf16x2_bits(float a, float b) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(b), "f"(a));
    return r;
}

// Chained plans: call cl's input rotated into x' (M bf16 rows of xk in the
// lanes' MMA order, xpos), by all consumer warps: warp w rotates the (token,
// group) pairs w, w + 16 and w + 32 (M * groups <= 48).  The arithmetic is
// that of the decode kernels: the group-256 transform in fp32 rounded to bf16
// (with U, of h = bf16(silu(X) * U) first).
template <int BITS>
__device__ __forceinline__ void chain_rotate(const CCall &cl, uint16_t *xs, int warp, int lane) {
    constexpr int KB = BITS == 8 ? 64 : 128;
    const int G = (cl.K + kGroup - 1) / kGroup;
    const int pairs = cl.M * G;
    // every load first: the rows come from L2, one round trip for all pairs
    uint4 raw[kCPairs], rawu[kCPairs];
#pragma unroll
    for (int j = 0; j < kCPairs; ++j) {
        const int q = warp + kGConsWarps * j;
        raw[j] = rawu[j] = make_uint4(0, 0, 0, 0);
        if (q < pairs) {
            const int m = q / G, g = q - m * G;
            const int64_t gk = static_cast<int64_t>(g) * kGroup;
            const int e = group_width(cl.K, gk) / 32;
            raw[j] = load_group_raw_cg(cl.X + m * cl.ldx + gk + lane * e, e);
            if (cl.U) rawu[j] = load_group_raw_cg(cl.U + m * cl.ldu + gk + lane * e, e);
        }
    }
#pragma unroll
    for (int j = 0; j < kCPairs; ++j) {
        const int q = warp + kGConsWarps * j;
        if (q < pairs) {
            const int m = q / G, g = q - m * G;
            const int gk = g * kGroup;
            const int n = group_width(cl.K, gk);
            if (cl.U) raw[j] = swiglu_raw(raw[j], rawu[j]);
            float v[8];
            const int E = fwht_group_raw(raw[j], n, v);
            uint16_t *row = xs + m * cl.xk;
            if (E == 8) {
                // a full group: the lane's 8 values land in two runs of 4
                // (xpos): 8-bit blocks of 64 hold k = 8l..8l+7 at q = 2(l&1)
                // and q + 1, each run (k0, k2, k1, k3); 4-bit blocks of 128 at
                // jj = 2(l&3) and jj + 1, runs (k0, k4, k1, k5), (k2, k6, k3, k7)
                uint16_t *p0, *p1;
                uint2 w0, w1;
                if constexpr (BITS == 8) {
                    p0 = row + gk + (lane >> 3) * 64 + ((lane & 1) * 2) * 16 + 4 * ((lane & 7) >> 1);
                    p1 = p0 + 16;
                    w0 = make_uint2(bf16x2_bits(v[0], v[2]), bf16x2_bits(v[1], v[3]));
                    w1 = make_uint2(bf16x2_bits(v[4], v[6]), bf16x2_bits(v[5], v[7]));
                } else {
                    p0 = row + gk + (lane >> 4) * 128 + (2 * (lane & 3)) * 16 + 4 * ((lane & 15) >> 2);
                    p1 = p0 + 16;
                    w0 = make_uint2(bf16x2_bits(v[0], v[4]), bf16x2_bits(v[1], v[5]));
                    w1 = make_uint2(bf16x2_bits(v[2], v[6]), bf16x2_bits(v[3], v[7]));
                }
                *reinterpret_cast<uint2 *>(p0) = w0;
                *reinterpret_cast<uint2 *>(p1) = w1;
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    if (e < E) {
                        const int kl = gk + lane * E + e;
                        row[(kl / KB) * KB + xpos<BITS>(kl % KB)] = f32_to_bf16_bits(v[e]);
                    }
                }
            }
        }
    }
    const int tail = cl.xk - cl.K;                  // zeros after K, up to the block edge
    for (int i = warp * 32 + lane; i < cl.M * tail; i += kGConsWarps * 32) {
        const int m = i / tail, kl = cl.K + (i - m * tail);
        xs[m * cl.xk + (kl / KB) * KB + xpos<BITS>(kl % KB)] = 0;
    }
    chain_sync();
}

// Wait with the thread suspended in the barrier between polls (up to ~1 us a
// poll, woken early when the phase completes): no issue slots spent spinning.
__device__ __forceinline__ bool mbar_wait_suspend(uint32_t bar, uint32_t parity) {
    const long long t0 = clock64();
    while (true) {
        uint32_t ok;
        asm volatile(
            "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
            "selp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(ok)
            : "r"(bar), "r"(parity), "r"(1000u)
            : "memory");
        if (ok) return true;
        if (clock64() - t0 > kA16WaitLimit) return false;
    }
}

// One K block (64 bytes of each of the lane's two rows) into the four
// accumulator chains.  HASB false: rows g + 8 do not exist (an 8-row item).
// BF: x' is the bf16 operand (chained plans), codes widened to bf16 pairs;
// else x' is the scaled fp16 form and the codes are widened with their bias
// as fp16 subnormals (4-bit: odd k x16); the sums then hold 2^-24 (sum c x' +
// bias sum x'), which the store corrects with the token's sum of x'.
template <int BITS, bool HASB, bool BF>
__device__ __forceinline__ void block_mma(float (&acc)[4][4], const unsigned char *pa,
                                          const unsigned char *pb, const uint16_t *xblk) {
    const uint4 wa = *reinterpret_cast<const uint4 *>(pa);
    const uint4 wb = HASB ? *reinterpret_cast<const uint4 *>(pb) : make_uint4(0, 0, 0, 0);
    const uint32_t A[4] = {wa.x, wa.y, wa.z, wa.w};
    const uint32_t B[4] = {wb.x, wb.y, wb.z, wb.w};
    if constexpr (BF && BITS == 8) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            uint32_t a0, a1 = 0, a2, a3 = 0;
            widen_i8(A[q], a0, a2);
            if (HASB) widen_i8(B[q], a1, a3);
            const uint2 bv = *reinterpret_cast<const uint2 *>(xblk + q * 16);
            mma_bf16(acc[q], a0, a1, a2, a3, bv.x, bv.y);
        }
    } else if constexpr (BF) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            uint32_t pa4[4], pb4[4] = {0, 0, 0, 0};
            widen_i4(A[q], pa4);
            if (HASB) widen_i4(B[q], pb4);
            const uint2 b0 = *reinterpret_cast<const uint2 *>(xblk + (2 * q) * 16);
            const uint2 b1 = *reinterpret_cast<const uint2 *>(xblk + (2 * q + 1) * 16);
            mma_bf16(acc[(2 * q) % 4], pa4[0], pb4[0], pa4[1], pb4[1], b0.x, b0.y);
            mma_bf16(acc[(2 * q + 1) % 4], pa4[2], pb4[2], pa4[3], pb4[3], b1.x, b1.y);
        }
    } else if constexpr (BITS == 8) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            uint32_t a0, a1 = 0, a2, a3 = 0;
            widen_i8_f16_biased(A[q], a0, a2);
            if (HASB) widen_i8_f16_biased(B[q], a1, a3);
            const uint2 bv = *reinterpret_cast<const uint2 *>(xblk + q * 16);
            mma_f16(acc[q], a0, a1, a2, a3, bv.x, bv.y);
        }
    } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            uint32_t pa4[4], pb4[4] = {0, 0, 0, 0};
            widen_i4_f16_biased(A[q], pa4);
            if (HASB) widen_i4_f16_biased(B[q], pb4);
            const uint2 b0 = *reinterpret_cast<const uint2 *>(xblk + (2 * q) * 16);
            const uint2 b1 = *reinterpret_cast<const uint2 *>(xblk + (2 * q + 1) * 16);
            mma_f16(acc[(2 * q) % 4], pa4[0], pb4[0], pa4[1], pb4[1], b0.x, b0.y);
            mma_f16(acc[(2 * q + 1) % 4], pa4[2], pb4[2], pa4[3], pb4[3], b1.x, b1.y);
        }
    }
}

// Blocks [b, bend) of one 16-row tile: fragment rows at pA (rows g) and pB
// (rows g + 8), x' of the lane at xb.  TILES: the tile form (chunks of two
// blocks cst bytes apart; the lane's 16-byte unit of an even / odd block at
// offE / offO within its swizzled row line); else rows of 64-byte blocks.
// Blocks go in pairs, so each step has two blocks' loads in flight.
template <int BITS, bool TILES, bool HASB, bool BF>
__device__ __forceinline__ void tile_blocks(float (&acc)[4][4], const unsigned char *pA,
                                            const unsigned char *pB, const uint16_t *xb, int b,
                                            int bend, int cst, int offE, int offO) {
    constexpr int KB = BITS == 8 ? 64 : 128;   // k per block
    auto off = [&](int blk) { return TILES ? (blk >> 1) * cst + ((blk & 1) ? offO : offE) : blk * 64; };
    if (TILES && b < bend && (b & 1)) {        // a run that starts on an odd block
        block_mma<BITS, HASB, BF>(acc, pA + off(b), pB + off(b), xb + b * KB);
        ++b;
    }
    for (; b + 1 < bend; b += 2) {
        const int o0 = TILES ? (b >> 1) * cst + offE : b * 64;
        const int o1 = TILES ? o0 - offE + offO : o0 + 64;
        block_mma<BITS, HASB, BF>(acc, pA + o0, pB + o0, xb + b * KB);
        block_mma<BITS, HASB, BF>(acc, pA + o1, pB + o1, xb + (b + 1) * KB);
    }
    if (b < bend) block_mma<BITS, HASB, BF>(acc, pA + off(b), pB + off(b), xb + b * KB);
}

// x' of one call (a CTA per call), in the order the product's lanes read it,
// as fp16 (for 4-bit weights, odd k divided by 16 as well, exactly): token
// row m is the bf16 rounding of the rotated row (the A16 operand), times 2^e
// with e chosen so that its largest magnitude lies in [2^14, 2^15).  The
// multiplication by a power of two is exact, and so is the fp16 form of every
// value not below 2^-31 of that largest one (smaller ones keep an absolute
// error under 2^-39 of it).  The product multiplies Y by 2^-e, read from the
// float after the M fp16 rows; the M floats after those hold each token's sum
// of x' as the product multiplies it (16 times the stored value at odd k for
// 4-bit weights), for the codes' bias.
// The eight warps share the call's (token, group) pairs: a first pass puts
// each pair's largest |x'| in shared memory, one warp turns them into the
// tokens' exponents, and a second pass transforms the pairs again (their
// rows are in L2 by then) and stores them scaled.  Every call's CTA runs at
// once, so the pass costs about one call's latency.
constexpr int kRotPairsMax = TQ_MAX_M_GROUPED * 64;   // tokens x groups (K <= 16384)

template <int BITS>
__global__ void __launch_bounds__(256)
k_rotate_grouped(const GCall *calls, int64_t ncalls) {
    constexpr int KB = BITS == 8 ? 64 : 128;
    __shared__ float pam[kRotPairsMax];
    __shared__ int tok_sh[TQ_MAX_M_GROUPED];
    if (blockIdx.x >= ncalls) return;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const GCall cl = calls[blockIdx.x];
    const int G = (cl.K + kGroup - 1) / kGroup;
    const int pairs = cl.M * G;
    if (pairs > kRotPairsMax) return;              // not reached: plans refuse such calls
    for (int q = warp; q < pairs; q += 8) {
        const int m = q / G, g = q - m * G;
        const int64_t gk = static_cast<int64_t>(g) * kGroup;
        const int n = group_width(cl.K, gk);
        float v[8];
        const int E = fwht_group_raw(load_group_raw(cl.X + m * cl.ldx + gk + lane * (n / 32), n / 32), n, v);
        float amax = 0.0f;
#pragma unroll
        for (int e = 0; e < 8; ++e)
            if (e < E) amax = fmaxf(amax, fabsf(bf16_bits_to_f32(f32_to_bf16_bits(v[e]))));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        if (lane == 0) pam[q] = amax;
    }
    __syncthreads();
    if (warp == 0) {
        for (int m = 0; m < cl.M; ++m) {
            float amax = 0.0f;
            for (int g2 = lane; g2 < G; g2 += 32) amax = fmaxf(amax, pam[m * G + g2]);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
            int ex = 0;
            if (amax > 0.0f) frexpf(amax, &ex);              // amax = f * 2^ex, f in [0.5, 1)
            if (lane == 0) tok_sh[m] = amax > 0.0f ? max(-100, min(100, 15 - ex)) : 0;
        }
    }
    __syncthreads();
    for (int q = warp; q < pairs; q += 8) {
        const int m = q / G, g = q - m * G;
        const int64_t gk = static_cast<int64_t>(g) * kGroup;
        const int n = group_width(cl.K, gk);
        float v[8];
        const int E = fwht_group_raw(load_group_raw(cl.X + m * cl.ldx + gk + lane * (n / 32), n / 32), n, v);
        const float up = ldexpf(1.0f, tok_sh[m]);
        uint16_t *row = cl.xq + static_cast<int64_t>(m) * cl.xk;
        float ls = 0.0f;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            if (e < E) {
                const int kl = static_cast<int>(gk) + lane * E + e;
                const float xb = bf16_bits_to_f32(f32_to_bf16_bits(v[e]));
                // 4-bit weights: odd k meets 16 times its code (widen_i4_f16_biased)
                const bool odd4 = BITS == 4 && (kl & 1);
                const __half h = __float2half_rn(xb * (odd4 ? up * 0.0625f : up));
                row[(kl / KB) * KB + xpos<BITS>(kl % KB)] = __half_as_ushort(h);
                ls += odd4 ? 16.0f * __half2float(h) : __half2float(h);
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ls += __shfl_xor_sync(0xffffffffu, ls, o);
        if (lane == 0) pam[q] = ls;       // the first pass's maxima are spent
    }
    const int tail = cl.xk - cl.K;                 // zeros after K, up to the block edge
    for (int i = threadIdx.x; i < cl.M * tail; i += 256) {
        const int m = i / tail, kl = cl.K + (i - m * tail);
        cl.xq[static_cast<int64_t>(m) * cl.xk + (kl / KB) * KB + xpos<BITS>(kl % KB)] = 0;
    }
    float *tailf = reinterpret_cast<float *>(cl.xq + static_cast<int64_t>(cl.M) * cl.xk);
    if (threadIdx.x < cl.M) tailf[threadIdx.x] = ldexpf(1.0f, -tok_sh[threadIdx.x]);
    __syncthreads();
    if (warp == 0) {   // the tokens' sums over their groups, in a fixed order
        for (int m = 0; m < cl.M; ++m) {
            float s = 0.0f;
            for (int g2 = lane; g2 < G; g2 += 32) s += pam[m * G + g2];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
            if (lane == 0) tailf[cl.M + m] = s;
        }
    }
}

template <int BITS, bool CHAIN>
__global__ void __launch_bounds__(kGThreads, 1)
k_gemv_grouped(const GroupedParams p) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    // stages on a 1024-byte boundary (the tensor copies' 128-byte swizzle)
    unsigned char *smem = smem_raw + ((1024 - (smem_addr(smem_raw) & 1023)) & 1023);
    constexpr int KB = BITS == 8 ? 64 : 128;   // k per block (16 bytes per lane)
    constexpr int RED = CHAIN ? kGRedChain : kGRedInd;
    constexpr int HDR_OFF = CHAIN ? kGHdrOff : kGHdrOffInd, BAR_OFF = CHAIN ? kGBarOff : kGBarOffInd;
    float *red = reinterpret_cast<float *>(smem + kGRedOff);
    unsigned char *hdr = smem + HDR_OFF;       // stage headers, 128 bytes apart
    const uint32_t full0 = smem_addr(smem + BAR_OFF);
    const uint32_t empty0 = full0 + 8 * kGStages;
    volatile int *abort_sh = reinterpret_cast<volatile int *>(smem + BAR_OFF + 2 * kGStages * 8);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t grid = gridDim.x;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kGStages; ++s) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(full0 + 8 * s));
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(empty0 + 8 * s));
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        *abort_sh = 0;
    }
    __syncthreads();

    if (warp == kGConsWarps) {
        // ------------------------------------------------ producer
        // Item k goes to stage k % kGStages once the consumers have released
        // the stage's previous item (this warp is the only waiter, in order).
        int64_t k = 0;
        GIssue nxt;                      // the next item's copy fields, loaded one item ahead
        if (blockIdx.x < p.nitems) nxt = issue_of(p.items + blockIdx.x);
        for (;; ++k) {
            const int64_t i = blockIdx.x + k * grid;
            const bool stop = __shfl_sync(0xffffffffu, *abort_sh, 0) != 0;   // one decision per warp
            if (i >= p.nitems || stop) break;
            const GIssue it = nxt;
            if (i + grid < p.nitems) nxt = issue_of(p.items + i + grid);
            const int s = static_cast<int>(k % kGStages);
            const int64_t u = k / kGStages;
            bool ok = true;
            if (lane == 0 && u > 0) ok = mbar_wait_suspend(empty0 + 8 * s, static_cast<uint32_t>((u - 1) & 1));
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) {
                if (lane == 0) {
                    *abort_sh = 1;
                    atomicOr(p.status, kStatusGroupedTimeout);
                }
                break;
            }
            unsigned char *st = smem + s * kGStageBytes;
            const uint32_t full = full0 + 8 * s;
            const int nch = (it.rbytes + 127) / 128;
            if (lane == 0) {
                // chained plans: no x' with the item (its consumers rotate the input)
                const uint32_t xbytes = CHAIN ? 0u : static_cast<uint32_t>(it.M) * it.xk * 2 + kXTail;
                // a tensor copy counts its whole box, zero fill included
                const uint32_t wbytes = it.tiles ? static_cast<uint32_t>(nch * it.rb * 128)
                                                 : static_cast<uint32_t>(it.rows * it.rbytes);
                asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(full),
                             "r"(wbytes + xbytes + static_cast<uint32_t>(sizeof(GItem)))
                             : "memory");
                // the record itself, into the stage's header
                asm volatile(
                    "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                    ::"r"(smem_addr(hdr + s * 128)), "l"(p.items + i), "r"(static_cast<uint32_t>(sizeof(GItem))),
                      "r"(full)
                    : "memory");
                if (!CHAIN)
                    asm volatile(
                        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                        ::"r"(smem_addr(st + it.xoff)), "l"(it.xq), "r"(xbytes), "r"(full)
                        : "memory");
            }
            __syncwarp();
            if (it.tiles) {
                for (int c = lane; c < nch; c += 32) {
                    asm volatile(
                        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes "
                        "[%0], [%1, {%2, %3}], [%4];"
                        ::"r"(smem_addr(st + c * it.rb * 128)), "l"(it.tmap), "r"(c * 128), "r"(it.n0),
                          "r"(full)
                        : "memory");
                }
            } else {
                for (int r = lane; r < it.rows; r += 32) {
                    asm volatile(
                        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                        ::"r"(smem_addr(st + r * it.ws)), "l"(it.w + static_cast<int64_t>(r) * it.rbytes),
                          "r"(static_cast<uint32_t>(it.rbytes)), "r"(full)
                        : "memory");
                }
            }
        }
        // never leave with copies still landing: wait for the last issued use
        // of every stage (already complete unless the consumers stopped)
        if (lane == 0) {
            for (int s = 0; s < kGStages; ++s) {
                const int64_t uses = k > s ? (k - s + kGStages - 1) / kGStages : 0;
                if (uses > 0) mbar_wait_bounded(full0 + 8 * s, static_cast<uint32_t>((uses - 1) & 1), kA16DrainLimit);
            }
        }
        return;
    }

    // ---------------------------------------------------- consumers
    // Units of an item are (16-row tile, K block), tile-major; warp w takes a
    // contiguous run of them and keeps one tile's sums in registers until its
    // run leaves the tile.  The partial sums of a row are then added over the
    // warps in warp order: the result does not depend on timing.
    const int g = lane >> 2, t = lane & 3;
    int cur = -1;                                  // chained plans: the call x' holds
    uint16_t *xs = reinterpret_cast<uint16_t *>(smem + kCXOff);
    for (int64_t k = 0;; ++k) {
        const int64_t i = blockIdx.x + k * grid;
        if (i >= p.nitems) break;
        const int s = static_cast<int>(k % kGStages);
        const bool ok = mbar_wait_suspend(full0 + 8 * s, static_cast<uint32_t>((k / kGStages) & 1));
        float *rd = red + (k & 1) * kGConsWarps * RED;
        // the header is read before the stage is released
        int rows = 0, rb = 0, ws = 0, xk = KB, M = 1, xoff = 0;
        uint32_t nbm = 1u << 20, rowm = 1u << 20;
        bool tiles = false;
        const float *swp = nullptr;
        void *y = nullptr;
        int64_t ldy = 0;
        int ci = 0;
        uint32_t cwait = 0;
        if (ok) {
            const GItem &h = *reinterpret_cast<const GItem *>(hdr + s * 128);
            rows = h.rows;
            rb = h.rb;
            ws = h.ws;
            xk = h.xk;
            M = h.M;
            xoff = h.xoff;
            tiles = h.tiles != 0;
            swp = h.sw;
            y = h.y;
            ldy = h.ldy;
            ci = h.call;
            cwait = h.wait;
            nbm = h.nbm;
            rowm = h.rowm;
        }
        if constexpr (CHAIN) {
            // the first item of a call in this CTA: wait for the previous
            // call, then rotate this call's input (every consumer holds the
            // same header once the barrier passes, or all of them stop)
            if (consumers_sync_any(!ok)) {
                if (threadIdx.x == 0) {
                    *abort_sh = 1;
                    atomicOr(p.status, kStatusGroupedTimeout);
                }
                break;
            }
            if (ci != cur) {
                const CCall cl = p.chain[ci];          // its load overlaps the wait
                bool dep = true;
                if (threadIdx.x == 0 && cwait > 0) dep = chain_wait(p.done + ci - 1, cwait + kChainWaitExtra);
                if (consumers_sync_any(!dep)) {
                    if (threadIdx.x == 0) {
                        *abort_sh = 1;
                        atomicOr(p.status, kStatusGroupedTimeout);
                    }
                    break;
                }
                chain_rotate<BITS>(cl, xs, warp, lane);
                cur = ci;
            }
        }
        const int NB = xk / KB, U = ((rb + 15) / 16) * NB;
        const int u0 = U * warp / kGConsWarps, u1 = U * (warp + 1) / kGConsWarps;
        // thread j < rows * M adds the partial sums of output (row j % rows,
        // token j / rows) after the barrier: the first warps do it while the
        // others already multiply the next item
        const int j = threadIdx.x;
        const bool store = ok && j < rows * M;
        const int m_st = store ? static_cast<int>((static_cast<uint32_t>(j) * rowm) >> 20) : 0;
        const int r_st = store ? j - m_st * rows : 0;
        // the warps whose runs touch the row's tile (read before the release)
        int w_lo = 0, w_hi = -1;
        if (store) {
            const GItem &h = *reinterpret_cast<const GItem *>(hdr + s * 128);
            w_lo = h.wf[r_st >> 4];
            w_hi = h.wl[r_st >> 4];
        }
        const float swv = store ? __ldg(swp + r_st) : 0.0f;
        // the token's 2^-e (after the x' rows), read before the stage is released
        const float *tailf = reinterpret_cast<const float *>(smem + s * kGStageBytes + xoff + M * xk * 2);
        const float dsc = (!store || CHAIN) ? 1.0f : tailf[m_st];
        // the codes' bias times the token's sum of x' (independent plans)
        const float bsum = (!store || CHAIN) ? 0.0f : (BITS == 8 ? 128.0f : 8.0f) * tailf[M + m_st];
        if (ok && u0 < u1) {
            const unsigned char *st = smem + s * kGStageBytes;
            const uint16_t *xb = (CHAIN ? xs : reinterpret_cast<const uint16_t *>(st + xoff)) + (g < M ? g : 0) * xk + 4 * t;
            // shared row of fragment row g: in the tile form the two rows a
            // quarter-warp reads are 4 apart, so their swizzled units fall in
            // opposite halves of the 128-byte line (no bank conflict)
            const int gr = tiles ? ((g >> 1) | ((g & 1) << 2)) : g;
            const int cst = rb * 128;
            // the run, one tile at a time: blocks [b, bend) of tile `tile`
            int tile = static_cast<int>((static_cast<uint32_t>(u0) * nbm) >> 20);
            for (int u = u0; u < u1; ++tile) {
                int b = u - tile * NB;
                const int bend = min(u1 - tile * NB, NB);
                u = tile * NB + bend;
                // rows g always exist (rb is a multiple of 8); rows g + 8 unless
                // the item has 8 rows
                const int rA = tile * 16 + gr, rB = rA + 8;
                const bool hasB = rB < rb;
                const unsigned char *pA = tiles ? st + rA * 128 : st + rA * ws + t * 16;
                const unsigned char *pB = tiles ? st + rB * 128 : st + rB * ws + t * 16;
                const int sw7 = rA & 7;          // = rB & 7
                const int offE = (t ^ sw7) << 4, offO = ((4 | t) ^ sw7) << 4;
                float acc[4][4];
#pragma unroll
                for (int c = 0; c < 4; ++c) acc[c][0] = acc[c][1] = acc[c][2] = acc[c][3] = 0.0f;
                if (tiles) {
                    if (hasB) tile_blocks<BITS, true, true, CHAIN>(acc, pA, pB, xb, b, bend, cst, offE, offO);
                    else tile_blocks<BITS, true, false, CHAIN>(acc, pA, pB, xb, b, bend, cst, offE, offO);
                } else {
                    if (hasB) tile_blocks<BITS, false, true, CHAIN>(acc, pA, pB, xb, b, bend, cst, offE, offO);
                    else tile_blocks<BITS, false, false, CHAIN>(acc, pA, pB, xb, b, bend, cst, offE, offO);
                }
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int row = tile * 16 + gr + 8 * h;
                    if (row >= rb) continue;
                    const float s0 = (acc[0][2 * h] + acc[1][2 * h]) + (acc[2][2 * h] + acc[3][2 * h]);
                    const float s1 = (acc[0][2 * h + 1] + acc[1][2 * h + 1]) + (acc[2][2 * h + 1] + acc[3][2 * h + 1]);
                    if (2 * t < M) rd[warp * RED + row * M + 2 * t] = s0;
                    if (2 * t + 1 < M) rd[warp * RED + row * M + 2 * t + 1] = s1;
                }
            }
        }
        // shared reads of the stage end here; the next bulk copy into it is
        // ordered after them by the proxy fence and the release below
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        if (consumers_sync_any(!ok)) {
            if (threadIdx.x == 0) {
                *abort_sh = 1;
                atomicOr(p.status, kStatusGroupedTimeout);
            }
            break;
        }
        if (threadIdx.x == 0)
            asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(empty0 + 8 * s) : "memory");
        if (store) {
            float sum = 0.0f;
            for (int w = w_lo; w <= w_hi; ++w) {
                // warps of a non-empty run in that range wrote a partial
                if (U * w / kGConsWarps < U * (w + 1) / kGConsWarps) sum += rd[w * RED + r_st * M + m_st];
            }
            const float yv = CHAIN ? swv * sum : swv * (dsc * fmaf(sum, 16777216.0f, -bsum));
            const int64_t off = static_cast<int64_t>(m_st) * ldy + r_st;
            if (p.ytype == 0)
                static_cast<float *>(y)[off] = yv;
            else
                static_cast<uint16_t *>(y)[off] = f32_to_bf16_bits(yv);
        }
        if constexpr (CHAIN) {
            // every output of the item is stored (the barrier orders them
            // before thread 0's release): count it done
            chain_sync();
            if (threadIdx.x == 0)
                asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p.done + ci), "r"(1u) : "memory");
        }
    }
}

}  // namespace

// Rows of one work item for calls of these sizes: the largest multiple of 16
// whose weight rows and the call's x' fit one stage (rows x tokens <= 160),
// else 8, else 0 (the call cannot be grouped).
int grouped_item_rows(int64_t M, int64_t K, int bits) {
    if (M < 1 || M > TQ_MAX_M_GROUPED || K < 1) return 0;
    const int64_t KB = bits == 8 ? 64 : 128;
    const int64_t rbytes = K * bits / 8;
    const int64_t ws = (rbytes + 127) / 128 * 128 + 64;
    const int64_t xbytes = M * ((K + KB - 1) / KB * KB) * 2 + kXTail;
    int64_t rb = (kGStageBytes - xbytes) / ws;
    if (rb > kGRedInd / M) rb = kGRedInd / M;
    return rb >= 16 ? static_cast<int>(rb / 16 * 16) : (rb >= 8 ? 8 : 0);
}

// Rows of one work item of a chained plan.  The stage holds weight rows only
// (the consumers rotate the input into x' of their own, which must hold the
// call: M * xk * 2 bytes, M * groups <= 48), and a call is spread over
// up to `grid` CTAs so that each call runs on as many SMs as it can: the
// fewest rows (8, else a multiple of 16) that deal the call over the grid,
// at most a stage's worth.  grid 0: 8 rows (the most items a call can have).
int chain_item_rows(int64_t M, int64_t K, int64_t N, int bits, int grid) {
    if (M < 1 || M > TQ_MAX_M_GROUPED || K < 1 || N < 1) return 0;
    const int64_t KB = bits == 8 ? 64 : 128;
    const int64_t xk = (K + KB - 1) / KB * KB;
    if (M * xk * 2 > kCXBytes) return 0;
    if (M * ((K + kGroup - 1) / kGroup) > kGConsWarps * kCPairs) return 0;
    const int64_t rbytes = K * bits / 8;
    const int64_t ws = (rbytes + 127) / 128 * 128 + 64;
    int64_t fit = kGStageBytes / ws;
    if (fit > kGRedChain / M) fit = kGRedChain / M;
    fit = fit >= 16 ? fit / 16 * 16 : (fit >= 8 ? 8 : 0);
    if (fit == 0) return 0;
    if (grid <= 0) return 8;
    int64_t want = (N + grid - 1) / grid;
    want = want <= 8 ? 8 : (want + 15) / 16 * 16;
    return static_cast<int>(want < fit ? want : fit);
}

}  // namespace tq

// The plan: where its tables and x' workspace sit in the caller's device
// buffer, and what a run launches.
struct tq_grouped_s {
    int device;
    int bits;
    int ytype;
    int grid;
    int64_t ncalls;       // calls with work (M > 0 and N > 0)
    int64_t nitems;
    tq::GCall *calls;
    tq::GItem *items;
    int64_t weight_bytes;
    int chain;            // 1: a chained plan (calls in order, one cooperative launch)
    int64_t nccalls;
    tq::CCall *ccalls;
    unsigned int *done;   // finished items per call, zeroed before each run
};

namespace tq {

namespace {

struct GroupedTables {
    std::vector<GCall> calls;
    std::vector<CCall> ccalls;         // chained plans
    std::vector<GItem> items;
    std::vector<CUtensorMap> maps;     // one per call in the tile form
    size_t calls_bytes = 0, items_bytes = 0, maps_bytes = 0, x_bytes = 0, ccalls_bytes = 0, done_bytes = 0;
    int64_t weight_bytes = 0;
    size_t total() const { return calls_bytes + items_bytes + maps_bytes + x_bytes + ccalls_bytes + done_bytes; }
};

// Host tables of a plan, with x' and tensor-map addresses as offsets into
// their areas.  `encode` false: sizes only (every short-row call counted in
// the tile form).  `chain` non-NULL: a chained plan of those calls (`calls`
// unused), its items sized for `grid` CTAs (0: the most items).
tq_status grouped_tables(const tq_a16_call *calls, const tq_chain_call *chain, int64_t n, int bits, int ytype,
                         bool encode, int grid, GroupedTables &t) {
    const int64_t KB = bits == 8 ? 64 : 128;
    uint32_t prev_items = 0, wait = 0;
    for (int64_t c = 0; c < n; ++c) {
        const tq_a16_call &a = chain ? chain[c].call : calls[c];
        if (a.M == 0 || a.N == 0) continue;
        const int rb = chain ? chain_item_rows(a.M, a.K, a.N, bits, grid) : grouped_item_rows(a.M, a.K, bits);
        if (rb == 0) return TQ_ERR_SHAPE;
        GCall g{};
        g.X = static_cast<const uint16_t *>(a.X);
        g.ldx = a.ldx;
        g.M = static_cast<int32_t>(a.M);
        g.K = static_cast<int32_t>(a.K);
        g.xk = static_cast<int32_t>((a.K + KB - 1) / KB * KB);
        if (chain) {
            CCall cc{};
            cc.X = g.X;
            cc.U = static_cast<const uint16_t *>(chain[c].U);
            cc.ldx = a.ldx;
            cc.ldu = chain[c].U ? chain[c].ldu : 0;
            cc.M = g.M;
            cc.K = g.K;
            cc.xk = g.xk;
            t.ccalls.push_back(cc);
            wait = prev_items;
            prev_items = static_cast<uint32_t>((a.N + rb - 1) / rb);
        } else {
            g.xq = reinterpret_cast<uint16_t *>(static_cast<uintptr_t>(t.x_bytes));
            t.calls.push_back(g);
            t.x_bytes += static_cast<size_t>(a.M) * g.xk * 2 + kXTail;   // a multiple of 32
        }
        const int64_t rbytes = a.K * bits / 8;
        const int64_t ws = (rbytes + 127) / 128 * 128 + 64;
        const int64_t nch = (rbytes + 127) / 128;
        t.weight_bytes += a.N * rbytes + 4 * a.N;
        // the tile form when its copies (one per 128-byte chunk) are fewer
        // than the rows of an item (sizes of a chained plan: its largest
        // items, so that every tensor map a plan may hold is counted)
        const int rb_form = chain && !encode ? chain_item_rows(a.M, a.K, a.N, bits, 1) : rb;
        bool tiles = nch < rb_form;
        const void *map_off = nullptr;
        if (tiles) {
            CUtensorMap m;
            if (encode && !make_map_u8(&m, a.Wq, a.N, rbytes, 128, rb, CU_TENSOR_MAP_SWIZZLE_128B)) {
                tiles = false;               // no encoder: rows instead
            } else {
                map_off = reinterpret_cast<const void *>(static_cast<uintptr_t>(t.maps.size() * sizeof(CUtensorMap)));
                t.maps.push_back(m);
            }
        }
        for (int64_t n0 = 0; n0 < a.N; n0 += rb) {
            GItem it{};
            it.w = static_cast<const uint8_t *>(a.Wq) + n0 * rbytes;
            it.tmap = map_off;
            it.n0 = static_cast<int32_t>(n0);
            it.tiles = tiles ? 1 : 0;
            it.xoff = static_cast<int32_t>(tiles ? nch * rb * 128 : rb * ws);
            it.xq = g.xq;
            it.sw = a.sw + n0;
            it.y = static_cast<unsigned char *>(a.Y) + n0 * (ytype == 0 ? 4 : 2);
            it.ldy = a.ldy;
            it.rows = static_cast<int32_t>(a.N - n0 < rb ? a.N - n0 : rb);
            it.rb = rb;
            it.rbytes = static_cast<int32_t>(rbytes);
            it.ws = static_cast<int32_t>(ws);
            it.xk = g.xk;
            it.M = static_cast<int16_t>(a.M);
            it.call = chain ? static_cast<int32_t>(t.ccalls.size() - 1) : 0;
            it.wait = chain ? wait : 0;
            // the consumers' divisions, done here: u / NB and j / rows by
            // multiplication are exact while u NB and j rows stay below 2^20
            // (a 96 KB stage keeps u NB under 2^15, and j rows <= 160^2)
            const int64_t NB = g.xk / KB, U = (rb + 15) / 16 * NB;
            it.nbm = static_cast<uint32_t>(((int64_t(1) << 20) + NB - 1) / NB);
            it.rowm = static_cast<uint32_t>(((int64_t(1) << 20) + it.rows - 1) / it.rows);
            // unit u belongs to the warp w with floor(U w / W) <= u < floor(U (w + 1) / W),
            // W = kGConsWarps: w = ceil(W (u + 1) / U) - 1
            auto owner = [&](int64_t u) { return (kGConsWarps * (u + 1) + U - 1) / U - 1; };
            for (int64_t tl = 0; tl < (rb + 15) / 16; ++tl) {
                it.wf[tl] = static_cast<uint8_t>(owner(tl * NB));
                it.wl[tl] = static_cast<uint8_t>(owner(tl * NB + NB - 1));
            }
            t.items.push_back(it);
        }
    }
    t.ccalls_bytes = (t.ccalls.size() * sizeof(CCall) + 255) / 256 * 256;
    t.done_bytes = (t.ccalls.size() * 4 + 255) / 256 * 256;
    t.calls_bytes = (t.calls.size() * sizeof(GCall) + 255) / 256 * 256;
    t.items_bytes = (t.items.size() * sizeof(GItem) + 255) / 256 * 256;
    t.maps_bytes = (t.maps.size() * sizeof(CUtensorMap) + 255) / 256 * 256;
    return TQ_OK;
}

}  // namespace

tq_status grouped_bytes(const tq_a16_call *calls, int64_t n, int bits, size_t *bytes) {
    GroupedTables t;
    const tq_status st = grouped_tables(calls, nullptr, n, bits, 0, false, 0, t);
    if (st == TQ_OK) *bytes = t.total();
    return st;
}

tq_status chain_bytes(const tq_chain_call *calls, int64_t n, int bits, size_t *bytes) {
    GroupedTables t;
    const tq_status st = grouped_tables(nullptr, calls, n, bits, 0, false, 0, t);
    if (st == TQ_OK) *bytes = t.total();
    return st;
}

namespace {

// Both kinds of plan: tables into `dmem` (calls, items, tensor maps, x' or
// the chained calls and their counters, in that order), then the handle.
tq_status plan_create(const tq_a16_call *calls, const tq_chain_call *chain, int64_t n, int bits, int ytype,
                      void *dmem, size_t dbytes, const DeviceInfo &dev, tq_grouped *out) {
    GroupedTables t;
    tq_status st = grouped_tables(calls, chain, n, bits, ytype, true, chain ? dev.sms : 0, t);
    if (st != TQ_OK) return st;
    if (t.total() > 0 && (!dmem || dbytes < t.total())) return TQ_ERR_WORKSPACE;
    unsigned char *base = static_cast<unsigned char *>(dmem);
    unsigned char *mbase = base + t.calls_bytes + t.items_bytes;
    unsigned char *xbase = mbase + t.maps_bytes;
    unsigned char *cbase = xbase + t.x_bytes;
    unsigned char *dbase = cbase + t.ccalls_bytes;
    for (GCall &g : t.calls) g.xq = reinterpret_cast<uint16_t *>(xbase + reinterpret_cast<uintptr_t>(g.xq));
    for (GItem &it : t.items) {
        it.xq = chain ? nullptr : reinterpret_cast<const uint16_t *>(xbase + reinterpret_cast<uintptr_t>(it.xq));
        if (it.tiles) it.tmap = mbase + reinterpret_cast<uintptr_t>(it.tmap);
    }
    cudaError_t e = cudaSuccess;
    if (!t.ccalls.empty())
        e = cudaMemcpy(cbase, t.ccalls.data(), t.ccalls.size() * sizeof(CCall), cudaMemcpyHostToDevice);
    if (e == cudaSuccess && !t.calls.empty())
        e = cudaMemcpy(base, t.calls.data(), t.calls.size() * sizeof(GCall), cudaMemcpyHostToDevice);
    if (e == cudaSuccess && !t.items.empty())
        e = cudaMemcpy(base + t.calls_bytes, t.items.data(), t.items.size() * sizeof(GItem),
                       cudaMemcpyHostToDevice);
    if (e == cudaSuccess && !t.maps.empty())
        e = cudaMemcpy(mbase, t.maps.data(), t.maps.size() * sizeof(CUtensorMap), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return cuda_fail(e);
    tq_grouped plan = new (std::nothrow) tq_grouped_s;
    if (!plan) return TQ_ERR_WORKSPACE;
    plan->device = dev.id;
    plan->bits = bits;
    plan->ytype = ytype;
    plan->ncalls = static_cast<int64_t>(t.calls.size());
    plan->nitems = static_cast<int64_t>(t.items.size());
    plan->grid = static_cast<int>(plan->nitems < dev.sms ? plan->nitems : dev.sms);
    plan->calls = reinterpret_cast<GCall *>(base);
    plan->items = reinterpret_cast<GItem *>(base + t.calls_bytes);
    plan->weight_bytes = t.weight_bytes;
    plan->chain = chain ? 1 : 0;
    plan->nccalls = static_cast<int64_t>(t.ccalls.size());
    plan->ccalls = reinterpret_cast<CCall *>(cbase);
    plan->done = reinterpret_cast<unsigned int *>(dbase);
    *out = plan;
    return TQ_OK;
}

}  // namespace

tq_status grouped_create(const tq_a16_call *calls, int64_t n, int bits, int ytype, void *dmem,
                         size_t dbytes, const DeviceInfo &dev, tq_grouped *out) {
    return plan_create(calls, nullptr, n, bits, ytype, dmem, dbytes, dev, out);
}

tq_status chain_create(const tq_chain_call *calls, int64_t n, int bits, int ytype, void *dmem,
                       size_t dbytes, const DeviceInfo &dev, tq_grouped *out) {
    return plan_create(nullptr, calls, n, bits, ytype, dmem, dbytes, dev, out);
}

namespace {

// A chained plan's run: the counters zeroed, then one cooperative launch
// (every CTA resident, as the waits between calls need).
tq_status chain_run(tq_grouped plan, const DeviceInfo &dev, cudaStream_t s) {
    auto kern = plan->bits == 8 ? k_gemv_grouped<8, true> : k_gemv_grouped<4, true>;
    static int configured_for[64][2] = {{0}};
    const int bi = plan->bits == 8 ? 0 : 1;
    if (dev.id < 0 || dev.id >= 64) return TQ_ERR_DEVICE;
    if (!configured_for[dev.id][bi]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kCSmem);
        if (e != cudaSuccess) return cuda_fail(e);
        int per_sm = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kGThreads, kCSmem);
        if (e != cudaSuccess) return cuda_fail(e);
        if (per_sm < 1) return TQ_ERR_DEVICE;
        configured_for[dev.id][bi] = 1;
    }
    if (plan->grid > dev.sms) return TQ_ERR_DEVICE;
    unsigned int *status = status_word();
    if (!status) return TQ_ERR_CUDA;
    cudaError_t e = cudaMemsetAsync(plan->done, 0, static_cast<size_t>(plan->nccalls) * 4, s);
    if (e != cudaSuccess) return cuda_fail(e);
    GroupedParams p;
    p.items = plan->items;
    p.nitems = plan->nitems;
    p.ytype = plan->ytype;
    p.status = status;
    p.chain = plan->ccalls;
    p.done = plan->done;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(plan->grid));
    cfg.blockDim = dim3(kGThreads);
    cfg.dynamicSmemBytes = kCSmem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, p);
    return e == cudaSuccess ? TQ_OK : cuda_fail(e);
}

}  // namespace

// phase 1: the rotation pre-pass; 2: the product; 3: both
tq_status grouped_run(tq_grouped plan, const DeviceInfo &dev, int phase, cudaStream_t s) {
    if (plan->device != dev.id) return TQ_ERR_DEVICE;
    if (plan->chain && phase != 3) return TQ_ERR_MODE;    // one launch: no phases to split
    if (plan->nitems == 0) return TQ_OK;
    if (plan->chain) return chain_run(plan, dev, s);
    auto rot = plan->bits == 8 ? k_rotate_grouped<8> : k_rotate_grouped<4>;
    auto kern = plan->bits == 8 ? k_gemv_grouped<8, false> : k_gemv_grouped<4, false>;
    static int configured_for[64][2] = {{0}};
    const int bi = plan->bits == 8 ? 0 : 1;
    if (dev.id >= 0 && dev.id < 64 && !configured_for[dev.id][bi]) {
        const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kGSmem);
        if (e != cudaSuccess) return cuda_fail(e);
        configured_for[dev.id][bi] = 1;
    }
    unsigned int *status = status_word();
    if (!status) return TQ_ERR_CUDA;
    if (phase & 1) {
        if (plan->ncalls > (1ll << 31) - 1) return TQ_ERR_OVERFLOW;
        rot<<<static_cast<unsigned>(plan->ncalls), 256, 0, s>>>(plan->calls, plan->ncalls);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return cuda_fail(e);
    }
    if (phase & 2) {
        GroupedParams p;
        p.items = plan->items;
        p.nitems = plan->nitems;
        p.ytype = plan->ytype;
        p.status = status;
        p.chain = nullptr;
        p.done = nullptr;
            kern<<<static_cast<unsigned>(plan->grid), kGThreads, kGSmem, s>>>(p);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return cuda_fail(e);
    }
    return TQ_OK;
}

void grouped_destroy(tq_grouped plan) { delete plan; }

int64_t grouped_weight_bytes(tq_grouped plan) { return plan->weight_bytes; }

}  // namespace tq
