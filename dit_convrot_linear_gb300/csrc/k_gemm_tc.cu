// A8 product on the 5th-generation tensor cores (tcgen05, TMEM accumulators):
//   acc[m][n] = sum_k Xq[m][k] * Wq[n][k]  (exact int32),
//   Y[m][n]   = (sx[m] * sw[n]) * acc[m][n].
// The DiT projections at large M are compute-bound (kvad-gpu internals,
// "Quantised weights on the GPU": beyond a prompt length of roughly a thousand
// tokens the arithmetic, not the weight stream, sets the time); they are about
// 80% of a denoising step (TensorFold PR #948, "What comes next").
//
// sm_103a has no integer tcgen05 MMA, so the codes are widened to fp16 (every
// int8 and int4 code is exact in fp16; every product, at most 127*127, is
// exact in fp32) and multiplied by tcgen05.mma kind::f16 into an fp32 TMEM
// accumulator.  An fp32 sum of integers stays exact while every partial sum
// is below 2^24, which 1024 products of int8 codes (1024 * 127^2 < 2^24) or
// 16384 products of int8 x int4 codes (16384 * 127 * 7 < 2^24) guarantee.  So
// the accumulator is drained every such chunk of K into an exact int32 running
// sum kept in a second TMEM region, and the result is bit-exact int32.
//
// A pair of CTAs (a cluster of 2, tcgen05 cta_group::2) computes a 256 x 256
// output tile: each CTA holds 128 rows of A (activations) and 128 rows of B
// (weights), and the MMA, issued by the even CTA, multiplies the pair's whole
// A by the pair's whole B, leaving each CTA its 128 rows x 256 columns in its
// own TMEM.  K steps of 64.  Per CTA:
//   warp 13     TMA producer: 2-D tensor copies of the raw int8 / packed int4
//               code tiles into a raw ring (64- or 32-byte swizzle, so the
//               converters' reads are bank-conflict free);
//   warps 0-7   convert raw codes to fp16 in the K-major 8x8 core-matrix
//               layout the MMA reads (operand ring), shared to shared, and
//               arrive on the even CTA's stage barrier; they work in groups
//               that take turns over the K steps, so one group's proxy fence
//               and cluster arrive overlap the others' conversions;
//   warp 8      allocates TMEM for the pair; in the even CTA, lane 0 issues
//               the MMAs and the commits (multicast to both CTAs);
//   warps 9-12  drain the accumulator (one TMEM lane quarter each) and write Y.
// Every wait is bounded: on expiry the CTA records the failure in the library
// status word, stops issuing work, lets in-flight MMAs finish (bounded), frees
// its TMEM and returns.

#include "tq_tc.cuh"

namespace tq {
namespace {

constexpr int HM = 128, BN = 256, HN = BN / 2, BK = 64;
constexpr int NCONV = 8, MMA_WARP = 8, TMA_WARP = 13, A_WARP = 14;
// The converter warps form CONV_GROUPS groups; group g converts the K steps
// it with it % CONV_GROUPS == g, so the fence-and-arrive latency at the end of
// one group's step overlaps the other groups' conversions.
#ifndef TQ_CONV_GROUPS
#define TQ_CONV_GROUPS 4
#endif
constexpr int CONV_GROUPS = TQ_CONV_GROUPS;
constexpr int WPG = NCONV / CONV_GROUPS;       // warps per group
constexpr int TPG = 32 * WPG;                  // threads per group
// Each use of a ring slot is converted by one group, so a slot's barriers
// count one group's warps whatever the ring depths are.
static_assert(NCONV % CONV_GROUPS == 0, "groups of whole warps");
constexpr int A_OP = HM * BK * 2;      // 16 KB fp16: this CTA's 128 rows of A
constexpr int B_OP = HN * BK * 2;      // 16 KB fp16: this CTA's 128 rows of B
constexpr int A_RAW = HM * BK;         // 8 KB int8 codes
constexpr int B_RAW = HN * BK;         // 8 KB int8 codes (int4: half used)
// Shared-memory plan of the operand sources (MODE):
//   0: raw A.  The TMA brings int8 codes of both operands and the converters
//      widen both;
//   1: pre-tiled A (AT).  The activations arrive as fp16 codes already in the
//      tensor core's layout, one 16 KB bulk copy per K step straight into the
//      operand ring (loaded by warp 14), and only B is widened;
//   2: pre-tiled A and B (BT).  The weights too were widened once into fp16
//      tiles (tq_tile_weights), so both arrive by tensor copies straight into
//      the operand ring, no converter runs, and the ring is one stage deeper.
template <int MODE>
struct Plan {
    static constexpr bool AT = MODE >= 1, BT = MODE == 2;
    static constexpr int BAND = BT ? 8 : 0;         // tile order (tile_m / tile_n)
    static constexpr int O = BT ? 6 : (AT ? 5 : 4);   // operand ring depth
    static constexpr int R = BT ? 0 : (AT ? 6 : 4);   // raw ring depth
    static constexpr int NWARPS = AT ? 15 : 14;
    static constexpr int THREADS = NWARPS * 32;
    static constexpr int RAW_A = AT ? 0 : A_RAW;    // raw A bytes per slot
    static constexpr int OP_BYTES = O * (A_OP + B_OP);
    static constexpr int RAW_BYTES = R * (RAW_A + B_RAW);
    static constexpr int SMEM_BYTES = OP_BYTES + RAW_BYTES + 1024;
    // A parity wait tells only two phases apart, so a waiter must know that
    // the phase before the one it waits for has completed.  A converter group
    // takes every CONV_GROUPS-th K step; for step j it waits first for its
    // operand stage to be free (step j - O consumed, in order, which implies
    // that every step up to j - O has landed and been converted), then for
    // its raw slot (previous use j - R, landed when R >= O) and, with pre-tiled
    // A, for the A tile (previous use j - O).  Its own previous step j - G
    // waited for step j - G - O to be consumed, so the stage wait cannot see
    // step j - 2O still pending when G <= O.
    static_assert(BT || R >= O, "raw slot's previous use covered by the stage wait");
    static_assert(BT || O >= CONV_GROUPS, "operand stages for every group");
};
constexpr uint32_t TMEM_COLS = 512;    // acc [0, 256) + running int32 sum [256, 512)
constexpr uint32_t RUN_COL = 256;
constexpr long long kWaitLimit = 4000000000ll;  // clock cycles, about 2 s
constexpr unsigned int kStatusGemmTimeout = 2u;
// instruction descriptor: D f32, A/B f16, K-major, N = 256, M = 256 (pair)
constexpr uint32_t IDESC = (1u << 4) | (uint32_t(BN >> 3) << 17) | (uint32_t(256 >> 4) << 24);

struct TcParams {
    const float *sx;
    int64_t M, K;
    const float *sw;
    int64_t N;
    void *Y;
    int64_t ldy;
    int ytype;            // 0 fp32, 1 bf16, 2 int32
    int mtiles, ntiles, ksteps, chunk_steps;
    unsigned int *status;
    const unsigned char *At;   // pre-tiled fp16 A codes (AT path), else null
    const unsigned int *a_trl;   // the tiled operand's trailer of bounds (word 0 the largest row
                                 // sum of |A codes|, word 6 of A codes squared), or null
    const unsigned int *w_sq;    // largest row sum of B codes squared (tiled weights), or null;
                                 // word 1 + j: per aligned window of 1024 * 2^j columns
                                 // (A's words 1 + j and 7 + j the same)
    // epilogue: Y = R + g[n] * (sx sw acc + b[n]); any of them may be absent
    const float *bias, *gate;
    const void *R;
    int64_t ldr;
    int rtype;                 // 0 fp32, 1 bf16
    int epi;                   // any of bias, gate, R given
    int vcols;                 // sw, bias, gate all 16-byte aligned (float4 loads)
    int vres;                  // R rows 16-byte aligned (16-byte loads)
    // Split tiles (stream-K).  Tiles [0, sk_dp_tiles) are computed whole,
    // tile = pair + i * pairs.  The K steps of the other tiles, sk_units in
    // all (tile-major, K fastest), are cut into one contiguous run per pair;
    // a pair takes its run from the top down.  A tile whose K steps fall to
    // several pairs is finished by the pair that holds its last K step: the
    // others store their exact int32 partial sums in their slot and raise
    // one flag per drain warp; the finisher waits for those flags, adds the
    // partials, writes Y and lowers the flags again.  sk_units == 0: every
    // tile is whole.
    int sk_dp_tiles;
    long long sk_units;
    unsigned int *sk_flags;    // [pairs][2 CTAs][kDrainWarps]
    int *sk_slots;             // [pairs][2 CTAs][128 rows][256 columns]
};

constexpr int kDrainWarps = 12;   // flags per CTA: the drain warps of the epilogue path
constexpr int kSlotInts = HM * BN;  // one CTA's partial tile

// The pieces of work of one pair, in order: whole tiles first, then the pieces
// of its run of split K steps from the top down.  kind 0: a whole tile; 1: a
// piece that does not hold the tile's last K step (stored as a partial); 2: a
// piece that does, with earlier pieces held by pairs first .. pair - 1.
struct Seg {
    int tile, k0, k1, kind, first;
};

// Pair owning K step x of the split run: the largest q with u0(q) <= x.
__device__ __forceinline__ int sk_owner(long long x, long long units, int pairs) {
    int q = static_cast<int>((x * pairs) / units);
    while (q + 1 < pairs && units * (q + 1) / pairs <= x) ++q;
    while (q > 0 && units * q / pairs > x) --q;
    return q;
}

struct SegIter {
    int pair, pairs, ksteps, dp_tiles, ntiles, i;
    long long units, u0, u;
    __device__ SegIter(const TcParams &p, int pair_, int pairs_)
        : pair(pair_), pairs(pairs_), ksteps(p.ksteps), dp_tiles(p.sk_units ? p.sk_dp_tiles : p.mtiles * p.ntiles),
          ntiles(p.mtiles * p.ntiles), i(0), units(p.sk_units) {
        u0 = units ? units * pair / pairs : 0;
        u = units ? units * (pair + 1) / pairs : 0;
    }
    __device__ bool next(Seg &s) {
        const int t = pair + i * pairs;
        if (t < dp_tiles) {
            s.tile = t; s.k0 = 0; s.k1 = ksteps; s.kind = 0; s.first = 0;
            ++i;
            return true;
        }
        if (u <= u0) return false;
        const long long tl = (u - 1) / ksteps, ts = tl * ksteps;
        s.tile = dp_tiles + static_cast<int>(tl);
        s.k0 = static_cast<int>((u0 > ts ? u0 : ts) - ts);
        s.k1 = static_cast<int>(u - ts);
        s.kind = (s.k0 == 0 && s.k1 == ksteps) ? 0 : (s.k1 < ksteps ? 1 : 2);
        s.first = s.kind == 2 ? sk_owner(ts, units, pairs) : 0;
        u = ts + s.k0;
        return true;
    }
};

__device__ __forceinline__ unsigned int ld_acquire(const unsigned int *p) {
    unsigned int v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Tile order: bands of BAND N-tiles (BAND 0: one band of all); inside a band
// N fastest, then M.  The tiles in flight at once (one per CTA pair) then
// share A strips (same M) and B strips (same band), so both stay in L2 while
// the fp32 output streams out.  Measured: bands of 8 for the both-tiled
// product, 1532 against 1402 TOPS on the DiT up projection; the converting
// products do best with one band.
template <int BAND>
__device__ __forceinline__ int tile_m(int tile, const TcParams &p) {
    if constexpr (BAND == 0) {
        return tile / p.ntiles;
    } else {
        const int band = tile / (BAND * p.mtiles), r = tile - band * (BAND * p.mtiles);
        return r / min(BAND, p.ntiles - band * BAND);
    }
}
template <int BAND>
__device__ __forceinline__ int tile_n(int tile, const TcParams &p) {
    if constexpr (BAND == 0) {
        return tile % p.ntiles;
    } else {
        const int band = tile / (BAND * p.mtiles), r = tile - band * (BAND * p.mtiles);
        const int w = min(BAND, p.ntiles - band * BAND);
        return band * BAND + r % w;
    }
}

// Converter thread (tid < TPG within its group) -> (row, 16-byte segment) of
// a 128-row tile for pass j.  Each run of 8 consecutive lanes (one shared-store
// phase) takes 8 consecutive rows of one segment, so its 16-byte stores fill
// one 128-byte core-matrix block (conflict-free), while a warp still loads
// whole sectors.
// 64-byte rows (int8 codes, 4 segments): passes 0 .. 512/TPG - 1
__device__ __forceinline__ void rows64(int tid, int j, int &r, int &seg) {
    const int lane = tid & 31, grp = (TPG * j + tid) >> 5;
    r = grp * 8 + (lane & 7);
    seg = lane >> 3;
}
// 32-byte rows (packed int4 codes, 2 segments): passes 0 .. 256/TPG - 1
__device__ __forceinline__ void rows32(int tid, int j, int &r, int &seg) {
    const int lane = tid & 31, grp = (TPG * j + tid) >> 5;
    r = grp * 16 + ((lane >> 4) << 3) + (lane & 7);
    seg = (lane >> 3) & 1;
}

// Bounded wait; on expiry raises the CTA abort flag and the status word.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int *abort,
                                          unsigned int *status) {
    const long long t0 = clock64();
    while (!mbar_try(bar, parity)) {
        if (*abort) return false;
        if (clock64() - t0 > kWaitLimit) {
            *abort = 1;
            atomicOr(status, kStatusGemmTimeout);
            return false;
        }
    }
    return true;
}

// arrive on the barrier at the same offset in CTA 0 of the cluster
__device__ __forceinline__ void mbar_arrive_leader(uint32_t bar) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, 0;" : "=r"(remote) : "r"(bar));
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(remote) : "memory");
}

__device__ __forceinline__ void commit_pair(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;"
        ::"r"(bar), "h"(static_cast<uint16_t>(3)) : "memory");
}

// A tensor copy of this CTA's half of a pair operand, completing on a barrier
// that may sit in the peer CTA (here the even CTA's stage barrier).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap *map, int c0, int c1,
                                                 uint32_t bar_cluster) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3}], [%4];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar_cluster)
        : "memory");
}

template <int BITS, int MODE, bool EPI = false>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(Plan<MODE>::THREADS, 1)
k_gemm_a8_tc(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
             const TcParams p) {
    using P = Plan<MODE>;
    constexpr bool AT = P::AT, BT = P::BT;
    constexpr int OSTAGES = P::O, RSTAGES = P::R;
    extern __shared__ __align__(1024) unsigned char smem[];
    unsigned char *opA = smem;                                       // [O][A_OP]
    unsigned char *opB = smem + OSTAGES * A_OP;                      // [O][B_OP]
    unsigned char *rawA = smem + P::OP_BYTES;                        // [R][RAW_A]
    unsigned char *rawB = smem + P::OP_BYTES + RSTAGES * P::RAW_A;   // [R][B_RAW]
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + P::OP_BYTES + P::RAW_BYTES);
    // bars: raw_full[R], raw_empty[R], op_full[O] (used in CTA 0), op_empty[O],
    //       acc_full[2], acc_empty[2] (CTA 0), done, a_full[O] (AT)
    __shared__ uint32_t tmem_base_sh;
    __shared__ volatile int abort_sh;
    __shared__ unsigned int a_bound[12];   // the A trailer's bounds, read once per CTA

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint32_t rank;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank));
    const uint32_t raw_full0 = smem_u32(bars), raw_empty0 = smem_u32(bars + RSTAGES);
    const uint32_t op_full0 = smem_u32(bars + 2 * RSTAGES);
    const uint32_t op_empty0 = smem_u32(bars + 2 * RSTAGES + OSTAGES);
    const uint32_t acc_full0 = smem_u32(bars + 2 * RSTAGES + 2 * OSTAGES);   // [2]
    const uint32_t acc_empty0 = acc_full0 + 16, done = acc_full0 + 32;        // [2], 1
    const uint32_t a_full0 = acc_full0 + 40;

    if (threadIdx.x == 0) {
        for (int s = 0; s < RSTAGES; ++s) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(raw_full0 + 8 * s));
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(raw_empty0 + 8 * s), "r"(WPG));
        }
        for (int s = 0; s < OSTAGES; ++s) {
            // the converter warps of both CTAs; with both operands tiled, the
            // even CTA's loader (its expected bytes cover both CTAs' copies)
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(op_full0 + 8 * s),
                         "r"(BT ? 1 : 2 * WPG));
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(op_empty0 + 8 * s));
        }
        for (int h = 0; h < 2; ++h) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(acc_full0 + 8 * h));
            // the drain warps of both CTAs
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(acc_empty0 + 8 * h),
                         "r"(EPI ? 24 : 8));
        }
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(done));
        if constexpr (AT && !BT) {
            for (int s = 0; s < OSTAGES; ++s)
                asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(a_full0 + 8 * s));
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        abort_sh = 0;
    }
    if (warp == 1 && lane < 12 && p.a_trl) a_bound[lane] = trailer_bound(p.a_trl, lane);
    if (warp == MMA_WARP) {
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(smem_u32(&tmem_base_sh)), "r"(TMEM_COLS));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    cluster_sync_all();  // barriers of both CTAs initialised, TMEM allocated
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = tmem_base_sh;

    // One fp32 accumulation per tile is exact when no partial sum can reach
    // 2^24: K within one chunk, or the tiled operand's largest row sum of
    // |codes| times the largest weight code, since any partial sum of
    // a_k * b_k is at most sum_k |a_k| * qmax (and some int8 weights reach it,
    // so the bound cannot be tightened without the weights).  Then two
    // accumulators [0, 256) and [256, 512) alternate between tiles and the
    // drain of one overlaps the MMAs of the next tile; otherwise one
    // accumulator is drained per chunk into the running sum.
    // The same bound per aligned window of K picks the longest chunk that
    // stays exact when one accumulation per tile does not.
    const double qmax = BITS == 8 ? 127.0 : 7.0;
    int cs = p.chunk_steps;
    bool single = p.ksteps <= cs;
    if (!single && p.a_trl) {
        single = static_cast<double>(a_bound[0]) * qmax < 16777216.0;
        // or by Cauchy-Schwarz: any partial sum is at most sum |a_k| |b_k| <=
        // |a|_2 |b|_2, so the largest row sums of squares on both sides with a
        // product below 2^48 keep every partial sum below 2^24 (the product of
        // two integers below 2^32 rounds in double, but not below 2^48 when
        // it is at least 2^48)
        if (!single && p.w_sq)
            single = static_cast<double>(a_bound[6]) * static_cast<double>(p.w_sq[0]) < 281474976710656.0;
        for (int j = 4; j >= 0 && !single; --j) {
            const int steps = (1024 << j) / BK;
            if (steps > cs && (static_cast<double>(a_bound[1 + j]) * qmax < 16777216.0 ||
                               (p.w_sq && static_cast<double>(a_bound[7 + j]) *
                                                  static_cast<double>(p.w_sq[1 + j]) < 281474976710656.0))) {
                cs = steps;
                break;
            }
        }
        single = single || p.ksteps <= cs;
    }
    const int cluster_id = blockIdx.x >> 1, nclusters = gridDim.x >> 1;
    constexpr int BRAW = BITS == 8 ? B_RAW : B_RAW / 2;   // bytes of one raw B tile

    // ---------------------------------------------------- epilogue (TMEM drain)
    // A drain warp reads the TMEM lanes of its quarter (warp % 4) and takes the
    // 32-column blocks slot, slot + nslots, ... of each tile.
    auto drain = [&](int slot, int nslots) {
        const int q = warp & 3;                       // TMEM lane quarter of this warp
        const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
        uint32_t ch = 0, tl = 0;
        const bool y16 = (reinterpret_cast<uintptr_t>(p.Y) & 15) == 0;
        const bool vec_ok = y16 && (p.ytype == 1 ? (p.ldy & 7) == 0 : (p.ldy & 3) == 0);
        // this warp's flag (one per drain warp; the same warp index drains the
        // same rows and columns in every CTA of the same rank)
        const int dw = warp < NCONV ? warp : NCONV + (warp - MMA_WARP - 1);
        const int prow = q * 32 + lane;               // this thread's row of the partial tile
        SegIter sit(p, cluster_id, nclusters);
        Seg sg;
        for (; !abort_sh && sit.next(sg); ++tl) {
            const int tile = sg.tile;
            const int64_t m0 = static_cast<int64_t>(tile_m<P::BAND>(tile, p)) * 2 * HM + rank * HM;
            const int64_t n0 = static_cast<int64_t>(tile_n<P::BAND>(tile, p)) * BN;
            const int64_t m = m0 + q * 32 + lane;
            const float xs = (p.ytype == 2 || m >= p.M) ? 1.0f : p.sx[m];
            // Y of this thread's row for output columns n0 + col .. + 31 from
            // their exact int32 sums
            auto y_block = [&](int col, const uint32_t (&r)[32]) {
                if (m >= p.M) return;
                const int64_t nb = n0 + col;
                if (p.ytype == 2) {
                    int32_t *y = static_cast<int32_t *>(p.Y) + m * p.ldy + nb;
                    if (vec_ok && nb + 32 <= p.N) {
#pragma unroll
                        for (int j = 0; j < 32; j += 4)
                            *reinterpret_cast<uint4 *>(y + j) = make_uint4(r[j], r[j + 1], r[j + 2], r[j + 3]);
                    } else {
                        for (int j = 0; j < 32; ++j)
                            if (nb + j < p.N) y[j] = static_cast<int32_t>(r[j]);
                    }
                    return;
                }
                if constexpr (!EPI) {
                    // all 32 scales loaded together, then the stores
                    float f[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int64_t n = nb + j;
                        const float wsc = n < p.N ? __ldg(p.sw + n) : 0.0f;
                        f[j] = (xs * wsc) * static_cast<float>(static_cast<int>(r[j]));
                    }
                    if (p.ytype == 0) {
                        float *y = static_cast<float *>(p.Y) + m * p.ldy + nb;
                        if (vec_ok && nb + 32 <= p.N) {
#pragma unroll
                            for (int j = 0; j < 32; j += 4)
                                *reinterpret_cast<float4 *>(y + j) = make_float4(f[j], f[j + 1], f[j + 2], f[j + 3]);
                        } else {
                            for (int j = 0; j < 32; ++j)
                                if (nb + j < p.N) y[j] = f[j];
                        }
                    } else {
                        uint16_t *y = static_cast<uint16_t *>(p.Y) + m * p.ldy + nb;
                        if (vec_ok && nb + 32 <= p.N) {
#pragma unroll
                            for (int j = 0; j < 32; j += 8) {
                                uint4 u;
                                u.x = f32_to_bf16_bits(f[j]) | (static_cast<uint32_t>(f32_to_bf16_bits(f[j + 1])) << 16);
                                u.y = f32_to_bf16_bits(f[j + 2]) | (static_cast<uint32_t>(f32_to_bf16_bits(f[j + 3])) << 16);
                                u.z = f32_to_bf16_bits(f[j + 4]) | (static_cast<uint32_t>(f32_to_bf16_bits(f[j + 5])) << 16);
                                u.w = f32_to_bf16_bits(f[j + 6]) | (static_cast<uint32_t>(f32_to_bf16_bits(f[j + 7])) << 16);
                                *reinterpret_cast<uint4 *>(y + j) = u;
                            }
                        } else {
                            for (int j = 0; j < 32; ++j)
                                if (nb + j < p.N) y[j] = f32_to_bf16_bits(f[j]);
                        }
                    }
                } else {
                // with the epilogue: eight columns at a time, values then their
                // stores (few registers live, so it does not spill).  (Reading
                // the block's whole residual first would spare an in-place
                // update (R = Y) the L1 misses its own stores cause, but
                // spills under the 128-register cap and costs more elsewhere.)
#pragma unroll
                for (int c = 0; c < 32; c += 8) {
                    const int64_t nc = nb + c;
                    float f[8];
                    {
                        // the chunk's loads issued together: column vectors as
                        // float4 pairs and the residual as one or two 16-byte
                        // loads when aligned, else element by element
                        const bool whole8 = nc + 8 <= p.N;
                        float wv[8], bv[8], gv[8], rv[8];
                        auto cols = [&](const float *v, float (&o)[8], float absent) {
                            if (v == nullptr) {
#pragma unroll
                                for (int j = 0; j < 8; ++j) o[j] = absent;
                            } else if (whole8 && p.vcols) {
                                const float4 a = __ldg(reinterpret_cast<const float4 *>(v + nc));
                                const float4 b = __ldg(reinterpret_cast<const float4 *>(v + nc + 4));
                                o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w;
                                o[4] = b.x; o[5] = b.y; o[6] = b.z; o[7] = b.w;
                            } else {
#pragma unroll
                                for (int j = 0; j < 8; ++j) o[j] = nc + j < p.N ? __ldg(v + nc + j) : absent;
                            }
                        };
                        cols(p.sw, wv, 0.0f);
                        cols(p.bias, bv, 0.0f);
                        cols(p.gate, gv, 1.0f);
                        // R may be Y itself: this thread reads each element before writing it
                        if (p.R == nullptr) {
#pragma unroll
                            for (int j = 0; j < 8; ++j) rv[j] = 0.0f;
                        } else if (p.rtype == 1) {
                            const uint16_t *rr = static_cast<const uint16_t *>(p.R) + m * p.ldr + nc;
                            if (whole8 && p.vres) {
                                const uint4 u = *reinterpret_cast<const uint4 *>(rr);
                                const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                                for (int j = 0; j < 4; ++j) {
                                    rv[2 * j] = __uint_as_float(w[j] << 16);
                                    rv[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
                                }
                            } else {
#pragma unroll
                                for (int j = 0; j < 8; ++j) rv[j] = nc + j < p.N ? bf16_bits_to_f32(rr[j]) : 0.0f;
                            }
                        } else {
                            const float *rr = static_cast<const float *>(p.R) + m * p.ldr + nc;
                            if (whole8 && p.vres) {
                                const float4 a = *reinterpret_cast<const float4 *>(rr);
                                const float4 b = *reinterpret_cast<const float4 *>(rr + 4);
                                rv[0] = a.x; rv[1] = a.y; rv[2] = a.z; rv[3] = a.w;
                                rv[4] = b.x; rv[5] = b.y; rv[6] = b.z; rv[7] = b.w;
                            } else {
#pragma unroll
                                for (int j = 0; j < 8; ++j) rv[j] = nc + j < p.N ? rr[j] : 0.0f;
                            }
                        }
                        // bias, then gate, then residual, in fp32
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            f[j] = rv[j] + gv[j] * ((xs * wv[j]) * static_cast<float>(static_cast<int>(r[c + j])) + bv[j]);
                    }
                    const bool whole = vec_ok && nc + 8 <= p.N;
                    if (p.ytype == 0) {
                        float *y = static_cast<float *>(p.Y) + m * p.ldy + nc;
                        if (whole) {
                            *reinterpret_cast<float4 *>(y) = make_float4(f[0], f[1], f[2], f[3]);
                            *reinterpret_cast<float4 *>(y + 4) = make_float4(f[4], f[5], f[6], f[7]);
                        } else {
                            for (int j = 0; j < 8; ++j)
                                if (nc + j < p.N) y[j] = f[j];
                        }
                    } else {
                        uint16_t *y = static_cast<uint16_t *>(p.Y) + m * p.ldy + nc;
                        if (whole) {
                            uint4 u;
                            u.x = f32_to_bf16_bits(f[0]) | (static_cast<uint32_t>(f32_to_bf16_bits(f[1])) << 16);
                            u.y = f32_to_bf16_bits(f[2]) | (static_cast<uint32_t>(f32_to_bf16_bits(f[3])) << 16);
                            u.z = f32_to_bf16_bits(f[4]) | (static_cast<uint32_t>(f32_to_bf16_bits(f[5])) << 16);
                            u.w = f32_to_bf16_bits(f[6]) | (static_cast<uint32_t>(f32_to_bf16_bits(f[7])) << 16);
                            *reinterpret_cast<uint4 *>(y) = u;
                        } else {
                            for (int j = 0; j < 8; ++j)
                                if (nc + j < p.N) y[j] = f32_to_bf16_bits(f[j]);
                        }
                    }
                }
                }
            };
            // A split tile: a piece without the last K step stores its exact
            // partial sums in this pair's slot; the piece with it first waits
            // until the earlier pieces' partials are stored (this warp's part
            // of them), then adds them before Y is written.
            // a partial tile in a slot: 16-byte chunk j of the 32-column block
            // col / 32 of row r at int4 index ((col / 32) * 8 + j) * 128 + r, so
            // the 32 lanes of a warp store or load 512 contiguous bytes
            int *my_slot = sg.kind == 1
                               ? p.sk_slots + (static_cast<int64_t>(cluster_id) * 2 + rank) * kSlotInts + prow * 4
                               : nullptr;
            auto wait_partials = [&]() -> bool {
                for (int c = sg.first; c < cluster_id; ++c) {
                    const unsigned int *f = p.sk_flags + (c * 2 + static_cast<int>(rank)) * kDrainWarps + dw;
                    const long long t0 = clock64();
                    while (ld_acquire(f) == 0u) {
                        if (abort_sh) return false;
                        if (clock64() - t0 > kWaitLimit) {
                            abort_sh = 1;
                            atomicOr(p.status, kStatusGemmTimeout);
                            return false;
                        }
                    }
                }
                return true;
            };
            auto finish = [&](int col, uint32_t (&r)[32]) {
                if (sg.kind == 1) {
                    int4 *d = reinterpret_cast<int4 *>(my_slot) + (col >> 5) * 8 * HM;
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        d[j * HM] = make_int4(static_cast<int>(r[4 * j]), static_cast<int>(r[4 * j + 1]),
                                              static_cast<int>(r[4 * j + 2]), static_cast<int>(r[4 * j + 3]));
                    return;
                }
                if (sg.kind == 2) {
                    for (int c = sg.first; c < cluster_id; ++c) {
                        const int4 *src = reinterpret_cast<const int4 *>(
                                              p.sk_slots + (static_cast<int64_t>(c) * 2 + rank) * kSlotInts + prow * 4) +
                                          (col >> 5) * 8 * HM;
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const int4 v = __ldcg(src + j * HM);
                            r[4 * j] += static_cast<uint32_t>(v.x);
                            r[4 * j + 1] += static_cast<uint32_t>(v.y);
                            r[4 * j + 2] += static_cast<uint32_t>(v.z);
                            r[4 * j + 3] += static_cast<uint32_t>(v.w);
                        }
                    }
                }
                y_block(col, r);
            };
            // after a piece: raise this warp's flag (stored partial) or lower
            // the flags it consumed, ready for the next launch
            auto settle = [&]() {
                if (sg.kind == 1) {
                    __threadfence();
                    __syncwarp();
                    if (lane == 0) {
                        unsigned int *f = p.sk_flags + (cluster_id * 2 + static_cast<int>(rank)) * kDrainWarps + dw;
                        asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(f), "r"(1u) : "memory");
                    }
                } else if (sg.kind == 2) {
                    __syncwarp();
                    if (lane == 0)
                        for (int c = sg.first; c < cluster_id; ++c)
                            p.sk_flags[(c * 2 + static_cast<int>(rank)) * kDrainWarps + dw] = 0u;
                }
            };
            if (single) {
                // the piece's one chunk: fp32 sums, exact integers
                const uint32_t buf = tl & 1;
                if (!mbar_wait(acc_full0 + 8 * buf, (tl >> 1) & 1, &abort_sh, p.status)) break;
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                if (sg.kind == 2 && !wait_partials()) break;
                for (int col = 32 * slot; col < BN; col += 32 * nslots) {
                    uint32_t v[32];
                    tmem_ld32(tmem + lane_base + 256u * buf + col, v);
                    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        v[j] = static_cast<uint32_t>(__float2int_rn(__uint_as_float(v[j])));
                    finish(col, v);
                }
                asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
                __syncwarp();
                if (lane == 0) mbar_arrive_leader(acc_empty0 + 8 * buf);
                settle();
                continue;
            }
            // chunks end at multiples of cs K steps (counted from K step 0,
            // so each lies inside one aligned window of the exactness bound)
            for (int c0 = sg.k0; c0 < sg.k1; ++ch) {
                const int c1 = min((c0 / cs + 1) * cs, sg.k1);
                const bool first = c0 == sg.k0;
                c0 = c1;
                if (!mbar_wait(acc_full0, ch & 1, &abort_sh, p.status)) break;
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                for (int col = 32 * slot; col < BN; col += 32 * nslots) {
                    uint32_t v[32], r[32];
                    tmem_ld32(tmem + lane_base + col, v);
                    if (!first) tmem_ld32(tmem + lane_base + RUN_COL + col, r);
                    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int x = __float2int_rn(__uint_as_float(v[j]));
                        r[j] = first ? static_cast<uint32_t>(x) : static_cast<uint32_t>(static_cast<int>(r[j]) + x);
                    }
                    tmem_st32(tmem + lane_base + RUN_COL + col, r);
                }
                asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
                __syncwarp();
                if (lane == 0) mbar_arrive_leader(acc_empty0);
            }
            if (abort_sh) break;
            // the piece's exact int32 sums are in the running region
            if (sg.kind == 2 && !wait_partials()) break;
            for (int col = 32 * slot; col < BN; col += 32 * nslots) {
                uint32_t r[32];
                tmem_ld32(tmem + lane_base + RUN_COL + col, r);
                asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
                finish(col, r);
            }
            settle();
        }
        };

    if (warp == TMA_WARP) {
        // ------------------------------------------------ TMA producer
        if (!BT && lane == 0) {
            uint32_t it = 0;
            SegIter sit(p, cluster_id, nclusters);
            Seg sg;
            while (!abort_sh && sit.next(sg)) {
                const int tile = sg.tile;
                const int m0 = tile_m<P::BAND>(tile, p) * 2 * HM + static_cast<int>(rank) * HM;
                const int n0 = tile_n<P::BAND>(tile, p) * BN + static_cast<int>(rank) * HN;
                for (int ks = sg.k0; ks < sg.k1; ++ks, ++it) {
                    const int s = it % (BT ? 1 : RSTAGES);
                    if (!mbar_wait(raw_empty0 + 8 * s, ((it / (BT ? 1 : RSTAGES)) & 1) ^ 1, &abort_sh, p.status)) break;
                    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                                 ::"r"(raw_full0 + 8 * s), "r"(static_cast<uint32_t>(P::RAW_A + BRAW)) : "memory");
                    if constexpr (!AT) tma_load_2d(smem_u32(rawA + s * A_RAW), &tmA, ks * BK, m0, raw_full0 + 8 * s);
                    tma_load_2d(smem_u32(rawB + s * B_RAW), &tmB, ks * BK * BITS / 8, n0, raw_full0 + 8 * s);
                }
            }
        }
        __syncwarp();
    } else if (AT && warp == A_WARP) {
        if constexpr (BT) {
            // -------------------------------------------- A and B loader (both tiled)
            // Tiles (mt, ks) of A and (nt, ks) of B are 16 KB rows of their
            // tensor maps.  Both CTAs copy their own halves; the copies
            // complete on the even CTA's stage barrier, whose expected bytes
            // (all four tiles) the even CTA posts.
            if (lane == 0) {
                uint32_t it = 0;
                SegIter sit(p, cluster_id, nclusters);
                Seg sg;
                while (!abort_sh && sit.next(sg)) {
                    const int tile = sg.tile;
                    const int mt = tile_m<P::BAND>(tile, p) * 2 + static_cast<int>(rank);
                    const int nt = tile_n<P::BAND>(tile, p) * 2 + static_cast<int>(rank);
                    for (int ks = sg.k0; ks < sg.k1; ++ks, ++it) {
                        const int s = it % OSTAGES;
                        if (!mbar_wait(op_empty0 + 8 * s, ((it / OSTAGES) & 1) ^ 1, &abort_sh, p.status)) break;
                        if (rank == 0)
                            asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                                         ::"r"(op_full0 + 8 * s), "r"(static_cast<uint32_t>(2 * (A_OP + B_OP)))
                                         : "memory");
                        uint32_t bar;
                        asm volatile("mapa.shared::cluster.u32 %0, %1, 0;" : "=r"(bar) : "r"(op_full0 + 8 * s));
                        tma_load_2d_pair(smem_u32(opA + s * A_OP), &tmA, 0, (mt * p.ksteps + ks) * 128, bar);
                        tma_load_2d_pair(smem_u32(opB + s * B_OP), &tmB, 0, (nt * p.ksteps + ks) * 128, bar);
                    }
                }
            }
            __syncwarp();
        } else {
        // ------------------------------------------------ A loader (pre-tiled fp16 codes)
        // Tile (mt, ks) of the activations is 16 KB contiguous, already in the
        // operand layout: one bulk copy into the stage once the MMA is done
        // with the stage's previous use.
        if (lane == 0) {
            uint32_t it = 0;
            SegIter sit(p, cluster_id, nclusters);
            Seg sg;
            while (!abort_sh && sit.next(sg)) {
                const int64_t mt = static_cast<int64_t>(tile_m<P::BAND>(sg.tile, p)) * 2 + rank;
                for (int ks = sg.k0; ks < sg.k1; ++ks, ++it) {
                    const int s = it % OSTAGES;
                    if (!mbar_wait(op_empty0 + 8 * s, ((it / OSTAGES) & 1) ^ 1, &abort_sh, p.status)) break;
                    const unsigned char *src = p.At + (mt * p.ksteps + ks) * static_cast<int64_t>(A_OP);
                    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                                 ::"r"(a_full0 + 8 * s), "r"(static_cast<uint32_t>(A_OP)) : "memory");
                    asm volatile(
                        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                        ::"r"(smem_u32(opA + s * A_OP)), "l"(src), "r"(static_cast<uint32_t>(A_OP)),
                          "r"(a_full0 + 8 * s)
                        : "memory");
                }
            }
        }
        __syncwarp();
        }
    } else if (warp < NCONV) {
        if constexpr (EPI) {
            // no conversion on this path: the converter warps help drain
            drain(1 + warp / 4, 3);
        }
        if constexpr (!BT) {
        // ------------------------------------------------ converters (shared -> shared)
        const int g = warp / WPG, tid = threadIdx.x % TPG;
        constexpr int NA = 512 / TPG;                          // A passes (and int8 B passes)
        constexpr int NB = BITS == 8 ? 512 / TPG : 256 / TPG;  // B passes
        uint32_t it = 0;
        SegIter sit(p, cluster_id, nclusters);
        Seg sg;
        while (!abort_sh && sit.next(sg)) {
            for (int ks = sg.k0; ks < sg.k1; ++ks, ++it) {
                if (static_cast<int>(it % CONV_GROUPS) != g) continue;
                const int rs = it % RSTAGES, os = it % OSTAGES;
                // stage first: see the ring plan for why the order matters
                if (!mbar_wait(op_empty0 + 8 * os, ((it / OSTAGES) & 1) ^ 1, &abort_sh, p.status)) break;
                if (!mbar_wait(raw_full0 + 8 * rs, (it / RSTAGES) & 1, &abort_sh, p.status)) break;
                const unsigned char *ra = rawA + rs * A_RAW;
                const unsigned char *rb = rawB + rs * B_RAW;
                unsigned char *oa = opA + os * A_OP;
                unsigned char *ob = opB + os * B_OP;
                if constexpr (!AT) {
                    uint4 a[NA];
#pragma unroll
                    for (int j = 0; j < NA; ++j) {
                        int r, seg;
                        rows64(tid, j, r, seg);
                        a[j] = *reinterpret_cast<const uint4 *>(ra + swz64(r, seg));
                    }
#pragma unroll
                    for (int j = 0; j < NA; ++j) {
                        int r, seg;
                        rows64(tid, j, r, seg);
                        store_i8x16(oa, r, seg, a[j]);
                    }
                }
                {
                    uint4 b[NB];
#pragma unroll
                    for (int j = 0; j < NB; ++j) {
                        int r, seg;
                        if constexpr (BITS == 8) {
                            rows64(tid, j, r, seg);
                            b[j] = *reinterpret_cast<const uint4 *>(rb + swz64(r, seg));
                        } else {
                            rows32(tid, j, r, seg);
                            b[j] = *reinterpret_cast<const uint4 *>(rb + swz32(r, seg));
                        }
                    }
#pragma unroll
                    for (int j = 0; j < NB; ++j) {
                        int r, seg;
                        if constexpr (BITS == 8) {
                            rows64(tid, j, r, seg);
                            store_i8x16(ob, r, seg, b[j]);
                        } else {
                            rows32(tid, j, r, seg);
                            store_i4x32(ob, r, seg, b[j]);
                        }
                    }
                }
                // One proxy fence serves both hand-offs: it makes this lane's
                // operand stores visible to the tensor core, and it orders this
                // lane's plain reads of the raw slot before the next TMA write
                // into that slot (both are async-proxy accesses; without the
                // fence the TMA was seen to overwrite a slot still being read).
                // The warp then arrives once on each barrier, after all its lanes.
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) {
                    // with pre-tiled A, the stage is complete once its bulk copy
                    // has landed too (this CTA's half; the even CTA's MMA cannot
                    // wait on the odd CTA's barrier, so the converters pass it on)
                    bool ok = true;
                    if constexpr (AT) ok = mbar_wait(a_full0 + 8 * os, (it / OSTAGES) & 1, &abort_sh, p.status);
                    if (ok) {
                        mbar_arrive_leader(op_full0 + 8 * os);
                        mbar_arrive_local(raw_empty0 + 8 * rs);
                    }
                }
            }
        }
        }
    } else if (warp == MMA_WARP) {
        // ------------------------------------------------ MMA issue (CTA 0, one thread)
        if (rank == 0 && lane == 0) {
            uint32_t it = 0, ch = 0, tl = 0;
            bool issued = false;
            SegIter sit(p, cluster_id, nclusters);
            Seg sg;
            for (; !abort_sh && sit.next(sg); ++tl) {
                // single: one chunk per piece into accumulator tl & 1;
                // else: chunks into accumulator 0, each drained before the next,
                // ending at multiples of cs K steps
                const uint32_t buf = single ? (tl & 1) : 0;
                for (int c0 = sg.k0, c1 = 0; c0 < sg.k1 && !abort_sh; c0 = c1) {
                    c1 = single ? sg.k1 : min((c0 / cs + 1) * cs, sg.k1);
                    const uint32_t use = single ? (tl >> 1) : ch;   // earlier uses of this accumulator
                    if (use > 0 && !mbar_wait(acc_empty0 + 8 * buf, (use - 1) & 1, &abort_sh, p.status)) break;
                    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                    for (int ks = c0; ks < c1; ++ks, ++it) {
                        const int s = it % OSTAGES;
                        if (!mbar_wait(op_full0 + 8 * s, (it / OSTAGES) & 1, &abort_sh, p.status)) break;
                        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                        const uint32_t a = smem_u32(opA + s * A_OP), b = smem_u32(opB + s * B_OP);
#pragma unroll
                        for (int kk = 0; kk < BK / 16; ++kk) {
                            const uint64_t ad = smem_desc(a + kk * 256), bd = smem_desc(b + kk * 256);
                            const uint32_t accum = (ks > c0 || kk > 0) ? 1u : 0u;
                            asm volatile(
                                "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
                                "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}\n"
                                ::"r"(tmem + 256u * buf), "l"(ad), "l"(bd), "r"(IDESC), "r"(accum));
                        }
                        issued = true;
                        commit_pair(op_empty0 + 8 * s);
                    }
                    if (abort_sh) break;
                    commit_pair(acc_full0 + 8 * buf);
                    ++ch;
                }
            }
            // let every issued MMA finish before the pair's TMEM is released
            if (issued) {
                asm volatile(
                    "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                    ::"r"(done) : "memory");
                const long long t0 = clock64();
                while (!mbar_try(done, 0) && clock64() - t0 < kWaitLimit) {
                }
            }
        }
        __syncwarp();
    } else {
        drain(0, EPI ? 3 : 1);
    }
    // nobody leaves while the peer may still arrive on this CTA's barriers or
    // while MMAs of the pair are in flight (CTA 0 waited for them above)
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    cluster_sync_all();
    if (warp == MMA_WARP) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS));
    }
}

// Shared launch of the operand paths (MODE as in Plan): Xq int8 codes (A
// through a tensor map), At pre-tiled fp16 codes, or At and Wt both pre-tiled
// (each read as rows of 128 bytes, one 16 KB tile a box).
// Split tiles (when the caller gives a split workspace) only where it was
// measured to pay: the tiles of a last wave that leaves pairs idle, and a long
// K.  Each piece costs a pipeline start, a drain and, for a partial, 128 KB
// stored or added per CTA, so short K and full waves lose: measured on 4-bit
// weights at M = 1024, 48 tiles, K = 12288: 70.9 -> 61.6 us; K = 3072: 29.9 ->
// 31.9 us; 384 tiles (five waves and four tiles), K = 3072: 106.3 -> 107.8
// us (the last wave's four tiles split: 144.9); 8-bit, M = 4032, 768 tiles,
// K = 3072: 186.4 -> 205.5 us.
constexpr double kSplitBelow = 0.85;
constexpr int kSplitMinKSteps = 96;

template <int MODE>
tq_status launch_tc(const int8_t *Xq, const unsigned char *At, const unsigned char *Wt, const float *sx,
                    int64_t M, int64_t K, const uint8_t *Wq, const float *sw, int64_t N, int bits, void *Y,
                    int ytype, int64_t ldy, const DeviceInfo &dev, cudaStream_t s,
                    const EpilogueArgs *ea = nullptr, void *split_ws = nullptr) {
    using P = Plan<MODE>;
    constexpr bool AT = P::AT;
    unsigned int *status = status_word();
    if (!status) return TQ_ERR_DEVICE;
    if (M > (1ll << 31) - 1 || N > (1ll << 31) - 1) return TQ_ERR_OVERFLOW;
    CUtensorMap tmA, tmB;
    if constexpr (MODE == 2) {
        if (!make_map_u8(&tmA, At, tiled_act_tiles_bytes(M, K) / 128, 128, 128, 128, CU_TENSOR_MAP_SWIZZLE_NONE) ||
            !make_map_u8(&tmB, Wt, (weights_tiled_bytes(N, K) - 256) / 128, 128, 128, 128, CU_TENSOR_MAP_SWIZZLE_NONE))
            return TQ_ERR_DEVICE;
    } else {
        const bool mapped = bits == 8 ? make_map_u8(&tmB, Wq, N, K, BK, 128, CU_TENSOR_MAP_SWIZZLE_64B)
                                      : make_map_u8(&tmB, Wq, N, K / 2, BK / 2, 128, CU_TENSOR_MAP_SWIZZLE_32B);
        if (!mapped) return TQ_ERR_DEVICE;
        if constexpr (AT) {
            tmA = tmB;   // not read on this path
        } else {
            if (!make_map_u8(&tmA, Xq, M, K, BK, 128, CU_TENSOR_MAP_SWIZZLE_64B)) return TQ_ERR_DEVICE;
        }
    }
    TcParams p{};
    p.sx = sx;
    p.M = M;
    p.K = K;
    p.sw = sw;
    p.N = N;
    p.Y = Y;
    p.ldy = ldy;
    p.ytype = ytype;
    p.mtiles = static_cast<int>((M + 2 * HM - 1) / (2 * HM));
    p.ntiles = static_cast<int>((N + BN - 1) / BN);
    p.ksteps = static_cast<int>((K + BK - 1) / BK);
    // K per exact fp32 chunk: 1024 * 127^2 < 2^24 (int8), 16384 * 127 * 7 < 2^24 (int4)
    p.chunk_steps = bits == 8 ? 1024 / BK : 16384 / BK;
    p.status = status;
    p.At = At;
    p.a_trl = AT ? tiled_act_trailer(const_cast<unsigned char *>(At), M, K) : nullptr;
    p.w_sq = (MODE == 2 && Wt) ? reinterpret_cast<const unsigned int *>(static_cast<const unsigned char *>(Wt) +
                                                                        weights_tiled_bytes(N, K) - 256)
                               : nullptr;
    if (ea) {
        p.bias = ea->bias;
        p.gate = ea->gate;
        p.R = ea->R;
        p.ldr = ea->ldr;
        p.rtype = ea->rtype;
    }
    p.epi = (p.bias || p.gate || p.R) ? 1 : 0;
    auto a16 = [](const void *q) { return (reinterpret_cast<uintptr_t>(q) & 15) == 0; };
    p.vcols = (a16(p.sw) && a16(p.bias) && a16(p.gate)) ? 1 : 0;
    p.vres = (p.R && a16(p.R) && (p.ldr * (p.rtype == 1 ? 2 : 4)) % 16 == 0) ? 1 : 0;
    const int64_t tiles = static_cast<int64_t>(p.mtiles) * p.ntiles;
    if (tiles > (1ll << 30)) return TQ_ERR_OVERFLOW;
    const bool epi = p.epi != 0;
    if (epi && MODE != 2) return TQ_ERR_MODE;   // the epilogue is built for the both-tiled product
    auto kern = MODE != 2 ? (bits == 8 ? k_gemm_a8_tc<8, MODE> : k_gemm_a8_tc<4, MODE>)
              : epi ? (bits == 8 ? k_gemm_a8_tc<8, MODE, MODE == 2> : k_gemm_a8_tc<4, MODE, MODE == 2>)
                    : (bits == 8 ? k_gemm_a8_tc<8, MODE> : k_gemm_a8_tc<4, MODE>);
    static bool configured_for[64][4] = {{false}};
    const int bi = (bits == 8 ? 0 : 1) + (epi ? 2 : 0);
    if (dev.id < 0 || dev.id >= 64) return TQ_ERR_DEVICE;
    if (!configured_for[dev.id][bi]) {
        const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   P::SMEM_BYTES);
        if (e != cudaSuccess) return cuda_fail(e);
        configured_for[dev.id][bi] = true;
    }
    const int64_t pmax = dev.sms / 2;
    int64_t pairs = tiles < pmax ? tiles : pmax;
    p.sk_dp_tiles = 0;
    p.sk_units = 0;
    p.sk_flags = nullptr;
    p.sk_slots = nullptr;
    if (split_ws && pmax > 0 && p.ksteps >= kSplitMinKSteps) {
        // The tiles of the whole waves stay whole; the K steps of the tiles of
        // a last wave that would leave more than 15% of the pairs idle are
        // split evenly over every pair (at least two K steps a pair).  With
        // fewer tiles than pairs that is every tile.  Measured on the DiT down
        // projection (192 tiles on 76 pairs, K = 12288, 8-bit): 189.5 against
        // 201.8 us; splitting one more wave, 198.7.
        const int64_t rem = tiles % pmax;
        if (rem > 0 && static_cast<double>(rem) < kSplitBelow * static_cast<double>(pmax)) {
            const int64_t dp = tiles - rem;
            const int64_t units = rem * p.ksteps;
            if (units >= 2 * pmax) {
                p.sk_dp_tiles = static_cast<int>(dp);
                p.sk_units = units;
                p.sk_flags = static_cast<unsigned int *>(split_ws);
                p.sk_slots = reinterpret_cast<int *>(static_cast<unsigned char *>(split_ws) + split_flag_bytes(dev));
                pairs = pmax;
            }
        }
    }
    kern<<<static_cast<unsigned>(2 * pairs), P::THREADS, P::SMEM_BYTES, s>>>(tmA, tmB, p);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? TQ_OK : cuda_fail(e);
}

}  // namespace

tq_status launch_gemm_a8(const int8_t *Xq, const float *sx, int64_t M, int64_t K,
                         const uint8_t *Wq, const float *sw, int64_t N, int bits,
                         void *Y, int ytype, int64_t ldy, const DeviceInfo &dev,
                         cudaStream_t s) {
    return launch_tc<0>(Xq, nullptr, nullptr, sx, M, K, Wq, sw, N, bits, Y, ytype, ldy, dev, s);
}

tq_status launch_gemm_a8_tiled(const void *At, const float *sx, int64_t M, int64_t K,
                               const uint8_t *Wq, const float *sw, int64_t N, int bits,
                               void *Y, int ytype, int64_t ldy, const DeviceInfo &dev,
                               cudaStream_t s) {
    return launch_tc<1>(nullptr, static_cast<const unsigned char *>(At), nullptr, sx, M, K, Wq, sw, N,
                        bits, Y, ytype, ldy, dev, s);
}

tq_status launch_gemm_a8_tt(const void *At, const float *sx, int64_t M, int64_t K, const void *Wt,
                            const float *sw, int64_t N, int bits, void *Y, int ytype, int64_t ldy,
                            const DeviceInfo &dev, cudaStream_t s, const EpilogueArgs *ea, void *split_ws) {
    return launch_tc<2>(nullptr, static_cast<const unsigned char *>(At), static_cast<const unsigned char *>(Wt),
                        sx, M, K, nullptr, sw, N, bits, Y, ytype, ldy, dev, s, ea, split_ws);
}

// Split workspace: the flags ([pairs][2 CTAs][kDrainWarps] words, rounded up to
// 256 bytes), then one partial tile per CTA ([pairs][2][128][256] int32).
size_t split_flag_bytes(const DeviceInfo &dev) {
    return (static_cast<size_t>(dev.sms / 2) * 2 * kDrainWarps * 4 + 255) / 256 * 256;
}

size_t split_workspace_bytes(const DeviceInfo &dev) {
    return split_flag_bytes(dev) + static_cast<size_t>(dev.sms / 2) * 2 * kSlotInts * 4;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
        cudaGetLastError();
    }
    return fn;
}

// 2-D map of a row-major byte matrix [rows][cols] (cols bytes per row), read in
// boxes of box_cols bytes x box_rows rows, out-of-range elements filled with zero.
bool make_map_u8(CUtensorMap *map, const void *base, int64_t rows, int64_t cols, int box_cols,
                 int box_rows, CUtensorMapSwizzle swz) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t estr[2] = {1u, 1u};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace tq
