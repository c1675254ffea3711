// Decode product for M <= 8 tokens, built for the shortest dependent path:
//   Y[m][n] = sw[n] * sum_k q_w[n][k] * x'_bf16[m][k],  fp32 sums,
// x' the group-256 Hadamard rotation of the token row rounded to bf16 (tensai
// docs, "画像生成" / Image generation, section "幅とメモリ").  Decode is bound by
// the weight stream (kvad-gpu internals, "Numbers"), but one call moves only a
// few MB, so what decides its time is the chain of latencies that must follow
// the previous call: read X, rotate, multiply, reduce, store.
//
// Layout of one call:
//   - A CTA owns RT = 16*WR weight rows and the whole of K: no cross-CTA
//     reduction.  Its 8 warps are WR row groups x WK = 8/WR K slices; a K
//     slice is a run of whole 256-groups.
//   - Before waiting for the previous kernel, the CTA bulk-copies its weight
//     slice (and row scales) into shared memory and releases the next launch
//     (programmatic dependent launch), so the weight stream of the following
//     calls overlaps this one.  Bulk copies read through the coherent L2, so
//     weights and scales must not be written by a kernel that may still be
//     running; only this library's product kernels trigger early, and they
//     write nothing but Y.
//   - After the wait, each warp reads and rotates only the groups of its own
//     K slice, keeping x' in its private shared memory (no block barrier),
//     widens weight codes to exact bf16 pairs and runs mma.sync m16n8k16 on
//     four independent accumulator chains.
//   - One barrier, then the K slices are added in a fixed order (deterministic)
//     and scaled.
// Waits are bounded: on expiry the status word is set and the call's output
// is left unwritten (tq_device_status reports it).

#include "tq_a16.cuh"

namespace tq {
namespace {

struct SmallParams {
    const uint16_t *X;
    int64_t ldx;
    const uint16_t *U;   // with U: the input row is h = bf16(silu(x) * u) (SwiGLU), else x
    int64_t ldu;
    int M;
    int64_t K;
    int G;
    const uint8_t *W;
    int64_t wld;
    const float *sw;
    int64_t N;
    void *Y;
    int64_t ldy;
    int ytype;
    int WR, WK;
    int gpw;        // most groups in any warp's K slice
    int WS;         // shared row stride of the weight slice (bytes, = 64 mod 128)
    int XS;         // per-warp x' row stride (bf16 elements, 2*XS = 32 mod 128)
    int w_off, x_off, r_off;
    unsigned int *status;
};

constexpr unsigned int kStatusSmallTimeout = 4u;
constexpr int NCH = 4;                          // accumulator chains per warp

// PRE: every warp's K slice is at most one group (256 columns), so the warp's
// weight fragments, widened to bf16 (16 MMA A-operands of 4 registers), fit in
// registers.  They are read and widened before the dependency wait, in the
// shadow of the previous kernel; after it only the x' loads and the MMAs remain.
template <int BITS, bool PRE>
__global__ void __launch_bounds__(kThreads)
k_gemv_small(const SmallParams p) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    constexpr int KB = BITS == 8 ? 64 : 128;  // k per block (one 16-byte chunk per lane)
    constexpr int BB = 64;                    // weight bytes per row per block
    constexpr int BPG = kGroup / KB;          // blocks per full group
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem_raw);
    float *sws = reinterpret_cast<float *>(smem_raw + 128);
    unsigned char *ws = smem_raw + p.w_off;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int RT = 16 * p.WR;
    const int64_t n0 = static_cast<int64_t>(blockIdx.x) * RT;
    const int rows = static_cast<int>(min(static_cast<int64_t>(RT), p.N - n0));
    const int rbytes = static_cast<int>(p.K * BITS / 8);
    const uint32_t wbar = smem_addr(bar);

    // ---- before the wait: weight slice and row scales of this tile
    if (warp == 0) {
        if (lane == 0) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(wbar));
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
            // A build for the library's own tests (TQ_TEST_UNSET_BYTES) expects
            // bytes that no copy brings, so the barrier's phase never completes
            // and the bounded waits on it expire: the expiry path is then taken
            // with every issued copy landed, the wait that a CTA keeps for its
            // copies before it exits runs to its full limit, and nothing else
            // changes.
#ifdef TQ_TEST_UNSET_BYTES
            constexpr uint32_t kUnset = TQ_TEST_UNSET_BYTES;
#else
            constexpr uint32_t kUnset = 0;
#endif
            asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(wbar),
                         "r"(static_cast<uint32_t>(rows * rbytes) + kUnset)
                         : "memory");
        }
        __syncwarp();
        for (int r = lane; r < rows; r += 32) {
            asm volatile(
                "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                ::"r"(smem_addr(ws + r * p.WS)), "l"(p.W + (n0 + r) * p.wld),
                  "r"(static_cast<uint32_t>(rbytes)), "r"(wbar)
                : "memory");
        }
    }
    if (threadIdx.x < rows) sws[threadIdx.x] = __ldg(p.sw + n0 + threadIdx.x);
    const int WR = p.WR, WK = p.WK;
    const int wr = warp % WR, wk = warp / WR;
    const int g0 = static_cast<int>(static_cast<int64_t>(p.G) * wk / WK);
    const int g1 = static_cast<int>(static_cast<int64_t>(p.G) * (wk + 1) / WK);
    if (wr == 0) {  // warm L2 with this slice's token rows (coherent: safe before the wait)
        for (int m = lane; m < p.M; m += 32) {
            const int64_t k0 = static_cast<int64_t>(g0) * kGroup;
            const int64_t k1 = min(static_cast<int64_t>(g1) * kGroup, p.K);
            if (k1 > k0) prefetch_l2(p.X + m * p.ldx + k0, static_cast<uint32_t>((k1 - k0) * 2));
            if (k1 > k0 && p.U) prefetch_l2(p.U + m * p.ldu + k0, static_cast<uint32_t>((k1 - k0) * 2));
        }
    }
    __syncthreads();  // barrier initialised; row scales in place
    pdl_launch_dependents();

    constexpr int QPB = BITS == 8 ? 4 : 8;          // MMAs per weight block
    constexpr int NBP = kGroup / KB;                // blocks in a one-group slice
    uint32_t fr[PRE ? NBP * QPB : 1][4];            // widened A operands
    bool have_w = false;
    if constexpr (PRE) {
        have_w = mbar_wait_bounded(wbar, 0);
        const int g = lane >> 2, t = lane & 3;
        const int rA = wr * 16 + g, rB = rA + 8;
        const bool okA = rA < rows, okB = rB < rows;
        const int nk0 = static_cast<int>(min(static_cast<int64_t>(g1) * kGroup, p.K) -
                                         static_cast<int64_t>(g0) * kGroup);
        const unsigned char *pA = ws + rA * p.WS + g0 * BPG * BB + t * 16;
        const unsigned char *pB = ws + rB * p.WS + g0 * BPG * BB + t * 16;
        const int sbytes = nk0 * BITS / 8;
#pragma unroll
        for (int blk = 0; blk < NBP; ++blk) {
            const int off = blk * BB;
            const bool in = have_w && off + t * 16 < sbytes;
            const uint4 wa = (in && okA) ? *reinterpret_cast<const uint4 *>(pA + off) : make_uint4(0, 0, 0, 0);
            const uint4 wb = (in && okB) ? *reinterpret_cast<const uint4 *>(pB + off) : make_uint4(0, 0, 0, 0);
            const uint32_t A[4] = {wa.x, wa.y, wa.z, wa.w};
            const uint32_t B[4] = {wb.x, wb.y, wb.z, wb.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                if constexpr (BITS == 8) {
                    uint32_t *f = fr[blk * QPB + q];
                    widen_i8(A[q], f[0], f[2]);
                    widen_i8(B[q], f[1], f[3]);
                } else {
                    uint32_t pa[4], pb[4];
                    widen_i4(A[q], pa);
                    widen_i4(B[q], pb);
                    uint32_t *f0 = fr[blk * QPB + 2 * q], *f1 = fr[blk * QPB + 2 * q + 1];
                    f0[0] = pa[0]; f0[1] = pb[0]; f0[2] = pa[1]; f0[3] = pb[1];
                    f1[0] = pa[2]; f1[1] = pb[2]; f1[2] = pa[3]; f1[3] = pb[3];
                }
            }
        }
    }
    pdl_wait();

    // ---- rotate this warp's groups into its private x' (token rows of XS)
    const int M = p.M, XS = p.XS;
    uint16_t *xw = reinterpret_cast<uint16_t *>(smem_raw + p.x_off) + static_cast<size_t>(warp) * M * XS;
    const int64_t kslice0 = static_cast<int64_t>(g0) * kGroup;
    const int nk = static_cast<int>(min(static_cast<int64_t>(g1) * kGroup, p.K) - kslice0);
    const int nblk = (nk + KB - 1) / KB;
    // groups are taken GB at a time: all their loads are issued before any
    // butterfly, so the row reads of a slice overlap instead of queueing
    constexpr int GB = 4;
    const int ng = g1 - g0;
    for (int m = 0; m < M; ++m) {
        uint16_t *xrow = xw + m * XS;
        for (int gb = 0; gb < ng; gb += GB) {
            uint4 raw[GB], rawu[GB];
#pragma unroll
            for (int u = 0; u < GB; ++u) {
                raw[u] = rawu[u] = make_uint4(0, 0, 0, 0);
                const int gi = gb + u;
                if (gi < ng) {
                    const int64_t gk = kslice0 + static_cast<int64_t>(gi) * kGroup;
                    const int E = group_width(p.K, gk) / 32;
                    raw[u] = load_group_raw(p.X + m * p.ldx + gk + lane * E, E);
                    if (p.U) rawu[u] = load_group_raw(p.U + m * p.ldu + gk + lane * E, E);
                }
            }
            if (p.U) {
#pragma unroll
                for (int u = 0; u < GB; ++u) raw[u] = swiglu_raw(raw[u], rawu[u]);
            }
#pragma unroll
            for (int u = 0; u < GB; ++u) {
                const int gi = gb + u;
                if (gi >= ng) break;
                const int64_t gk = kslice0 + static_cast<int64_t>(gi) * kGroup;
                float v[8] = {};
                const int E = fwht_group_raw(raw[u], group_width(p.K, gk), v);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    if (e < E) {
                        const int kl = gi * kGroup + lane * E + e;
                        xrow[(kl / KB) * KB + xpos<BITS>(kl % KB)] = f32_to_bf16_bits(v[e]);
                    }
                }
            }
        }
        for (int kl = nk + lane; kl < nblk * KB; kl += 32)   // padding of a partial last block
            xrow[(kl / KB) * KB + xpos<BITS>(kl % KB)] = 0;
    }
    __syncwarp();

    // ---- products: this warp's 16 rows x its K slice
    if constexpr (!PRE) have_w = mbar_wait_bounded(wbar, 0);
    if (!have_w && lane == 0) atomicOr(p.status, kStatusSmallTimeout);
    const int g = lane >> 2, t = lane & 3;
    const int rA = wr * 16 + g, rB = rA + 8;
    const bool okA = rA < rows, okB = rB < rows;
    const int boff0 = g0 * BPG * BB;   // byte offset of the slice in a weight row
    const unsigned char *pA = ws + rA * p.WS + boff0 + t * 16;
    const unsigned char *pB = ws + rB * p.WS + boff0 + t * 16;
    const bool xin = g < M;            // this lane's token (B column) exists
    const uint16_t *xb = xw + (xin ? g : 0) * XS + 4 * t;
    const int slice_bytes = nk * BITS / 8;

    float acc[NCH][4];
#pragma unroll
    for (int c = 0; c < NCH; ++c) acc[c][0] = acc[c][1] = acc[c][2] = acc[c][3] = 0.0f;
    if (PRE && have_w) {
#pragma unroll
        for (int blk = 0; blk < NBP; ++blk) {
            if (blk < nblk) {
                const uint16_t *xblk = xb + blk * KB;
#pragma unroll
                for (int q = 0; q < QPB; ++q) {
                    // token columns >= M read row 0 (valid); their outputs are dropped
                    const uint2 bv = *reinterpret_cast<const uint2 *>(xblk + q * 16);
                    const uint32_t *f = fr[blk * QPB + q];
                    mma_bf16(acc[q % NCH], f[0], f[1], f[2], f[3], bv.x, bv.y);
                }
            }
        }
    } else if (have_w) {
        for (int blk = 0; blk < nblk; ++blk) {
            const int off = blk * BB;
            const bool in = off + t * 16 < slice_bytes;
            const uint4 wa = (in && okA) ? *reinterpret_cast<const uint4 *>(pA + off) : make_uint4(0, 0, 0, 0);
            const uint4 wb = (in && okB) ? *reinterpret_cast<const uint4 *>(pB + off) : make_uint4(0, 0, 0, 0);
            const uint32_t A[4] = {wa.x, wa.y, wa.z, wa.w};
            const uint32_t B[4] = {wb.x, wb.y, wb.z, wb.w};
            const uint16_t *xblk = xb + blk * KB;
            if constexpr (BITS == 8) {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    uint32_t a0, a1, a2, a3;
                    widen_i8(A[q], a0, a2);
                    widen_i8(B[q], a1, a3);
                    uint2 bv = make_uint2(0, 0);
                    if (xin) bv = *reinterpret_cast<const uint2 *>(xblk + q * 16);
                    mma_bf16(acc[q], a0, a1, a2, a3, bv.x, bv.y);
                }
            } else {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    uint32_t pa[4], pb[4];
                    widen_i4(A[q], pa);
                    widen_i4(B[q], pb);
                    uint2 b0 = make_uint2(0, 0), b1 = make_uint2(0, 0);
                    if (xin) {
                        b0 = *reinterpret_cast<const uint2 *>(xblk + (2 * q) * 16);
                        b1 = *reinterpret_cast<const uint2 *>(xblk + (2 * q + 1) * 16);
                    }
                    mma_bf16(acc[(2 * q) % NCH], pa[0], pb[0], pa[1], pb[1], b0.x, b0.y);
                    mma_bf16(acc[(2 * q + 1) % NCH], pa[2], pb[2], pa[3], pb[3], b1.x, b1.y);
                }
            }
        }
    }

    // ---- fixed-order sum over the K slices, scale, store
    float *red = reinterpret_cast<float *>(smem_raw + p.r_off);   // [WK][RT][M]
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int row = wr * 16 + g + 8 * h;
        const int m0 = 2 * t;
        float s0 = 0.0f, s1 = 0.0f;
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
            s0 += acc[c][2 * h];
            s1 += acc[c][2 * h + 1];
        }
        if (m0 < M) red[(wk * RT + row) * M + m0] = s0;
        if (m0 + 1 < M) red[(wk * RT + row) * M + m0 + 1] = s1;
    }
    __syncthreads();
    if (have_w) {
        for (int idx = threadIdx.x; idx < rows * M; idx += kThreads) {
            const int m = idx / rows, r = idx % rows;   // consecutive threads -> consecutive n
            float s = 0.0f;
            for (int k = 0; k < WK; ++k) s += red[(k * RT + r) * M + m];
            const float y = sws[r] * s;
            const int64_t n = n0 + r;
            if (p.ytype == 0)
                static_cast<float *>(p.Y)[m * p.ldy + n] = y;
            else
                static_cast<uint16_t *>(p.Y)[m * p.ldy + n] = f32_to_bf16_bits(y);
        }
    } else {
        mbar_wait_bounded(wbar, 0, kA16DrainLimit);  // never leave with copies landing in shared memory
    }
}

// Eight output rows per CTA, for products whose 16-row CTAs would leave most
// SMs idle and whose K is too long for 16-row fragments to fit in registers
// (down projection of the decode workload: N = 896, K = 4864 gives 112 CTAs
// instead of 56).  The MMA's rows 8..15 are zeros.  Before the dependency
// wait each warp reads and widens the weights of its run of K blocks into
// registers (at most RB_NF MMA operands of two registers); after it the eight
// warps rotate the token rows' groups into one shared x' (one barrier) and
// each multiplies its run.  M <= 2.
constexpr int RB_ROWS = 8;
constexpr int RB_NF = 40;

struct Rows8Params {
    const uint16_t *X;
    int64_t ldx;
    const uint16_t *U;   // as SmallParams
    int64_t ldu;
    int M;
    int64_t K;
    const uint8_t *W;
    int64_t wld;
    const float *sw;
    int64_t N;
    void *Y;
    int64_t ldy;
    int ytype;
    int WS;                     // shared row stride of the weights (bytes)
    int XK;                     // x' row length (K rounded up to whole blocks)
    int w_off, x_off, r_off;
    unsigned int *status;
};

template <int BITS>
__global__ void __launch_bounds__(kThreads, 2)
k_gemv_rows8(const Rows8Params p) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    constexpr int KB = BITS == 8 ? 64 : 128;    // k per block (one 16-byte chunk per lane)
    constexpr int BB = 64;                      // weight bytes per row per block
    constexpr int QPB = BITS == 8 ? 4 : 8;      // MMAs per block
    constexpr int NBW = RB_NF / QPB;            // blocks per warp at most
    constexpr int W = kThreads / 32;
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem_raw);
    float *sws = reinterpret_cast<float *>(smem_raw + 16);
    unsigned char *ws = smem_raw + p.w_off;
    uint16_t *xs = reinterpret_cast<uint16_t *>(smem_raw + p.x_off);
    float *red = reinterpret_cast<float *>(smem_raw + p.r_off);    // [W][8][M]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t n0 = static_cast<int64_t>(blockIdx.x) * RB_ROWS;
    const int rows = static_cast<int>(min(static_cast<int64_t>(RB_ROWS), p.N - n0));
    const int rbytes = static_cast<int>(p.K * BITS / 8);
    const uint32_t wbar = smem_addr(bar);
    const int nbt = static_cast<int>((p.K + KB - 1) / KB);           // blocks in K
    const int b0 = nbt * warp / W, b1 = nbt * (warp + 1) / W;         // this warp's run
    const int G = static_cast<int>((p.K + kGroup - 1) / kGroup);

    // ---- before the wait: weights, row scales, token rows warmed in L2
    if (warp == 0) {
        if (lane == 0) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(wbar));
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
            // A build for the library's own tests (TQ_TEST_UNSET_BYTES) expects
            // bytes that no copy brings, so the barrier's phase never completes
            // and the bounded waits on it expire: the expiry path is then taken
            // with every issued copy landed, the wait that a CTA keeps for its
            // copies before it exits runs to its full limit, and nothing else
            // changes.
#ifdef TQ_TEST_UNSET_BYTES
            constexpr uint32_t kUnset = TQ_TEST_UNSET_BYTES;
#else
            constexpr uint32_t kUnset = 0;
#endif
            asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(wbar),
                         "r"(static_cast<uint32_t>(rows * rbytes) + kUnset)
                         : "memory");
        }
        __syncwarp();
        for (int r = lane; r < rows; r += 32) {
            asm volatile(
                "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                ::"r"(smem_addr(ws + r * p.WS)), "l"(p.W + (n0 + r) * p.wld),
                  "r"(static_cast<uint32_t>(rbytes)), "r"(wbar)
                : "memory");
        }
    }
    if (threadIdx.x < rows) sws[threadIdx.x] = __ldg(p.sw + n0 + threadIdx.x);
    for (int g = warp; g < G; g += W) {   // coherent L2 prefetch: safe before the wait
        const int64_t k0 = static_cast<int64_t>(g) * kGroup;
        const int64_t k1 = min(k0 + kGroup, p.K);
        for (int m = lane; m < p.M; m += 32) {
            prefetch_l2(p.X + m * p.ldx + k0, static_cast<uint32_t>((k1 - k0) * 2));
            if (p.U) prefetch_l2(p.U + m * p.ldu + k0, static_cast<uint32_t>((k1 - k0) * 2));
        }
    }
    __syncthreads();
    pdl_launch_dependents();

    const bool have_w = mbar_wait_bounded(wbar, 0);
    const int g = lane >> 2, t = lane & 3;
    uint32_t fr[RB_NF][2];                      // row g's widened codes, two k halves
    {
        const bool okA = g < rows;
        const unsigned char *pA = ws + g * p.WS + t * 16;
#pragma unroll
        for (int i = 0; i < NBW; ++i) {
            const int blk = b0 + i;
            const bool in = have_w && okA && blk < b1 && blk * BB + t * 16 < rbytes;
            const uint4 wa = in ? *reinterpret_cast<const uint4 *>(pA + blk * BB) : make_uint4(0, 0, 0, 0);
            const uint32_t A[4] = {wa.x, wa.y, wa.z, wa.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                if constexpr (BITS == 8) {
                    widen_i8(A[q], fr[i * QPB + q][0], fr[i * QPB + q][1]);
                } else {
                    uint32_t pa[4];
                    widen_i4(A[q], pa);
                    fr[i * QPB + 2 * q][0] = pa[0];
                    fr[i * QPB + 2 * q][1] = pa[1];
                    fr[i * QPB + 2 * q + 1][0] = pa[2];
                    fr[i * QPB + 2 * q + 1][1] = pa[3];
                }
            }
        }
    }
    pdl_wait();

    // ---- rotate: warp w takes groups w, w + 8, ... (all their loads first)
    const int M = p.M, XK = p.XK;
    constexpr int GW = 3;                       // groups per warp at most (K <= 24 groups)
    for (int m = 0; m < M; ++m) {
        uint16_t *xrow = xs + m * XK;
        uint4 raw[GW], rawu[GW];
#pragma unroll
        for (int u = 0; u < GW; ++u) {
            const int gi = warp + u * W;
            raw[u] = rawu[u] = make_uint4(0, 0, 0, 0);
            if (gi < G) {
                const int64_t gk = static_cast<int64_t>(gi) * kGroup;
                const int E = group_width(p.K, gk) / 32;
                raw[u] = load_group_raw(p.X + m * p.ldx + gk + lane * E, E);
                if (p.U) rawu[u] = load_group_raw(p.U + m * p.ldu + gk + lane * E, E);
            }
        }
        if (p.U) {
#pragma unroll
            for (int u = 0; u < GW; ++u) raw[u] = swiglu_raw(raw[u], rawu[u]);
        }
#pragma unroll
        for (int u = 0; u < GW; ++u) {
            const int gi = warp + u * W;
            if (gi >= G) break;
            const int gk = gi * kGroup;
            float v[8] = {};
            const int E = fwht_group_raw(raw[u], group_width(p.K, gk), v);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                if (e < E) {
                    const int k = gk + lane * E + e;
                    xrow[(k / KB) * KB + xpos<BITS>(k % KB)] = f32_to_bf16_bits(v[e]);
                }
            }
        }
    }
    const int pad = XK - static_cast<int>(p.K);   // columns of the last block past K
    if (pad > 0) {
        for (int idx = threadIdx.x; idx < M * pad; idx += kThreads) {
            const int m = idx / pad, k = static_cast<int>(p.K) + idx % pad;
            xs[m * XK + (k / KB) * KB + xpos<BITS>(k % KB)] = 0;
        }
    }
    __syncthreads();

    // ---- products on the register fragments
    float acc[NCH][4];
#pragma unroll
    for (int c = 0; c < NCH; ++c) acc[c][0] = acc[c][1] = acc[c][2] = acc[c][3] = 0.0f;
    // token columns >= M read row 0 (valid); their outputs are dropped
    const uint16_t *xb = xs + (g < M ? g : 0) * XK + 4 * t;
    if (have_w) {
#pragma unroll
        for (int i = 0; i < NBW; ++i) {
            const int blk = b0 + i;
            if (blk < b1) {
                const uint16_t *xblk = xb + blk * KB;
#pragma unroll
                for (int q = 0; q < QPB; ++q) {
                    const uint2 bv = *reinterpret_cast<const uint2 *>(xblk + q * 16);
                    mma_bf16(acc[q % NCH], fr[i * QPB + q][0], 0u, fr[i * QPB + q][1], 0u, bv.x, bv.y);
                }
            }
        }
    } else if (lane == 0) {
        atomicOr(p.status, kStatusSmallTimeout);
    }

    // ---- fixed-order sum over the warps' runs, scale, store (rows g; g + 8 are the zero rows)
    {
        const int m0 = 2 * t;
        float s0 = 0.0f, s1 = 0.0f;
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
            s0 += acc[c][0];
            s1 += acc[c][1];
        }
        if (m0 < M) red[(warp * RB_ROWS + g) * M + m0] = s0;
        if (m0 + 1 < M) red[(warp * RB_ROWS + g) * M + m0 + 1] = s1;
    }
    __syncthreads();
    if (have_w) {
        for (int idx = threadIdx.x; idx < rows * M; idx += kThreads) {
            const int m = idx / rows, r = idx % rows;
            float sum = 0.0f;
            for (int w2 = 0; w2 < W; ++w2) sum += red[(w2 * RB_ROWS + r) * M + m];
            const float y = sws[r] * sum;
            const int64_t n = n0 + r;
            if (p.ytype == 0)
                static_cast<float *>(p.Y)[m * p.ldy + n] = y;
            else
                static_cast<uint16_t *>(p.Y)[m * p.ldy + n] = f32_to_bf16_bits(y);
        }
    } else {
        mbar_wait_bounded(wbar, 0, kA16DrainLimit);  // never leave with copies landing in shared memory
    }
}

struct SmallPlan {
    int WR, WK, gpw, WS, XS, w_off, x_off, r_off;
    size_t smem;
};

constexpr size_t kSmallSmemMax = 200 * 1024;

SmallPlan plan_small(int64_t M, int64_t N, int64_t K, int bits, const DeviceInfo &dev) {
    const int64_t G = (K + kGroup - 1) / kGroup;
    SmallPlan pl{};
    // rows per CTA: the most (up to 128) that still give one CTA per SM
    int WR = 1;
    while (WR < 8 && (N + 32 * WR - 1) / (32 * WR) >= dev.sms) WR *= 2;
    pl.WR = WR;
    pl.WK = 8 / WR;
    pl.gpw = static_cast<int>((G + pl.WK - 1) / pl.WK);
    const int RT = 16 * WR;
    const int64_t rb = K * bits / 8;
    pl.WS = static_cast<int>((rb + 127) / 128 * 128 + 64);
    pl.XS = pl.gpw * kGroup + 16;
    pl.w_off = 128 + (4 * RT + 127) / 128 * 128;
    pl.x_off = pl.w_off + RT * pl.WS;
    pl.r_off = pl.x_off + static_cast<int>(8 * M * pl.XS * 2);
    pl.r_off = (pl.r_off + 15) / 16 * 16;
    pl.smem = static_cast<size_t>(pl.r_off) + static_cast<size_t>(pl.WK) * RT * M * 4;
    return pl;
}

struct Rows8Plan {
    int WS, XK, w_off, x_off, r_off;
    size_t smem;
    bool ok;
};

// The eight-row kernel takes M <= 2, K within eight warps' runs of blocks and
// at most three groups per warp, and few enough rows to stay within two CTAs
// per SM.
Rows8Plan plan_rows8(int64_t M, int64_t N, int64_t K, int bits, const DeviceInfo &dev) {
    Rows8Plan pl{};
    const int64_t KB = bits == 8 ? 64 : 128;
    const int64_t nbt = (K + KB - 1) / KB;
    const int64_t nbw = RB_NF / (bits == 8 ? 4 : 8);
    const int64_t G = (K + kGroup - 1) / kGroup;
    pl.ok = M >= 1 && M <= 2 && nbt <= 8 * nbw && G <= 24 &&
            (N + RB_ROWS - 1) / RB_ROWS <= 2 * static_cast<int64_t>(dev.sms);
    const int64_t rb = K * bits / 8;
    pl.WS = static_cast<int>((rb + 127) / 128 * 128 + 64);
    pl.XK = static_cast<int>(nbt * KB);
    pl.w_off = 128;
    pl.x_off = pl.w_off + RB_ROWS * pl.WS;
    pl.r_off = (pl.x_off + static_cast<int>(M * pl.XK * 2) + 15) / 16 * 16;
    pl.smem = static_cast<size_t>(pl.r_off) + static_cast<size_t>(kThreads / 32) * RB_ROWS * M * 4;
    pl.ok = pl.ok && pl.smem <= kSmallSmemMax;
    return pl;
}

tq_status launch_rows8(const uint16_t *X, int64_t M, int64_t K, int64_t ldx, const uint8_t *Wq,
                       const float *sw, int64_t N, int bits, void *Y, int ytype, int64_t ldy,
                       const Rows8Plan &pl, const DeviceInfo &dev, cudaStream_t s, const uint16_t *U,
                       int64_t ldu) {
    unsigned int *status = status_word();
    if (!status) return TQ_ERR_DEVICE;
    Rows8Params p{};
    p.X = X;
    p.ldx = ldx;
    p.U = U;
    p.ldu = ldu;
    p.M = static_cast<int>(M);
    p.K = K;
    p.W = Wq;
    p.wld = bits == 8 ? K : K / 2;
    p.sw = sw;
    p.N = N;
    p.Y = Y;
    p.ldy = ldy;
    p.ytype = ytype;
    p.WS = pl.WS;
    p.XK = pl.XK;
    p.w_off = pl.w_off;
    p.x_off = pl.x_off;
    p.r_off = pl.r_off;
    p.status = status;
    auto kern = bits == 8 ? k_gemv_rows8<8> : k_gemv_rows8<4>;
    static int configured_for[64][2] = {{0}};
    const int bi = bits == 8 ? 0 : 1;
    if (dev.id < 0 || dev.id >= 64) return TQ_ERR_DEVICE;
    if (!configured_for[dev.id][bi]) {
        const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   static_cast<int>(kSmallSmemMax));
        if (e != cudaSuccess) return cuda_fail(e);
        configured_for[dev.id][bi] = 1;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>((N + RB_ROWS - 1) / RB_ROWS), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = pl.smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, p);
    return e == cudaSuccess ? TQ_OK : cuda_fail(e);
}

}  // namespace

bool gemv_small_fits(int64_t M, int64_t N, int64_t K, int bits, const DeviceInfo &dev) {
    if (M < 1 || M > 8) return false;
    return plan_small(M, N, K, bits, dev).smem <= kSmallSmemMax;
}

bool gemv_decode_fits(int64_t M, int64_t N, int64_t K, int bits, const DeviceInfo &dev) {
    if (M < 1 || M > 8) return false;
    const SmallPlan pl = plan_small(M, N, K, bits, dev);
    if (pl.gpw > 1 && plan_rows8(M, N, K, bits, dev).ok) return true;
    return pl.smem <= kSmallSmemMax;
}

tq_status launch_gemv_small(const uint16_t *X, int64_t M, int64_t K, int64_t ldx,
                            const uint8_t *Wq, const float *sw, int64_t N, int bits,
                            void *Y, int ytype, int64_t ldy, const DeviceInfo &dev,
                            cudaStream_t s, const uint16_t *U, int64_t ldu) {
    const SmallPlan pl = plan_small(M, N, K, bits, dev);
    if (pl.gpw > 1) {   // 16-row fragments would not fit: eight rows per CTA if the shape allows
        const Rows8Plan r8 = plan_rows8(M, N, K, bits, dev);
        if (r8.ok) return launch_rows8(X, M, K, ldx, Wq, sw, N, bits, Y, ytype, ldy, r8, dev, s, U, ldu);
    }
    if (pl.smem > kSmallSmemMax) return TQ_ERR_SHAPE;
    unsigned int *status = status_word();
    if (!status) return TQ_ERR_DEVICE;
    SmallParams p{};
    p.X = X;
    p.ldx = ldx;
    p.U = U;
    p.ldu = ldu;
    p.M = static_cast<int>(M);
    p.K = K;
    p.G = static_cast<int>((K + kGroup - 1) / kGroup);
    p.W = Wq;
    p.wld = bits == 8 ? K : K / 2;
    p.sw = sw;
    p.N = N;
    p.Y = Y;
    p.ldy = ldy;
    p.ytype = ytype;
    p.WR = pl.WR;
    p.WK = pl.WK;
    p.gpw = pl.gpw;
    p.WS = pl.WS;
    p.XS = pl.XS;
    p.w_off = pl.w_off;
    p.x_off = pl.x_off;
    p.r_off = pl.r_off;
    p.status = status;
    // weight fragments in registers when every warp's slice is one group
    const bool pre = pl.gpw == 1;
    auto kern = bits == 8 ? (pre ? k_gemv_small<8, true> : k_gemv_small<8, false>)
                          : (pre ? k_gemv_small<4, true> : k_gemv_small<4, false>);
    static int configured_for[64][4] = {{0}};
    const int bi = (bits == 8 ? 0 : 2) + (pre ? 1 : 0);
    if (dev.id >= 0 && dev.id < 64 && !configured_for[dev.id][bi]) {
        const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   static_cast<int>(kSmallSmemMax));
        if (e != cudaSuccess) return cuda_fail(e);
        configured_for[dev.id][bi] = 1;
    }
    const int64_t tiles = (N + 16 * pl.WR - 1) / (16 * pl.WR);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(tiles), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = pl.smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, p);
    return e == cudaSuccess ? TQ_OK : cuda_fail(e);
}

}  // namespace tq
