/*
 * tq.h -- rotated low-bit linear projection on GB300 (sm_103a), C ABI.
 *
 * The method.  Weight rows are rotated by a normalised Hadamard matrix over
 * every group of 256 input columns and quantised to int8 (or int4) with one
 * fp32 scale per output row; the matching input rows get the same rotation,
 * so the product is unchanged (tensai docs, "画像生成" / Image generation,
 * sections "チェックポイントの入手" and "幅とメモリ").  The formats are
 * TensorPencil's "INT8 ConvRot" and "INT4 ConvRot" (README, "Details").
 *
 * Readings where the pages are silent, fixed by this library:
 *   - H is Sylvester's matrix, Hs[i][j] = (-1)^popcount(i & j), times
 *     c_n = 1/sqrt(n), so H is symmetric and orthogonal.
 *   - K is 256*q + t with t in {0, 32, 64, 128}; the last group of width
 *     t < 256 uses its own H_t.
 *   - Quantisation is symmetric, nearest-even: s = fp32(amax / qmax),
 *     q = clamp(rint(v' / s), -qmax, qmax), qmax = 127 (8-bit) or 7 (4-bit).
 *     A zero row (or one whose scale rounds to 0 in fp32) has s = 0 and all
 *     codes 0.
 *   - int4 codes are packed two per byte along K: byte k/2 holds code k (even
 *     k) in its low nibble and code k+1 in its high nibble, two's complement.
 *   - A8 activations: one int8 scale per token row over all of K (the pages
 *     say only that the device quantises each product's activations finely;
 *     tensai docs, section "GPU").
 *   - A16 activations: the rotated row rounded to bf16 (nearest even).
 *
 * Conventions for every entry point.
 *   - Every pointer is device memory owned by the caller (allocated, for
 *     example, by PyTorch).  The library never allocates or frees device
 *     memory and runs everything asynchronously on `stream` (0 = the legacy
 *     default stream).  Two calls synchronise the host, and only they: the
 *     set-up call tq_grouped_create (it copies its tables into the caller's
 *     buffer) and tq_device_status (it waits for `stream` before it reads
 *     the status word).  Every product and quantiser call returns as soon as
 *     its launches are queued.
 *   - All checks (null pointers, shapes, strides, alignment, 64-bit size
 *     overflow, enum values) happen on the host before any launch; a refused
 *     call launches nothing and returns the status naming the reason.
 *   - A launch error is returned as TQ_ERR_CUDA; tq_last_cuda_error() gives
 *     the CUDA error code.
 *   - M == 0 or N == 0 is an empty call: TQ_OK, nothing launched.
 *   - Inputs must be finite; non-finite bf16 inputs give unspecified codes.
 *   - Strided inputs are honoured: X row m starts at X + m * ldx elements.
 *   - Results are deterministic: the same inputs give the same bytes.
 */
#ifndef TQ_H
#define TQ_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    TQ_OK = 0,
    TQ_ERR_NULL = 1,        /* a required pointer is NULL */
    TQ_ERR_SHAPE = 2,       /* M, N, K, a stride or the group width is not allowed */
    TQ_ERR_BITS = 3,        /* bits is not 8 or 4 */
    TQ_ERR_MODE = 4,        /* unknown mode / output type, bits disagree with mode, or eps out of range */
    TQ_ERR_OVERFLOW = 5,    /* a size product overflows 64 bits or a kernel index */
    TQ_ERR_ALIGN = 6,       /* a pointer or stride breaks the alignment rule */
    TQ_ERR_WORKSPACE = 7,   /* workspace missing or smaller than required */
    TQ_ERR_CUDA = 8,        /* a CUDA call failed (see tq_last_cuda_error) */
    TQ_ERR_DEVICE_TIMEOUT = 9, /* a bounded device-side wait expired */
    TQ_ERR_DEVICE = 10      /* no usable sm_103 device is current */
} tq_status;

typedef enum {
    TQ_W8A16 = 0,  /* int8 weights x rotated bf16 activations, fp32 sums */
    TQ_W4A16 = 1,  /* int4 weights x rotated bf16 activations, fp32 sums */
    TQ_W8A8 = 2    /* int8 (bits=8) or int4 (bits=4) weights x int8 activations */
} tq_mode;

typedef enum {
    TQ_OUT_F32 = 0,
    TQ_OUT_BF16 = 1,
    TQ_OUT_I32 = 2  /* tq_linear_q8 and tq_linear_tiled only: the raw int32 sums */
} tq_out;

/* Largest K any entry point accepts. */
#define TQ_MAX_K 65536
/* Largest M the A16 modes accept (the skinny decode kernel). */
#define TQ_MAX_M_A16 64

/*
 * Human-readable name of a status, naming the refused condition (the pages
 * refuse a size a format cannot take by name before any work starts: kvad-gpu
 * internals, "Quantised weights on the GPU"; TensorFold PR #948, review
 * follow-up: overflowing size products refused by name).  Never NULL.
 */
const char *tq_status_str(tq_status s);

/* CUDA error code of the most recent TQ_ERR_CUDA on this host thread. */
int tq_last_cuda_error(void);

/* Library version, major * 10000 + minor * 100 + patch. */
int tq_version(void);

/*
 * Weight rotate + quantise + pack (one-time; tensai docs, "画像生成",
 * section "チェックポイントの入手").
 *
 *   W       bf16 [N, K], row n at W + n * ldw elements; ldw >= K,
 *           ldw % 8 == 0, W 16-byte aligned.
 *   bits    8 or 4.
 *   group   must be 256 (the group width of the method).
 *   codes   bits = 8: int8 [N, K] dense (row stride K).
 *           bits = 4: packed bytes [N, K / 2] dense, layout above.
 *           16-byte aligned.
 *   scales  fp32 [N], 4-byte aligned.
 * Codes and scales are bit-exact with an fp64 explicit-product reference for
 * every row whose group sums are exact in fp64 (true whenever a group's
 * nonzero magnitudes span fewer than about 37 binades).
 */
tq_status tq_quantize_weights(const void *W, int64_t N, int64_t K, int64_t ldw,
                              int bits, int group, void *codes, float *scales,
                              cudaStream_t stream);

/*
 * Activation rotation (256-wide fast Walsh-Hadamard transform, fp32) fused
 * with per-token symmetric int8 quantisation (tensai docs, "画像生成", sections
 * "幅とメモリ" and "GPU").
 *
 *   X   bf16 [M, K], row m at X + m * ldx; ldx >= K, ldx % 8 == 0,
 *       X 16-byte aligned.
 *   Xq  int8 [M, K] dense, 16-byte aligned.
 *   sx  fp32 [M]: the token scales, s = amax / 127.
 * The transform sums in fp32, so a code may differ by one from the fp64
 * reference where the sum lands within rounding of a .5 boundary.
 */
tq_status tq_rotate_quant_act(const void *X, int64_t M, int64_t K, int64_t ldx,
                              int8_t *Xq, float *sx, cudaStream_t stream);

/*
 * Activation rotation rounded to bf16: the A16 operand (same passages).
 *   X   as tq_rotate_quant_act.
 *   Xr  bf16 [M, K] dense, 16-byte aligned.
 */
tq_status tq_rotate_act_bf16(const void *X, int64_t M, int64_t K, int64_t ldx,
                             void *Xr, cudaStream_t stream);

/*
 * Bytes of workspace tq_linear needs for these sizes (0 when none; for the
 * A16 modes, the bytes of the optional tensor-core operand).  The
 * projections are about 80% of a DiT step's GPU time (TensorFold PR #948,
 * "What comes next" and "Receipts").
 */
size_t tq_linear_workspace_bytes(int64_t M, int64_t K, int64_t N, int bits,
                                 tq_mode mode);

/*
 * The rotated low-bit linear projection: Y[m][n] = sum_k W[n][k] x[m][k],
 * computed on the rotated, quantised operands.
 *
 *   X        bf16 [M, K] (unrotated), layout as tq_rotate_quant_act.
 *   Wq, sw   codes and row scales from tq_quantize_weights with `bits`.
 *   mode     TQ_W8A16 (bits = 8) or TQ_W4A16 (bits = 4): M <= 64; the
 *            rotated activations are rounded to bf16 and multiplied with the
 *            weight codes in fp32, Y = sw[n] * sum_k q_w x'_bf16.
 *            TQ_W8A8 (bits = 8 or 4): activations are quantised per token
 *            (tq_rotate_quant_act) and Y = sx[m] * sw[n] * acc[m][n], acc the
 *            exact int32 sum of code products.
 *   Y        fp32 or bf16 [M, N], row m at Y + m * ldy; ldy >= N; Y aligned
 *            to its element size.
 *   workspace, ws_bytes   device scratch of at least
 *            tq_linear_workspace_bytes(M, K, N, bits, mode) bytes, 256-byte
 *            aligned (may be NULL when that is 0).  Its contents on entry do
 *            not matter; the call overwrites it.
 *            TQ_W8A8: required.  A16 modes: optional.  Up to 16 token rows
 *            over weights of at least 2^24 codes that fill the GPU in one
 *            wave run the split-K product (clusters of CTAs along K, each
 *            rotating its own run of the input; no workspace).  Otherwise,
 *            with the workspace, products of more than 8 token rows, or of
 *            such weights with 3 to 8 token rows, run on the tensor cores
 *            (the rotated rows are first written to the workspace as fp16
 *            tiles, each token scaled by a power of two, which keeps every
 *            bf16 value exact); without it (or smaller than that size) the
 *            CUDA-core kernels run.  All compute the same Y within fp32
 *            rounding.  Calls in order on one stream may share a workspace
 *            (the next call's weights stream early, but its operand is
 *            written only after this call ends); calls on different streams
 *            need their own.
 */
tq_status tq_linear(const void *X, int64_t M, int64_t K, int64_t ldx,
                    const void *Wq, const float *sw, int64_t N, int bits,
                    tq_mode mode, void *Y, tq_out ytype, int64_t ldy,
                    void *workspace, size_t ws_bytes, cudaStream_t stream);

/*
 * The A8 product on activations that are already rotated and quantised
 * (tq_rotate_quant_act): Y = sx[m] * sw[n] * acc[m][n].  The int8 x int8
 * product of the rotated operands (tensai docs, "画像生成", section "幅とメモリ":
 * both operands rotated, so the product is unchanged; section "GPU": the
 * device quantises each product's activations).  Splitting the rotation and
 * the product lets one quantised input serve several products.
 *   Xq   int8 [M, K] dense, 16-byte aligned;  sx fp32 [M].
 *   ytype TQ_OUT_I32 writes acc itself (int32 [M, N], ldy as for fp32).
 */
tq_status tq_linear_q8(const int8_t *Xq, const float *sx, int64_t M, int64_t K,
                       const void *Wq, const float *sw, int64_t N, int bits,
                       void *Y, tq_out ytype, int64_t ldy, cudaStream_t stream);

/* Longest row (K) the tiled activation operand takes. */
#define TQ_MAX_K_TILED 16384

/*
 * Bytes of the tiled activation operand of an M x K input: 0 when K is not a
 * valid row length or is above TQ_MAX_K_TILED.
 */
size_t tq_act_tiled_bytes(int64_t M, int64_t K);

/*
 * tq_rotate_quant_act writing its codes in the A8 product's own operand form
 * ("tiled"): the same codes and token scales (same passages), stored as fp16
 * in 128-row x 64-column tiles laid out as the tensor cores read them, so the
 * product loads each tile with one copy.  A caller that multiplies one input
 * by several weight matrices (the query/key/value or gate/up projections of a
 * DiT block) rotates and quantises it once.
 *   X        as tq_rotate_quant_act; K <= TQ_MAX_K_TILED.
 *   At       at least tq_act_tiled_bytes(M, K) bytes, 256-byte aligned; its
 *            layout is private to this library (read it only through
 *            tq_linear_tiled).
 *   sx       fp32 [M]: the token scales.
 */
tq_status tq_rotate_quant_act_tiled(const void *X, int64_t M, int64_t K, int64_t ldx, void *At,
                                    size_t at_bytes, float *sx, cudaStream_t stream);

/*
 * The SwiGLU row kernel fused with tq_rotate_quant_act_tiled: the input of a
 * down projection, h = bf16(silu(G) * U) with silu(g) = g / (1 + e^-g) (the
 * gated unit of Shazeer, "GLU Variants Improve Transformer", 2020), rotated
 * and quantised per token into the tiled operand.  The pages name SwiGLU among
 * the row kernels next to the projections, candidates for fusion (TensorFold
 * PR #948, "What comes next").  Fused, h (bf16 [M, K]) is neither written nor
 * read again.  silu and the product are computed in fp32 and rounded to bf16,
 * as an unfused SwiGLU kernel would store h.  So a code may differ by one from
 * the fp64 reference, as for tq_rotate_quant_act.
 *   G, U   bf16 [M, K], rows at G + m * ldg and U + m * ldu (for example the
 *          two halves of a fused gate/up product's output: U = G + K, both
 *          strides 2K); each follows tq_rotate_quant_act's rules for X.
 *   At, at_bytes, sx   as tq_rotate_quant_act_tiled.
 */
tq_status tq_swiglu_quant_act_tiled(const void *G, int64_t ldg, const void *U, int64_t ldu, int64_t M,
                                    int64_t K, void *At, size_t at_bytes, float *sx, cudaStream_t stream);

/*
 * The modulated layer norm fused with tq_rotate_quant_act_tiled: the input of
 * a DiT block's query/key/value or gate/up projection,
 *   h = bf16((x - mu) / sqrt(var + eps) * (1 + scale) + shift),
 * mu and var the mean and biased variance of the row x (a layer norm with no
 * affine parameters of its own, modulated as in the adaptive layer norm of
 * Peebles and Xie, "Scalable Diffusion Models with Transformers", 2023),
 * rotated and quantised per token into the tiled operand.  The pages name the
 * modulated layer norm among the row kernels next to the projections,
 * candidates for fusion, and keep norms in fp32 (TensorFold PR #948, "What
 * comes next" and its precision list); the modulation is shared by every
 * block (same PR, "What it adds").  Fused, h (bf16 [M, K]) is neither
 * written nor read again.  mu, var and h are computed in fp32 (two passes
 * over the row held in registers) and h is rounded to bf16, as an unfused
 * norm kernel would store it.  So a code may differ by one from the fp64
 * reference, as for tq_rotate_quant_act.
 *   X          as tq_rotate_quant_act; K <= TQ_MAX_K_TILED.
 *   shift, scale  fp32 [K], 16-byte aligned: one modulation for all M rows
 *              (rows with different modulations, such as the prompt rows and
 *              image rows of a step, are separate calls).
 *   eps        added to the variance; finite and >= 0, else TQ_ERR_MODE
 *              (DiT blocks use 1e-6).
 *   At, at_bytes, sx   as tq_rotate_quant_act_tiled.
 */
tq_status tq_modnorm_quant_act_tiled(const void *X, int64_t M, int64_t K, int64_t ldx, const float *shift,
                                     const float *scale, float eps, void *At, size_t at_bytes, float *sx,
                                     cudaStream_t stream);

/*
 * The decode product (A16 modes, M <= 8 tokens) of the SwiGLU of two rows:
 * Y = the rotated low-bit product of h = bf16(silu(G) * U), silu(g) =
 * g / (1 + e^-g), with (Wq, sw).  The down projection of a gated FFN layer
 * takes h made from its gate and up outputs; fused, h is formed as the
 * decode kernel loads its input (the same arithmetic as
 * tq_swiglu_quant_act_tiled), so a layer's gate+up call can feed its down
 * call directly.  The pages name SwiGLU among the row kernels beside the
 * projections, candidates for fusion (TensorFold PR #948, "What comes
 * next"), and decode as one projection at a time, each input the previous
 * output (kvad-gpu internals, "Numbers").
 *   G, U     bf16 [M, K], rows at G + m * ldg and U + m * ldu (for example
 *            the two halves of a fused gate+up output row: U = G + K); each
 *            follows tq_rotate_quant_act's rules for X.
 *   mode     TQ_W8A16 or TQ_W4A16 (bits to match); other arguments as
 *            tq_linear.  Shapes the decode kernels do not take (M > 8, or K
 *            past their shared-memory plan) are refused with TQ_ERR_SHAPE.
 */
tq_status tq_linear_swiglu(const void *G, int64_t ldg, const void *U, int64_t ldu, int64_t M, int64_t K,
                           const void *Wq, const float *sw, int64_t N, int bits, tq_mode mode, void *Y,
                           tq_out ytype, int64_t ldy, cudaStream_t stream);

/*
 * The A8 product on a tiled operand: as tq_linear_q8 with At, sx from
 * tq_rotate_quant_act_tiled (same M and K) in place of Xq, sx.
 */
tq_status tq_linear_tiled(const void *At, const float *sx, int64_t M, int64_t K, const void *Wq,
                          const float *sw, int64_t N, int bits, void *Y, tq_out ytype, int64_t ldy,
                          cudaStream_t stream);

/*
 * Bytes of the tiled weight operand (tq_tile_weights) of an N x K matrix: 0
 * when K is not a valid row length or is above TQ_MAX_K_TILED.
 */
size_t tq_weights_tiled_bytes(int64_t N, int64_t K);

/*
 * The weight codes of tq_quantize_weights (with `bits`) widened once into the
 * A8 product's own operand form.  The values are fp16, which holds the small
 * integer codes exactly.  They sit in 128-row x 64-column tiles laid out as the
 * tensor cores read them, with rows padded to 256 and columns to 64 by zeros.
 * sm_103a has no integer tensor-core MMA, so the product otherwise widens the
 * codes of every weight tile for every tile of activations.  With the tiled
 * form it copies both operands straight into its stages instead.  The cost is
 * device memory: twice the bytes of 8-bit codes, four times those of 4-bit
 * codes.  A set-up step, run once per weight matrix like tq_quantize_weights;
 * the pages have no counterpart.
 *   Wq      codes [N, K] as written by tq_quantize_weights, 16-byte aligned.
 *   Wt      at least tq_weights_tiled_bytes(N, K) bytes, 256-byte aligned; its
 *           layout is private to this library (read it through tq_linear_tt).
 *           After the tiles it records the rows' largest sum of codes
 *           squared. With the activations' own, the product then knows when
 *           one fp32 accumulation over all of K stays exact (Cauchy-Schwarz).
 */
tq_status tq_tile_weights(const void *Wq, int64_t N, int64_t K, int bits, void *Wt,
                          size_t wt_bytes, cudaStream_t stream);

/*
 * The A8 product with both operands in the tiled form: as tq_linear_tiled,
 * with Wt from tq_tile_weights (same N, K and bits) in place of Wq.  The
 * results are the same: the exact int32 sums and Y = sx[m] * sw[n] * acc.
 */
tq_status tq_linear_tt(const void *At, const float *sx, int64_t M, int64_t K, const void *Wt,
                       const float *sw, int64_t N, int bits, void *Y, tq_out ytype, int64_t ldy,
                       cudaStream_t stream);

/*
 * Optional epilogue of the A8 product (tq_linear_tt_ex), computed in fp32:
 *   Y[m][n] = R[m][n] + gate[n] * (sx[m] * sw[n] * acc[m][n] + bias[n]).
 * Each of bias, gate and R may be absent: absent bias adds 0, absent gate is
 * 1, absent R is 0.  This is a DiT block's gated residual, one of the row
 * kernels next to the projections that the pages list as candidates for
 * fusion (TensorFold PR #948, "What comes next").  Fused, the projection's
 * output is never written and re-read by a separate kernel.
 */
typedef struct {
    const float *bias;      /* fp32 [N], or NULL; 4-byte aligned */
    const float *gate;      /* fp32 [N], or NULL; 4-byte aligned */
    const void *residual;   /* [M, N] of rtype, row m at residual + m * ldr, or NULL.  It may
                               be Y itself (an in-place update; then ldr == ldy and rtype ==
                               ytype), but must not otherwise overlap Y */
    int64_t ldr;            /* residual row stride (elements), >= N */
    tq_out rtype;           /* TQ_OUT_F32 or TQ_OUT_BF16 */
} tq_epilogue;

/*
 * tq_linear_tt with an epilogue.  epi == NULL is tq_linear_tt itself; with an
 * epilogue, ytype is TQ_OUT_F32 or TQ_OUT_BF16 (not the raw int32 sums).
 */
tq_status tq_linear_tt_ex(const void *At, const float *sx, int64_t M, int64_t K, const void *Wt,
                          const float *sw, int64_t N, int bits, const tq_epilogue *epi, void *Y,
                          tq_out ytype, int64_t ldy, cudaStream_t stream);

/*
 * Bytes of the split workspace of tq_linear_tt_split on the current device (0
 * when no usable device is current).  It does not depend on the sizes of a
 * call: one workspace serves every product that runs on one stream.
 */
size_t tq_split_workspace_bytes(void);

/*
 * tq_linear_tt_ex with the tiles of the last wave split along K.  The
 * projections are most of a DiT step (TensorFold PR #948, "What comes next":
 * about 80% of the GPU time); a product whose 256 x 256 output tiles leave the
 * last wave of CTA pairs partly idle (the down projection of a 1024-token
 * block is 48 tiles, of a 4032-token one 192 = 2 x 76 + 40) spends that share
 * of its time with part of the tensor cores unused.  With a workspace, the
 * tiles of the whole waves stay whole and the K steps of the last wave's
 * tiles are shared evenly by every pair; a pair that holds only part of a
 * tile stores its exact int32 partial sums, and the pair that holds the
 * tile's last K step adds them before the epilogue.  The sums are integers, so
 * the result is bit-identical to tq_linear_tt_ex, whatever the split (the
 * library decides it from the tile count and K: long K only, where it was
 * measured to pay).
 *
 *   workspace  tq_split_workspace_bytes() bytes of device memory, 256-byte
 *              aligned, ZEROED before its first use (cudaMemsetAsync).  Every
 *              call that completes leaves it zeroed again.  After a call
 *              returned TQ_ERR_DEVICE_TIMEOUT from tq_device_status, zero it
 *              again before reuse.  Calls that may run at the same time on
 *              the GPU (different streams) need workspaces of their own.
 *              NULL: no split (tq_linear_tt_ex).
 * Other arguments as tq_linear_tt_ex.  TQ_ERR_WORKSPACE if ws_bytes is too
 * small, TQ_ERR_ALIGN if the workspace is not 256-byte aligned.
 */
tq_status tq_linear_tt_split(const void *At, const float *sx, int64_t M, int64_t K, const void *Wt,
                             const float *sw, int64_t N, int bits, const tq_epilogue *epi, void *Y,
                             tq_out ytype, int64_t ldy, void *workspace, size_t ws_bytes,
                             cudaStream_t stream);

/*
 * Block-scaled weights: one fp32 scale per block of G input columns instead
 * of one per row.  These are the blocks with a shared scale of the GGML
 * formats (Q8_0 and Q4_0, 32 wide) and of kvad's own q8 (an fp32 scale per 32
 * weights; kvad-gpu internals, "Quantised weights on the GPU").  On rotated
 * weights they win back the 4-bit accuracy that one scale per row loses,
 * since the rotation lowers 4-bit's error less than 8-bit's (tensai docs,
 * "画像生成", section "幅とメモリ").
 *
 * The blocks are taken either of the rotated row (rotate = 1, the rotation of
 * tq_quantize_weights) or of the bf16 weights as they are (rotate = 0, the
 * unrotated format).  Block b of row n gets s = fp32(amax_b / qmax) and
 * codes rint(v / s), exactly as tq_quantize_weights does for a whole row, so
 * the codes and scales are bit-exact with the fp64 reference under the same
 * condition.
 *
 *   W       as tq_quantize_weights.
 *   K       a valid row length (K = 256 q + t, t in {0, 32, 64, 128}), with
 *           K % G == 0.
 *   bits    8 or 4.
 *   G       32, 64, 128 or 256.  Other values give TQ_ERR_SHAPE.
 *   rotate  1 or 0.  Other values give TQ_ERR_MODE.
 *   codes   as tq_quantize_weights.
 *   scales  fp32 [N, K / G], row n at scales + n * (K / G); 4-byte aligned.
 */
tq_status tq_quantize_weights_blocked(const void *W, int64_t N, int64_t K, int64_t ldw, int bits, int G,
                                      int rotate, void *codes, float *scales, cudaStream_t stream);

/* Largest M tq_linear_blocked accepts. */
#define TQ_MAX_M_BLOCKED 8

/*
 * Decode product on block-scaled weights:
 *   Y[m][n] = sum_b s[n][b] * sum_{k in block b} q[n][k] * x[m][k]
 * with fp32 sums.  x is the token row's rotation rounded to bf16 when
 * rotate = 1 (the product's own rotation, as tq_rotate_act_bf16 computes it),
 * and the bf16 row itself when rotate = 0.  rotate and G must be those the
 * weights were quantised with.
 *
 *   X        bf16 [M, K] (unrotated), layout as tq_rotate_quant_act;
 *            0 <= M <= TQ_MAX_M_BLOCKED.
 *   Wq, sw   from tq_quantize_weights_blocked.
 *   Y        fp32 or bf16 [M, N], row m at Y + m * ldy; ldy >= N; aligned to
 *            its element size.
 * The token rows are held in shared memory as fp32: the M rounded up to a
 * power of two, times K, times 4 bytes, must fit one CTA's shared memory
 * (227 KB on sm_103), else TQ_ERR_SHAPE.  M == 0 or N == 0 is no work.
 */
tq_status tq_linear_blocked(const void *X, int64_t M, int64_t K, int64_t ldx, const void *Wq, const float *sw,
                            int G, int64_t N, int bits, int rotate, void *Y, tq_out ytype, int64_t ldy,
                            cudaStream_t stream);

/*
 * Synchronises `stream`, then reads and clears the library's device status
 * word on the current device.  Returns TQ_ERR_DEVICE_TIMEOUT if a bounded
 * device-side wait expired in any call since the last check (that call's
 * output is then invalid), TQ_ERR_CUDA on a CUDA error, else TQ_OK.
 *
 * The pages' runtimes report a failure as a named error the caller can act
 * on rather than stopping (TensorFold PR #948, review follow-up: errors such
 * as error.ScratchTooLarge returned by name).  A device-side wait cannot
 * return to the host, so the kernels record an expired wait here instead of
 * trapping, which keeps the CUDA context usable.  This is the one call
 * besides tq_grouped_create that synchronises the host.
 */
tq_status tq_device_status(cudaStream_t stream);

/* Bytes of device memory the library keeps for tq_linear_a8_static. */
#define TQ_STATIC_SCRATCH_BYTES (16u << 20)

/*
 * tq_linear in mode TQ_W8A8 (bits = 8 or 4) without a workspace argument,
 * for callers that cannot allocate device memory.  The pages have no
 * counterpart: this is a library convenience.
 *
 * tq_linear needs scratch for the quantised activations and expects the
 * caller to pass it.  A plugin whose host application owns every device
 * allocation, or a service that reserves all device memory at start-up and
 * may not allocate afterwards, has none to pass.  This entry point instead
 * uses one fixed array of TQ_STATIC_SCRATCH_BYTES compiled into the library;
 * each GPU that loads the library holds that memory until the process exits.
 * It allocates nothing and frees nothing.
 *
 *   Arguments and results are those of tq_linear with mode TQ_W8A8.
 *   Limit: the int8 codes (M * K bytes) and the token scales (4 * M bytes),
 *   each rounded up to 256 bytes, must fit in TQ_STATIC_SCRATCH_BYTES; larger
 *   calls are refused with TQ_ERR_WORKSPACE before any launch.
 *   Set-up: the first call on a device looks up the array's device address
 *   (with that device current); make that first call before any stream
 *   capture.  The lookup is repeated if the device's CUDA context has been
 *   replaced since (after cudaDeviceReset, for example).
 *   Sharing: every call uses the same array and leaves its contents there.
 *   Nothing in it has to start at zero (each call writes what it reads), but
 *   calls that overlap on the GPU (for example on two streams) race on it:
 *   keep them ordered, for example on one stream.
 */
tq_status tq_linear_a8_static(const void *X, int64_t M, int64_t K, int64_t ldx,
                              const void *Wq, const float *sw, int64_t N, int bits,
                              void *Y, tq_out ytype, int64_t ldy,
                              cudaStream_t stream);

/*
 * Grouped A16 product: many independent calls of tq_linear in mode TQ_W8A16
 * or TQ_W4A16 run as one pass over their weights.
 *
 * Decode is bound by the weight stream (kvad-gpu internals, "Numbers"), but a
 * call of a small model moves a few MB, and a call launched on its own must
 * wait for the previous one before it reads its input: at that size the chain
 * of waits, not the stream, sets the time.  Calls that do not depend on one
 * another (the gate and up projections of a layer, or the calls of a batch of
 * independent requests) can share one stream: the plan rotates every call's
 * input once, then one CTA per SM streams the calls' weight rows through
 * shared memory while the others compute.  The pages have no counterpart;
 * the arithmetic of each call is that of tq_linear.
 *
 * Each call computes Y[m][n] = sw[n] * sum_k q_w[n][k] x'_bf16[m][k] with
 * fp32 sums (same passages as tq_linear).  The order of the fp32 sums differs
 * from tq_linear's, so the two agree to rounding, not bit for bit; a plan
 * gives the same bytes on every run.
 */

/* Most token rows of one call in a grouped plan. */
#define TQ_MAX_M_GROUPED 8

/* One call of a grouped plan: the arguments of tq_linear in an A16 mode. */
typedef struct {
    const void *X;      /* bf16 [M, K], rules of tq_linear (16-byte aligned, ldx % 8 == 0) */
    int64_t ldx;
    const void *Wq;     /* codes from tq_quantize_weights with the plan's bits */
    const float *sw;    /* fp32 [N] row scales */
    void *Y;            /* [M, N] of the plan's output type, row m at Y + m * ldy */
    int64_t ldy;
    int64_t M, N, K;    /* 0 <= M <= TQ_MAX_M_GROUPED; M == 0 or N == 0: no work */
} tq_a16_call;

/* A plan (host handle; its device tables live in the caller's buffer). */
typedef struct tq_grouped_s *tq_grouped;

/*
 * Bytes of device memory a plan of these calls needs (tables and the rotated
 * inputs, about 128 bytes per 96 KB of weights plus 2 * M * K bytes per call).
 * Refusals are those of tq_grouped_create (no device is needed).
 */
tq_status tq_grouped_bytes(const tq_a16_call *calls, int64_t ncalls, int bits, size_t *bytes);

/*
 * Checks every call and writes the plan's tables into `dmem`.
 *   calls, ncalls  host array of the calls (copied; the array may be reused).
 *   bits           8 (TQ_W8A16) or 4 (TQ_W4A16) for every call.
 *   ytype          TQ_OUT_F32 or TQ_OUT_BF16 for every call.
 *   dmem, dbytes   device buffer of at least tq_grouped_bytes(...) bytes,
 *                  256-byte aligned, owned by the caller; it must outlive the
 *                  plan and not be touched while the plan exists.
 *   plan           receives the handle.
 * Each call follows tq_linear's rules for X, Wq, sw, Y and its strides, with
 * M <= TQ_MAX_M_GROUPED; in addition one work item (8 weight rows and the
 * call's rotated input, 2 * M * K bytes, K rounded up to 64 for 8-bit and
 * 128 for 4-bit weights) must fit 96 KB, or the call is refused with
 * TQ_ERR_SHAPE (for M = 1: K up to 9728 with 8-bit weights, 16128 with
 * 4-bit).  The calls' pointers are kept: their buffers must stay allocated at
 * the same addresses while the plan is used.
 * A set-up call: it copies its tables with cudaMemcpy (the host waits), so
 * make it outside stream capture.  The device is the current one; runs on
 * another device are refused.
 */
tq_status tq_grouped_create(const tq_a16_call *calls, int64_t ncalls, int bits, tq_out ytype,
                            void *dmem, size_t dbytes, tq_grouped *plan);

/*
 * Runs every call of the plan on `stream` (two launches: the input rotation,
 * then the product; capturable in a CUDA graph).  Requirements:
 *   - the calls are independent: no call's Y overlaps any call's X, Wq, sw or
 *     another call's Y;
 *   - runs of one plan are ordered (they share the plan's rotated inputs).
 */
tq_status tq_grouped_run(tq_grouped plan, cudaStream_t stream);

/*
 * The two launches of tq_grouped_run on their own, in this order on one
 * stream (or ordered by events): tq_grouped_rotate reads every call's X and
 * writes the plan's rotated inputs; tq_grouped_product reads them and the
 * weights and writes every Y.  The inputs may change between the two only if
 * the rotation is run again.
 */
tq_status tq_grouped_rotate(tq_grouped plan, cudaStream_t stream);
tq_status tq_grouped_product(tq_grouped plan, cudaStream_t stream);

/* Algorithmic bytes one run streams: every call's weight codes and row scales. */
int64_t tq_grouped_weight_bytes(tq_grouped plan);

/* Frees the host handle (the device buffer stays the caller's).  NULL is ignored. */
void tq_grouped_destroy(tq_grouped plan);

/*
 * Chained plans: decode calls that depend on one another, run in order in
 * one launch, the way a decoder walks its layers (kvad-gpu internals,
 * "Numbers": decode runs one projection at a time, each input the previous
 * output, and is bound by the weight stream).  Call c starts only after every
 * earlier call has finished, so its X (and U) may be any earlier call's Y.
 * The launch keeps streaming later calls' weights into shared memory while
 * earlier calls finish; between calls its CTAs wait on counters in the plan's
 * buffer (bounded waits: on expiry tq_device_status reports
 * TQ_ERR_DEVICE_TIMEOUT and the outputs of unfinished calls are unwritten).
 * The launch is cooperative: it needs every SM free of other work while it
 * runs (another kernel on the device delays its start).
 *
 * Each call is a grouped call, optionally with the SwiGLU of two rows as its
 * input: with U set, the product reads h = bf16(silu(X) * U), silu(g) =
 * g / (1 + e^-g) (the arithmetic of tq_linear_swiglu), as a gated FFN's down
 * projection takes the two halves of its gate+up output.
 */
typedef struct {
    tq_a16_call call;   /* as in a grouped plan; X holds the gate rows when U is set */
    const void *U;      /* NULL, or bf16 [M, K] up rows at U + m * ldu (X's rules) */
    int64_t ldu;
} tq_chain_call;

/* Bytes of device memory a chained plan of these calls needs (no device
 * needed; the refusals of tq_chain_create). */
tq_status tq_chain_bytes(const tq_chain_call *calls, int64_t ncalls, int bits, size_t *bytes);

/*
 * Checks every call and writes the chained plan's tables into `dmem`;
 * arguments and ownership as tq_grouped_create.  Each call follows
 * tq_linear's rules for X, U, Wq, sw, Y and strides, with M <= 8; in
 * addition its rotated input must fit the launch's own buffer (2 * M * K
 * bytes, K rounded up to 64 for 8-bit and 128 for 4-bit weights, at most
 * 17984) and eight weight rows a 96 KB stage, or the call is refused with
 * TQ_ERR_SHAPE (for M = 1: K up to 8960 with 8- or 4-bit weights).
 * A call's Y must not overlap its own X or U, nor any call's Wq or sw; it
 * may overlap an earlier call's X, U or Y (later calls run after them).
 * Run the plan with tq_grouped_run (the counters are zeroed, then one
 * launch; capturable in a CUDA graph); tq_grouped_rotate and
 * tq_grouped_product refuse a chained plan with TQ_ERR_MODE.  Runs of one
 * plan are ordered (they share its counters).
 */
tq_status tq_chain_create(const tq_chain_call *calls, int64_t ncalls, int bits, tq_out ytype,
                          void *dmem, size_t dbytes, tq_grouped *plan);

#ifdef __cplusplus
}
#endif
#endif /* TQ_H */
