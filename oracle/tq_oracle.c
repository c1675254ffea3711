/*
 * CPU oracle for the rotated low-bit linear projection.
 *
 * TEST INFRASTRUCTURE ONLY.  The tests, the smoke check and the benchmark's
 * CPU-baseline leg are the only callers.  The product path (the CUDA library)
 * never links, loads or calls this file, and this file uses nothing of it.
 *
 * What it computes, and where the pages say so:
 *   - Weights are rotated by a Hadamard matrix over every group of 256 input
 *     columns, then quantised to int8 with one scale per row
 *     (tensai docs, "画像生成" / Image generation, section "チェックポイントの入手",
 *     Getting the checkpoints).
 *   - The matrix is orthogonal, so the product is unchanged when the matching
 *     input rows get the same rotation; the rotation of an input row views it as
 *     groups of 256 and takes one product with H per group
 *     (same page, section "幅とメモリ", Width and memory).
 *   - 8-bit by default, 4-bit with -q4 (same section; flag list "フラグ").
 *     INT8 and INT4 "ConvRot" are the two formats of TensorPencil's README
 *     ("Details", format table).
 *   - On the device the activations of each product are quantised per product
 *     (same page, section "GPU"); the oracle takes one symmetric int8 scale per
 *     token row over all of K.
 *
 * Steps (numbered as the oracle's own):
 *   O1 bf16 bits -> fp64, exactly.
 *   O2 per row and group: S = Hs_n . v by an explicit n x n product in fp64,
 *      Hs_n[i][j] = (-1)^popcount(i & j) (Sylvester's construction), then
 *      v' = c_n * S with c_n = sqrt(1/n) correctly rounded.
 *   O3 per row: amax = max |v'|; s = fp32(amax / qmax); q = clamp(rint(v'/s)).
 *   O4 activations (A8): O3 with qmax = 127 over the whole row.
 *   O4' activations (A16): v' rounded to the nearest bf16, ties to even.
 *   O5 A8 product: int64 sum of code products (asserted to fit int32),
 *      Y = s_x * s_w * acc in fp64.
 *   O6 A16 product: Y = s_w * sum_k q_w * x'_bf16 in fp64.
 *   O7 int4 packing: byte k/2 of a row holds code k (even) in its low nibble and
 *      code k+1 in its high nibble, two's complement.
 *   O8 SwiGLU (the row kernel between a gate/up product and the down product;
 *      the pages name it among the row kernels next to the projections,
 *      TensorFold PR #948, "What comes next"): h = silu(g) * u with
 *      silu(g) = g / (1 + e^-g), the gated unit of Shazeer, "GLU Variants
 *      Improve Transformer" (2020), in fp64 from bf16 g and u, then rounded
 *      to the nearest bf16 (the activations are bf16).
 *   O9 block-scaled weights (a scale per block of G columns instead of per
 *      row: the blocks with a shared scale of the GGML formats, Q8_0 and Q4_0
 *      32 wide, and kvad's own q8 with an fp32 scale per 32 weights; kvad-gpu
 *      internals, "Quantised weights on the GPU"; used on the rotated weights
 *      to recover 4-bit accuracy, whose error the rotation lowers less than
 *      8-bit's, tensai docs, "画像生成", section "幅とメモリ"): O3 applied to
 *      every block on its own, s_b = fp32(amax_b / qmax), q = rint(v / s_b).
 *      The blocks are taken of v' (rotated) or of the bf16 weights themselves
 *      (the unrotated format).
 *   O10 block-scaled A16 product: Y = sum_b s_b * sum_{k in block b} q_w * x
 *      in fp64, x the bf16 activations (rotated and rounded as in O4' when
 *      the weights were rotated, else as given).
 *   O11 modulated layer norm (the row kernel in front of a DiT block's
 *      query/key/value and gate/up products; the pages name "the modulated
 *      layer norm" among the row kernels next to the projections, with fp32
 *      norms, TensorFold PR #948, "What comes next" and the precision list of
 *      its summary; the modulation is shared by every block, same PR, "What it
 *      adds", host.zig): per row, mu = mean(x), var = mean((x - mu)^2) (the
 *      biased variance: a layer norm divides by K), and
 *      h = (x - mu) / sqrt(var + eps) * (1 + scale) + shift, in fp64 from bf16
 *      x and fp32 shift, scale [K] (one modulation for all rows), then
 *      rounded to the nearest bf16.  The form LN(x) (1 + scale) + shift with no
 *      affine parameters of its own is the adaptive layer norm of Peebles and
 *      Xie, "Scalable Diffusion Models with Transformers" (2023).
 *
 * Readings where the pages are silent (each listed in the design notes):
 *   Sylvester order and 1/sqrt(n) normalisation; a last group narrower than
 *   256 (a power of two >= 32) uses its own H_t; nearest-even rounding; codes
 *   symmetric in [-qmax, qmax]; a zero row (or a scale that rounds to zero in
 *   fp32) has scale 0 and all-zero codes.
 */
#include <fenv.h>
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* -------------------------------------------------------------------------- */
/* small thread pool: run fn(arg, i0, i1) over [0, n) split into ranges        */

typedef void (*range_fn)(void *arg, int64_t i0, int64_t i1);

typedef struct {
    range_fn fn;
    void *arg;
    int64_t i0, i1;
} range_job;

static void *range_worker(void *p) {
    range_job *j = (range_job *)p;
    fesetround(FE_TONEAREST);
    j->fn(j->arg, j->i0, j->i1);
    return NULL;
}

static void parallel_for(int64_t n, int nthreads, range_fn fn, void *arg) {
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if (n < nthreads) nthreads = n > 0 ? (int)n : 1;
    pthread_t th[256];
    range_job jobs[256];
    int created[256] = {0};
    for (int t = 0; t < nthreads; ++t) {
        jobs[t].fn = fn;
        jobs[t].arg = arg;
        jobs[t].i0 = n * t / nthreads;
        jobs[t].i1 = n * (t + 1) / nthreads;
    }
    for (int t = 1; t < nthreads; ++t) {
        if (pthread_create(&th[t], NULL, range_worker, &jobs[t]) == 0)
            created[t] = 1;
        else
            range_worker(&jobs[t]);
    }
    range_worker(&jobs[0]);
    for (int t = 1; t < nthreads; ++t)
        if (created[t]) pthread_join(th[t], NULL);
}

/* -------------------------------------------------------------------------- */
/* O1 and O4': bf16 <-> fp64                                                   */

double or_bf16_to_f64(uint16_t b) {
    uint32_t bits = (uint32_t)b << 16;
    float f;
    memcpy(&f, &bits, 4);
    return (double)f;
}

/* Nearest bf16 to x, ties to even, in one rounding from fp64. */
uint16_t or_f64_to_bf16(double x) {
    if (isnan(x)) return 0x7FC0;
    const uint16_t sign = signbit(x) ? 0x8000 : 0;
    const double a = fabs(x);
    if (a == 0.0) return sign;
    int e;
    frexp(a, &e);                  /* a = f * 2^e with f in [0.5, 1) */
    int q = e - 8;                 /* bf16 keeps 8 significant bits */
    if (q < -133) q = -133;        /* smallest bf16 step (subnormal range) */
    const double v = ldexp(nearbyint(ldexp(a, -q)), q);
    if (v > 0x1.FEp127) return sign | 0x7F80;
    float f = (float)v;            /* exact: at most 8 significant bits */
    uint32_t bits;
    memcpy(&bits, &f, 4);
    return sign | (uint16_t)((bits >> 16) & 0x7FFF);
}

int or_round_bf16(const double *v, int64_t n, uint16_t *out) {
    fesetround(FE_TONEAREST);
    for (int64_t i = 0; i < n; ++i) out[i] = or_f64_to_bf16(v[i]);
    return 0;
}

/* -------------------------------------------------------------------------- */
/* Hadamard matrices and the group layout of a row                             */

static int popcount_u32(uint32_t x) {
    int c = 0;
    while (x) {
        c += (int)(x & 1u);
        x >>= 1;
    }
    return c;
}

/* Hs_n[i][j] = (-1)^popcount(i & j), n a power of two (Sylvester). */
int or_sylvester(int n, int8_t *H) {
    if (n < 1 || (n & (n - 1)) || n > 4096) return 1;
    for (int i = 0; i < n; ++i)
        for (int j = 0; j < n; ++j)
            H[(int64_t)i * n + j] = (popcount_u32((uint32_t)(i & j)) & 1) ? -1 : 1;
    return 0;
}

/* c_n = 1/sqrt(n), correctly rounded: sqrt of the exact 1/n (n a power of 2). */
double or_hadamard_norm(int n) { return sqrt(1.0 / (double)n); }

/* Width of the group that starts at column g0 of a K-wide row: 256, or the
 * power-of-two tail K - g0 when fewer than 256 columns remain.  Returns 0 when
 * K is not 256*q + t with t in {0, 32, 64, 128}. */
int or_group_width(int64_t K, int64_t g0) {
    const int64_t rest = K - g0;
    if (rest >= 256) return 256;
    if (rest == 128 || rest == 64 || rest == 32) return (int)rest;
    return 0;
}

int or_valid_k(int64_t K) {
    if (K <= 0) return 0;
    const int64_t t = K % 256;
    return t == 0 || t == 32 || t == 64 || t == 128;
}

/* -------------------------------------------------------------------------- */
/* O2: rotation by explicit products                                           */

typedef struct {
    const uint16_t *X;
    int64_t K, ld;
    double *out;
    const int8_t *H256, *H128, *H64, *H32;
    volatile int bad_group;
} rot_arg;

static const int8_t *pick_h(const rot_arg *a, int n) {
    return n == 256 ? a->H256 : n == 128 ? a->H128 : n == 64 ? a->H64 : a->H32;
}

static void rot_rows(void *p, int64_t r0, int64_t r1) {
    rot_arg *a = (rot_arg *)p;
    double v[256];
    for (int64_t r = r0; r < r1; ++r) {
        const uint16_t *row = a->X + r * a->ld;
        double *o = a->out + r * a->K;
        for (int64_t g0 = 0; g0 < a->K;) {
            const int n = or_group_width(a->K, g0);
            if (n == 0) { /* no valid group starts here: refuse the row */
                a->bad_group = 1;
                break;
            }
            const int8_t *H = pick_h(a, n);
            const double c = or_hadamard_norm(n);
            for (int j = 0; j < n; ++j) v[j] = or_bf16_to_f64(row[g0 + j]); /* O1 */
            for (int i = 0; i < n; ++i) {
                double s = 0.0;
                for (int j = 0; j < n; ++j) s += (double)H[i * n + j] * v[j];
                o[g0 + i] = c * s;
            }
            g0 += n;
        }
    }
}

/* out[r][k] (fp64, dense [R, K]) = rotation of bf16 rows X[r * ld + k]. */
int or_rotate_rows(const uint16_t *X, int64_t R, int64_t K, int64_t ld,
                   double *out, int nthreads) {
    if (!or_valid_k(K) || ld < K || R < 0) return 2;
    if (R == 0) return 0;
    if (!X || !out) return 1;
    int8_t *H256 = (int8_t *)malloc(256 * 256 + 128 * 128 + 64 * 64 + 32 * 32);
    if (!H256) return 4;
    int8_t *H128 = H256 + 256 * 256, *H64 = H128 + 128 * 128, *H32 = H64 + 64 * 64;
    or_sylvester(256, H256);
    or_sylvester(128, H128);
    or_sylvester(64, H64);
    or_sylvester(32, H32);
    rot_arg a = {X, K, ld, out, H256, H128, H64, H32, 0};
    parallel_for(R, nthreads, rot_rows, &a);
    free(H256);
    return a.bad_group ? 2 : 0;
}

/* -------------------------------------------------------------------------- */
/* O3 / O4: per-row symmetric quantisation                                     */

int or_quantize_rows(const double *V, int64_t R, int64_t K, int qmax,
                     int8_t *codes, float *scales) {
    if (R < 0 || K < 0 || qmax < 1 || qmax > 127) return 2;
    fesetround(FE_TONEAREST);
    for (int64_t r = 0; r < R; ++r) {
        const double *v = V + r * K;
        double amax = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            const double a = fabs(v[k]);
            if (a > amax) amax = a;
        }
        const float s = (float)(amax / (double)qmax);
        scales[r] = s;
        for (int64_t k = 0; k < K; ++k) {
            if (s == 0.0f) {
                codes[r * K + k] = 0;
                continue;
            }
            double q = nearbyint(v[k] / (double)s);
            if (q > qmax) q = qmax;
            if (q < -qmax) q = -qmax;
            codes[r * K + k] = (int8_t)q;
        }
    }
    return 0;
}

/* -------------------------------------------------------------------------- */
/* O7: int4 packing                                                            */

int or_pack_int4(const int8_t *codes, int64_t R, int64_t K, uint8_t *packed) {
    if (K % 2) return 2;
    for (int64_t r = 0; r < R; ++r)
        for (int64_t k = 0; k < K; k += 2) {
            const uint8_t lo = (uint8_t)codes[r * K + k] & 0xF;
            const uint8_t hi = (uint8_t)codes[r * K + k + 1] & 0xF;
            packed[r * (K / 2) + k / 2] = (uint8_t)(lo | (hi << 4));
        }
    return 0;
}

int or_unpack_int4(const uint8_t *packed, int64_t R, int64_t K, int8_t *codes) {
    if (K % 2) return 2;
    for (int64_t r = 0; r < R; ++r)
        for (int64_t k = 0; k < K; k += 2) {
            const uint8_t b = packed[r * (K / 2) + k / 2];
            int lo = b & 0xF, hi = b >> 4;
            codes[r * K + k] = (int8_t)(lo >= 8 ? lo - 16 : lo);
            codes[r * K + k + 1] = (int8_t)(hi >= 8 ? hi - 16 : hi);
        }
    return 0;
}

/* -------------------------------------------------------------------------- */
/* O5: A8 product (int8 activation codes x int8/int4 weight codes)            */

typedef struct {
    const int8_t *Xq;
    const float *sx;
    int64_t M, K;
    const int8_t *Wq;
    const float *sw;
    int64_t N;
    int32_t *acc;
    double *Y;
    const int64_t *pm, *pn;
    const uint16_t *Xr;
    volatile int overflow;
} lin_arg;

static int64_t dot_i8(const int8_t *x, const int8_t *w, int64_t K) {
    int64_t s = 0;
    for (int64_t k = 0; k < K; ++k) s += (int64_t)x[k] * (int64_t)w[k];
    return s;
}

static void a8_one(lin_arg *a, int64_t m, int64_t n, int64_t out_idx) {
    const int64_t s = dot_i8(a->Xq + m * a->K, a->Wq + n * a->K, a->K);
    if (s > INT32_MAX || s < INT32_MIN) a->overflow = 1;
    if (a->acc) a->acc[out_idx] = (int32_t)s;
    if (a->Y) a->Y[out_idx] = (double)a->sx[m] * (double)a->sw[n] * (double)s;
}

static void a8_cols(void *p, int64_t n0, int64_t n1) {
    lin_arg *a = (lin_arg *)p;
    for (int64_t m = 0; m < a->M; ++m)
        for (int64_t n = n0; n < n1; ++n) a8_one(a, m, n, m * a->N + n);
}

static void a8_pairs(void *p, int64_t i0, int64_t i1) {
    lin_arg *a = (lin_arg *)p;
    for (int64_t i = i0; i < i1; ++i) a8_one(a, a->pm[i], a->pn[i], i);
}

/* acc[m][n] (may be NULL) and Y[m][n] (may be NULL), dense [M, N]. */
int or_linear_a8(const int8_t *Xq, const float *sx, int64_t M, int64_t K,
                 const int8_t *Wq, const float *sw, int64_t N, int32_t *acc,
                 double *Y, int nthreads) {
    lin_arg a = {Xq, sx, M, K, Wq, sw, N, acc, Y, NULL, NULL, NULL, 0};
    parallel_for(N, nthreads, a8_cols, &a);
    return a.overflow ? 3 : 0;
}

/* The same at listed (m, n) pairs only: out[i] for (pm[i], pn[i]). */
int or_linear_a8_pairs(const int8_t *Xq, const float *sx, int64_t M, int64_t K,
                       const int8_t *Wq, const float *sw, int64_t N,
                       const int64_t *pm, const int64_t *pn, int64_t count,
                       int32_t *acc, double *Y, int nthreads) {
    for (int64_t i = 0; i < count; ++i)
        if (pm[i] < 0 || pm[i] >= M || pn[i] < 0 || pn[i] >= N) return 2;
    lin_arg a = {Xq, sx, M, K, Wq, sw, N, acc, Y, pm, pn, NULL, 0};
    parallel_for(count, nthreads, a8_pairs, &a);
    return a.overflow ? 3 : 0;
}

/* -------------------------------------------------------------------------- */
/* O6: A16 product (bf16 rotated activations x int8/int4 weight codes)        */

static void a16_one(lin_arg *a, int64_t m, int64_t n, int64_t out_idx) {
    const uint16_t *x = a->Xr + m * a->K;
    const int8_t *w = a->Wq + n * a->K;
    double s = 0.0;
    for (int64_t k = 0; k < a->K; ++k) s += (double)w[k] * or_bf16_to_f64(x[k]);
    a->Y[out_idx] = (double)a->sw[n] * s;
}

static void a16_cols(void *p, int64_t n0, int64_t n1) {
    lin_arg *a = (lin_arg *)p;
    for (int64_t m = 0; m < a->M; ++m)
        for (int64_t n = n0; n < n1; ++n) a16_one(a, m, n, m * a->N + n);
}

static void a16_pairs(void *p, int64_t i0, int64_t i1) {
    lin_arg *a = (lin_arg *)p;
    for (int64_t i = i0; i < i1; ++i) a16_one(a, a->pm[i], a->pn[i], i);
}

int or_linear_a16(const uint16_t *Xr, int64_t M, int64_t K, const int8_t *Wq,
                  const float *sw, int64_t N, double *Y, int nthreads) {
    lin_arg a = {NULL, NULL, M, K, Wq, sw, N, NULL, Y, NULL, NULL, Xr, 0};
    parallel_for(N, nthreads, a16_cols, &a);
    return 0;
}

int or_linear_a16_pairs(const uint16_t *Xr, int64_t M, int64_t K,
                        const int8_t *Wq, const float *sw, int64_t N,
                        const int64_t *pm, const int64_t *pn, int64_t count,
                        double *Y, int nthreads) {
    for (int64_t i = 0; i < count; ++i)
        if (pm[i] < 0 || pm[i] >= M || pn[i] < 0 || pn[i] >= N) return 2;
    lin_arg a = {NULL, NULL, M, K, Wq, sw, N, NULL, Y, pm, pn, Xr, 0};
    parallel_for(count, nthreads, a16_pairs, &a);
    return 0;
}

/* -------------------------------------------------------------------------- */
/* Plain fp64 product Y = A . B^T (A [M,K], B [N,K]) for the invariance pins. */

typedef struct {
    const double *A, *B;
    int64_t M, K, N;
    double *Y;
} mm_arg;

static void mm_cols(void *p, int64_t n0, int64_t n1) {
    const mm_arg *a = (const mm_arg *)p;
    for (int64_t m = 0; m < a->M; ++m)
        for (int64_t n = n0; n < n1; ++n) {
            double s = 0.0;
            for (int64_t k = 0; k < a->K; ++k) s += a->A[m * a->K + k] * a->B[n * a->K + k];
            a->Y[m * a->N + n] = s;
        }
}

int or_matmul_f64(const double *A, int64_t M, int64_t K, const double *B,
                  int64_t N, double *Y, int nthreads) {
    mm_arg a = {A, B, M, K, N, Y};
    parallel_for(N, nthreads, mm_cols, &a);
    return 0;
}

/* -------------------------------------------------------------------------- */
/* O8 SwiGLU                                                                   */

int or_swiglu_f64(const double *g, const double *u, int64_t n, double *h) {
    for (int64_t i = 0; i < n; ++i) h[i] = g[i] / (1.0 + exp(-g[i])) * u[i];
    return 0;
}

/* H [M, K] dense bf16 bits from bf16 G, U [M, K] with row strides ldg, ldu. */
int or_swiglu_bf16(const uint16_t *G, int64_t ldg, const uint16_t *U, int64_t ldu, int64_t M,
                   int64_t K, uint16_t *H) {
    fesetround(FE_TONEAREST);
    for (int64_t m = 0; m < M; ++m)
        for (int64_t k = 0; k < K; ++k) {
            const double g = or_bf16_to_f64(G[m * ldg + k]), u = or_bf16_to_f64(U[m * ldu + k]);
            double h;
            or_swiglu_f64(&g, &u, 1, &h);
            H[m * K + k] = or_f64_to_bf16(h);
        }
    return 0;
}

/* -------------------------------------------------------------------------- */
/* O11 modulated layer norm                                                    */

/* One row: h = (x - mu) / sqrt(var + eps) * (1 + scale) + shift in fp64. */
int or_modnorm_f64(const double *x, int64_t K, const double *shift, const double *scale, double eps,
                   double *h) {
    if (K <= 0) return 1;
    double mu = 0.0;
    for (int64_t k = 0; k < K; ++k) mu += x[k];
    mu /= (double)K;
    double var = 0.0;
    for (int64_t k = 0; k < K; ++k) var += (x[k] - mu) * (x[k] - mu);
    var /= (double)K;
    const double rstd = 1.0 / sqrt(var + eps);
    for (int64_t k = 0; k < K; ++k) h[k] = (x[k] - mu) * rstd * (1.0 + scale[k]) + shift[k];
    return 0;
}

/* H [M, K] dense bf16 bits from bf16 X [M, K] (row stride ldx), fp32 shift and
 * scale [K] and eps. */
int or_modnorm_bf16(const uint16_t *X, int64_t ldx, int64_t M, int64_t K, const float *shift,
                    const float *scale, float eps, uint16_t *H) {
    if (K <= 0) return 1;
    fesetround(FE_TONEAREST);
    double *x = malloc(sizeof(double) * (size_t)K * 4);
    if (!x) return 2;
    double *sh = x + K, *sc = x + 2 * K, *h = x + 3 * K;
    for (int64_t k = 0; k < K; ++k) {
        sh[k] = (double)shift[k];
        sc[k] = (double)scale[k];
    }
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t k = 0; k < K; ++k) x[k] = or_bf16_to_f64(X[m * ldx + k]);
        or_modnorm_f64(x, K, sh, sc, (double)eps, h);
        for (int64_t k = 0; k < K; ++k) H[m * K + k] = or_f64_to_bf16(h[k]);
    }
    free(x);
    return 0;
}

/* -------------------------------------------------------------------------- */
/* O9 block-scaled quantisation: O3 applied to every block of G columns of a   */
/* row on its own (one scale per block instead of one per row).               */

int or_quantize_blocks(const double *V, int64_t R, int64_t K, int64_t G, int qmax,
                       int8_t *codes, float *scales) {
    if (R < 0 || K < 0 || G < 1 || K % G || qmax < 1 || qmax > 127) return 2;
    fesetround(FE_TONEAREST);
    const int64_t nb = K / G;
    for (int64_t r = 0; r < R; ++r)
        for (int64_t b = 0; b < nb; ++b) {
            const double *v = V + r * K + b * G;
            int8_t *q = codes + r * K + b * G;
            double amax = 0.0;
            for (int64_t k = 0; k < G; ++k) {
                const double a = fabs(v[k]);
                if (a > amax) amax = a;
            }
            const float s = (float)(amax / (double)qmax);
            scales[r * nb + b] = s;
            for (int64_t k = 0; k < G; ++k) {
                if (s == 0.0f) {
                    q[k] = 0;
                    continue;
                }
                double c = nearbyint(v[k] / (double)s);
                if (c > qmax) c = qmax;
                if (c < -qmax) c = -qmax;
                q[k] = (int8_t)c;
            }
        }
    return 0;
}

/* -------------------------------------------------------------------------- */
/* O10 block-scaled A16 product: Y[m][n] = sum_b s[n][b] * sum_{k in b} q * x  */
/* in fp64, x the bf16 activation row as given (rotated or not).              */

typedef struct {
    const uint16_t *X;
    int64_t M, K, G;
    const int8_t *Wq;
    const float *sw;
    int64_t N;
    double *Y;
} blk_arg;

static void blk_cols(void *p, int64_t n0, int64_t n1) {
    const blk_arg *a = (const blk_arg *)p;
    const int64_t nb = a->K / a->G;
    for (int64_t m = 0; m < a->M; ++m)
        for (int64_t n = n0; n < n1; ++n) {
            const uint16_t *x = a->X + m * a->K;
            const int8_t *w = a->Wq + n * a->K;
            double y = 0.0;
            for (int64_t b = 0; b < nb; ++b) {
                double part = 0.0;
                for (int64_t k = b * a->G; k < (b + 1) * a->G; ++k)
                    part += (double)w[k] * or_bf16_to_f64(x[k]);
                y += (double)a->sw[n * nb + b] * part;
            }
            a->Y[m * a->N + n] = y;
        }
}

int or_linear_a16_blocked(const uint16_t *X, int64_t M, int64_t K, const int8_t *Wq,
                          const float *sw, int64_t G, int64_t N, double *Y, int nthreads) {
    if (M < 0 || N < 0 || K < 0 || G < 1 || K % G) return 2;
    blk_arg a = {X, M, K, G, Wq, sw, N, Y};
    parallel_for(N, nthreads, blk_cols, &a);
    return 0;
}
