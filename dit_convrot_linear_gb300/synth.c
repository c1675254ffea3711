/*
 * Seeded synthetic inputs for the rotated low-bit linear projection.
 *
 * This file holds input generation only: no step of the projection itself
 * (no rotation, no quantisation, no product).  Both the CUDA path's harness
 * and the CPU oracle's tests draw their inputs from here, so the two sides see
 * the same bf16 tensors.
 *
 * Recipe (every tensor):
 *   key      = SplitMix64 finaliser of (FNV-1a-64(name) XOR seed)
 *   U(i)     = top 53 bits of SplitMix64(key + (i+1) * golden) / 2^53, in [0,1)
 *              (counter-based SplitMix64: Steele, Lea and Flood, "Fast
 *              splittable pseudorandom number generators", OOPSLA 2014)
 *   Z(i)     = sqrt(-2 ln(1 - U(2i))) * cos(2 pi U(2i+1))     (Box and Muller,
 *              "A note on the generation of random normal deviates", 1958)
 *   x[r][c]  = Z(r*cols + c) * sigma * (c is an outlier column ? mult : 1)
 *   stored   = x rounded to the nearest bf16, ties to even (one rounding)
 * Outlier columns are the first `count` entries of the column indices sorted
 * by the SplitMix64 hash of a second key, returned in ascending order.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define GOLDEN 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

uint64_t synth_key(const char *name, uint64_t seed) {
    uint64_t h = 0xcbf29ce484222325ULL; /* FNV-1a 64 offset basis */
    for (const unsigned char *p = (const unsigned char *)name; *p; ++p) {
        h ^= *p;
        h *= 0x100000001b3ULL; /* FNV-1a 64 prime */
    }
    return mix64(h ^ seed);
}

static inline double uniform01(uint64_t key, uint64_t i) {
    return (double)(mix64(key + (i + 1) * GOLDEN) >> 11) * 0x1.0p-53;
}

static inline double normal_at(uint64_t key, uint64_t i) {
    const double u1 = 1.0 - uniform01(key, 2 * i); /* (0, 1] */
    const double u2 = uniform01(key, 2 * i + 1);
    return sqrt(-2.0 * log(u1)) * cos(6.283185307179586 * u2);
}

/* fp64 -> bf16 bits, nearest, ties to even, in one rounding. */
static uint16_t to_bf16(double x) {
    if (isnan(x)) return 0x7FC0;
    const uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs(x);
    if (a == 0.0) return sign;
    int e;
    frexp(a, &e);                       /* a = f * 2^e, f in [0.5, 1) */
    int q = e - 8;                      /* quantum of an 8-bit significand */
    if (q < -133) q = -133;             /* bf16 subnormal quantum 2^-133 */
    double r = rint(ldexp(a, -q));      /* exact scaling, then ties-to-even */
    double v = ldexp(r, q);
    if (v > 0x1.FEp127) return sign | 0x7F80; /* beyond the largest finite bf16 */
    float f = (float)v;                 /* exact: v has at most 8 significant bits */
    uint32_t bits;
    memcpy(&bits, &f, 4);
    return sign | (uint16_t)((bits >> 16) & 0x7FFF);
}

typedef struct {
    uint64_t key;
    int64_t r0, r1, cols;
    double sigma, mult;
    const uint8_t *is_out;
    uint16_t *out;
} fill_job;

static void *fill_worker(void *arg) {
    fill_job *j = (fill_job *)arg;
    for (int64_t r = j->r0; r < j->r1; ++r) {
        for (int64_t c = 0; c < j->cols; ++c) {
            double v = normal_at(j->key, (uint64_t)(r * j->cols + c)) * j->sigma;
            if (j->is_out && j->is_out[c]) v *= j->mult;
            j->out[r * j->cols + c] = to_bf16(v);
        }
    }
    return NULL;
}

/* Fill out[rows][cols] (bf16 bits).  out_cols lists the outlier columns. */
int synth_fill_bf16(uint64_t key, int64_t rows, int64_t cols, double sigma,
                    const int64_t *out_cols, int64_t n_out, double mult,
                    uint16_t *out, int nthreads) {
    if (rows < 0 || cols < 0 || (rows * cols > 0 && !out)) return 1;
    uint8_t *is_out = NULL;
    if (n_out > 0) {
        is_out = (uint8_t *)calloc((size_t)cols, 1);
        if (!is_out) return 2;
        for (int64_t i = 0; i < n_out; ++i)
            if (out_cols[i] >= 0 && out_cols[i] < cols) is_out[out_cols[i]] = 1;
    }
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if (rows < nthreads) nthreads = rows > 0 ? (int)rows : 1;
    pthread_t th[256];
    fill_job jobs[256];
    for (int t = 0; t < nthreads; ++t) {
        jobs[t].key = key;
        jobs[t].r0 = rows * t / nthreads;
        jobs[t].r1 = rows * (t + 1) / nthreads;
        jobs[t].cols = cols;
        jobs[t].sigma = sigma;
        jobs[t].mult = mult;
        jobs[t].is_out = is_out;
        jobs[t].out = out;
    }
    int created[256] = {0};
    for (int t = 1; t < nthreads; ++t) {
        if (pthread_create(&th[t], NULL, fill_worker, &jobs[t]) == 0)
            created[t] = 1;
        else
            fill_worker(&jobs[t]); /* run inline if a thread cannot start */
    }
    fill_worker(&jobs[0]);
    for (int t = 1; t < nthreads; ++t)
        if (created[t]) pthread_join(th[t], NULL);
    free(is_out);
    return 0;
}

typedef struct { uint64_t h; int64_t c; } keyed;

static int cmp_keyed(const void *a, const void *b) {
    const keyed *x = (const keyed *)a, *y = (const keyed *)b;
    if (x->h != y->h) return x->h < y->h ? -1 : 1;
    return x->c < y->c ? -1 : (x->c > y->c);
}

static int cmp_i64(const void *a, const void *b) {
    int64_t x = *(const int64_t *)a, y = *(const int64_t *)b;
    return x < y ? -1 : (x > y);
}

/* count distinct columns of [0, cols), seeded, ascending. */
int synth_choose_columns(uint64_t key, int64_t cols, int64_t count, int64_t *out) {
    if (count < 0 || count > cols) return 1;
    keyed *k = (keyed *)malloc(sizeof(keyed) * (size_t)(cols > 0 ? cols : 1));
    if (!k) return 2;
    for (int64_t c = 0; c < cols; ++c) {
        k[c].h = mix64(key + ((uint64_t)c + 1) * GOLDEN);
        k[c].c = c;
    }
    qsort(k, (size_t)cols, sizeof(keyed), cmp_keyed);
    for (int64_t i = 0; i < count; ++i) out[i] = k[i].c;
    qsort(out, (size_t)count, sizeof(int64_t), cmp_i64);
    free(k);
    return 0;
}
