/*
 * synth.c -- seeded synthetic inputs shared by the oracle tests and the GPU path.
 *
 * This file draws random numbers and lays out sparsity patterns (row lengths,
 * distinct sorted column indices per row, values, dense vectors).  It holds no
 * arithmetic of the sparse products themselves: it never builds row offsets,
 * transposes, blocks or sums anything that the library or the oracle computes.
 *
 * Random numbers: counter-based SplitMix64 (Steele, Lea, Flood, "Fast
 * splittable pseudorandom number generators", OOPSLA 2014).  Value i of a
 * stream with key k is mix(k + (i+1)*0x9E3779B97F4A7C15); streams are keyed by
 * (seed, tag), so every array is reproducible on any machine regardless of the
 * order in which it is generated.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define GOLDEN 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}
static inline uint64_t stream_key(uint64_t seed, uint64_t tag) {
    return mix64(mix64(seed + GOLDEN) ^ (tag * 0xD1B54A32D192ED03ULL));
}
static inline uint64_t draw(uint64_t key, uint64_t i) { return mix64(key + (i + 1) * GOLDEN); }
/* uniform double in [0, 1) with 53 random bits */
static inline double u01(uint64_t z) { return (double)(z >> 11) * 0x1.0p-53; }
/* uniform integer in [0, n) */
static inline int64_t below(uint64_t z, int64_t n) { return (int64_t)(u01(z) * (double)n); }

uint64_t synth_raw(uint64_t seed, uint64_t tag, uint64_t i) { return draw(stream_key(seed, tag), i); }

/* out[i] = lo + (hi - lo) * u_i, rounded to fp32 */
void synth_uniform_f32(uint64_t seed, uint64_t tag, int64_t n, double lo, double hi, float* out) {
    uint64_t k = stream_key(seed, tag);
    for (int64_t i = 0; i < n; ++i) out[i] = (float)(lo + (hi - lo) * u01(draw(k, (uint64_t)i)));
}

/* Box-Muller: one normal per pair of uniforms. */
static inline double normal_at(uint64_t k, int64_t i) {
    double u1 = u01(draw(k, 2 * (uint64_t)i));
    double u2 = u01(draw(k, 2 * (uint64_t)i + 1));
    double r = sqrt(-2.0 * log(1.0 - u1)); /* 1 - u1 in (0, 1] */
    return r * cos(6.283185307179586 * u2);
}

void synth_normal_f32(uint64_t seed, uint64_t tag, int64_t n, double sigma, float* out) {
    uint64_t k = stream_key(seed, tag);
    for (int64_t i = 0; i < n; ++i) out[i] = (float)(sigma * normal_at(k, i));
}

static inline uint16_t f32_to_bf16_rne(float f) {
    uint32_t b;
    memcpy(&b, &f, 4);
    b += 0x7FFFu + ((b >> 16) & 1u);
    return (uint16_t)(b >> 16);
}

/* N(0, sigma) drawn in fp64, rounded to fp32, then to bf16 (round to nearest even). */
void synth_normal_bf16(uint64_t seed, uint64_t tag, int64_t n, double sigma, uint16_t* out) {
    uint64_t k = stream_key(seed, tag);
    for (int64_t i = 0; i < n; ++i) out[i] = f32_to_bf16_rne((float)(sigma * normal_at(k, i)));
}

/* fp32 -> bf16 bits (round to nearest even), for test inputs built from fp32 data. */
void synth_f32_to_bf16(int64_t n, const float* in, uint16_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = f32_to_bf16_rne(in[i]);
}

/* ---------------------------------------------------------------- lengths */

/* row lengths uniform in {a, ..., b}; returns the total */
int64_t synth_lengths_uniform(uint64_t seed, uint64_t tag, int64_t M, int32_t a, int32_t b, int32_t* len) {
    uint64_t k = stream_key(seed, tag);
    int64_t tot = 0;
    for (int64_t i = 0; i < M; ++i) {
        len[i] = a + (int32_t)below(draw(k, (uint64_t)i), (int64_t)b - a + 1);
        tot += len[i];
    }
    return tot;
}

/* Poisson(lambda) by inversion of the cumulative distribution. */
int64_t synth_lengths_poisson(uint64_t seed, uint64_t tag, int64_t M, double lambda, int32_t* len) {
    int kmax = (int)(lambda + 40.0 * sqrt(lambda) + 40.0);
    double* cdf = (double*)malloc(sizeof(double) * (size_t)(kmax + 1));
    double p = exp(-lambda), c = 0.0;
    for (int k = 0; k <= kmax; ++k) {
        c += p;
        cdf[k] = c;
        p *= lambda / (double)(k + 1);
    }
    uint64_t key = stream_key(seed, tag);
    int64_t tot = 0;
    for (int64_t i = 0; i < M; ++i) {
        double u = u01(draw(key, (uint64_t)i));
        int lo = 0, hi = kmax; /* first k with cdf[k] > u */
        while (lo < hi) {
            int mid = (lo + hi) / 2;
            if (cdf[mid] > u) hi = mid; else lo = mid + 1;
        }
        len[i] = lo;
        tot += lo;
    }
    free(cdf);
    return tot;
}

/*
 * Zipf(expo) on {1..lmax} by inversion, then every draw L is rescaled to
 * clamp(rint(s*L), 1, lmax) with the smallest s (bisection, 64 steps) whose
 * mean reaches target_mean.  Returns the total; *s_out receives s.
 */
int64_t synth_lengths_zipf(uint64_t seed, uint64_t tag, int64_t M, double expo, int32_t lmax,
                           double target_mean, int32_t* len, double* s_out) {
    double* cdf = (double*)malloc(sizeof(double) * (size_t)lmax);
    double c = 0.0;
    for (int32_t k = 1; k <= lmax; ++k) {
        c += pow((double)k, -expo);
        cdf[k - 1] = c;
    }
    for (int32_t k = 0; k < lmax; ++k) cdf[k] /= c;
    uint64_t key = stream_key(seed, tag);
    for (int64_t i = 0; i < M; ++i) {
        double u = u01(draw(key, (uint64_t)i));
        int32_t lo = 0, hi = lmax - 1;
        while (lo < hi) {
            int32_t mid = lo + (hi - lo) / 2;
            if (cdf[mid] > u) hi = mid; else lo = mid + 1;
        }
        len[i] = lo + 1;
    }
    free(cdf);
    double slo = 0.0, shi = target_mean > 1.0 ? target_mean : 1.0;
    double goal = target_mean * (double)M;
    for (int it = 0; it < 64; ++it) {
        double mid = 0.5 * (slo + shi);
        double tot = 0.0;
        for (int64_t i = 0; i < M; ++i) {
            double v = rint(mid * (double)len[i]);
            if (v < 1.0) v = 1.0;
            if (v > (double)lmax) v = (double)lmax;
            tot += v;
        }
        if (tot < goal) slo = mid; else shi = mid;
    }
    int64_t tot = 0;
    for (int64_t i = 0; i < M; ++i) {
        double v = rint(shi * (double)len[i]);
        if (v < 1.0) v = 1.0;
        if (v > (double)lmax) v = (double)lmax;
        len[i] = (int32_t)v;
        tot += len[i];
    }
    if (s_out) *s_out = shi;
    return tot;
}

/* ---------------------------------------------------------------- columns */

static int cmp_i32(const void* a, const void* b) {
    int32_t x = *(const int32_t*)a, y = *(const int32_t*)b;
    return (x > y) - (x < y);
}
/* ascending sort of non-negative ints: insertion sort when short, else an
   LSD radix sort (8-bit digits) through `tmp` (n ints) */
static void sort_i32(int32_t* a, int64_t n, int32_t* tmp) {
    if (n <= 24) {
        for (int64_t i = 1; i < n; ++i) {
            int32_t v = a[i];
            int64_t j = i - 1;
            while (j >= 0 && a[j] > v) { a[j + 1] = a[j]; --j; }
            a[j + 1] = v;
        }
        return;
    }
    if (!tmp) { qsort(a, (size_t)n, sizeof(int32_t), cmp_i32); return; }
    int32_t *src = a, *dst = tmp;
    for (int shift = 0; shift < 32; shift += 8) {
        int64_t cnt[257];
        memset(cnt, 0, sizeof(cnt));
        for (int64_t i = 0; i < n; ++i) cnt[(((uint32_t)src[i]) >> shift & 255u) + 1]++;
        for (int d = 0; d < 256; ++d) cnt[d + 1] += cnt[d];
        for (int64_t i = 0; i < n; ++i) dst[cnt[((uint32_t)src[i]) >> shift & 255u]++] = src[i];
        int32_t* t = src; src = dst; dst = t;
    }
    /* four passes: the result is back in a */
}
/* merge sorted a[0..na) and sorted b[0..nb) into out (no aliasing with b) */
static void merge_i32(const int32_t* a, int64_t na, const int32_t* b, int64_t nb, int32_t* out) {
    int64_t i = 0, j = 0, k = 0;
    while (i < na && j < nb) out[k++] = (b[j] < a[i]) ? b[j++] : a[i++];
    while (i < na) out[k++] = a[i++];
    while (j < nb) out[k++] = b[j++];
}
static int64_t unique_sorted(int32_t* a, int64_t n) {
    if (n == 0) return 0;
    int64_t m = 1;
    for (int64_t i = 1; i < n; ++i)
        if (a[i] != a[m - 1]) a[m++] = a[i];
    return m;
}

/*
 * l distinct sorted integers uniform over [lo, hi), written to out.
 * Sparse rows: draw, sort, drop repeats and redraw the shortfall (attempt a
 * uses counter block a), merging the new draws into the kept ones.
 * Dense rows (l > range/4): partial Fisher-Yates.
 * `scratch` must hold 4*l ints (the dense case has range < 4*l).
 */
static void distinct_sorted(uint64_t rowkey, int64_t lo, int64_t hi, int64_t l, int32_t* out, int32_t* scratch) {
    int64_t range = hi - lo;
    if (l <= 0) return;
    if (l * 4 > range) {
        for (int64_t i = 0; i < range; ++i) scratch[i] = (int32_t)(lo + i);
        for (int64_t i = 0; i < l; ++i) {
            int64_t j = i + below(draw(rowkey, (uint64_t)i), range - i);
            int32_t t = scratch[i]; scratch[i] = scratch[j]; scratch[j] = t;
        }
        memcpy(out, scratch, sizeof(int32_t) * (size_t)l);
        sort_i32(out, l, scratch + l);
        return;
    }
    int32_t* fresh = scratch;       /* l ints */
    int32_t* tmp = scratch + l;     /* l ints: radix buffer */
    int32_t* merged = scratch + 2 * l; /* l ints */
    int64_t have = 0;
    uint64_t attempt = 0;
    while (have < l) {
        int64_t need = l - have;
        for (int64_t i = 0; i < need; ++i)
            fresh[i] = (int32_t)(lo + below(draw(rowkey, (attempt << 32) | (uint64_t)i), range));
        sort_i32(fresh, need, tmp);
        merge_i32(out, have, fresh, need, merged);
        have = unique_sorted(merged, l);
        memcpy(out, merged, sizeof(int32_t) * (size_t)have);
        ++attempt;
    }
}

/* Row i gets len[i] distinct sorted columns uniform over [0, K).  Output is
   COO in row-major order: row_out[p] = i, col_out[p] = column. */
void synth_cols_uniform(uint64_t seed, uint64_t tag, int64_t M, int64_t K, const int32_t* len,
                        int32_t* row_out, int32_t* col_out) {
    uint64_t key = stream_key(seed, tag);
    int64_t mx = 0;
    for (int64_t i = 0; i < M; ++i) if (len[i] > mx) mx = len[i];
    int32_t* scratch = (int32_t*)malloc(sizeof(int32_t) * (size_t)(4 * mx + 1));
    int64_t p = 0;
    for (int64_t i = 0; i < M; ++i) {
        uint64_t rk = mix64(key ^ ((uint64_t)i * 0xA24BAED4963EE407ULL));
        distinct_sorted(rk, 0, K, len[i], col_out + p, scratch);
        for (int64_t q = 0; q < len[i]; ++q) row_out[p + q] = (int32_t)i;
        p += len[i];
    }
    free(scratch);
}

/*
 * Banded rows with outliers: each entry of row i is, with probability
 * `outlier`, uniform over [0, K); otherwise uniform over the band
 * [c - half, c + half) clipped to [0, K), with c = floor(i * num / den).
 * Repeats are redrawn (same rule, next attempt); columns end sorted.
 */
void synth_cols_band(uint64_t seed, uint64_t tag, int64_t M, int64_t K, const int32_t* len, int64_t half,
                     double outlier, int64_t num, int64_t den, int32_t* row_out, int32_t* col_out) {
    uint64_t key = stream_key(seed, tag);
    int64_t p = 0;
    for (int64_t i = 0; i < M; ++i) {
        uint64_t rk = mix64(key ^ ((uint64_t)i * 0xA24BAED4963EE407ULL));
        int64_t c = (i * num) / den;
        int64_t lo = c - half < 0 ? 0 : c - half;
        int64_t hi = c + half > K ? K : c + half;
        int64_t l = len[i];
        int32_t* out = col_out + p;
        int64_t have = 0;
        uint64_t attempt = 0;
        while (have < l) {
            int64_t need = l - have;
            for (int64_t q = 0; q < need; ++q) {
                uint64_t ctr = (attempt << 33) | ((uint64_t)q << 1);
                double u = u01(draw(rk, ctr));
                uint64_t z = draw(rk, ctr | 1u);
                out[have + q] = (int32_t)(u < outlier ? below(z, K) : lo + below(z, hi - lo));
            }
            sort_i32(out, l, NULL);
            have = unique_sorted(out, l);
            ++attempt;
        }
        for (int64_t q = 0; q < l; ++q) row_out[p + q] = (int32_t)i;
        p += l;
    }
}

/*
 * 4x4-clustered columns.  Rows come in groups of four (4g .. 4g+3).  Each
 * group draws a sequence of distinct column quads q in [0, K/4) (quad q is
 * columns 4q .. 4q+3); row i takes the first ceil(len[i]/4) quads of its
 * group's sequence, the last one cut to the first (len[i] mod 4) columns when
 * len[i] is not a multiple of 4.  Columns end sorted.  Needs K % 4 == 0 and
 * 4*ceil(len/4) <= K.
 */
void synth_cols_quads(uint64_t seed, uint64_t tag, int64_t M, int64_t K, const int32_t* len,
                      int32_t* row_out, int32_t* col_out) {
    uint64_t key = stream_key(seed, tag);
    int64_t nq = K / 4;
    int64_t mx = 0;
    for (int64_t i = 0; i < M; ++i) if (len[i] > mx) mx = len[i];
    int64_t mq = (mx + 3) / 4;
    int32_t* seq = (int32_t*)malloc(sizeof(int32_t) * (size_t)(mq + 1));
    int32_t* tmp = (int32_t*)malloc(sizeof(int32_t) * (size_t)(4 * mq + 4));
    int64_t p = 0;
    for (int64_t g = 0; g * 4 < M; ++g) {
        int64_t r0 = 4 * g, r1 = r0 + 4 < M ? r0 + 4 : M;
        int64_t need = 0;
        for (int64_t i = r0; i < r1; ++i) { int64_t t = (len[i] + 3) / 4; if (t > need) need = t; }
        uint64_t gk = mix64(key ^ ((uint64_t)g * 0xA24BAED4963EE407ULL));
        /* sequence of distinct quads, in draw order; repeats are skipped */
        int64_t have = 0;
        uint64_t ctr = 0;
        while (have < need) {
            int32_t q = (int32_t)below(draw(gk, ctr++), nq);
            int dup = 0;
            for (int64_t t = 0; t < have; ++t) if (seq[t] == q) { dup = 1; break; }
            if (!dup) seq[have++] = q;
        }
        for (int64_t i = r0; i < r1; ++i) {
            int64_t l = len[i], full = l / 4, rem = l % 4, nqr = (l + 3) / 4;
            int64_t n = 0;
            for (int64_t t = 0; t < nqr; ++t) {
                int64_t w = (t < full) ? 4 : rem;
                for (int64_t c = 0; c < w; ++c) tmp[n++] = 4 * seq[t] + (int32_t)c;
            }
            sort_i32(tmp, n, NULL);
            memcpy(col_out + p, tmp, sizeof(int32_t) * (size_t)n);
            for (int64_t q = 0; q < n; ++q) row_out[p + q] = (int32_t)i;
            p += n;
        }
    }
    free(seq); free(tmp);
}

/*
 * Block pattern: for each of the MB block-rows, `per_row` distinct block
 * columns uniform over [0, KB) without replacement, sorted; bcol_out has
 * MB*per_row entries.
 */
void synth_block_cols(uint64_t seed, uint64_t tag, int64_t MB, int64_t KB, int64_t per_row, int32_t* bcol_out) {
    uint64_t key = stream_key(seed, tag);
    int32_t* scratch = (int32_t*)malloc(sizeof(int32_t) * (size_t)(4 * per_row + 1));
    for (int64_t I = 0; I < MB; ++I) {
        uint64_t rk = mix64(key ^ ((uint64_t)I * 0xA24BAED4963EE407ULL));
        distinct_sorted(rk, 0, KB, per_row, bcol_out + I * per_row, scratch);
    }
    free(scratch);
}

/* Fisher-Yates permutation of 0..n-1 (for shuffled COO inputs). */
void synth_permutation(uint64_t seed, uint64_t tag, int64_t n, int64_t* perm) {
    uint64_t key = stream_key(seed, tag);
    for (int64_t i = 0; i < n; ++i) perm[i] = i;
    for (int64_t i = n - 1; i > 0; --i) {
        int64_t j = below(draw(key, (uint64_t)i), i + 1);
        int64_t t = perm[i]; perm[i] = perm[j]; perm[j] = t;
    }
}
