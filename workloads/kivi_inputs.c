/*
 * kivi_inputs.c -- seeded synthetic K/V tensors for tests and benchmarks.
 *
 * This module only draws random numbers; it holds none of the quantizer's
 * arithmetic.  Both the oracle and the CUDA library are fed from it.
 *
 * Every element is a pure function of (seed, tensor, bh, token, channel):
 * a counter-based generator (the SplitMix64 finaliser applied to a counter),
 * so a tensor is bit-identical for any thread count, any token window and
 * any chunking, and tokens appended later in a sequence are the same values
 * whichever window generated them.
 *
 * Distributions (double precision, then rounded to IEEE binary16, saturated
 * at +-65504):
 *   normal     Box-Muller (cosine branch) from two uniforms
 *   student-t  Z / sqrt(chi2_nu / nu) with chi2_nu a sum of nu squared normals
 *              (integer nu)
 *   laplace    inverse CDF, scale 1
 * Key structure: per (tensor, head) a set of outlier channels (partial
 * Fisher-Yates draw, or a fixed list) multiplied by a constant, and an
 * optional per (head, channel) offset drawn from U(-amp, amp).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { KG_NORMAL = 0, KG_STUDENT_T = 1, KG_LAPLACE = 2 };

typedef struct {
    uint64_t seed;            /* workload seed */
    uint64_t tensor;          /* layer * 2 + (0 keys | 1 values) */
    int32_t dist;             /* KG_* */
    int32_t nu;               /* student-t degrees of freedom */
    double sigma;             /* scale applied to the base draw */
    int32_t heads;            /* kv heads: head = bh % heads */
    int32_t n_outliers;       /* outlier channels per head */
    double outlier_mult;      /* multiplier of outlier channels */
    const int32_t *fixed_outliers; /* non-NULL: this list for every head */
    double offset_amp;        /* per (head, channel) offset U(-amp, amp); 0 = none */
} kivi_gen_spec;

static uint64_t mix64(uint64_t z)
{
    z += 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

/* uniform in (0, 1] with 53 random bits */
static double unit(uint64_t r) { return ((double)(r >> 11) + 1.0) * 0x1.0p-53; }

static uint64_t stream_key(const kivi_gen_spec *s, uint64_t purpose)
{
    return mix64(mix64(s->seed * 0xD1B54A32D192ED03ull + purpose) ^ (s->tensor * 0x8CB92BA72F3D8DD7ull));
}

static double normal_at(uint64_t key, uint64_t ctr, int j)
{
    const double u1 = unit(mix64(key + ctr * 32u + 2u * (uint64_t)j));
    const double u2 = unit(mix64(key + ctr * 32u + 2u * (uint64_t)j + 1u));
    return sqrt(-2.0 * log(u1)) * cos(6.283185307179586 * u2);
}

static double draw(const kivi_gen_spec *s, uint64_t key, uint64_t ctr)
{
    switch (s->dist) {
    case KG_STUDENT_T: {
        const double z = normal_at(key, ctr, 0);
        double chi2 = 0.0;
        for (int k = 0; k < s->nu; ++k) {
            const double n = normal_at(key, ctr, 1 + k);
            chi2 += n * n;
        }
        return z / sqrt(chi2 / (double)s->nu);
    }
    case KG_LAPLACE: {
        const double u = unit(mix64(key + ctr * 32u)) - 0x1.0p-54;  /* (0, 1) */
        return u < 0.5 ? log(2.0 * u) : -log(2.0 * (1.0 - u));
    }
    default:
        return normal_at(key, ctr, 0);
    }
}

static uint16_t to_half_bits(double v)
{
    if (v > 65504.0) v = 65504.0;
    if (v < -65504.0) v = -65504.0;
    _Float16 h = (_Float16)v;
    uint16_t b;
    memcpy(&b, &h, sizeof b);
    return b;
}

typedef struct {
    const kivi_gen_spec *spec;
    uint16_t *out;
    int64_t r0, r1;               /* flat (bh, token) row range */
    int64_t bh0;                  /* bh index of the first output slice */
    int64_t tok0, n_tok, d, out_bh_stride;
    const uint8_t *outlier_mask;  /* [heads][d] */
    const double *offset;         /* [heads][d] or NULL */
} job_t;

static void *fill_range(void *arg)
{
    const job_t *j = (const job_t *)arg;
    const kivi_gen_spec *s = j->spec;
    const uint64_t key = stream_key(s, 1);
    for (int64_t r = j->r0; r < j->r1; ++r) {
        const int64_t b = r / j->n_tok, i = r % j->n_tok;
        const int64_t gb = j->bh0 + b;            /* bh index in the whole tensor */
        const int64_t head = gb % s->heads;
        const uint64_t t = (uint64_t)(j->tok0 + i);
        uint16_t *row = j->out + b * j->out_bh_stride + i * j->d;
        for (int64_t c = 0; c < j->d; ++c) {
            const uint64_t ctr = ((uint64_t)gb << 40) ^ (t << 16) ^ (uint64_t)c;
            double v = s->sigma * draw(s, key, ctr);
            if (j->outlier_mask[head * j->d + c]) v *= s->outlier_mult;
            if (j->offset) v += j->offset[head * j->d + c];
            row[c] = to_half_bits(v);
        }
    }
    return NULL;
}

/* Fill out[b * out_bh_stride + i * d + c] for b < bh, i < n_tok, c < d with
 * the value of bh slice bh0 + b at sequence position tok0 + i.  Returns 0, or
 * -1 on bad input. */
int kivi_gen_fill_range(const kivi_gen_spec *spec, uint16_t *out, int64_t bh0, int64_t bh,
                        int64_t tok0, int64_t n_tok, int64_t d, int64_t out_bh_stride,
                        int n_threads)
{
    if (!spec || !out || bh0 < 0 || bh < 0 || tok0 < 0 || n_tok < 0 || d <= 0 || d >= 65536)
        return -1;
    if (spec->heads <= 0 || spec->n_outliers < 0 || spec->n_outliers > d) return -1;
    /* the counter packs bh, token and channel into disjoint bit fields */
    if (bh0 + bh >= ((int64_t)1 << 19) || tok0 + n_tok >= ((int64_t)1 << 24)) return -1;
    if (out_bh_stride < n_tok * d) return -1;
    if (n_threads < 1) n_threads = 1;

    uint8_t *mask = (uint8_t *)calloc((size_t)spec->heads * (size_t)d, 1);
    double *offset = NULL;
    int32_t *perm = (int32_t *)malloc(sizeof(int32_t) * (size_t)d);
    if (!mask || !perm) { free(mask); free(perm); return -1; }

    const uint64_t okey = stream_key(spec, 2);
    for (int h = 0; h < spec->heads; ++h) {
        if (spec->fixed_outliers) {
            for (int k = 0; k < spec->n_outliers; ++k) {
                const int32_t c = spec->fixed_outliers[k];
                if (c < 0 || c >= d) { free(mask); free(perm); return -1; }
                mask[(size_t)h * d + c] = 1;
            }
        } else {
            for (int64_t c = 0; c < d; ++c) perm[c] = (int32_t)c;
            for (int k = 0; k < spec->n_outliers; ++k) {
                const uint64_t r = mix64(okey + (uint64_t)h * 4096u + (uint64_t)k);
                const int64_t jx = k + (int64_t)(r % (uint64_t)(d - k));
                const int32_t tmp = perm[k]; perm[k] = perm[jx]; perm[jx] = tmp;
                mask[(size_t)h * d + perm[k]] = 1;
            }
        }
    }
    if (spec->offset_amp > 0.0) {
        offset = (double *)malloc(sizeof(double) * (size_t)spec->heads * (size_t)d);
        if (!offset) { free(mask); free(perm); return -1; }
        const uint64_t fkey = stream_key(spec, 3);
        for (int h = 0; h < spec->heads; ++h)
            for (int64_t c = 0; c < d; ++c) {
                const double u = unit(mix64(fkey + (uint64_t)h * 65536u + (uint64_t)c));
                offset[(size_t)h * d + c] = spec->offset_amp * (2.0 * u - 1.0);
            }
    }

    const int64_t rows = bh * n_tok;
    if (rows == 0) { free(mask); free(offset); free(perm); return 0; }
    if (n_threads > rows) n_threads = (int)rows;
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)n_threads);
    job_t *jobs = (job_t *)malloc(sizeof(job_t) * (size_t)n_threads);
    int rc = 0;
    if (!th || !jobs) rc = -1;
    if (rc == 0) {
        for (int k = 0; k < n_threads; ++k) {
            jobs[k] = (job_t){spec, out, rows * k / n_threads, rows * (k + 1) / n_threads,
                              bh0, tok0, n_tok, d, out_bh_stride, mask, offset};
        }
        if (n_threads == 1) {
            fill_range(&jobs[0]);
        } else {
            int started = 0;
            for (int k = 0; k < n_threads; ++k) {
                if (pthread_create(&th[k], NULL, fill_range, &jobs[k]) != 0) { rc = -1; break; }
                ++started;
            }
            for (int k = 0; k < started; ++k) pthread_join(th[k], NULL);
            if (rc != 0) {  /* finish whatever was not started, serially */
                for (int k = started; k < n_threads; ++k) fill_range(&jobs[k]);
                rc = 0;
            }
        }
    }
    free(th); free(jobs); free(mask); free(offset); free(perm);
    return rc;
}

/* kivi_gen_fill_range from bh slice 0. */
int kivi_gen_fill(const kivi_gen_spec *spec, uint16_t *out, int64_t bh, int64_t tok0,
                  int64_t n_tok, int64_t d, int64_t out_bh_stride, int n_threads)
{
    return kivi_gen_fill_range(spec, out, 0, bh, tok0, n_tok, d, out_bh_stride, n_threads);
}

/* The outlier channel set of one head (for tests): writes n_outliers indices. */
int kivi_gen_outliers(const kivi_gen_spec *spec, int64_t d, int head, int32_t *out)
{
    if (!spec || d <= 0 || spec->n_outliers > d) return -1;
    if (spec->fixed_outliers) {
        for (int k = 0; k < spec->n_outliers; ++k) out[k] = spec->fixed_outliers[k];
        return 0;
    }
    int32_t *perm = (int32_t *)malloc(sizeof(int32_t) * (size_t)d);
    if (!perm) return -1;
    for (int64_t c = 0; c < d; ++c) perm[c] = (int32_t)c;
    const uint64_t okey = stream_key(spec, 2);
    for (int k = 0; k < spec->n_outliers; ++k) {
        const uint64_t r = mix64(okey + (uint64_t)head * 4096u + (uint64_t)k);
        const int64_t jx = k + (int64_t)(r % (uint64_t)(d - k));
        const int32_t tmp = perm[k]; perm[k] = perm[jx]; perm[jx] = tmp;
        out[k] = perm[k];
    }
    free(perm);
    return 0;
}
