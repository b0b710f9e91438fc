/*
 * kivi_oracle.c -- plain CPU oracle for the KIVI KV-cache flush.
 *
 * TEST INFRASTRUCTURE ONLY: used by the tests, the smoke check and the
 * benchmark's CPU-baseline leg; never by the product path.  It shares no code
 * with the CUDA library.
 *
 * Written for a reader checking it against the pages by eye: one group at a
 * time, one element at a time, in the order the method is stated
 * (VeloxQuant-MLX blog post "How I fused KIVI's KV-cache quantization into two
 * bit-exact Metal kernels ..." -- sections "What we're actually optimizing",
 * "The layout problem that shapes everything", "Three ways to be off by one
 * bit"; release post "VeloxQuant-MLX 0.8.0 adds KIVI" -- "What KIVI is").
 *
 * Build: a C11 compiler with -O2 -ffp-contract=off -fno-fast-math so that
 * every binary32 operation below is a single IEEE operation.
 */
#include "kivi_oracle.h"

#include <fenv.h>
#include <math.h>
#include <stdlib.h>
#include <string.h>

#define KIVI_ORACLE_MAX_GROUP 128

static int valid_bits(int bits) { return bits == 2 || bits == 4 || bits == 8; }
static int valid_group(int g) { return g == 16 || g == 32 || g == 64 || g == 128; }
static uint32_t qmax_of(int bits) { return (1u << bits) - 1u; }
static int codes_per_word(int bits) { return 32 / bits; }

/* ------------------------------------------------------------------------ */
/* IEEE binary16 <-> binary32                                               */
/* ------------------------------------------------------------------------ */

/* binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.
 * Exponent field 0 encodes zero and subnormals (fraction * 2^-24), field 31
 * encodes infinity (fraction 0) and NaN. */
float kivi_oracle_half_to_float(uint16_t h)
{
    const int sign = (h >> 15) & 1;
    const int efield = (h >> 10) & 0x1F;
    const int frac = h & 0x3FF;
    float mag;
    if (efield == 0) {
        mag = ldexpf((float)frac, -24);                 /* exact */
    } else if (efield == 31) {
        mag = frac ? NAN : INFINITY;
    } else {
        mag = ldexpf((float)(1024 + frac), efield - 25); /* exact */
    }
    return sign ? -mag : mag;
}

/* Round |f| to the binary16 grid: find the binade exponent e of |f| (never
 * below -14, the subnormal binade), express |f| in units of that binade's
 * spacing 2^(e-10) (an exact power-of-two scaling), round that unit count to
 * the nearest integer with ties to even, and re-normalise if rounding carried
 * into the next binade.  Values past the largest finite half round to
 * infinity exactly as the unbounded-exponent rounding would. */
uint16_t kivi_oracle_float_to_half(float f)
{
    uint32_t fb;
    memcpy(&fb, &f, sizeof fb);
    const uint16_t sign = (uint16_t)((fb >> 16) & 0x8000u);
    if (isnan(f)) return (uint16_t)(sign | 0x7E00u);
    const float a = fabsf(f);
    if (isinf(a)) return (uint16_t)(sign | 0x7C00u);
    if (a == 0.0f) return sign;

    int k;
    (void)frexpf(a, &k);            /* a = m * 2^k, m in [0.5, 1) */
    int e = k - 1;                  /* 2^e <= a < 2^(e+1) */
    if (e < -14) e = -14;
    const float units = ldexpf(a, 10 - e);   /* exact */
    float n = nearbyintf(units);    /* ties to even under FE_TONEAREST */
    if (n >= 2048.0f) {             /* carried into the next binade */
        n = 1024.0f;
        e += 1;
    }
    if (e > 15) return (uint16_t)(sign | 0x7C00u);
    const uint32_t ni = (uint32_t)n;
    if (ni < 1024u) return (uint16_t)(sign | ni);     /* subnormal (e == -14) */
    return (uint16_t)(sign | (uint32_t)((e + 15) << 10) | (ni - 1024u));
}

void kivi_oracle_halves_to_floats(const uint16_t *h, float *f, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) f[i] = kivi_oracle_half_to_float(h[i]);
}

void kivi_oracle_floats_to_halves(const float *f, uint16_t *h, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) h[i] = kivi_oracle_float_to_half(f[i]);
}

/* ------------------------------------------------------------------------ */
/* The quantizer                                                            */
/* ------------------------------------------------------------------------ */

int kivi_oracle_group_params(const float *vals, int64_t n, int bits,
                             float *scale, float *zero)
{
    if (!valid_bits(bits) || n <= 0) return -1;
    if (fegetround() != FE_TONEAREST) return -1;
    for (int64_t i = 0; i < n; ++i)
        if (!isfinite(vals[i])) return -1;

    float mn = vals[0];
    float mx = vals[0];
    for (int64_t i = 1; i < n; ++i) {
        if (vals[i] < mn) mn = vals[i];
        if (vals[i] > mx) mx = vals[i];
    }
    /* A zero extreme may be -0 or +0 depending on which was seen first; adding
     * +0 makes it +0 either way, so the result does not depend on order. */
    mn = mn + 0.0f;
    mx = mx + 0.0f;

    *zero = mn;
    *scale = (mx - mn) / (float)qmax_of(bits);
    return 0;
}

uint32_t kivi_oracle_code(float x, float scale, float zero, int bits)
{
    if (!valid_bits(bits)) return 0xFFFFFFFFu;
    if (scale == 0.0f) return 0u;                 /* max == min */
    const float t = x - zero;
    const float u = t / scale;
    float r = nearbyintf(u);                      /* round half to even */
    if (r < 0.0f) r = 0.0f;                       /* clip */
    if (r > (float)qmax_of(bits)) r = (float)qmax_of(bits);
    return (uint32_t)r;
}

uint16_t kivi_oracle_recon(uint32_t q, float scale, float zero)
{
    /* Two roundings: the product is rounded to binary32 before the add. */
    volatile float prod = (float)q * scale;
    const float r = prod + zero;
    return kivi_oracle_float_to_half(r);
}

/* Quantize G gathered values of one group into codes q[0..G). */
static int quantize_group(const float *vals, int group, int bits,
                          uint32_t *q, float *scale, float *zero)
{
    if (kivi_oracle_group_params(vals, group, bits, scale, zero) != 0) return -1;
    for (int i = 0; i < group; ++i) q[i] = kivi_oracle_code(vals[i], *scale, *zero, bits);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Keys: one (scale, zero) per channel per group of G tokens                */
/* ------------------------------------------------------------------------ */

/* Token i of group g of channel c, with the ragged tail padded by repeating
 * the last token ([POST] "3. Padding semantics"). */
static float key_value(const uint16_t *x_bh, int64_t s, int64_t d,
                       int64_t g, int64_t c, int group, int i)
{
    int64_t t = g * group + i;
    if (t > s - 1) t = s - 1;
    return kivi_oracle_half_to_float(x_bh[t * d + c]);
}

int kivi_oracle_key_group(const uint16_t *x_bh, int64_t s, int64_t d,
                          int64_t g, int64_t c, int group, int bits,
                          uint32_t *words, float *scale, float *zero)
{
    if (!valid_bits(bits) || !valid_group(group) || s <= 0 || d <= 0) return -1;
    if (g < 0 || g * group >= s || c < 0 || c >= d) return -1;
    float vals[KIVI_ORACLE_MAX_GROUP];
    uint32_t q[KIVI_ORACLE_MAX_GROUP];
    for (int i = 0; i < group; ++i) vals[i] = key_value(x_bh, s, d, g, c, group, i);
    if (quantize_group(vals, group, bits, q, scale, zero) != 0) return -1;
    const int w = codes_per_word(bits);
    for (int j = 0; j < group / w; ++j) words[j] = 0u;
    for (int i = 0; i < group; ++i) words[i / w] |= q[i] << ((i % w) * bits);
    return 0;
}

int kivi_oracle_quantize_keys(const uint16_t *x, int64_t bh, int64_t s, int64_t d,
                              int group, int bits,
                              uint32_t *codes, float *scale, float *zero)
{
    if (!valid_bits(bits) || !valid_group(group) || bh < 0 || s < 0 || d <= 0) return -1;
    if (bh == 0 || s == 0) return 0;
    const int w = codes_per_word(bits);
    const int64_t ng = (s + group - 1) / group;
    const int64_t rows = ng * group / w;           /* code word rows per bh */
    uint32_t words[KIVI_ORACLE_MAX_GROUP];
    for (int64_t b = 0; b < bh; ++b) {
        const uint16_t *x_bh = x + b * s * d;
        for (int64_t g = 0; g < ng; ++g) {
            for (int64_t c = 0; c < d; ++c) {
                float sc, ze;
                if (kivi_oracle_key_group(x_bh, s, d, g, c, group, bits, words, &sc, &ze) != 0)
                    return -1;
                scale[(b * ng + g) * d + c] = sc;
                zero[(b * ng + g) * d + c] = ze;
                for (int j = 0; j < group / w; ++j)
                    codes[(b * rows + g * (group / w) + j) * d + c] = words[j];
            }
        }
    }
    return 0;
}

int kivi_oracle_dequantize_keys(const uint32_t *codes, const float *scale,
                                const float *zero, int64_t bh, int64_t s, int64_t d,
                                int group, int bits, uint16_t *y)
{
    if (!valid_bits(bits) || !valid_group(group) || bh < 0 || s < 0 || d <= 0) return -1;
    const int w = codes_per_word(bits);
    const int64_t ng = (s + group - 1) / group;
    const int64_t rows = ng * group / w;
    for (int64_t b = 0; b < bh; ++b)
        for (int64_t t = 0; t < s; ++t)
            for (int64_t c = 0; c < d; ++c) {
                const uint32_t word = codes[(b * rows + t / w) * d + c];
                const uint32_t q = (word >> ((t % w) * bits)) & qmax_of(bits);
                const int64_t p = (b * ng + t / group) * d + c;
                y[(b * s + t) * d + c] = kivi_oracle_recon(q, scale[p], zero[p]);
            }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Values: one (scale, zero) per token per group of G channels              */
/* ------------------------------------------------------------------------ */

int kivi_oracle_value_row(const uint16_t *x_row, int64_t d, int group, int bits,
                          uint32_t *words, float *scale, float *zero)
{
    if (!valid_bits(bits) || !valid_group(group) || d <= 0 || d % group != 0) return -1;
    const int w = codes_per_word(bits);
    float vals[KIVI_ORACLE_MAX_GROUP];
    uint32_t q[KIVI_ORACLE_MAX_GROUP];
    for (int64_t j = 0; j < d / w; ++j) words[j] = 0u;
    for (int64_t g = 0; g < d / group; ++g) {
        for (int i = 0; i < group; ++i) vals[i] = kivi_oracle_half_to_float(x_row[g * group + i]);
        if (quantize_group(vals, group, bits, q, &scale[g], &zero[g]) != 0) return -1;
        for (int i = 0; i < group; ++i) {
            const int64_t c = g * group + i;
            words[c / w] |= q[i] << ((c % w) * bits);
        }
    }
    return 0;
}

int kivi_oracle_quantize_values(const uint16_t *x, int64_t bh, int64_t s, int64_t d,
                                int group, int bits,
                                uint32_t *codes, float *scale, float *zero)
{
    if (!valid_bits(bits) || !valid_group(group) || bh < 0 || s < 0 || d <= 0) return -1;
    if (d % group != 0) return -1;
    const int w = codes_per_word(bits);
    for (int64_t r = 0; r < bh * s; ++r) {
        if (kivi_oracle_value_row(x + r * d, d, group, bits, codes + r * (d / w),
                                  scale + r * (d / group), zero + r * (d / group)) != 0)
            return -1;
    }
    return 0;
}

int kivi_oracle_dequantize_values(const uint32_t *codes, const float *scale,
                                  const float *zero, int64_t bh, int64_t s, int64_t d,
                                  int group, int bits, uint16_t *y)
{
    if (!valid_bits(bits) || !valid_group(group) || bh < 0 || s < 0 || d <= 0) return -1;
    if (d % group != 0) return -1;
    const int w = codes_per_word(bits);
    for (int64_t r = 0; r < bh * s; ++r)
        for (int64_t c = 0; c < d; ++c) {
            const uint32_t word = codes[r * (d / w) + c / w];
            const uint32_t q = (word >> ((c % w) * bits)) & qmax_of(bits);
            const int64_t p = r * (d / group) + c / group;
            y[r * d + c] = kivi_oracle_recon(q, scale[p], zero[p]);
        }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Residual window and flush                                                */
/* ------------------------------------------------------------------------ */

int64_t kivi_oracle_flush_size(int64_t n_res, int residual, int group)
{
    if (group <= 0 || residual < 0 || n_res < 0) return -1;
    if (n_res < (int64_t)residual + group) return 0;
    return ((n_res - residual) / group) * group;
}

int kivi_oracle_append(uint16_t *k_res, uint16_t *v_res, int64_t bh, int64_t d, int64_t r_cap,
                       int64_t res_head, int64_t *n_res, const uint16_t *k_new,
                       const uint16_t *v_new, int64_t n)
{
    if (bh < 0 || d <= 0 || r_cap <= 0 || n < 0) return -1;
    if (res_head < 0 || res_head >= r_cap || *n_res < 0 || *n_res > r_cap) return -1;
    if (*n_res + n > r_cap) return -3;
    for (int64_t b = 0; b < bh; ++b) {
        for (int64_t i = 0; i < n; ++i) {
            /* new token i becomes logical residual token n_res + i */
            const int64_t row = (res_head + *n_res + i) % r_cap;
            for (int64_t c = 0; c < d; ++c) {
                k_res[(b * r_cap + row) * d + c] = k_new[(b * n + i) * d + c];
                v_res[(b * r_cap + row) * d + c] = v_new[(b * n + i) * d + c];
            }
        }
    }
    *n_res += n;
    return 0;
}

int64_t kivi_oracle_flush(const uint16_t *k_res, const uint16_t *v_res,
                          int64_t bh, int64_t d, int64_t r_cap, int64_t cap,
                          int group, int bits, int residual,
                          uint32_t *k_codes, float *k_scale, float *k_zero,
                          uint32_t *v_codes, float *v_scale, float *v_zero,
                          int64_t *s_q, int64_t *res_head, int64_t *n_res)
{
    if (!valid_bits(bits) || !valid_group(group) || residual < 0) return -1;
    if (bh < 0 || d <= 0 || d % group != 0 || r_cap <= 0 || cap < 0) return -1;
    if (*s_q < 0 || *s_q % group != 0 || *n_res < 0 || *n_res > r_cap) return -1;
    if (*res_head < 0 || *res_head >= r_cap) return -1;

    const int64_t n = kivi_oracle_flush_size(*n_res, residual, group);
    if (n == 0) return 0;
    if (*s_q + n > cap) return -3;

    const int w = codes_per_word(bits);
    const int64_t head = *res_head;
    float vals[KIVI_ORACLE_MAX_GROUP];
    uint32_t q[KIVI_ORACLE_MAX_GROUP];

    for (int64_t b = 0; b < bh; ++b) {
        /* keys: group j of the flushed tokens, channel c */
        for (int64_t j = 0; j < n / group; ++j) {
            for (int64_t c = 0; c < d; ++c) {
                for (int i = 0; i < group; ++i) {
                    const int64_t row = (head + j * group + i) % r_cap;
                    vals[i] = kivi_oracle_half_to_float(k_res[(b * r_cap + row) * d + c]);
                }
                float sc, ze;
                if (quantize_group(vals, group, bits, q, &sc, &ze) != 0) return -1;
                const int64_t gq = *s_q / group + j;            /* store group */
                k_scale[(b * (cap / group) + gq) * d + c] = sc;
                k_zero[(b * (cap / group) + gq) * d + c] = ze;
                for (int i = 0; i < group; ++i) {
                    const int64_t t = gq * group + i;            /* store token */
                    uint32_t *word = &k_codes[(b * (cap / w) + t / w) * d + c];
                    if (i % w == 0) *word = 0u;
                    *word |= q[i] << ((t % w) * bits);
                }
            }
        }
        /* values: each flushed token's row */
        for (int64_t i = 0; i < n; ++i) {
            const int64_t row = (head + i) % r_cap;
            const int64_t t = *s_q + i;
            if (kivi_oracle_value_row(v_res + (b * r_cap + row) * d, d, group, bits,
                                      v_codes + (b * cap + t) * (d / w),
                                      v_scale + (b * cap + t) * (d / group),
                                      v_zero + (b * cap + t) * (d / group)) != 0)
                return -1;
        }
    }
    *s_q += n;
    *res_head = (head + n) % r_cap;
    *n_res -= n;
    return n;
}

/* ------------------------------------------------------------------------ */
/* Decode attention over the reconstructed cache (binary64)                  */
/* ------------------------------------------------------------------------ */

int kivi_oracle_attention(const uint16_t *q, int64_t r, const uint16_t *k,
                          const uint16_t *v, int64_t n, int64_t d, double scale,
                          double *out) {
    if (n < 1 || r < 1 || d < 1) return -1;
    double *s = (double *)malloc((size_t)n * sizeof(double));
    if (!s) return -1;
    for (int64_t h = 0; h < r; ++h) {
        /* scores */
        double mx = -INFINITY;
        for (int64_t t = 0; t < n; ++t) {
            double dot = 0.0;
            for (int64_t c = 0; c < d; ++c)
                dot += (double)kivi_oracle_half_to_float(q[h * d + c]) *
                       (double)kivi_oracle_half_to_float(k[t * d + c]);
            s[t] = scale * dot;
            if (s[t] > mx) mx = s[t];
        }
        /* softmax weights */
        double den = 0.0;
        for (int64_t t = 0; t < n; ++t) {
            s[t] = exp(s[t] - mx);
            den += s[t];
        }
        /* weighted sum of the values */
        for (int64_t c = 0; c < d; ++c) {
            double acc = 0.0;
            for (int64_t t = 0; t < n; ++t)
                acc += (s[t] / den) * (double)kivi_oracle_half_to_float(v[t * d + c]);
            out[h * d + c] = acc;
        }
    }
    free(s);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* KIVI-Sink: high key-norm tokens kept fp16 and out of the calibration     */
/* (VeloxQuant-MLX project description, "KVSink-adapted sink protection")   */
/* ------------------------------------------------------------------------ */

int kivi_oracle_sink_scores(const uint16_t *k, int64_t batch, int64_t heads, int64_t n,
                            int64_t d, int64_t bh_stride, float *score)
{
    if (batch < 0 || heads <= 0 || n < 0 || d <= 0 || bh_stride < n * d) return -1;
    for (int64_t b = 0; b < batch; ++b)
        for (int64_t t = 0; t < n; ++t) {
            float sum = 0.0f;
            for (int64_t h = 0; h < heads; ++h) {
                const uint16_t *row = k + (b * heads + h) * bh_stride + t * d;
                float acc = 0.0f;                      /* squared L2 norm, in channel order */
                for (int64_t c = 0; c < d; ++c) {
                    const float x = kivi_oracle_half_to_float(row[c]);
                    acc = fmaf(x, x, acc);
                }
                sum = sum + sqrtf(acc);                /* norms summed in head order */
            }
            score[b * n + t] = sum / (float)heads;    /* mean over the KV heads */
        }
    return 0;
}

/* a before b in the ranking: larger score, then smaller position */
static int ranks_before(float sa, int64_t pa, float sb, int64_t pb)
{
    return sa > sb || (sa == sb && pa < pb);
}

int kivi_oracle_sink_topk(int64_t k, int64_t *pos, float *score, int64_t *count,
                          const float *cand, int64_t p0, int64_t n)
{
    if (k < 0 || n < 0 || *count < 0 || *count > k) return -1;
    const int64_t total = *count + n;
    int64_t *ap = (int64_t *)malloc(sizeof(int64_t) * (size_t)(total > 0 ? total : 1));
    float *as = (float *)malloc(sizeof(float) * (size_t)(total > 0 ? total : 1));
    char *used = (char *)calloc((size_t)(total > 0 ? total : 1), 1);
    if (!ap || !as || !used) { free(ap); free(as); free(used); return -1; }
    for (int64_t i = 0; i < *count; ++i) { ap[i] = pos[i]; as[i] = score[i]; }
    for (int64_t i = 0; i < n; ++i) {
        if (!isfinite(cand[i])) { free(ap); free(as); free(used); return -1; }
        ap[*count + i] = p0 + i;
        as[*count + i] = cand[i];
    }
    /* selection: k times the best entry not yet taken */
    const int64_t keep = total < k ? total : k;
    for (int64_t j = 0; j < keep; ++j) {
        int64_t best = -1;
        for (int64_t i = 0; i < total; ++i) {
            if (used[i]) continue;
            if (best < 0 || ranks_before(as[i], ap[i], as[best], ap[best])) best = i;
        }
        used[best] = 1;
        pos[j] = ap[best];
        score[j] = as[best];
    }
    *count = keep;
    free(ap); free(as); free(used);
    return 0;
}

static int is_sink(const int64_t *top, int64_t n_top, int64_t p)
{
    for (int64_t i = 0; i < n_top; ++i)
        if (top[i] == p) return 1;
    return 0;
}

int64_t kivi_oracle_flush_sink(const uint16_t *k_res, const uint16_t *v_res,
                               int64_t batch, int64_t heads, int64_t d, int64_t r_cap,
                               int64_t cap, int group, int bits, int residual,
                               uint32_t *k_codes, float *k_scale, float *k_zero,
                               uint32_t *v_codes, float *v_scale, float *v_zero,
                               int64_t *s_q, int64_t *res_head, int64_t *n_res,
                               int64_t k_top, const int64_t *top_pos, const int64_t *top_count,
                               int64_t sink_cap, int64_t *sink_pos, int64_t *sink_count,
                               uint16_t *sink_k, uint16_t *sink_v)
{
    if (!valid_bits(bits) || !valid_group(group) || batch < 0 || heads <= 0 || d <= 0) return -1;
    if (r_cap <= 0 || r_cap % group || cap % group || *s_q % group || *res_head % group) return -1;
    if (d % group != 0 || d % codes_per_word(bits) != 0 || k_top < 0 || sink_cap < 0) return -1;
    const int64_t n = kivi_oracle_flush_size(*n_res, residual, group);
    if (n <= 0) return n < 0 ? -1 : 0;
    if (*s_q + n > cap) return -3;
    const int64_t bh = batch * heads;
    const int w = codes_per_word(bits);
    const int64_t head = *res_head;
    /* sinks among the flushed tokens: every one must fit into the sink store */
    for (int64_t b = 0; b < batch; ++b) {
        int64_t add = 0;
        for (int64_t i = 0; i < n; ++i)
            add += is_sink(top_pos + b * k_top, top_count[b], *s_q + i);
        if (sink_count[b] + add > sink_cap) return -3;
    }
    float vals[KIVI_ORACLE_MAX_GROUP];
    int keep_idx[KIVI_ORACLE_MAX_GROUP];
    for (int64_t bb = 0; bb < bh; ++bb) {
        const int64_t b = bb / heads;
        const int64_t *top = top_pos + b * k_top;
        /* keys: per channel and group, the non-sink tokens set the parameters */
        for (int64_t j = 0; j < n / group; ++j) {
            for (int64_t c = 0; c < d; ++c) {
                int kept = 0;
                for (int i = 0; i < group; ++i) {
                    const int64_t li = j * group + i;                 /* logical residual token */
                    if (is_sink(top, top_count[b], *s_q + li)) continue;
                    const int64_t row = (head + li) % r_cap;
                    vals[kept] = kivi_oracle_half_to_float(k_res[(bb * r_cap + row) * d + c]);
                    keep_idx[kept] = i;
                    ++kept;
                }
                float sc = 0.0f, ze = 0.0f;           /* a group of sinks only: both 0 */
                if (kept > 0 && kivi_oracle_group_params(vals, kept, bits, &sc, &ze) != 0) return -1;
                const int64_t gq = *s_q / group + j;
                k_scale[(bb * (cap / group) + gq) * d + c] = sc;
                k_zero[(bb * (cap / group) + gq) * d + c] = ze;
                uint32_t q[KIVI_ORACLE_MAX_GROUP];
                for (int i = 0; i < group; ++i) q[i] = 0u;            /* sink tokens: code 0 */
                for (int e = 0; e < kept; ++e) q[keep_idx[e]] = kivi_oracle_code(vals[e], sc, ze, bits);
                for (int i = 0; i < group; ++i) {
                    const int64_t t = gq * group + i;
                    uint32_t *word = &k_codes[(bb * (cap / w) + t / w) * d + c];
                    if (i % w == 0) *word = 0u;
                    *word |= q[i] << ((t % w) * bits);
                }
            }
        }
        /* values: a sink token's row is not quantized (codes, scales, zeros 0) */
        for (int64_t i = 0; i < n; ++i) {
            const int64_t row = (head + i) % r_cap;
            const int64_t t = *s_q + i;
            uint32_t *vw = v_codes + (bb * cap + t) * (d / w);
            float *vs = v_scale + (bb * cap + t) * (d / group);
            float *vz = v_zero + (bb * cap + t) * (d / group);
            if (is_sink(top, top_count[b], t)) {
                for (int64_t j2 = 0; j2 < d / w; ++j2) vw[j2] = 0u;
                for (int64_t g2 = 0; g2 < d / group; ++g2) { vs[g2] = 0.0f; vz[g2] = 0.0f; }
                continue;
            }
            if (kivi_oracle_value_row(v_res + (bb * r_cap + row) * d, d, group, bits, vw, vs, vz) != 0)
                return -1;
        }
    }
    /* the sink tokens' fp16 rows, in position order, for every head */
    for (int64_t b = 0; b < batch; ++b) {
        for (int64_t i = 0; i < n; ++i) {
            const int64_t t = *s_q + i;
            if (!is_sink(top_pos + b * k_top, top_count[b], t)) continue;
            const int64_t slot = sink_count[b]++;
            sink_pos[b * sink_cap + slot] = t;
            const int64_t row = (head + i) % r_cap;
            for (int64_t h = 0; h < heads; ++h) {
                const int64_t bb = b * heads + h;
                memcpy(sink_k + (bb * sink_cap + slot) * d, k_res + (bb * r_cap + row) * d,
                       sizeof(uint16_t) * (size_t)d);
                memcpy(sink_v + (bb * sink_cap + slot) * d, v_res + (bb * r_cap + row) * d,
                       sizeof(uint16_t) * (size_t)d);
            }
        }
    }
    *s_q += n;
    *res_head = (head + n) % r_cap;
    *n_res -= n;
    return n;
}

int kivi_oracle_sink_restore(uint16_t *k, uint16_t *v, int64_t batch, int64_t heads, int64_t s,
                             int64_t d, int64_t sink_cap, const int64_t *sink_pos,
                             const int64_t *sink_count, const uint16_t *sink_k,
                             const uint16_t *sink_v)
{
    if (batch < 0 || heads <= 0 || s < 0 || d <= 0 || sink_cap < 0) return -1;
    for (int64_t b = 0; b < batch; ++b)
        for (int64_t j = 0; j < sink_count[b]; ++j) {
            const int64_t t = sink_pos[b * sink_cap + j];
            if (t < 0 || t >= s) continue;              /* not in the dequantized range */
            for (int64_t h = 0; h < heads; ++h) {
                const int64_t bb = b * heads + h;
                memcpy(k + (bb * s + t) * d, sink_k + (bb * sink_cap + j) * d,
                       sizeof(uint16_t) * (size_t)d);
                memcpy(v + (bb * s + t) * d, sink_v + (bb * sink_cap + j) * d,
                       sizeof(uint16_t) * (size_t)d);
            }
        }
    return 0;
}
