/*
 * kivi_oracle.h -- plain, single-threaded CPU oracle for the KIVI KV-cache flush.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link or
 * call this library: only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code with the CUDA library.
 *
 * Sources (VeloxQuant-MLX documentation pages):
 *   [POST]    blog post "How I fused KIVI's KV-cache quantization into two
 *             bit-exact Metal kernels ..." (veloxquant-mlx.netlify.app/docs/blog)
 *   [RELEASE] blog post "VeloxQuant-MLX 0.8.0 adds KIVI", section "What KIVI is"
 *   [README]  VeloxQuant-MLX 0.24.1 project description (pypi.org),
 *             section "KIVI -- tuning-free asymmetric 2-bit baseline"
 *   [BITPACK] blog post on the library's Metal kernels, section
 *             "Kernel 1: Bit-Packing" (LSB-first code order)
 *
 * Arithmetic: IEEE binary32 throughout, no fused multiply-add, no flush to
 * zero, round-half-to-even.  Inputs and reconstructions are IEEE binary16,
 * passed as raw uint16_t bit patterns.
 *
 * Layouts (all row-contiguous, bh = batch*kv_heads flattened):
 *   x            fp16   [bh][s][d]
 *   key codes    u32    [bh][ng*G/W][d]   word (bh, t/W, c) holds tokens
 *                                         t..t+W-1 of channel c, token t at
 *                                         bits [(t%W)*b, (t%W+1)*b)
 *   key scale    f32    [bh][ng][d]       one (scale, zero) per channel per
 *   key zero     f32    [bh][ng][d]       group of G tokens
 *   value codes  u32    [bh][s][d/W]      word (bh, s, c/W) holds channels
 *                                         c..c+W-1 of token s
 *   value scale  f32    [bh][s][d/G]      one (scale, zero) per token per
 *   value zero   f32    [bh][s][d/G]      group of G channels
 * with W = 32/b codes per word and ng = ceil(s/G).
 *
 * Return values: 0 on success, -1 on an argument the operation does not
 * define (bits not in {2,4,8}, G not in {16,32,64,128}, d not divisible as
 * required, non-finite input).  Functions never allocate caller memory.
 */
#ifndef KIVI_ORACLE_H
#define KIVI_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* binary16 <-> binary32 conversions written from the IEEE 754 format
 * definition.  half -> float is exact; float -> half rounds to nearest,
 * ties to even, and overflows to infinity. */
float    kivi_oracle_half_to_float(uint16_t h);
uint16_t kivi_oracle_float_to_half(float f);
/* Element-wise array forms of the two conversions (n elements). */
void kivi_oracle_halves_to_floats(const uint16_t *h, float *f, int64_t n);
void kivi_oracle_floats_to_halves(const float *f, uint16_t *h, int64_t n);

/* Asymmetric min/max parameters of one group of n fp32 values
 * ([POST] "What we're actually optimizing"; [RELEASE] "What KIVI is"):
 *   zero = min(group), scale = (max(group) - min(group)) / (2^bits - 1).
 * min and max are canonicalised so that a zero extreme is +0. */
int kivi_oracle_group_params(const float *vals, int64_t n, int bits,
                             float *scale, float *zero);

/* Code of one value: q = clip(round_half_even((x - zero) / scale), 0, 2^b-1),
 * q = 0 when scale == 0.  Returns 0xFFFFFFFF for an invalid bit width. */
uint32_t kivi_oracle_code(float x, float scale, float zero, int bits);

/* Reconstruction of one code: fp16(round(round(q*scale) + zero)) with two
 * separately rounded binary32 operations ([POST] "1. FMA contraction"). */
uint16_t kivi_oracle_recon(uint32_t q, float scale, float zero);

/* Full-tensor operations on contiguous buffers (layouts above). */
int kivi_oracle_quantize_keys(const uint16_t *x, int64_t bh, int64_t s, int64_t d,
                              int group, int bits,
                              uint32_t *codes, float *scale, float *zero);
int kivi_oracle_quantize_values(const uint16_t *x, int64_t bh, int64_t s, int64_t d,
                                int group, int bits,
                                uint32_t *codes, float *scale, float *zero);
int kivi_oracle_dequantize_keys(const uint32_t *codes, const float *scale,
                                const float *zero, int64_t bh, int64_t s, int64_t d,
                                int group, int bits, uint16_t *y);
int kivi_oracle_dequantize_values(const uint32_t *codes, const float *scale,
                                  const float *zero, int64_t bh, int64_t s, int64_t d,
                                  int group, int bits, uint16_t *y);

/* One key group (channel c, token group g) of one bh slice x_bh [s][d]:
 * writes G/W code words (token order), its scale and zero.  Lets tests check
 * sampled outputs of tensors too large for the full-tensor calls. */
int kivi_oracle_key_group(const uint16_t *x_bh, int64_t s, int64_t d,
                          int64_t g, int64_t c, int group, int bits,
                          uint32_t *words, float *scale, float *zero);
/* One value row (token s of x_bh [s][d]): writes d/W words and d/G scales
 * and zeros. */
int kivi_oracle_value_row(const uint16_t *x_row, int64_t d, int group, int bits,
                          uint32_t *words, float *scale, float *zero);

/* Residual-window flush size ([POST] "What we're actually optimizing": the
 * newest residual tokens stay fp16, aged-out tokens are quantized as a batch;
 * pinned by the "flush/layer" column of the [POST] Generation 1 table):
 *   n_flush = floor((n_res - R) / G) * G  if n_res >= R + G, else 0. */
int64_t kivi_oracle_flush_size(int64_t n_res, int residual, int group);

/* Append of n new tokens behind the residual of one layer ([POST] "What
 * we're actually optimizing": the newest tokens enter the fp16 residual
 * window and age out of it by flushes).  New token i of k_new, v_new
 * (fp16 [bh][n][d]) becomes logical residual token *n_res + i, stored at
 * ring row (res_head + *n_res + i) % r_cap of k_res, v_res ([bh][r_cap][d]);
 * then *n_res += n.  Returns 0, -1 (invalid arguments) or -3 (the ring
 * would hold more than r_cap tokens; nothing written). */
int kivi_oracle_append(uint16_t *k_res, uint16_t *v_res, int64_t bh, int64_t d, int64_t r_cap,
                       int64_t res_head, int64_t *n_res, const uint16_t *k_new,
                       const uint16_t *v_new, int64_t n);

/* Flush of one layer (keys and values) from an fp16 residual ring into the
 * quantized store.
 *   k_res, v_res   fp16 [bh][r_cap][d]; logical residual token i (0 = oldest)
 *                  sits at ring row (res_head + i) % r_cap
 *   store          key codes [bh][cap/W][d], key scale/zero [bh][cap/G][d],
 *                  value codes [bh][cap][d/W], value scale/zero [bh][cap][d/G]
 *   *s_q           tokens already in the store (multiple of G); advanced
 *   *res_head      ring row of the oldest residual token; advanced
 *   *n_res         residual token count; reduced
 * The oldest n_flush tokens are quantized (keys per channel, values per
 * token) and written at store token offset *s_q.  Returns the number of
 * tokens flushed, or -1 (invalid arguments) / -3 (store capacity exceeded). */
int64_t kivi_oracle_flush(const uint16_t *k_res, const uint16_t *v_res,
                          int64_t bh, int64_t d, int64_t r_cap, int64_t cap,
                          int group, int bits, int residual,
                          uint32_t *k_codes, float *k_scale, float *k_zero,
                          uint32_t *v_codes, float *v_scale, float *v_zero,
                          int64_t *s_q, int64_t *res_head, int64_t *n_res);

/* Decode attention of r query heads against the n cached tokens of one KV
 * head, reading the keys and values as the fp16 values the cache holds
 * (dequantized store tokens followed by the fp16 residual tokens; [POST]
 * last section: attention that reads the packed codes expands them in
 * registers, so what it computes is attention over the reconstruction):
 *   s[h][t] = scale * sum_c q[h][c] * k[t][c]
 *   p[h][t] = exp(s[h][t] - max_t s[h][t]) / sum_t exp(s[h][t] - max_t s[h][t])
 *   out[h][c] = sum_t p[h][t] * v[t][c]
 * q fp16 [r][d], k and v fp16 [n][d], out binary64 [r][d].  Every product,
 * sum, exponential and quotient is binary64 (the fp16 inputs convert
 * exactly).  Subtracting the maximum leaves the softmax unchanged in exact
 * arithmetic and keeps exp() finite.  Returns -1 for n < 1, r < 1 or d < 1. */
int kivi_oracle_attention(const uint16_t *q, int64_t r, const uint16_t *k,
                          const uint16_t *v, int64_t n, int64_t d, double scale,
                          double *out);

/* KIVI-Sink (VeloxQuant-MLX project description, section "KVSink-adapted
 * sink protection"): tokens with anomalously high key L2-norm (mean over the
 * KV heads; a running top-k of token positions) are kept fp16 and excluded
 * from the quantization-parameter calibration.
 *
 * Score of token t of sequence b (keys k: [batch*heads] slices, bh stride
 * bh_stride elements, n rows of d):
 *     score = (sum_h sqrt(sum_c k_c^2)) / heads
 * in binary32: the squared norm accumulated with fmaf in channel order,
 * sqrtf, the norms summed in head order, one division.  score[b*n + t]. */
int kivi_oracle_sink_scores(const uint16_t *k, int64_t batch, int64_t heads, int64_t n,
                            int64_t d, int64_t bh_stride, float *score);

/* Running top-k of one sequence: merges candidates (position p0 + i, score
 * cand[i]) into (pos, score)[0 .. *count), keeping the k best ranked by
 * larger score, then smaller position; the result is sorted in that order.
 * Returns -1 for bad sizes or a non-finite score. */
int kivi_oracle_sink_topk(int64_t k, int64_t *pos, float *score, int64_t *count,
                          const float *cand, int64_t p0, int64_t n);

/* kivi_oracle_flush with sink protection (bh = batch * heads; flushed
 * logical residual token i of sequence b has position *s_q + i).  A flushed
 * token whose position is in its sequence's top set (top_pos[b][0 ..
 * top_count[b])) is a sink:
 *   keys    excluded from its groups' min/max (a group of sinks only gets
 *           scale 0 and zero 0); its code slots hold 0
 *   values  its row gets codes 0, scales 0, zeros 0
 *   store   its position and its fp16 key and value rows (every head) are
 *           appended to the sink store: sink_pos [batch][sink_cap],
 *           sink_count [batch], sink_k / sink_v [bh][sink_cap][d]
 * With no top positions it equals kivi_oracle_flush.  Returns the tokens
 * flushed, -1 (bad arguments) or -3 (store or sink store capacity). */
int64_t kivi_oracle_flush_sink(const uint16_t *k_res, const uint16_t *v_res,
                               int64_t batch, int64_t heads, int64_t d, int64_t r_cap,
                               int64_t cap, int group, int bits, int residual,
                               uint32_t *k_codes, float *k_scale, float *k_zero,
                               uint32_t *v_codes, float *v_scale, float *v_zero,
                               int64_t *s_q, int64_t *res_head, int64_t *n_res,
                               int64_t k_top, const int64_t *top_pos, const int64_t *top_count,
                               int64_t sink_cap, int64_t *sink_pos, int64_t *sink_count,
                               uint16_t *sink_k, uint16_t *sink_v);

/* Puts the sink tokens' fp16 rows back into dequantized keys and values
 * [bh][s][d] (positions >= s are skipped). */
int kivi_oracle_sink_restore(uint16_t *k, uint16_t *v, int64_t batch, int64_t heads, int64_t s,
                             int64_t d, int64_t sink_cap, const int64_t *sink_pos,
                             const int64_t *sink_count, const uint16_t *sink_k,
                             const uint16_t *sink_v);

#ifdef __cplusplus
}
#endif

#endif /* KIVI_ORACLE_H */
