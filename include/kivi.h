/*
 * kivi.h -- C ABI of the GB300 KIVI KV-cache codec (libkivi.so).
 *
 * KIVI quantizes keys per channel and values per token with asymmetric
 * min/max groups, keeps the newest tokens in fp16 and folds aged-out tokens
 * into a compressed store (VeloxQuant-MLX blog post "How I fused KIVI's
 * KV-cache quantization into two bit-exact Metal kernels ...", sections
 * "What we're actually optimizing" and "The layout problem that shapes
 * everything"; release post "VeloxQuant-MLX 0.8.0 adds KIVI", section "What
 * KIVI is").  For every group:
 *
 *     zero  = min(group)                      (binary32; a zero extreme is +0)
 *     scale = (max(group) - min(group)) / (2^bits - 1)      (IEEE division)
 *     q     = clip(round_half_even((x - zero) / scale), 0, 2^bits - 1)
 *             (q = 0 when scale == 0, i.e. max == min)
 *     recon = fp16_rn( fp32(q * scale) + zero )   (two roundings, no FMA)
 *
 * All arithmetic is IEEE binary32 and matches the CPU oracle bit for bit.
 *
 * Tensors are row-contiguous [bh][s][d] IEEE binary16 (bh = batch * kv_heads,
 * s = tokens, d = head_dim), element (b, t, c) at b*bh_stride + t*d + c.
 * With G = group, b = bits, W = 32 / b codes per uint32 word and
 * ng = ceil(s / G):
 *
 *   keys    codes  u32 [bh][ng*G/W][d]  word (b, t/W, c) holds tokens t..t+W-1
 *                                       of channel c; token t at bits
 *                                       [(t%W)*b, (t%W+1)*b) (LSB first)
 *           scale  f32 [bh][ng][d]      one (scale, zero) per channel per
 *           zero   f32 [bh][ng][d]      group of G tokens
 *   values  codes  u32 [bh][s][d/W]     word (b, t, c/W) holds channels
 *                                       c..c+W-1 of token t (LSB first)
 *           scale  f32 [bh][s][d/G]     one (scale, zero) per token per
 *           zero   f32 [bh][s][d/G]     group of G channels
 *
 * A key group that runs past the last token is padded by repeating the last
 * token (fused-kernel post, "3. Padding semantics"); its padding slots hold
 * that token's code.
 *
 * Common rules for every call:
 *   - Pointers marked "device" are CUDA device pointers owned by the caller;
 *     the library allocates no device or host memory and keeps no pointer
 *     after the call returns.
 *   - Calls are asynchronous on `stream` (NULL = the legacy default stream);
 *     outputs are complete when the stream reaches that point.  Calls that
 *     overlap on the GPU with writes to their inputs or outputs race.
 *   - Supported: bits in {2, 4, 8}; group in {16, 32, 64, 128}; 8 <= d <= 256
 *     with d % 8 == 0 for keys and d % group == 0, d % 32 == 0 for values.
 *   - Alignment (KIVI_ERR_ALIGN otherwise): every base pointer 16-byte
 *     aligned; bh strides of fp16 tensors and of key codes multiples of 16
 *     bytes; key scale/zero bh strides multiples of 8 bytes (16 for
 *     dequantization); value code bh strides multiples of 8 bytes at 2 bits
 *     and 16 bytes at 4 and 8 bits; value scale/zero strides unrestricted.
 *     The contiguous layouts above always satisfy these rules.
 *   - Arguments are validated on the host before any launch; a call that
 *     returns an error launched nothing and wrote nothing.  bh == 0 or
 *     s == 0 is a valid empty call.
 *   - Inputs must be finite; results for NaN or infinite inputs are
 *     unspecified (but every write stays inside the stated output ranges).
 */
#ifndef KIVI_H
#define KIVI_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Symbols of this header are the library's only exported symbols. */
#if defined(__GNUC__)
#define KIVI_API __attribute__((visibility("default")))
#else
#define KIVI_API
#endif

/* A cudaStream_t, declared without the CUDA headers. */
typedef struct CUstream_st *kivi_stream_t;

typedef enum {
    KIVI_OK = 0,
    KIVI_ERR_INVAL = 1,     /* argument outside the supported set */
    KIVI_ERR_ALIGN = 2,     /* pointer or bh stride breaks 16-byte alignment */
    KIVI_ERR_CAPACITY = 3,  /* flush would overrun the store */
    KIVI_ERR_CUDA = 4       /* a CUDA runtime call failed; see kivi_last_cuda_error */
} kivi_status;

/* Most layers one batched call takes (kivi_flush, kivi_dequantize_cache). */
#define KIVI_MAX_LAYERS 128

/* ------------------------------------------------------------------------ */
/* Full-tensor quantization                                                 */
/* ------------------------------------------------------------------------ */

/* Keys, quantized per channel over groups of `group` tokens (fused-kernel
 * post, "The layout problem": the group runs along the strided token axis).
 *   x        device fp16 [bh][s][d], bh stride x_bh_stride >= s*d elements
 *   codes    device u32, bh stride codes_bh_stride >= ng*group/W*d words
 *   scale,   device f32, bh stride sz_bh_stride >= ng*d floats
 *   zero
 * Returns KIVI_OK, KIVI_ERR_INVAL, KIVI_ERR_ALIGN or KIVI_ERR_CUDA. */
KIVI_API kivi_status kivi_quantize_keys(const void *x, int64_t bh, int64_t s, int64_t d,
                               int64_t x_bh_stride, int group, int bits,
                               uint32_t *codes, int64_t codes_bh_stride,
                               float *scale, float *zero, int64_t sz_bh_stride,
                               kivi_stream_t stream);

/* Values, quantized per token over groups of `group` channels (the group
 * runs along the contiguous head_dim axis).
 *   x        device fp16 [bh][s][d], bh stride x_bh_stride >= s*d elements
 *   codes    device u32, bh stride codes_bh_stride >= s*d/W words
 *   scale,   device f32, bh stride sz_bh_stride >= s*d/group floats
 *   zero
 * Returns KIVI_OK, KIVI_ERR_INVAL, KIVI_ERR_ALIGN or KIVI_ERR_CUDA. */
KIVI_API kivi_status kivi_quantize_values(const void *x, int64_t bh, int64_t s, int64_t d,
                                 int64_t x_bh_stride, int group, int bits,
                                 uint32_t *codes, int64_t codes_bh_stride,
                                 float *scale, float *zero, int64_t sz_bh_stride,
                                 kivi_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Dequantization (fused-kernel post, "1. FMA contraction": the product is  */
/* rounded before the add)                                                  */
/* ------------------------------------------------------------------------ */

/* Keys: codes/scale/zero in the key layout above (same strides as the
 * quantize call) -> y device fp16 [bh][s][d], bh stride y_bh_stride >= s*d.
 * Returns KIVI_OK, KIVI_ERR_INVAL, KIVI_ERR_ALIGN or KIVI_ERR_CUDA. */
KIVI_API kivi_status kivi_dequantize_keys(const uint32_t *codes, int64_t codes_bh_stride,
                                 const float *scale, const float *zero,
                                 int64_t sz_bh_stride, int64_t bh, int64_t s, int64_t d,
                                 int group, int bits, void *y, int64_t y_bh_stride,
                                 kivi_stream_t stream);

/* Values: codes/scale/zero in the value layout above -> y fp16 [bh][s][d].
 * Returns KIVI_OK, KIVI_ERR_INVAL, KIVI_ERR_ALIGN or KIVI_ERR_CUDA. */
KIVI_API kivi_status kivi_dequantize_values(const uint32_t *codes, int64_t codes_bh_stride,
                                   const float *scale, const float *zero,
                                   int64_t sz_bh_stride, int64_t bh, int64_t s, int64_t d,
                                   int group, int bits, void *y, int64_t y_bh_stride,
                                   kivi_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Fused fake quantization: quantize and dequantize in one pass             */
/* ------------------------------------------------------------------------ */

/* The fp16 reconstruction y = dequantize(quantize(x)) written in the same
 * pass that makes the codes, with no round trip of the codes through memory
 * (fused-kernel post, "What we're actually optimizing" and "1. FMA
 * contraction": its kernels quantize and dequantize in one dispatch and
 * return the reconstruction).  y is bit-identical to kivi_quantize_* followed
 * by kivi_dequantize_* on the same arguments.  For keys of a ragged last
 * group only the real tokens are written (the padding exists only inside
 * the group's statistics).
 *   x      device fp16 [bh][s][d], bh stride x_bh_stride >= s*d
 *   y      device fp16 [bh][s][d], bh stride y_bh_stride >= s*d; must not
 *          overlap x
 *   codes, scale, zero, codes_bh_stride, sz_bh_stride
 *          as for kivi_quantize_keys / kivi_quantize_values, written too; or
 *          all three NULL (strides ignored) for the reconstruction alone
 * Returns KIVI_OK, KIVI_ERR_INVAL (also when only some of codes, scale,
 * zero are NULL), KIVI_ERR_ALIGN or KIVI_ERR_CUDA. */
KIVI_API kivi_status kivi_fakequant_keys(const void *x, int64_t bh, int64_t s, int64_t d,
                                         int64_t x_bh_stride, int group, int bits, void *y,
                                         int64_t y_bh_stride, uint32_t *codes,
                                         int64_t codes_bh_stride, float *scale, float *zero,
                                         int64_t sz_bh_stride, kivi_stream_t stream);
KIVI_API kivi_status kivi_fakequant_values(const void *x, int64_t bh, int64_t s, int64_t d,
                                           int64_t x_bh_stride, int group, int bits, void *y,
                                           int64_t y_bh_stride, uint32_t *codes,
                                           int64_t codes_bh_stride, float *scale, float *zero,
                                           int64_t sz_bh_stride, kivi_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Residual window and flush                                                */
/* ------------------------------------------------------------------------ */

/* One layer's buffers (all device, caller-owned, contiguous per bh):
 *   k_res, v_res   fp16 [bh][r_cap][d] residual rings: logical residual
 *                  token i (0 = oldest) lives at ring row (res_head + i) % r_cap
 *                  (written by kivi_append, read by the flushes)
 *   k_codes        u32 [bh][cap/W][d]      store, key layout with s = cap
 *   k_scale,k_zero f32 [bh][cap/G][d]
 *   v_codes        u32 [bh][cap][d/W]      store, value layout with s = cap
 *   v_scale,v_zero f32 [bh][cap][d/G] */
typedef struct {
    const void *k_res;
    const void *v_res;
    uint32_t *k_codes;
    float *k_scale;
    float *k_zero;
    uint32_t *v_codes;
    float *v_scale;
    float *v_zero;
} kivi_layer;

/* Geometry and state shared by every layer of a cache (every layer flushes
 * together).  r_cap and cap are multiples of `group`; s_q and res_head stay
 * multiples of `group`; 0 <= n_res <= r_cap. */
typedef struct {
    int64_t bh, d;        /* batch * kv_heads, head_dim */
    int64_t r_cap;        /* residual ring capacity, tokens */
    int64_t cap;          /* store capacity, tokens */
    int32_t group, bits;  /* group size G, code width b */
    int32_t residual;     /* R: newest tokens kept fp16 */
    int32_t reserved;     /* must be 0 */
    int64_t s_q;          /* tokens in the store */
    int64_t res_head;     /* ring row of the oldest residual token */
    int64_t n_res;        /* tokens in the residual ring */
} kivi_cache;

/* Tokens one flush moves: floor((n_res - residual) / group) * group when
 * n_res >= residual + group, else 0 (fused-kernel post, "What we're actually
 * optimizing": the newest residual tokens stay fp16 and whole groups of
 * aged-out tokens are quantized as a batch; the "flush/layer" column of its
 * "Generation 1" table fixes the rule).  Returns -1 for a negative argument
 * or group <= 0. */
KIVI_API int64_t kivi_flush_size(int64_t n_res, int residual, int group);

/* Append: n new tokens of every layer enter the fp16 residual window behind
 * the tokens already there (fused-kernel post, "What we're actually
 * optimizing": the newest tokens stay fp16 until whole groups of them age
 * out).  Token i (0 <= i < n) of bh slice b of layer l is read from
 * k_new[l] + b * new_bh_stride + i * d (likewise v_new[l]) and written to
 * ring row (res_head + n_res + i) % r_cap of layers[l].k_res (v_res); then
 * n_res += n.  Nothing else moves: rows of the ring wrap, tokens are never
 * shifted.  One launch covers every layer.
 *   k_new, v_new    host arrays of n_layers device pointers, each fp16
 *                   [bh][n][d] rows with bh stride new_bh_stride >= n*d
 *                   elements (a multiple of 8); they must not overlap the
 *                   rings
 *   cache           host memory, updated in place on success (n_res)
 * The store pointers of `layers` are not used (they may be NULL).
 * n == 0 (or bh == 0) launches nothing and only advances n_res.
 * Returns KIVI_OK, KIVI_ERR_INVAL, KIVI_ERR_ALIGN, KIVI_ERR_CAPACITY (the
 * ring would hold more than r_cap tokens; nothing launched, state
 * unchanged) or KIVI_ERR_CUDA. */
KIVI_API kivi_status kivi_append(const kivi_layer *layers, int n_layers, kivi_cache *cache,
                                 const void *const *k_new, const void *const *v_new,
                                 int64_t new_bh_stride, int64_t n, kivi_stream_t stream);

/* Flush: quantize the oldest kivi_flush_size(n_res, residual, group) residual
 * tokens of every layer (keys per channel, values per token) into the store
 * at token offset s_q, then advance the state: s_q += n, res_head =
 * (res_head + n) % r_cap, n_res -= n.  The residual rings are only read; no
 * token is copied.  `layers` is a host array of n_layers (1..KIVI_MAX_LAYERS)
 * entries; `cache` is host memory updated in place on success; `n_flushed`
 * (host, may be NULL) receives n.  n == 0 launches nothing.
 * Returns KIVI_OK, KIVI_ERR_INVAL, KIVI_ERR_ALIGN, KIVI_ERR_CAPACITY (state
 * unchanged, nothing launched) or KIVI_ERR_CUDA. */
KIVI_API kivi_status kivi_flush(const kivi_layer *layers, int n_layers, kivi_cache *cache,
                       int64_t *n_flushed, kivi_stream_t stream);

/* Fused fake-quant flush: kivi_flush that also writes the fp16
 * reconstruction of the n flushed tokens of every layer into k_hat[l],
 * v_hat[l] (host arrays of n_layers device pointers, each fp16
 * [bh][cap][d] contiguous), at token rows s_q .. s_q + n - 1: the
 * dequantized store kept as fp16, filled in the flush's own pass (the
 * post's cache holds exactly this reconstruction).  A layer's three key
 * store pointers (k_codes, k_scale, k_zero) may all be NULL, and likewise
 * its three value store pointers: that store is then not written.  The rows
 * written equal those kivi_dequantize_cache would produce from the store.
 * events: as for kivi_flush_timed (may be NULL).
 * Returns KIVI_OK, KIVI_ERR_INVAL, KIVI_ERR_ALIGN, KIVI_ERR_CAPACITY or
 * KIVI_ERR_CUDA, with the state rules of kivi_flush. */
KIVI_API kivi_status kivi_flush_fakequant(const kivi_layer *layers, int n_layers,
                                          kivi_cache *cache, void *const *k_hat,
                                          void *const *v_hat, int64_t *n_flushed,
                                          kivi_stream_t stream, void *const events[3]);

/* A decode step's append and flush in one call: kivi_append of the n new
 * tokens of every layer, then kivi_flush (same arguments, results, state
 * updates and errors; every argument of both steps is checked before the
 * first launch, so an error launches nothing and changes no state).  When
 * the tokens the flush moves were all in the ring before the append (the
 * usual decode step: n_res >= the flush size), the flush's kernels do not
 * read what the append writes, and their launches overlap the append's tail
 * on the GPU (programmatic dependent launch) instead of waiting for it;
 * stream order is kept: the call's work is complete when the stream reaches
 * its end.  The store pointers of `layers` must be given (no NULL store).
 * events: NULL, or 4 cudaEvent_t recorded before the append, before the key
 * launch, between the key and the value launch and after it (NULL entries
 * skipped); when the flush moves nothing only the first is recorded. */
KIVI_API kivi_status kivi_append_flush(const kivi_layer *layers, int n_layers, kivi_cache *cache,
                                       const void *const *k_new, const void *const *v_new,
                                       int64_t new_bh_stride, int64_t n, int64_t *n_flushed,
                                       kivi_stream_t stream, void *const events[4]);

/* Dequantize the first cache->s_q tokens of every layer's store into
 * k_out[l], v_out[l] (host arrays of n_layers device pointers, each fp16
 * [bh][s_q][d] contiguous).  Equivalent to kivi_dequantize_keys and
 * kivi_dequantize_values on each layer's store, in two launches.
 * Returns KIVI_OK, KIVI_ERR_INVAL, KIVI_ERR_ALIGN or KIVI_ERR_CUDA. */
KIVI_API kivi_status kivi_dequantize_cache(const kivi_layer *layers, int n_layers,
                                  const kivi_cache *cache, void *const *k_out,
                                  void *const *v_out, kivi_stream_t stream);

/* The two batched calls with per-launch timing points: when `events` is not
 * NULL, events[0] is recorded on `stream` before the key launch, events[1]
 * between the key and the value launch and events[2] after the value launch
 * (each a cudaEvent_t created by the caller; NULL entries are skipped).
 * Otherwise identical to kivi_flush / kivi_dequantize_cache; a flush that
 * moves nothing records nothing. */
KIVI_API kivi_status kivi_flush_timed(const kivi_layer *layers, int n_layers,
                                      kivi_cache *cache, int64_t *n_flushed,
                                      kivi_stream_t stream, void *const events[3]);
KIVI_API kivi_status kivi_dequantize_cache_timed(const kivi_layer *layers, int n_layers,
                                                 const kivi_cache *cache, void *const *k_out,
                                                 void *const *v_out, kivi_stream_t stream,
                                                 void *const events[3]);

/* ------------------------------------------------------------------------ */
/* KIVI-Sink: high key-norm tokens kept fp16                                */
/* ------------------------------------------------------------------------ */

/* KIVI-Sink (VeloxQuant-MLX project description, section "KVSink-adapted
 * sink protection"): every token is scored by its key L2 norm averaged over
 * the KV heads, a running top-k of token positions is kept per sequence, and
 * a flushed token that is in it is kept fp16 in a sink store and left out of
 * its groups' quantization parameters.  With k_top == 0 the flush is plain
 * KIVI, bit for bit.  Scores are binary32: squared norm by fused
 * multiply-adds in channel order, correctly rounded square root, norms added
 * in head order, one division; ranking by larger score, then smaller
 * position.  A token's position is its index in the sequence: residual token
 * i (0 = oldest) has position s_q + i. */

/* One layer's KIVI-Sink state, all device memory owned by the caller:
 *   top_pos    int64 [batch][k_top]  running top-k positions, ranked
 *   top_score  f32   [batch][k_top]  their scores
 *   top_count  int32 [batch]         entries in use (start at 0)
 *   sink_pos   int64 [batch][sink_cap]  positions of the stored sinks, in
 *                                       flush order (ascending)
 *   sink_count int32 [batch]         sinks stored (start at 0)
 *   sink_k,    fp16  [bh][sink_cap][d]  the sinks' key / value rows
 *   sink_v
 *   mask       u32   [batch][ceil(r_cap/32)]  scratch of the flush
 *   scores     f32   [batch][r_cap]     scratch of the update */
typedef struct {
    int64_t *top_pos;
    float *top_score;
    int32_t *top_count;
    int64_t *sink_pos;
    int32_t *sink_count;
    void *sink_k;
    void *sink_v;
    uint32_t *mask;
    float *scores;
} kivi_sink_layer;

/* batch: sequences (cache->bh / batch KV heads each); k_top: 0..64;
 * sink_cap: sink store capacity per sequence; reserved must be 0.  Every
 * sink call also requires n_layers * batch * r_cap and
 * n_layers * bh * sink_cap * d / 8 to stay below 2^31 (KIVI_ERR_INVAL). */
typedef struct {
    int64_t batch;
    int32_t k_top;
    int32_t sink_cap;
    int32_t reserved;
    int32_t reserved2;
} kivi_sink_cfg;

/* Scores residual tokens i0 .. i0+n-1 (already in the rings) of every layer
 * and merges them into the layers' running top-k.  Call once per token, in
 * order (after appending, before flushing).  KIVI_ERR_INVAL if the range is
 * not inside the residual. */
KIVI_API kivi_status kivi_sink_update(const kivi_layer *layers, const kivi_sink_layer *sinks,
                                      int n_layers, const kivi_cache *cache,
                                      const kivi_sink_cfg *cfg, int64_t i0, int64_t n,
                                      kivi_stream_t stream);

/* kivi_flush with sink protection: flushed tokens in their sequence's top-k
 * are left out of the key groups' min/max (a group of sinks only gets scale
 * and zero 0) with code 0, their value rows get codes, scales and zeros 0,
 * and their positions and fp16 key / value rows (every head) are appended
 * to the sink store.  A sink store that would overflow keeps the earliest
 * flushed sinks that fit and sets bit 1 of the device fault word
 * (kivi_device_fault); the flushed top-k tokens that did not fit are
 * quantized as plain tokens (codes, scales and zeros of plain KIVI), so no
 * token's value is lost.
 * Returns as kivi_flush. */
KIVI_API kivi_status kivi_flush_sink(const kivi_layer *layers, const kivi_sink_layer *sinks,
                                     int n_layers, kivi_cache *cache,
                                     const kivi_sink_cfg *cfg, int64_t *n_flushed,
                                     kivi_stream_t stream);

/* Puts the stored sinks' fp16 rows back into dequantized store tensors
 * k_out[l], v_out[l] (fp16 [bh][s_q][d], as kivi_dequantize_cache writes
 * them), at their positions. */
KIVI_API kivi_status kivi_sink_restore(const kivi_sink_layer *sinks, int n_layers,
                                       const kivi_cache *cache, const kivi_sink_cfg *cfg,
                                       void *const *k_out, void *const *v_out,
                                       kivi_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Decode attention over the packed cache                                    */
/* ------------------------------------------------------------------------ */

/* Attention of one new query token per sequence over everything a cache
 * holds, reading the packed store directly: the codes are expanded in
 * registers and never written out as fp16 (fused-kernel post, closing
 * section: packed storage plus attention that reads the packed codes is
 * where the memory and speed win of the method lives).  For every layer l,
 * sequence b and query head h (r = h_q / h_kv query heads share KV head
 * j = h / r, h_kv = cache->bh / batch):
 *     out[l][b][h] = sum_t softmax_t(sm_scale * q[l][b][h] . k_t) v_t
 * over t = the cache->s_q store tokens, whose keys and values are exactly
 * the fp16 reconstructions kivi_dequantize_cache produces, followed by the
 * cache->n_res residual tokens of the fp16 rings (bh slice b*h_kv + j).
 * The arithmetic is binary32 with the scores and the value products on
 * tensor cores (fp16 inputs, binary32 accumulation; the probabilities enter
 * as a high and a low fp16 part), so results agree with an exact evaluation
 * to a relative error of about 1e-5 of the softmax-weighted value magnitudes.
 *   layers, cache   as for kivi_flush (store and rings); cache is only read
 *   batch           sequences (cache->bh must be a multiple)
 *   h_q             query heads per sequence; h_q / h_kv in 1..8
 *   q, out          host arrays of n_layers device pointers: q fp16
 *                   [batch][h_q][d], out fp32 [batch][h_q][d], contiguous
 *   n_split         1..64: token ranges per (layer, bh) processed by separate
 *                   blocks (kivi_decode_attention_splits suggests one); with
 *                   n_split > 1 the partial results go to `workspace`
 *                   (device, kivi_decode_attention_workspace floats) and a
 *                   second launch combines them
 * Supported: d in {64, 128, 256} (G dividing d).  s_q + n_res must be at
 * least 1.
 * Kernel: matrix products on the register-operand tensor-core path by
 * default.  With the environment variable KIVI_ATTENTION_KERNEL=tcgen05
 * (read at every call) calls at d == 128 and G >= 32 with at most 8 query
 * heads per KV head and without a sink store run on the tensor-memory
 * kernel instead (warp-specialised and persistent: tcgen05 matrix
 * multiplies issued by one thread, accumulators in tensor memory); the
 * results agree to the same bound, and on a GB300 it measured slower than
 * the default at every bits x G, so it is not the default.
 * Returns KIVI_OK, KIVI_ERR_INVAL, KIVI_ERR_ALIGN or KIVI_ERR_CUDA. */
KIVI_API kivi_status kivi_decode_attention(const kivi_layer *layers, int n_layers,
                                           const kivi_cache *cache, int64_t batch, int32_t h_q,
                                           float sm_scale, const void *const *q,
                                           float *const *out, int32_t n_split,
                                           float *workspace, int64_t workspace_floats,
                                           kivi_stream_t stream);

/* A split count for kivi_decode_attention that fills the current device
 * (about two waves of blocks); 1 when the (layer, bh) pairs alone do. */
KIVI_API int32_t kivi_decode_attention_splits(const kivi_cache *cache, int n_layers,
                                              int64_t batch);

/* Workspace floats kivi_decode_attention needs with n_split splits (0 for
 * n_split == 1); -1 for arguments it would reject. */
KIVI_API int64_t kivi_decode_attention_workspace(const kivi_cache *cache, int n_layers,
                                                 int64_t batch, int32_t h_q, int32_t n_split);

/* kivi_decode_attention without a caller workspace and without allocating,
 * for callers that cannot obtain device memory at the point of the call: a
 * plug-in handed only the cache's pointers and no allocator, a runtime
 * whose memory is planned once up front, or a decode loop that must not
 * pay cudaMalloc's implicit device synchronisation.  The paper has no
 * counterpart; this is a deployment variant of the call above.  With
 * n_split > 1 the partial results go to a fixed device array inside the
 * library (2^24 floats = 64 MiB, held on every device that loads the
 * library until the process exits).  Its device address is looked up on
 * the first call on a device (and again after that device is reset); that
 * first call makes runtime calls, so it should come before any stream
 * capture.  A call whose kivi_decode_attention_workspace size exceeds the
 * array returns KIVI_ERR_CAPACITY before any CUDA call.  Every partial a
 * call reads is written earlier in the same call, so the array is never
 * cleared.  Calls that overlap on the device (different streams, or
 * different host threads without ordering) share the array and race: order
 * them on one stream.  Otherwise identical to kivi_decode_attention,
 * including its results.
 * Returns KIVI_OK, KIVI_ERR_INVAL, KIVI_ERR_ALIGN, KIVI_ERR_CAPACITY or
 * KIVI_ERR_CUDA. */
KIVI_API kivi_status kivi_decode_attention_noalloc(const kivi_layer *layers, int n_layers,
                                                   const kivi_cache *cache, int64_t batch,
                                                   int32_t h_q, float sm_scale,
                                                   const void *const *q, float *const *out,
                                                   int32_t n_split, kivi_stream_t stream);

/* kivi_decode_attention over a cache whose flushes were sink-protected
 * (kivi_flush_sink): the store slots of each sequence's stored sinks (code 0)
 * are replaced by the sinks' exact fp16 key and value rows from the sink
 * store, so the keys and values attended are those of the restored cache
 * (kivi_dequantize_cache then kivi_sink_restore).  sinks, cfg as for
 * kivi_flush_sink; cfg->batch must equal batch; the sink stores are only
 * read.  Other arguments, results and errors as kivi_decode_attention. */
KIVI_API kivi_status kivi_decode_attention_sinks(const kivi_layer *layers,
                                                 const kivi_sink_layer *sinks, int n_layers,
                                                 const kivi_cache *cache,
                                                 const kivi_sink_cfg *cfg, int64_t batch,
                                                 int32_t h_q, float sm_scale,
                                                 const void *const *q, float *const *out,
                                                 int32_t n_split, float *workspace,
                                                 int64_t workspace_floats, kivi_stream_t stream);

/* The device word in which kernels record that a pipeline wait (a bulk copy
 * that never arrived) gave up after its time limit (bit 0: decode
 * attention; bit 1: a sink store overflow, see kivi_flush_sink; bit 2: the
 * self-test below); read and cleared by this call (synchronous).  Results
 * of a call that set bit 0 are unspecified. */
KIVI_API kivi_status kivi_device_fault(uint32_t *fault);

/* Self-test of the bounded-wait path: one warp waits, with the same bounded
 * mbarrier wait as the decode-attention pipeline, on a barrier phase that
 * nothing completes; after limit_us microseconds (1 .. 1000000) the wait
 * gives up and bit 2 of the device fault word is set.  Asynchronous on the
 * stream; touches no other memory.  KIVI_ERR_INVAL for a limit out of
 * range. */
KIVI_API kivi_status kivi_selftest_wait_timeout(uint32_t limit_us, kivi_stream_t stream);

/* ------------------------------------------------------------------------ */
/* Sizes and diagnostics                                                    */
/* ------------------------------------------------------------------------ */

/* uint32 words of one bh slice of key codes (ceil(s/G)*G/W*d) or value
 * codes (s*d/W); -1 for unsupported group/bits or negative sizes. */
KIVI_API int64_t kivi_key_code_words(int64_t s, int64_t d, int group, int bits);
KIVI_API int64_t kivi_value_code_words(int64_t s, int64_t d, int group, int bits);

/* Static description of a status code. */
KIVI_API const char *kivi_status_string(kivi_status status);

/* The cudaError_t value behind the last KIVI_ERR_CUDA returned on the calling
 * host thread (0 if none). */
KIVI_API int kivi_last_cuda_error(void);

/* ABI version of this header (KIVI_ABI_VERSION). */
#define KIVI_ABI_VERSION 1
KIVI_API int kivi_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KIVI_H */
