// kivi_launch.h -- parameters shared by the host entry points and the kernels.
//
// Every kernel takes one parameter block (passed by value, __grid_constant__)
// that lists up to KIVI_MAX_LAYERS tensors ("jobs") of identical geometry, so
// one launch covers every layer of a cache.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kivi.h"

namespace kivi_impl {

// Division of unsigned n < 2^31 by a fixed divisor d >= 1 without a divide:
// with l = ceil(log2 d) and m = floor(2^32 (2^l - d) / d) + 1,
// n / d = (umulhi(n, m) + n) >> l  (Granlund and Montgomery, "Division by
// invariant integers using multiplication", 1994).  n + umulhi(n, m) stays
// below 2^32 because n < 2^31.
struct FastDiv {
  uint32_t d, m, l;
  static FastDiv make(uint32_t d) {
    FastDiv f;
    f.d = d;
    f.l = 0;
    while ((uint64_t{1} << f.l) < d) ++f.l;
    f.m = static_cast<uint32_t>(((uint64_t{1} << 32) * ((uint64_t{1} << f.l) - d)) / d + 1);
    return f;
  }
#ifdef __CUDACC__
  __device__ __forceinline__ uint32_t div(uint32_t n) const {
    return (__umulhi(n, m) + n) >> l;
  }
#endif
};

// One fp16 tensor quantized into one code/scale/zero set, and (fused
// fake-quant calls) its fp16 reconstruction y.  codes/scale/zero may be null
// in the fake-quant full-tensor calls (then only y is written).
struct QuantJob {
  const void *x;
  uint32_t *codes;
  float *scale;
  float *zero;
  void *y;
  const uint32_t *mask;  // sink mode: [batch][mask_words] bit r = logical row r is a sink
};

// Quantization of n_jobs tensors [bh][*][d].
//   rows         tokens to quantize (logical rows 0 .. rows-1)
//   ring, head   ring == 0: logical row r is stored row r;  ring > 0: logical
//                row r is stored row (head + r) % ring (residual ring)
//   out0         keys: group index in the output of logical group 0
//                values: row index in the output of logical row 0
struct QuantParams {
  int32_t n_jobs;
  int32_t d;
  // 1: the launch's inputs do not depend on the previous grid in the stream
  // (programmatic dependent launch): the kernel starts its work at once and
  // waits for that grid only before it ends, so its blocks fill the SMs the
  // previous grid's tail leaves idle while stream order is kept
  int32_t defer_wait;
  int32_t pad0;
  int64_t bh;
  int64_t rows;
  int64_t x_bh_stride;      // fp16 elements
  int64_t codes_bh_stride;  // uint32 words
  int64_t sz_bh_stride;     // floats
  int64_t ring;
  int64_t head;
  int64_t out0;
  int64_t y_bh_stride;      // fp16 elements (reconstruction)
  int64_t y_row0;           // row of the reconstruction of logical row 0
  int64_t heads;            // sink mode: bh slices per sequence (sequence = bh / heads)
  int64_t mask_words;       // sink mode: mask words per sequence
  unsigned int *fault;      // the device fault word (staged kernels, bit 3: a pipeline wait
                            // timed out; debug builds, bit 4: an index check failed);
                            // filled by the launchers that use it
  // filled by the launchers: divisors of the kernels' unit index
  FastDiv div_chunks, div_rows, div_bh;
  QuantJob jobs[KIVI_MAX_LAYERS];
};

struct DequantJob {
  const uint32_t *codes;
  const float *scale;
  const float *zero;
  void *y;
};

// Dequantization of n_jobs code sets into fp16 [bh][rows][d].
struct DequantParams {
  int32_t n_jobs;
  int32_t d;
  int32_t defer_wait;   // as QuantParams::defer_wait
  int32_t pad0;
  int64_t bh;
  int64_t rows;
  int64_t codes_bh_stride;
  int64_t sz_bh_stride;
  int64_t y_bh_stride;
  FastDiv div_chunks, div_rows, div_bh;  // filled by the launcher
  unsigned int *fault;                  // debug builds: the device fault word (bit 4)
  DequantJob jobs[KIVI_MAX_LAYERS];
};

// Append of n new tokens of every layer behind its residual: token i of
// bh slice b of job l goes from new[b * new_bh_stride + i * d ..] to ring row
// (row0 + i) % r_cap of the layer's rings (row0 = (res_head + n_res) % r_cap).
struct AppendJob {
  const void *k_new;   // fp16 [bh][n][d] (bh stride new_bh_stride)
  const void *v_new;
  void *k_res;         // fp16 rings [bh][r_cap][d]
  void *v_res;
};
struct AppendParams {
  int32_t n_jobs;
  int32_t d;
  int64_t bh;
  int64_t n;
  int64_t r_cap;
  int64_t row0;
  int64_t new_bh_stride;  // fp16 elements
  FastDiv div_chunks, div_n, div_bh;  // filled by the launcher
  unsigned int *fault;                // debug builds: the device fault word (bit 4)
  AppendJob jobs[KIVI_MAX_LAYERS];
};
cudaError_t launch_append(const AppendParams &p, cudaStream_t stream);

// Decode attention over one layer's cache: the packed store (key and value
// codes, scales, zeros) and the fp16 residual rings, queries fp16
// [batch][h_q][d], output fp32 [batch][h_q][d].
struct AttnJob {
  const uint32_t *k_codes;
  const float *k_scale;
  const float *k_zero;
  const uint32_t *v_codes;
  const float *v_scale;
  const float *v_zero;
  const void *k_res;
  const void *v_res;
  const void *q;
  float *out;
  // KIVI-Sink store of the layer (all null without sinks): per sequence the
  // positions (ascending) and count, per bh the fp16 key / value rows
  const int64_t *sink_pos;    // [batch][sink_cap]
  const int32_t *sink_count;  // [batch]
  const void *sink_k;         // fp16 [bh][sink_cap][d]
  const void *sink_v;
};

// Work item = (job, bh, split): split s covers store tiles [s*tps, (s+1)*tps)
// (tiles of 32 tokens; with G = 16 the last one may hold 16) and the last
// split also the residual tiles.
struct AttnParams {
  int32_t n_jobs;
  int32_t d;          // head_dim: 64, 128 or 256
  int32_t r;          // query heads per KV head
  int32_t h_kv;       // KV heads per sequence (bh = batch * h_kv)
  int32_t n_split;
  int32_t tiles_store;
  int32_t tiles_res;
  int32_t tiles_per_split;
  int32_t tail_half;  // 1: the last store tile holds 16 tokens (G = 16, s_q = 16 mod 32)
  int64_t bh;
  int64_t cap;        // store capacity (tokens)
  int64_t r_cap;      // ring capacity (tokens)
  int64_t res_head;
  int64_t n_res;
  float scale_log2;   // softmax scale * log2(e)
  int32_t sink_cap;   // > 0: the jobs' sink stores are read (see AttnJob)
  float *ws;          // n_split > 1: partial results, see kivi_attention_kernel.cuh
  unsigned int *fault;   // device fault word (filled by the launchers)
  AttnJob jobs[KIVI_MAX_LAYERS];
};

// KIVI-Sink state of one layer (device arrays) and the call's parameters.
constexpr int kMaxSinkTop = 64;   // largest running top-k
struct SinkJob {
  const void *k_res;      // fp16 rings [bh][r_cap][d]
  const void *v_res;
  int64_t *top_pos;       // [batch][k_top] running top-k positions, ranked
  float *top_score;       // [batch][k_top]
  int32_t *top_count;     // [batch]
  int64_t *sink_pos;      // [batch][sink_cap] positions of the stored sinks
  int32_t *sink_count;    // [batch]
  void *sink_k;           // fp16 [bh][sink_cap][d]
  void *sink_v;
  uint32_t *mask;         // [batch][mask_words] flush scratch
  float *scores;          // [batch][r_cap] update scratch
  void *k_out;            // restore: fp16 [bh][out_rows][d]
  void *v_out;
};
struct SinkParams {
  int32_t n_jobs;
  int32_t k_top;
  int32_t sink_cap;
  int32_t pad;
  int64_t batch;
  int64_t heads;
  int64_t d;
  int64_t r_cap;
  int64_t res_head;
  int64_t s_q;            // store tokens before the call (positions of residual token i: s_q + i)
  int64_t i0, n;          // update: residual tokens i0 .. i0+n-1; flush: n tokens flushed
  int64_t mask_words;
  int64_t out_rows;       // restore: rows of k_out / v_out
  unsigned int *fault;    // the device fault word (bit 1: sink store overflow)
  SinkJob jobs[KIVI_MAX_LAYERS];
};
cudaError_t launch_sink_update(const SinkParams &p, cudaStream_t stream);
cudaError_t launch_sink_prepare(const SinkParams &p, cudaStream_t stream);
cudaError_t launch_sink_restore(const SinkParams &p, cudaStream_t stream);

// Launchers (one per kernel family); they pick the template instance for
// (group, bits), size the grid from the device's SM count and occupancy,
// and return the launch's cudaError_t.
// mode kQuantPlain: codes, scales, zeros; kQuantRecon: also the fp16
// reconstruction of every quantized element (jobs[i].y, p.y_bh_stride,
// p.y_row0); kQuantSink: rows flagged in jobs[i].mask are left out of the
// key groups' min/max and get code 0 (value rows: codes, scales, zeros 0).
enum { kQuantPlain = 0, kQuantRecon = 1, kQuantSink = 2 };
cudaError_t launch_key_quant(const QuantParams &p, int group, int bits, int mode,
                             cudaStream_t stream);
cudaError_t launch_value_quant(const QuantParams &p, int group, int bits, int mode,
                               cudaStream_t stream);
cudaError_t launch_key_dequant(const DequantParams &p, int group, int bits, cudaStream_t stream);
// The staged key quantizer (head_dim 128, G >= 32, plain and fused modes):
// whole G x 128 tiles streamed into a shared-memory ring by bulk copies.
// Sets *handled = false (and launches nothing) for arguments it does not take.
cudaError_t launch_key_quant_staged(const QuantParams &p, int group, int bits, int mode,
                                    cudaStream_t stream, bool *handled);
// Decode attention (head_dim 64, 128 or 256): the main kernel, then
// (n_split > 1) the combine kernel.  The register-MMA kernel
// (kivi_attention_kernel.cuh) serves every call; with
// KIVI_ATTENTION_KERNEL=tcgen05 in the environment the tensor-memory kernel
// (kivi_attention_ws.cu) serves the calls at head_dim 128 without a sink
// store at G >= 32.
cudaError_t launch_decode_attention(const AttnParams &p, int group, int bits,
                                    cudaStream_t stream);
// The register-operand kernels at head_dim 64 and 256 (each in its own
// translation unit; 128 is in kivi_attention.cu).
cudaError_t launch_decode_attention_d64(const AttnParams &p, int group, int bits,
                                        cudaStream_t stream);
cudaError_t launch_decode_attention_d256(const AttnParams &p, int group, int bits,
                                         cudaStream_t stream);
// The warp-specialised persistent tensor-memory kernel (kivi_attention_ws.cu;
// head_dim 128, G >= 32, no sink store, r <= 8): sets *handled = false (and
// launches nothing) for arguments it does not take.
cudaError_t launch_decode_attention_ws(const AttnParams &p, int group, int bits,
                                       cudaStream_t stream, bool *handled);
// The split combine (n_split > 1): out = sum_s e^(m_s - M) o_s / sum_s
// e^(m_s - M) l_s per (layer, sequence, query head, channel) from p.ws.
cudaError_t launch_attention_combine(const AttnParams &p, cudaStream_t stream);
// Recommended number of splits for `items` (job, bh) pairs of `tiles_store`
// store tiles each on the current device.
int attention_splits(int64_t items, int64_t tiles_store, int group, int bits);
// The file-scope device workspace of the allocation-free decode attention:
// its address on the current device (looked up once per device) and size.
cudaError_t attention_scratch(float **ptr, int64_t *max_floats);
int64_t attention_scratch_floats();
// SM count of the current device (looked up once per device).
int current_sm_count();
// Launch of a grid-stride kernel that starts with grid_dependency_wait():
// with programmatic stream serialization, so that its blocks are scheduled
// while the previous kernel in the stream drains and start their work the
// moment it completes (the ordering is that of a plain launch).
template <typename P>
cudaError_t launch_dependent(void (*kern)(P), int64_t grid, int threads, cudaStream_t stream,
                             const P &params, size_t dynamic_smem = 0) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(static_cast<unsigned>(threads));
  cfg.dynamicSmemBytes = dynamic_smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, params);
}
// Grid of one block per `threads` units for a grid-stride kernel, clamped to
// the launch limit of 2^31 - 1 blocks in x (at least one block).
inline int64_t flat_grid(int64_t units, int threads) {
  const int64_t blocks = (units + threads - 1) / threads;
  return blocks < 1 ? 1 : (blocks > 2147483647 ? 2147483647 : blocks);
}
// Address of the device fault word on the current device (looked up once
// per device), for kernels of other translation units.
cudaError_t fault_word_address(unsigned int **ptr);
// The fault word for the index checks of the debug build; nullptr (and no
// lookup) in release builds.
inline cudaError_t debug_fault_word(unsigned int **ptr) {
#ifdef KIVI_DEBUG_BOUNDS
  return fault_word_address(ptr);
#else
  *ptr = nullptr;
  return cudaSuccess;
#endif
}
// Reads and clears the device word in which kernels record a pipeline wait
// that timed out (bit 0: decode attention).
cudaError_t read_and_clear_fault(uint32_t *fault);
// One warp's bounded wait on a phase that nothing completes (bit 2 of the
// fault word once it gives up).
cudaError_t launch_wait_timeout_selftest(uint64_t limit_ns, cudaStream_t stream);
cudaError_t launch_value_dequant(const DequantParams &p, int group, int bits,
                                 cudaStream_t stream);

}  // namespace kivi_impl
