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
  int64_t bh;
  int64_t rows;
  int64_t codes_bh_stride;
  int64_t sz_bh_stride;
  int64_t y_bh_stride;
  FastDiv div_chunks, div_rows, div_bh;  // filled by the launcher
  DequantJob jobs[KIVI_MAX_LAYERS];
};

// Launchers (one per kernel family); they pick the template instance for
// (group, bits), size the grid from the device's SM count and occupancy,
// and return the launch's cudaError_t.
// recon: also write the fp16 reconstruction of every quantized element
// (jobs[i].y, p.y_bh_stride, p.y_row0).
cudaError_t launch_key_quant(const QuantParams &p, int group, int bits, bool recon,
                             cudaStream_t stream);
cudaError_t launch_value_quant(const QuantParams &p, int group, int bits, bool recon,
                               cudaStream_t stream);
cudaError_t launch_key_dequant(const DequantParams &p, int group, int bits, cudaStream_t stream);
cudaError_t launch_value_dequant(const DequantParams &p, int group, int bits,
                                 cudaStream_t stream);

}  // namespace kivi_impl
