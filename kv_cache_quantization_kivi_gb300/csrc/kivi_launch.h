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

// One fp16 tensor quantized into one code/scale/zero set.
struct QuantJob {
  const void *x;
  uint32_t *codes;
  float *scale;
  float *zero;
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
  DequantJob jobs[KIVI_MAX_LAYERS];
};

// Launchers (one per kernel family); they pick the template instance for
// (group, bits), size the grid from the device's SM count and occupancy,
// and return the launch's cudaError_t.
cudaError_t launch_key_quant(const QuantParams &p, int group, int bits, cudaStream_t stream);
cudaError_t launch_value_quant(const QuantParams &p, int group, int bits, cudaStream_t stream);
cudaError_t launch_key_dequant(const DequantParams &p, int group, int bits, cudaStream_t stream);
cudaError_t launch_value_dequant(const DequantParams &p, int group, int bits,
                                 cudaStream_t stream);

// Reads and clears the key kernel's fault record (synchronous).
cudaError_t read_and_clear_key_fault(uint32_t *fault);

}  // namespace kivi_impl
