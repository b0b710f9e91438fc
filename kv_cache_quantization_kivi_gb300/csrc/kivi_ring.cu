// kivi_ring.cu -- the residual ring's append: new tokens of every layer
// written behind the residual window in one launch.
//
// The newest tokens of a KIVI cache stay fp16 in a residual window and age
// out of it in whole groups by flushes (VeloxQuant-MLX KIVI fused-kernel
// post, "What we're actually optimizing").  Here the window is a ring of
// r_cap rows per bh slice; logical residual token i lives at ring row
// (res_head + i) % r_cap, so appending n tokens writes rows
// (res_head + n_res + j) % r_cap, j < n, and moves nothing else.
//
// One thread copies one 16-byte piece (8 channels) of one token of one bh
// slice of one layer, for keys and values: a warp reads 512 contiguous bytes
// of the new tokens and writes 512 contiguous bytes of a ring row (whole
// rows at d = 128; the ring's wrap only moves whole rows).
#include <cuda_runtime.h>

#include "kivi_device.cuh"
#include "kivi_launch.h"

namespace kivi_impl {
namespace {

constexpr int kAppendThreads = 256;

// unit = ((job * bh + b) * n + i) * (d / 8) + c   (< 2^31, host-checked)
__global__ void __launch_bounds__(kAppendThreads)
    append_kernel(const __grid_constant__ AppendParams p) {
  kivi_dev::grid_dependency_wait();
  kivi_dev::grid_launch_dependents();
  const uint32_t total = static_cast<uint32_t>(p.n_jobs) * p.div_bh.d * p.div_n.d *
                         p.div_chunks.d;
  const uint32_t stride = gridDim.x * blockDim.x;
#pragma unroll 1
  for (uint32_t u = blockIdx.x * blockDim.x + threadIdx.x; u < total; u += stride) {
    const uint32_t row_all = p.div_chunks.div(u);
    const uint32_t c = u - row_all * p.div_chunks.d;
    const uint32_t jb = p.div_n.div(row_all);
    const uint32_t i = row_all - jb * p.div_n.d;
    const uint32_t job = p.div_bh.div(jb);
    const uint32_t b = jb - job * p.div_bh.d;
    const AppendJob &J = p.jobs[job];
    int64_t row = p.row0 + i;            // row0 < r_cap and i < r_cap
    if (row >= p.r_cap) row -= p.r_cap;
    const int64_t src = static_cast<int64_t>(b) * p.new_bh_stride +
                        static_cast<int64_t>(i) * p.d + 8 * c;
    const int64_t dst = (static_cast<int64_t>(b) * p.r_cap + row) * p.d + 8 * c;
    // debug builds: both rows lie inside their bh slices
    if (!KIVI_BOUND(p.fault, b < p.bh && static_cast<int64_t>(i) * p.d + 8 * c + 8 <=
                                 p.new_bh_stride && row >= 0 && row < p.r_cap))
      continue;
    const uint4 kv = kivi_dev::ld_stream(static_cast<const uint16_t *>(J.k_new) + src);
    const uint4 vv = kivi_dev::ld_stream(static_cast<const uint16_t *>(J.v_new) + src);
    *reinterpret_cast<uint4 *>(static_cast<uint16_t *>(J.k_res) + dst) = kv;
    *reinterpret_cast<uint4 *>(static_cast<uint16_t *>(J.v_res) + dst) = vv;
  }
}

}  // namespace

cudaError_t launch_append(const AppendParams &p, cudaStream_t stream) {
  AppendParams q = p;
  q.div_chunks = FastDiv::make(static_cast<uint32_t>(p.d / 8));
  q.div_n = FastDiv::make(static_cast<uint32_t>(p.n));
  q.div_bh = FastDiv::make(static_cast<uint32_t>(p.bh));
  const int64_t units = static_cast<int64_t>(p.n_jobs) * p.bh * p.n * (p.d / 8);
  const cudaError_t e = debug_fault_word(&q.fault);
  if (e != cudaSuccess) return e;
  return launch_dependent(append_kernel, flat_grid(units, kAppendThreads), kAppendThreads,
                          stream, q);
}

}  // namespace kivi_impl
