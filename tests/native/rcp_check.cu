// GPU check of the quantize kernels' reciprocal (kivi_arith.cuh, rcp_rn):
// bit-identical to __frcp_rn for every normal b in [2^-126, 2^126).  Prints
// the count checked and the mismatches; exit status 1 if any.
#include <cstdio>

#include <cuda_runtime.h>

#include "../../kv_cache_quantization_kivi_gb300/csrc/kivi_arith.cuh"

__global__ void check(unsigned long long *bad, unsigned int lo, unsigned int hi) {
  unsigned long long n = 0;
  for (unsigned int u = lo + blockIdx.x * blockDim.x + threadIdx.x; u < hi;
       u += gridDim.x * blockDim.x) {
    const float b = __uint_as_float(u);
    n += __float_as_uint(kivi_dev::rcp_rn(b)) != __float_as_uint(__frcp_rn(b));
  }
  atomicAdd(bad, n);
}

int main() {
  unsigned long long *d = nullptr, h = 0;
  if (cudaMalloc(&d, sizeof(h)) != cudaSuccess) return 2;
  cudaMemset(d, 0, sizeof(h));
  const unsigned int lo = 0x00800000u, hi = 0x7E800000u;
  int sms = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
  check<<<sms * 8, 256>>>(d, lo, hi);
  const cudaError_t e = cudaMemcpy(&h, d, sizeof(h), cudaMemcpyDeviceToHost);
  cudaFree(d);
  if (e != cudaSuccess) {
    std::printf("cuda error %s\n", cudaGetErrorString(e));
    return 2;
  }
  std::printf("checked=%u mismatches=%llu\n", hi - lo, h);
  return h != 0;
}
