// GPU check of the quantize kernels' per-element code (kivi_device.cuh)
// against the literal definition with the IEEE division (exact_code), on
// random binary16 groups and on elements placed next to a rounding midpoint
// (k + 1/2) * scale, for Q = 3, 15, 255, for both fast paths: codes2 (the
// fused multiply-add form with its literal-division fallback) and
// codes2_diff_nobranch (difference first; every code it accepts must be the
// defined one, the pairs it declines are counted).  Prints the samples,
// mismatches and declined pairs per path and mode; exit status 1 if any
// mismatch.
#include <cstdio>

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "../../kv_cache_quantization_kivi_gb300/csrc/kivi_device.cuh"

using namespace kivi_dev;

__device__ __forceinline__ unsigned long long mix(unsigned long long z) {
  z += 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

// a finite binary16 value from 16 random bits (an exponent field of 31 -- inf
// or NaN -- is folded to 30)
__device__ __forceinline__ float rand_half(unsigned int bits) {
  unsigned short u = static_cast<unsigned short>(bits);
  if ((u & 0x7C00u) == 0x7C00u) u &= 0xFBFFu;
  return __half2float(__ushort_as_half(u));
}

__global__ void check(unsigned long long *bad, unsigned long long iters, int mode, int path) {
  unsigned long long n_bad = 0, n_declined = 0;
  const unsigned long long tid = blockIdx.x * static_cast<unsigned long long>(blockDim.x) + threadIdx.x;
  for (unsigned long long i = 0; i < iters; ++i) {
    const unsigned long long h = mix(tid * 0x100000001B3ull + i * 0x9E3779B97F4A7C15ull + mode);
    const float qf = (h & 3) == 0 ? 3.0f : (h & 3) == 1 ? 15.0f : (h & 3) == 2 ? 255.0f : 3.0f;
    float a = rand_half(static_cast<unsigned int>(h >> 8));
    float b = rand_half(static_cast<unsigned int>(h >> 24));
    if ((h >> 60) == 0) {                      // narrow groups (kept finite)
      const float nb = __half2float(__float2half_rn(a * 1.0009765625f));
      b = fabsf(nb) <= 65504.0f ? nb : a;
    }
    const float mn = fminf(a, b), mx = fmaxf(a, b);
    const GroupQ g = make_group(mn, mx, qf);
    float x[2];
    for (int e = 0; e < 2; ++e) {
      const unsigned long long h2 = mix(h + e + 1);
      float v;
      if (mode == 0) {
        v = rand_half(static_cast<unsigned int>(h2));
      } else {   // next to a midpoint k + 1/2 of the grid
        const float k = static_cast<float>(static_cast<unsigned int>(h2 >> 20) % static_cast<unsigned int>(qf)) + 0.5f;
        const float m = __fadd_rn(g.zero, __fmul_rn(k, g.scale));
        const unsigned short hm = __half_as_ushort(__float2half_rn(m));
        const int d = static_cast<int>((h2 >> 40) % 5) - 2;
        v = __half2float(__ushort_as_half(static_cast<unsigned short>(hm + d)));
        if (!(v == v) || fabsf(v) > 65504.0f) v = mn;
      }
      x[e] = fminf(fmaxf(v, mn), mx);   // inside the group's range, as every element is
    }
    const float q0 = static_cast<float>(exact_code(x[0], g, qf));
    const float q1 = static_cast<float>(exact_code(x[1], g, qf));
    if (path == 0) {
      const GroupQ2 g2 = make_group2(g, g);
      const uint64_t xs = f2_pack(x[0], x[1]);
      const uint64_t n = qf == 3.0f    ? codes2<2, false>(xs, g2, mn, mx, mn, mx)
                         : qf == 15.0f ? codes2<4, false>(xs, g2, mn, mx, mn, mx)
                                       : codes2<8, false>(xs, g2, mn, mx, mn, mx);
      n_bad += __uint_as_float(f2_lo_bits(n)) != q0;
      n_bad += __uint_as_float(f2_hi_bits(n)) != q1;
    } else {
      // difference first: accepted codes must be the defined ones, and a
      // declined pair (the caller then takes the literal division) is counted
      const GroupD2 gd = make_group_d2(g, g);
      const uint32_t x2 = static_cast<uint32_t>(__half_as_ushort(__float2half_rn(x[0]))) |
                          (static_cast<uint32_t>(__half_as_ushort(__float2half_rn(x[1]))) << 16);
      uint32_t acc = 0xFFFFFFFFu;
      const uint64_t n = qf == 3.0f    ? codes2_diff_nobranch<2>(x2, gd, acc)
                         : qf == 15.0f ? codes2_diff_nobranch<4>(x2, gd, acc)
                                       : codes2_diff_nobranch<8>(x2, gd, acc);
      if (acc >> 31) {
        n_bad += __uint_as_float(f2_lo_bits(n)) != q0;
        n_bad += __uint_as_float(f2_hi_bits(n)) != q1;
      } else {
        ++n_declined;
      }
    }
  }
  atomicAdd(bad, n_bad);
  atomicAdd(bad + 1, n_declined);
}

int main() {
  unsigned long long *d = nullptr, h[2] = {0, 0};
  if (cudaMalloc(&d, sizeof(h)) != cudaSuccess) return 2;
  int sms = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
  const int blocks = sms * 8, threads = 256;
  const unsigned long long iters = 1024;
  int failed = 0;
  for (int path = 0; path < 2; ++path) {
    for (int mode = 0; mode < 2; ++mode) {
      cudaMemset(d, 0, sizeof(h));
      check<<<blocks, threads>>>(d, iters, mode, path);
      if (cudaMemcpy(h, d, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return 2;
      std::printf("path=%s mode=%s samples=%llu mismatches=%llu declined=%llu\n",
                  path ? "difference-first" : "fma", mode ? "near-midpoint" : "random",
                  2ull * blocks * threads * iters, h[0], h[1]);
      failed |= h[0] != 0;
    }
  }
  cudaFree(d);
  return failed;
}
