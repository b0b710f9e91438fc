// kivi_expand.cuh -- expansion of packed KIVI codes into fp16
// reconstructions, shared by the decode-attention kernels: the same
// arithmetic as the dequantize kernels, fp16(RN(RN(q * scale) + zero)) (the
// product inside a fused multiply-add with an exact addend, so nothing is
// contracted), and for 2-bit codes a four-entry fp16 table per (scale, zero)
// looked up with byte permutes (bit-identical results).
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

#include "kivi_device.cuh"

namespace kivi_dev {

// 2^23 + q as floats for the codes of one word, in code order.  Codes are
// spread four to a register (one byte each) by a shift and a mask, then a
// byte permute puts each byte under the exponent of 2^23.
template <int BITS>
__device__ __forceinline__ void word_magics(uint32_t w, float *m) {
  constexpr uint32_t M = 0x4B000000u;
  if (BITS == 8) {
#pragma unroll
    for (int k = 0; k < 4; ++k) m[k] = __uint_as_float(__byte_perm(w, M, 0x7650u + k));
  } else {
    constexpr int PER_BYTE = 8 / BITS;                      // codes per byte
    constexpr uint32_t MASK = BITS == 2 ? 0x03030303u : 0x0F0F0F0Fu;
#pragma unroll
    for (int j = 0; j < PER_BYTE; ++j) {
      const uint32_t y = (w >> (j * BITS)) & MASK;         // byte k: code k*PER_BYTE + j
#pragma unroll
      for (int k = 0; k < 4; ++k)
        m[k * PER_BYTE + j] = __uint_as_float(__byte_perm(y, M, 0x7650u + k));
    }
  }
}

// 2^23 + q floats of 16 consecutive codes: one word (2 bits), two (4 bits)
// or four (8 bits), in code order.
template <int BITS>
__device__ __forceinline__ void magics16(const uint32_t *w, float (&m)[16]) {
  constexpr int W = 32 / BITS;
#pragma unroll
  for (int i = 0; i < 16 / W; ++i) word_magics<BITS>(w[i], m + i * W);
}

// fp16 reconstructions of 8 consecutive codes (as magic floats) sharing one
// (scale, -2^23 scale, zero): fp16(RN(RN(q scale) + zero)), the product made
// inside an FMA with an exact addend (nothing to contract), the add rounded
// separately.
__device__ __forceinline__ uint4 deq8(const float *m, uint64_t s2, uint64_t ns2, uint64_t z2) {
  uint32_t h[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint64_t r = f2_add(f2_fma(f2_pack(m[2 * i], m[2 * i + 1]), s2, ns2), z2);
    h[i] = h2_as_u32(__floats2half2_rn(__uint_as_float(static_cast<uint32_t>(r)),
                                       __uint_as_float(static_cast<uint32_t>(r >> 32))));
  }
  return make_uint4(h[0], h[1], h[2], h[3]);
}

__device__ __forceinline__ void scale_consts(float s, float z, uint64_t &s2, uint64_t &ns2,
                                             uint64_t &z2) {
  const float ns = __fmul_rn(s, -8388608.0f);   // -2^23 s, exact
  s2 = f2_pack(s, s);
  ns2 = f2_pack(ns, ns);
  z2 = f2_pack(z, z);
}

// 2-bit codes: the four possible reconstructions of a unit (one scale and
// zero) as an fp16 table in two registers (lo = codes 0, 1; hi = codes 2, 3),
// and the 16 codes of a word looked up with byte permutes.  A code q spread
// into a byte becomes the byte pair selector 0x22 q + 0x10 (bytes 2q, 2q+1 of
// the table) by one integer multiply-add over four bytes at once.  Output
// order: half2 word i of chunk k holds codes 8k + i and 8k + i + 4, i.e.
// position p of a chunk holds code kPerm[p] (see perm8 below).
__device__ __forceinline__ void lut2(float s, float z, uint32_t &lo, uint32_t &hi) {
  uint64_t s2, ns2, z2;
  scale_consts(s, z, s2, ns2, z2);
  const uint64_t m01 = f2_pack(__uint_as_float(0x4B000000u), __uint_as_float(0x4B000001u));
  const uint64_t m23 = f2_pack(__uint_as_float(0x4B000002u), __uint_as_float(0x4B000003u));
  const uint64_t r01 = f2_add(f2_fma(m01, s2, ns2), z2);
  const uint64_t r23 = f2_add(f2_fma(m23, s2, ns2), z2);
  lo = h2_as_u32(__floats2half2_rn(__uint_as_float(static_cast<uint32_t>(r01)),
                                   __uint_as_float(static_cast<uint32_t>(r01 >> 32))));
  hi = h2_as_u32(__floats2half2_rn(__uint_as_float(static_cast<uint32_t>(r23)),
                                   __uint_as_float(static_cast<uint32_t>(r23 >> 32))));
}
__device__ __forceinline__ void lookup16(uint32_t w, uint32_t lo, uint32_t hi, uint4 &c0,
                                         uint4 &c1) {
  uint32_t h[8];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t y = (w >> (2 * j)) & 0x03030303u;   // byte k: code 4k + j
    const uint32_t sel = y * 0x22u + 0x10101010u;       // byte pair selectors
    h[j] = __byte_perm(lo, hi, sel);                    // codes j, j + 4
    h[4 + j] = __byte_perm(lo, hi, sel >> 16);          // codes j + 8, j + 12
  }
  c0 = make_uint4(h[0], h[1], h[2], h[3]);
  c1 = make_uint4(h[4], h[5], h[6], h[7]);
}
// Within each 8-element chunk the 2-bit path stores element perm8(p) at
// position p: p = 2i holds i, p = 2i + 1 holds i + 4; its inverse places
// element e at 2e (e < 4) or 2(e - 4) + 1.
__device__ __forceinline__ int perm8(int p) { return (p >> 1) + ((p & 1) << 2); }
__device__ __forceinline__ int perm8_inv(int e) { return ((e & 3) << 1) | (e >> 2); }


}  // namespace kivi_dev
