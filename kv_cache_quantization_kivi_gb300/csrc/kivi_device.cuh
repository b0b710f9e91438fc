// kivi_device.cuh -- device helpers shared by the KIVI kernels: the group
// quantizer with its exact rounding decision, packed binary32 (f32x2)
// arithmetic written as inline PTX, and streaming loads / stores.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

#include "kivi_arith.cuh"

namespace kivi_dev {

// Index checks of the debug build (compiled with -DKIVI_DEBUG_BOUNDS): every
// global access of the flush and full-tensor kernels first checks its offset
// against the extent of its bh slice that the host validated (and its slice
// and layer against the launch); a failed check records bit 4 of the device
// fault word and the access is skipped.  Release builds compile every check
// to `true`.
#ifdef KIVI_DEBUG_BOUNDS
__device__ __forceinline__ bool bound_check(bool ok, unsigned int *fault) {
  if (!ok && fault != nullptr) atomicOr(fault, 16u);
  return ok;
}
#define KIVI_BOUND(fault, cond) (::kivi_dev::bound_check((cond), (fault)))
#else
#define KIVI_BOUND(fault, cond) (true)
#endif

// ---------------------------------------------------------------------------
// Group quantizer
// ---------------------------------------------------------------------------
//
// Definition (per group, IEEE binary32; the VeloxQuant-MLX KIVI fused-kernel
// post, "What we're actually optimizing" and "2. Rounding mode"):
//   zero = min, scale = (max - min) / Q with Q = 2^b - 1,
//   q = clip(rint((x - zero) / scale), 0, Q), q = 0 when scale == 0,
// where both the subtraction and the division are rounded to binary32 and
// rint rounds half to even.
//
// Fast path.  Dividing every element costs a correctly rounded division.
// Instead each group precomputes r = RN(1/scale) and c = RN(-zero * r), and
// each element evaluates v = RN(x * r + c) with one fused multiply-add.
// With eps = 2^-24, T = RN(x - zero) / scale (the exact quotient of the
// rounded difference) and u = RN(T) (the quotient the definition rounds):
//   x*r + c = T (1+a)/(1+g) + e_c,  |a|,|g| <= eps,  |e_c| <= eps |zero*r|
//   v = (x*r + c)(1+h),             |h| <= eps
//   |T| <= Q (1 + 2 eps)            (x - zero <= max - min and monotone rounding)
// so |v - u| <= eps (4.001 Q + 1.001 |c|) =: E.  Let n = rint(v).  If
// |v - n| < 1/2 - E then u lies strictly within 1/2 of the integer n, so
// rint(u) = n and no tie is possible: the fast code is the defined code.
// Otherwise (v within E of a half-integer, about one element in 10^5 for
// b = 2) the caller recomputes the element with the exact division.  The
// group constants below use a threshold 1/2 - 2E, which also absorbs the
// rounding of the threshold's own computation.
//
// rint(v) for |v| < 2^22 comes from y = RN(v + 1.5*2^23): y lies in
// [2^23, 2^24) where the binary32 spacing is 1, so the addition itself
// rounds v to an integer with ties to even, and n = y - 1.5*2^23 is that
// integer, exactly.  codes2 below evaluates this for a pair of elements with
// packed f32x2 operations.

constexpr float kRoundMagic = 12582912.0f;  // 1.5 * 2^23

template <int BITS>
struct CodeFmt {
  static constexpr int W = 32 / BITS;            // codes per uint32 word
  static constexpr uint32_t Q = (1u << BITS) - 1u;
};

struct GroupQ {
  float scale;  // binary32 scale (0 when max == min)
  float zero;   // binary32 zero point (min, canonical +0)
  float r;      // RN(1/scale), 0 when scale == 0
  float c;      // RN(-zero * r)
  float thr;    // fast-path acceptance threshold on |v - rint(v)|
};

__device__ __forceinline__ GroupQ make_group(float mn, float mx, float qf) {
  GroupQ g;
  // A zero extreme may arrive as -0 or +0; adding +0 gives +0 either way.
  mn = __fadd_rn(mn, 0.0f);
  mx = __fadd_rn(mx, 0.0f);
  g.zero = mn;
  g.scale = div_by_q(__fsub_rn(mx, mn), qf);   // = RN((mx - mn) / Q)
  if (g.scale > 0.0f) {
    g.r = rcp_rn(g.scale);                      // = RN(1 / scale)
    g.c = __fmul_rn(-mn, g.r);
    // 2E = 2^-23 (4.01 Q + 1.01 |c|)
    const float two_e = __fmul_rn(__fmaf_rn(1.01f, fabsf(g.c), __fmul_rn(4.01f, qf)), 0x1p-23f);
    g.thr = __fsub_rn(0.5f, two_e);
  } else {
    g.r = 0.0f;     // v = 0 for every element: code 0, exact
    g.c = 0.0f;
    g.thr = 1.0f;
  }
  return g;
}

// The defined code, computed literally (used when the fast path declines).
__device__ __forceinline__ uint32_t exact_code(float x, const GroupQ &g, float qf) {
  if (g.scale == 0.0f) return 0u;
  const float t = __fsub_rn(x, g.zero);
  const float u = __fdiv_rn(t, g.scale);
  float r = rintf(u);
  r = fminf(fmaxf(r, 0.0f), qf);
  return static_cast<uint32_t>(r);
}

// ---------------------------------------------------------------------------
// Half-precision min / max.  binary16 -> binary32 conversion is exact and
// monotone, so min/max taken in binary16 equal min/max of the converted
// values; only the sign of a zero extreme can differ, and make_group
// canonicalises it.
// ---------------------------------------------------------------------------

__device__ __forceinline__ __half2 u32_as_h2(uint32_t u) {
  __half2 h;
  memcpy(&h, &u, 4);
  return h;
}
__device__ __forceinline__ uint32_t h2_as_u32(__half2 h) {
  uint32_t u;
  memcpy(&u, &h, 4);
  return u;
}

// ---------------------------------------------------------------------------
// Packed binary32 pairs (Blackwell f32x2 arithmetic: two IEEE operations,
// each rounded on its own, per instruction).  A pair is a 64-bit value with
// the first element in the low 32 bits.
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ uint32_t f2_lo_bits(uint64_t v) { return static_cast<uint32_t>(v); }
__device__ __forceinline__ uint32_t f2_hi_bits(uint64_t v) {
  return static_cast<uint32_t>(v >> 32);
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_const(float c) { return f2_pack(c, c); }
__device__ __forceinline__ uint64_t h2_to_f2(__half2 h) {
  const float2 f = __half22float2(h);
  return f2_pack(f.x, f.y);
}

// Constants of two groups (one per element of a pair) for the packed fast path.
struct GroupQ2 {
  uint64_t r;        // (r0, r1)
  uint64_t c;        // (c0, c1)
  uint64_t neg_thr2; // -(thr'^2) with thr' slightly below thr (see fast_codes2)
};

__device__ __forceinline__ float thr_sq_below(float thr) {
  // thr' = thr (1 - 2^-20) and RN(thr'^2) <= thr^2, so d^2 < RN(thr'^2)
  // implies |d| < thr.  A non-positive threshold rejects everything.
  if (!(thr > 0.0f)) return 0.0f;
  const float t = __fmul_rn(thr, 0.99999904632568359375f);
  return __fmul_rn(t, t);
}

__device__ __forceinline__ GroupQ2 make_group2(const GroupQ &a, const GroupQ &b) {
  GroupQ2 g;
  g.r = f2_pack(a.r, b.r);
  g.c = f2_pack(a.c, b.c);
  g.neg_thr2 = f2_pack(-thr_sq_below(a.thr), -thr_sq_below(b.thr));
  return g;
}

// The defined codes of a pair, computed literally, as an f32x2 pair of
// integer-valued floats.  It runs only for the rare pairs the fast path
// declines (mostly exact .5 ties, which fp16 data produce often).
template <int BITS>
__device__ __forceinline__ uint64_t exact_codes2_inline(float x0, float x1, float mn0, float mx0,
                                                     float mn1, float mx1) {
  const float qf = static_cast<float>((1u << BITS) - 1u);
  const GroupQ g0 = make_group(mn0, mx0, qf);
  const GroupQ g1 = make_group(mn1, mx1, qf);
  return f2_pack(static_cast<float>(exact_code(x0, g0, qf)),
                 static_cast<float>(exact_code(x1, g1, qf)));
}
template <int BITS>
__device__ __noinline__ uint64_t exact_codes2_outline(float x0, float x1, float mn0, float mx0,
                                                      float mn1, float mx1) {
  return exact_codes2_inline<BITS>(x0, x1, mn0, mx0, mn1, mx1);
}

// Codes of a pair as integer-valued floats (q0, q1).  y = RN(v + 1.5*2^23)
// rounds v to an integer, n = y - 1.5*2^23 is that integer exactly, and the
// acceptance test |v - n| < thr is evaluated as RN(d*d - RN(thr'^2)) < 0
// (sign bit set); a pair with an element outside it is recomputed by the
// literal division (out of line when OUTLINE, where register pressure makes
// inlined copies spill).  (mn0, mx0) and (mn1, mx1) are the extremes of the
// two elements' groups.
template <int BITS, bool OUTLINE>
__device__ __forceinline__ uint64_t codes2(uint64_t x, const GroupQ2 &g, float mn0, float mx0,
                                           float mn1, float mx1) {
  const uint64_t magic = f2_pack(kRoundMagic, kRoundMagic);
  const uint64_t v = f2_fma(x, g.r, g.c);
  const uint64_t y = f2_add(v, magic);
  const uint64_t n = f2_sub(y, magic);
  const uint64_t d = f2_sub(v, n);
  const uint64_t e = f2_fma(d, d, g.neg_thr2);
  if ((f2_lo_bits(e) & f2_hi_bits(e)) >> 31) return n;
  const float x0 = __uint_as_float(f2_lo_bits(x)), x1 = __uint_as_float(f2_hi_bits(x));
  return OUTLINE ? exact_codes2_outline<BITS>(x0, x1, mn0, mx0, mn1, mx1)
                 : exact_codes2_inline<BITS>(x0, x1, mn0, mx0, mn1, mx1);
}

// The same without a branch: the sign bits of the acceptance test are AND-ed
// into neg_acc (its top bit ends clear if some element needs the exact path),
// so a whole word of pairs is one basic block and its instructions
// interleave; a word whose flag is clear is recomputed with codes2.
__device__ __forceinline__ uint64_t codes2_nobranch(uint64_t x, const GroupQ2 &g,
                                                    uint32_t &neg_acc) {
  const uint64_t magic = f2_pack(kRoundMagic, kRoundMagic);
  const uint64_t v = f2_fma(x, g.r, g.c);
  const uint64_t y = f2_add(v, magic);
  const uint64_t n = f2_sub(y, magic);
  const uint64_t d = f2_sub(v, n);
  const uint64_t e = f2_fma(d, d, g.neg_thr2);
  neg_acc &= f2_lo_bits(e) & f2_hi_bits(e);
  return n;
}

// ---------------------------------------------------------------------------
// Fast path from the binary16 input ("difference first")
// ---------------------------------------------------------------------------
//
// The definition's first step, t = RN(x - zero), is one mixed-precision add
// from the binary16 input (add.rn.f32.f16: the exact binary16 -> binary32
// conversion and one rounded addition of -zero), so no separate conversion
// is needed.  Then v = RN(t * r) with r = RN(1/scale).  With eps = 2^-24,
// T = t / scale (exact) and u = RN(T) (the quotient the definition rounds):
//   t * r = T (1 + a),   v = T (1 + a)(1 + b),   u = T (1 + g),  |a|,|b|,|g| <= eps
//   0 <= T <= Q (1 + 2 eps)       (t <= RN(max - min), scale >= (max - min)(1 - eps) / Q)
// so |v - u| <= Q (1 + 2 eps)(3 eps + 3 eps^2) <= 3.0001 Q eps =: E, a bound
// that depends on the code width alone.  As for the fast path above, if
// |v - n| < 1/2 - E for n = rint(v) then rint(u) = n (and u < Q + 1/2, so
// no clip is needed); the test is run against 1/2 - 2E, here a compile-time
// constant per code width.  A group with scale == 0 has r = 0: v = 0 and
// every code 0, as defined.

struct GroupD2 {
  uint64_t r;    // (RN(1/scale0), RN(1/scale1)), 0 for a zero scale
  float nz0;     // -zero0
  float nz1;     // -zero1
};

__host__ __device__ constexpr double diff_thr(double q) {
  return 0.5 - 2.0 * 3.0001 * q * 5.9604644775390625e-8;   // 1/2 - 2E, E = 3.0001 Q 2^-24
}
// -(thr')^2 with thr' = thr (1 - 2^-20): the float rounding of the square
// (relative 2^-24) stays far inside the 2^-20 margin, so d^2 < thr'^2
// implies |d| < thr.
template <int BITS>
__host__ __device__ constexpr float diff_neg_thr2() {
  return -static_cast<float>(diff_thr((1 << BITS) - 1) * (1.0 - 9.5367431640625e-7) *
                             diff_thr((1 << BITS) - 1) * (1.0 - 9.5367431640625e-7));
}

// A group's scale, zero and reciprocal only (the difference-first path
// needs no other constant); the same arithmetic as make_group.
__device__ __forceinline__ GroupQ make_group_szr(float mn, float mx, float qf) {
  GroupQ g;
  mn = __fadd_rn(mn, 0.0f);
  mx = __fadd_rn(mx, 0.0f);
  g.zero = mn;
  g.scale = div_by_q(__fsub_rn(mx, mn), qf);
  g.r = g.scale > 0.0f ? rcp_rn(g.scale) : 0.0f;
  g.c = 0.0f;
  g.thr = 0.0f;
  return g;
}

__device__ __forceinline__ GroupD2 make_group_d2(const GroupQ &a, const GroupQ &b) {
  GroupD2 g;
  g.r = f2_pack(a.r, b.r);
  g.nz0 = -a.zero;
  g.nz1 = -b.zero;
  return g;
}

__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

// (RN(x0 - zero0), RN(x1 - zero1)) from a pair of binary16 values.
__device__ __forceinline__ uint64_t diff_pair(uint32_t x2, float nz0, float nz1) {
  float t0, t1;
  asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
      "add.rn.f32.f16 %0, lo, %3;\n\tadd.rn.f32.f16 %1, hi, %4;\n\t}"
      : "=f"(t0), "=f"(t1)
      : "r"(x2), "f"(nz0), "f"(nz1));
  return f2_pack(t0, t1);
}

// Codes of a pair as integer-valued floats, branch-free; the sign bits of the
// acceptance test are AND-ed into neg_acc (its top bit ends clear if some
// element needs the literal division).
template <int BITS>
__device__ __forceinline__ uint64_t codes2_diff_nobranch(uint32_t x2, const GroupD2 &g,
                                                         uint32_t &neg_acc) {
  const uint64_t magic = f2_pack(kRoundMagic, kRoundMagic);
  const uint64_t v = f2_mul(diff_pair(x2, g.nz0, g.nz1), g.r);
  const uint64_t y = f2_add(v, magic);
  const uint64_t n = f2_sub(y, magic);
  const uint64_t d = f2_sub(v, n);
  const uint64_t e = f2_fma(d, d, f2_const(diff_neg_thr2<BITS>()));
  neg_acc &= f2_lo_bits(e) & f2_hi_bits(e);
  return n;
}

// The defined codes of a pair with the literal division, from the groups'
// scale and zero (the rare pairs the difference-first path declines).
__device__ __noinline__ inline uint64_t exact_pair_sz(uint32_t x2, float s0, float z0, float s1,
                                                      float z1, float qf) {
  GroupQ a, b;
  a.scale = s0;
  a.zero = z0;
  b.scale = s1;
  b.zero = z1;
  const float2 x = __half22float2(u32_as_h2(x2));
  return f2_pack(static_cast<float>(exact_code(x.x, a, qf)),
                 static_cast<float>(exact_code(x.y, b, qf)));
}

// Codes of a pair: the difference-first fast path, or the literal division
// behind a branch per pair (almost never taken).
template <int BITS>
__device__ __forceinline__ uint64_t codes2_diff(uint32_t x2, const GroupD2 &g, float s0, float z0,
                                                float s1, float z1, float qf) {
  uint32_t ok = 0xFFFFFFFFu;
  const uint64_t n = codes2_diff_nobranch<BITS>(x2, g, ok);
  if (ok >> 31) return n;
  return exact_pair_sz(x2, s0, z0, s1, z1, qf);
}

// Packing.  Codes are small integers held exactly in binary32, so sums
// q_a + q_b * 2^k (k a multiple of the code width) below 2^24 are exact; a
// binary tree of such fused multiply-adds assembles a 16-bit half-word of
// codes, y = half + 2^23 then holds it in its low 16 mantissa bits, and one
// byte permute joins two half-words into a 32-bit code word (LSB first).

// Two 16-bit halves (as integer-valued floats) -> one word: lo | hi << 16.
__device__ __forceinline__ uint32_t join_halves(float lo, float hi) {
  const uint64_t b = f2_add(f2_pack(lo, hi), f2_const(8388608.0f));  // + 2^23
  return __byte_perm(f2_lo_bits(b), f2_hi_bits(b), 0x5410);
}
// The same for two pairs of halves (elementwise): returns (lo.x | hi.x << 16,
// lo.y | hi.y << 16).
__device__ __forceinline__ uint2 join_halves2(uint64_t lo, uint64_t hi) {
  const uint64_t a = f2_add(lo, f2_const(8388608.0f));
  const uint64_t b = f2_add(hi, f2_const(8388608.0f));
  return make_uint2(__byte_perm(f2_lo_bits(a), f2_lo_bits(b), 0x5410),
                    __byte_perm(f2_hi_bits(a), f2_hi_bits(b), 0x5410));
}

// ---------------------------------------------------------------------------
// Reconstruction: fp16(RN(RN(q * scale) + zero))  (fused-kernel post,
// "1. FMA contraction": the product is rounded before the add).
//
// q is turned into a float without a conversion instruction: m = the float
// with bits 0x4B000000 | q equals 2^23 + q.  Then RN(m*scale - 2^23*scale)
// with one fused multiply-add equals RN(q*scale) exactly: 2^23*scale is an
// exact power-of-two multiple, the real value m*scale - 2^23*scale is q*scale,
// and the fused operation rounds it once.  The add of zero is a separate,
// separately rounded operation.
// ---------------------------------------------------------------------------

__device__ __forceinline__ float recon_f32(uint32_t q, float scale, float neg_scale_2p23,
                                           float zero) {
  const float m = __uint_as_float(0x4B000000u | q);
  const float prod = __fmaf_rn(m, scale, neg_scale_2p23);
  return __fadd_rn(prod, zero);
}

// Reconstruction of a pair of integer-valued float codes n = (q0, q1) with
// per-element (scale, zero) pairs: fp16(RN(RN(q*scale) + zero)).  The product
// is formed as in recon_f32, inside an explicit fused multiply-add on
// m = 2^23 + q with the exact addend -2^23*scale (neg_scale2_2p23), because a
// packed multiply followed by a packed add may be contracted by the compiler
// into one fused multiply-add that rounds once (it was, and the result then
// differs in the last fp16 bit for about 3 in 10^4 elements).  An FMA result
// followed by an add offers nothing to contract.
__device__ __forceinline__ uint32_t recon_pair(uint64_t n, uint64_t scale2,
                                               uint64_t neg_scale2_2p23, uint64_t zero2) {
  const uint64_t m = f2_add(n, f2_pack(8388608.0f, 8388608.0f));  // 2^23 + q, exact
  const uint64_t r = f2_add(f2_fma(m, scale2, neg_scale2_2p23), zero2);
  const __half2 h = __floats2half2_rn(__uint_as_float(static_cast<uint32_t>(r)),
                                      __uint_as_float(static_cast<uint32_t>(r >> 32)));
  uint32_t u;
  memcpy(&u, &h, 4);
  return u;
}
// (-2^23 * s0, -2^23 * s1): exact, a power-of-two multiple.
__device__ __forceinline__ uint64_t neg_scale_2p23_pair(float s0, float s1) {
  return f2_pack(__fmul_rn(s0, -8388608.0f), __fmul_rn(s1, -8388608.0f));
}

// ---------------------------------------------------------------------------
// Streaming global loads / stores (data touched once)
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint4 ld_stream(const void *p) {
  return __ldcs(reinterpret_cast<const uint4 *>(p));
}
__device__ __forceinline__ void st_stream(void *p, uint4 v) {
  __stcs(reinterpret_cast<uint4 *>(p), v);
}
__device__ __forceinline__ void st_stream(void *p, uint2 v) {
  __stcs(reinterpret_cast<uint2 *>(p), v);
}

// ---------------------------------------------------------------------------
// Shared-memory pipeline: mbarrier and bulk asynchronous copies (the
// non-tensor form of the tensor memory accelerator), written as inline PTX.
// ---------------------------------------------------------------------------

// Programmatic dependent launch: a kernel launched with programmatic stream
// serialization may be scheduled while the previous grid in its stream
// drains; griddepcontrol.wait (a no-op without such a dependency) holds it
// until that grid has completed and its memory operations are visible, and
// launch_dependents lets the next grid be scheduled early in turn.
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Makes barrier initialisation visible to the asynchronous proxy.
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Orders this thread's earlier generic-proxy shared-memory accesses before
// later asynchronous-proxy accesses (a bulk copy into a buffer just read).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0u;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait for the phase of `bar` with the given parity to complete, giving up
// after `limit_ns` nanoseconds of wall-clock time.  Returns false on timeout.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  uint64_t limit_ns) {
#pragma unroll 1
  for (int i = 0; i < 32; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
#pragma unroll 1
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 > limit_ns) return false;
  }
}

// L2 policy for data read exactly once.
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// Bulk copy of `bytes` (a multiple of 16; both addresses 16-byte aligned)
// from global memory into this CTA's shared memory; completion is signalled
// on the mbarrier as transaction bytes.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes,
                                          uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

// ---------------------------------------------------------------------------
// Warp-level matrix multiply-accumulate (fp16 inputs, fp32 accumulation) and
// the 8x8 16-bit fragment transpose.
// ---------------------------------------------------------------------------

// d += a * b for one m16n8k16 tile: a = 4 registers of half2 (row-major
// 16x16), b = 2 registers (16x8, column-major), d = 4 fp32.
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                          uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Fragment of the transpose of an 8x8 matrix of 16-bit values held in the
// accumulator layout (lane l: row l/4, columns 2(l%4), 2(l%4)+1).
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t a) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
  return d;
}

}  // namespace kivi_dev
