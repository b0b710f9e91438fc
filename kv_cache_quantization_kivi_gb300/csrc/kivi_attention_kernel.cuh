// kivi_attention_kernel.cuh -- the register-operand decode-attention kernel
// that reads the packed KIVI store, templated on head_dim D in {64, 128, 256}
// (each D instantiated in its own translation unit: kivi_attention.cu for
// 128, kivi_attention_d64.cu and kivi_attention_d256.cu).
//
// The fused-kernel post's closing section names the step after the fused
// quantizer: attention that reads the packed codes directly, so that the
// fp16 expansion happens in registers and never in memory.  This kernel
// computes, for every layer, sequence and query head,
//   out = softmax(scale * q K^T) V
// over the cache's s_q store tokens (dequantized in registers, bit-identical
// to the fp16 reconstruction of the dequantize kernels) followed by its n_res
// fp16 residual tokens.  Query head h of a sequence reads KV head h / r.
//
// Work item (one CTA of 4 warps) = (layer, bh, split).  Its store tiles (32
// tokens each; at G = 16 the last may hold 16) and, in the last split, its
// residual tiles are dealt to the
// warps round-robin; each warp streams its store tiles' key codes, key
// scale/zero rows, value codes and value scales/zeros (six contiguous pieces)
// into a private shared-memory ring with bulk asynchronous copies completed
// on per-stage mbarriers, so no CTA barrier is needed until the end.  Per
// tile the warp expands the codes cooperatively -- each lane one key channel
// (four of them) or one value token, so a code word's scale is loaded once
// and its codes are spread four to a register with one shift, one mask and
// byte permutes -- into an fp16 tile in its own shared-memory buffer
// (swizzled so that 16-byte stores and ldmatrix rows avoid bank conflicts),
// then:
//   S^T = K Q^T     m16n8k16 tensor-core MMAs: A = key tile (16 tokens x 16
//                   channels, ldmatrix), B = the query heads
//   online softmax  per head column, base-2 exponent with the scale folded in
//                   (the hardware's approximate exponential, well inside the
//                   error the result's bound allows it); the reference moves
//                   only when a score exceeds it by > 2^3
//   O^T += V^T P^T  A = value tile (16 channels x 16 tokens, ldmatrix), B =
//                   P^T from the score accumulators through movmatrix
// P is scaled by 2^12 and split into fp16 high and low parts (two MMAs), so
// the probabilities keep ~22 bits; the scale cancels against the softmax
// denominator accumulated in fp32 from the same values.  The 4 warps' states
// are combined through shared memory; with several splits the partial
// (max, sum, unnormalised output) go to the caller's workspace and a second
// kernel combines them.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>

#include "kivi_device.cuh"
#include "kivi_expand.cuh"
#include "kivi_launch.h"

namespace kivi_impl {

namespace {

using namespace kivi_dev;

constexpr int kWarps = 4;
constexpr int kThreads = 32 * kWarps;
constexpr int kTile = 32;          // tokens per tile (one pipeline stage)
constexpr int kHalf = 16;          // tokens expanded and attended at a time
constexpr float kPScale = 4096.0f; // P * 2^12 stays a normal fp16 down to P = 2^-26
constexpr float kTau = 3.0f;       // a score at most 2^3 above the reference: P * 2^12 <= 2^15
constexpr uint64_t kWaitLimitNs = 200000000ull;  // 0.2 s per pipeline wait

// 2^x by the hardware's approximate base-2 exponential (results below the
// normal range flush to zero)
__device__ __forceinline__ float ex2_fast(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Shared-memory stage of one store tile (byte offsets).
template <int BITS, int G, int D>
struct StageFmt {
  static constexpr int KR = G < 32 ? kTile / G : 1; // key groups per tile
  static constexpr int kKc = BITS * D * 4;         // key codes: 32/W rows x D words
  static constexpr int kKs = KR * D * 4;           // key scale (or zero) rows of the groups
  static constexpr int kVc = BITS * D * 4;         // value codes: 32 rows x D/W words
  static constexpr int kVs = kTile * (D / G) * 4;  // value scales (or zeros) of 32 tokens
  static constexpr int oKs = kKc, oKz = oKs + kKs, oVc = oKz + kKs, oVs = oVc + kVc,
                       oVz = oVs + kVs;
  static constexpr int kBytes = oVz + kVs;
  static constexpr int kBuf = kHalf * D * 2;       // fp16 half tile per warp
  static constexpr int kQ = (D / 16) * 32 * 8;     // [D/16][32] query fragments
  // stages per warp: two, or one where two do not fit (D = 256, 8 bits, G = 16)
  static constexpr int NS =
      kWarps * 2 * kBytes + kWarps * kBuf + kWarps * 2 * 8 + kQ <= 227 * 1024 ? 2 : 1;
  static constexpr int kRing = kWarps * NS * kBytes;
  static constexpr int kBufs = kRing;              // [warp] fp16 half tiles
  static constexpr int kBars = kBufs + kWarps * kBuf;
  static constexpr int kQsm = kBars + kWarps * NS * 8;
  static constexpr int kSmem = kQsm + kQ;
  // the closing combine's exchange (maxima, sums, outputs in rows padded to
  // D + 4 floats so that the four lanes of a channel row hit four banks)
  // reuses the ring and tile buffers, below the mbarriers
  static constexpr int kRowO = D + 4;
  static constexpr int kRed = (2 * kWarps * 8 + kWarps * 8 * kRowO) * 4;
  static_assert(kRed <= kBars && kSmem <= 227 * 1024, "shared-memory plan");
};

// ---------------------------------------------------------------------------
// fp16 half-tile layouts in a warp's buffer (4 KB = 16 tokens x 128 channels)
//   row-major [token][channel]  (values; residual keys): row 256 B, its
//     16-byte chunk j stored at chunk (j ^ (j >> 3)) ^ (token & 7)
//   transposed [channel][token] (store keys): row 32 B, chunk j stored at
//     chunk j ^ ((channel >> 2) & 1)
// so that every 8-lane phase of the 16-byte stores (the value expansion's 8
// lanes write the even, then the odd chunks of one token; the others one
// chunk of 8 rows) and of ldmatrix (8 rows, one chunk column) touches 8
// distinct bank groups.
// ---------------------------------------------------------------------------
template <int D>
__device__ __forceinline__ uint32_t tok_major(int tok, int chunk) {
  return static_cast<uint32_t>(tok * (2 * D) + (((chunk ^ (chunk >> 3)) ^ (tok & 7)) << 4));
}
__device__ __forceinline__ uint32_t ch_major(int ch, int chunk) {
  return static_cast<uint32_t>(ch * 32 + ((chunk ^ ((ch >> 2) & 1)) << 4));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&a)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&a)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3])
               : "r"(addr));
}
__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

// Keys of tokens 16 hb .. 16 hb + 15 of a store tile -> transposed fp16 half
// tile.  Unit = those 16 tokens of one channel; lane takes channels
// lane + 32 i.
template <int BITS, int D>
__device__ __forceinline__ void expand_keys(const uint32_t *kc, const float *ks, const float *kz,
                                            int hb, uint32_t buf, int lane) {
  constexpr int W = 32 / BITS;
#pragma unroll
  for (int i = 0; i < D / 32; ++i) {
    const int c = lane + 32 * i;
    if constexpr (BITS == 2) {   // tokens of each chunk in perm8 order
      uint32_t lo, hi;
      lut2(ks[c], kz[c], lo, hi);
      uint4 c0, c1;
      lookup16(kc[hb * D + c], lo, hi, c0, c1);
      sts128(buf + ch_major(c, 0), c0);
      sts128(buf + ch_major(c, 1), c1);
    } else {
      uint64_t s2, ns2, z2;
      scale_consts(ks[c], kz[c], s2, ns2, z2);
      uint32_t w[16 / W];
#pragma unroll
      for (int k = 0; k < 16 / W; ++k) w[k] = kc[(hb * (16 / W) + k) * D + c];
      float m[16];
      magics16<BITS>(w, m);
      sts128(buf + ch_major(c, 0), deq8(m, s2, ns2, z2));
      sts128(buf + ch_major(c, 1), deq8(m + 8, s2, ns2, z2));
    }
  }
}

// 2-bit keys with tables built once per tile (G >= 32: one scale and zero per
// channel for the whole tile): lo/hi of channels lane + 32 i.
template <int D>
__device__ __forceinline__ void expand_keys2_lut(const uint32_t *kc, const uint32_t (&lo)[D / 32],
                                                 const uint32_t (&hi)[D / 32], int hb,
                                                 uint32_t buf, int lane) {
#pragma unroll
  for (int i = 0; i < D / 32; ++i) {
    const int c = lane + 32 * i;
    uint4 c0, c1;
    lookup16(kc[hb * D + c], lo[i], hi[i], c0, c1);
    sts128(buf + ch_major(c, 0), c0);
    sts128(buf + ch_major(c, 1), c1);
  }
}

// Values of tokens 16 hb .. of a store tile -> row-major fp16 half tile.
// Unit = 16 channels of one token (the 16/W consecutive words of channels
// 16 cu ..); consecutive lanes take consecutive units, so their word loads
// are consecutive too.
template <int BITS, int G, int D>
__device__ __forceinline__ void expand_values(const uint32_t *vc, const float *vs, const float *vz,
                                              int hb, uint32_t buf, int lane) {
  constexpr int W = 32 / BITS;
  constexpr int RW = D / W;           // words per token
  constexpr int NG = D / G;
  constexpr int WU = 16 / W;          // words per unit
#pragma unroll
  for (int k = 0; k < D / 32; ++k) {
    const int u = lane + 32 * k;
    const int tok = u / (D / 16), cu = u % (D / 16);   // token of the half, 16-channel unit
    const int trow = 16 * hb + tok;               // token of the tile
    const int grp = (16 * cu) / G;
    if constexpr (BITS == 2) {
      // the key half tile holds this half's tokens in perm8 order: so do the
      // value rows; the channels of each chunk come out in perm8 order too
      uint32_t lo, hi;
      lut2(vs[trow * NG + grp], vz[trow * NG + grp], lo, hi);
      uint4 c0, c1;
      lookup16(vc[trow * RW + cu], lo, hi, c0, c1);
      const int row = (tok & 8) | perm8_inv(tok & 7);
      sts128(buf + tok_major<D>(row, 2 * cu), c0);
      sts128(buf + tok_major<D>(row, 2 * cu + 1), c1);
      continue;
    }
    uint64_t s2, ns2, z2;
    scale_consts(vs[trow * NG + grp], vz[trow * NG + grp], s2, ns2, z2);
    const uint32_t *src = vc + trow * RW + cu * WU;
    uint32_t w[WU];
    if constexpr (WU == 4) {
      const uint4 v = *reinterpret_cast<const uint4 *>(src);
      w[0] = v.x; w[1 % WU] = v.y; w[2 % WU] = v.z; w[3 % WU] = v.w;
    } else if constexpr (WU == 2) {
      const uint2 v = *reinterpret_cast<const uint2 *>(src);
      w[0] = v.x; w[1 % WU] = v.y;
    } else {
      w[0] = src[0];
    }
    float m[16];
    magics16<BITS>(w, m);
    sts128(buf + tok_major<D>(tok, 2 * cu), deq8(m, s2, ns2, z2));
    sts128(buf + tok_major<D>(tok, 2 * cu + 1), deq8(m + 8, s2, ns2, z2));
  }
}

// KIVI-Sink: the store slots of sink tokens hold code 0; their exact fp16
// rows, kept in the sink store, replace them in the expanded half tiles
// before the tensor cores read the tiles.  Token tt (0..15) of a half is, in
// the transposed key tile, element perm(tt & 7) of chunk tt >> 3 of every
// channel row, and in the value tile row (tt & 8) | perm(tt & 7) with the
// channels of each chunk in perm8 order (2 bits: the order the table lookups
// produce; other widths: natural order).
__device__ __forceinline__ void sts16(uint32_t addr, unsigned short v) {
  asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}
template <int BITS, int D>
__device__ __forceinline__ void sink_key_column(uint32_t buf, const __half *row, int tt, int lane) {
  const int chunk = tt >> 3;
  const int pos = BITS == 2 ? perm8_inv(tt & 7) : (tt & 7);
#pragma unroll
  for (int i = 0; i < D / 32; ++i) {
    const int c = lane + 32 * i;
    sts16(buf + ch_major(c, chunk) + 2 * pos, __half_as_ushort(row[c]));
  }
}
template <int BITS, int D>
__device__ __forceinline__ void sink_value_row(uint32_t buf, const __half *row, int tt, int lane) {
  if (lane < D / 8) {
    uint4 v = *reinterpret_cast<const uint4 *>(row + 8 * lane);
    int r = tt;
    if (BITS == 2) {   // rows and chunk channels in perm8 order: (0,4) (1,5) (2,6) (3,7)
      r = (tt & 8) | perm8_inv(tt & 7);
      v = make_uint4(__byte_perm(v.x, v.z, 0x5410u), __byte_perm(v.x, v.z, 0x7632u),
                     __byte_perm(v.y, v.w, 0x5410u), __byte_perm(v.y, v.w, 0x7632u));
    }
    sts128(buf + tok_major<D>(r, lane), v);
  }
}

// 2-bit values with G >= 32: unit = 32 channels of one token (one group, so
// one table, and two code words); lane takes units lane and lane + 32 (token
// u / 4, channels 32 (u % 4) ..).  Rows and channel chunks in perm8 order as
// in expand_values; each 8-lane phase of a 16-byte store covers two token
// rows whose permuted indices differ by 2, whose chunk sets are
// complementary under the swizzle, so the stores are conflict-free.
template <int G, int D>
__device__ __forceinline__ void expand_values2_32(const uint32_t *vc, const float *vs,
                                                  const float *vz, int hb, uint32_t buf, int lane) {
  constexpr int RW = D / 16;          // words per token
  constexpr int NG = D / G;
#pragma unroll
  for (int k = 0; k < D / 64; ++k) {
    const int u = lane + 32 * k;
    const int tok = u / (D / 32), cq = u % (D / 32);
    const int trow = 16 * hb + tok;
    const int grp = (32 * cq) / G;
    uint32_t lo, hi;
    lut2(vs[trow * NG + grp], vz[trow * NG + grp], lo, hi);
    const uint2 w = *reinterpret_cast<const uint2 *>(vc + trow * RW + 2 * cq);
    const int row = (tok & 8) | perm8_inv(tok & 7);
    uint4 c0, c1;
    lookup16(w.x, lo, hi, c0, c1);
    sts128(buf + tok_major<D>(row, 4 * cq), c0);
    sts128(buf + tok_major<D>(row, 4 * cq + 1), c1);
    lookup16(w.y, lo, hi, c0, c1);
    sts128(buf + tok_major<D>(row, 4 * cq + 2), c0);
    sts128(buf + tok_major<D>(row, 4 * cq + 3), c1);
  }
}

// Residual half tile (fp16 ring rows tok0 .. tok0 + 15) -> row-major fp16
// half tile; rows past `valid` (counted from tok0) are zero.  Two lanes per
// token (lanes l and l + 16), eight chunks each.
template <bool PERM, int D>
__device__ __forceinline__ void load_residual(const __half *base, int64_t r_cap, int64_t head,
                                              int tok0, int valid, uint32_t buf, int lane) {
  const int tok = lane & 15, c0 = (lane >> 4) * (D / 16);
  const bool ok = tok < valid;
  const uint4 *src = nullptr;
  if (ok) {
    const int64_t rr = (head + tok0 + tok) % r_cap;
    src = reinterpret_cast<const uint4 *>(base + rr * D);
  }
#pragma unroll
  for (int ch = 0; ch < D / 16; ++ch) {
    uint4 v = ok ? src[c0 + ch] : make_uint4(0u, 0u, 0u, 0u);
    if (PERM) {   // channels of the chunk in perm8 order: (0,4) (1,5) (2,6) (3,7)
      v = make_uint4(__byte_perm(v.x, v.z, 0x5410u), __byte_perm(v.x, v.z, 0x7632u),
                     __byte_perm(v.y, v.w, 0x5410u), __byte_perm(v.y, v.w, 0x7632u));
    }
    sts128(buf + tok_major<D>(tok, c0 + ch), v);
  }
}

// Per-thread online-softmax state for heads 2t, 2t+1 (t = lane % 4).
template <int D>
struct SoftState {
  float m[2];
  float l[2];
  float o[D / 16][4];  // O^T accumulators: channel block mc, (ch g, h 2t), (g, 2t+1), (g+8, 2t), (g+8, 2t+1)
};

// Scores of 16 tokens x 8 heads from the key half tile in `buf` (transposed
// layout for store tiles, row-major for residual tiles); the 8 channel steps
// accumulate in four independent chains.
template <bool KEYS_T, int D>
__device__ __forceinline__ void half_scores(uint32_t buf, const uint2 *qsm, int lane,
                                            float (&s)[4]) {
  float acc[4][4];
#pragma unroll
  for (int j = 0; j < 4; ++j)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[j][i] = 0.0f;
  const int mat = lane >> 3, row = lane & 7;
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint2 qb = qsm[kk * 32 + lane];
    // matrices (tokens tb.., channels cb..) in A order: (0,0) (8,0) (0,8) (8,8)
    const int tb = (mat & 1) * 8, cb = 16 * kk + (mat >> 1) * 8;
    uint32_t a[4];
    if (KEYS_T)
      ldsm_x4_trans(buf + ch_major(cb + row, tb >> 3), a);
    else
      ldsm_x4(buf + tok_major<D>(tb + row, cb >> 3), a);
    mma_16816(acc[kk & 3], a, qb.x, qb.y);
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) s[i] = (acc[0][i] + acc[1][i]) + (acc[2][i] + acc[3][i]);
}

// Online softmax update with 16 tokens' scores (the first `valid` real);
// returns the P^T fragments (x 2^12, fp16 high and low parts).
template <int D>
__device__ __forceinline__ void half_softmax(SoftState<D> &st, float (&s)[4], float scale_log2,
                                             int valid, int g, uint32_t (&phi)[2],
                                             uint32_t (&plo)[2]) {
  // The reference m of a head column moves only when a score of the half
  // exceeds it by more than kTau (one warp vote; always at the first half):
  // then it becomes the running maximum and the output and sum are
  // rescaled.  P = 2^(s - m) * 2^12 <= 2^15 stays a finite fp16, and o and l
  // are relative to the same m, so the result is that of any reference.
  bool over = false;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int tok = g + (i >= 2 ? 8 : 0);
    const float v = tok < valid ? s[i] * scale_log2 : -INFINITY;
    s[i] = v;
    over |= v > st.m[i & 1] + kTau;
  }
  if (__any_sync(0xffffffffu, over)) {
    float mt[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int i = 0; i < 4; ++i) mt[i & 1] = fmaxf(mt[i & 1], s[i]);
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      mt[0] = fmaxf(mt[0], __shfl_xor_sync(0xffffffffu, mt[0], off));
      mt[1] = fmaxf(mt[1], __shfl_xor_sync(0xffffffffu, mt[1], off));
    }
    float alpha[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const float mn = fmaxf(st.m[j], mt[j]);
      alpha[j] = mn == -INFINITY ? 1.0f : exp2f(st.m[j] - mn);
      st.m[j] = mn;
      st.l[j] *= alpha[j];
    }
#pragma unroll
    for (int mc = 0; mc < D / 16; ++mc) {
      st.o[mc][0] *= alpha[0];
      st.o[mc][1] *= alpha[1];
      st.o[mc][2] *= alpha[0];
      st.o[mc][3] *= alpha[1];
    }
  }
  float p[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float m = st.m[i & 1];
    p[i] = m == -INFINITY ? 0.0f : ex2_fast(s[i] - m) * kPScale;
  }
  const __half2 h0 = __floats2half2_rn(p[0], p[1]);   // token g: heads 2t, 2t+1
  const __half2 h1 = __floats2half2_rn(p[2], p[3]);   // token g+8
  const __half2 l0 = __floats2half2_rn(p[0] - __low2float(h0), p[1] - __high2float(h0));
  const __half2 l1 = __floats2half2_rn(p[2] - __low2float(h1), p[3] - __high2float(h1));
  phi[0] = movmatrix_trans(h2_as_u32(h0));
  phi[1] = movmatrix_trans(h2_as_u32(h1));
  plo[0] = movmatrix_trans(h2_as_u32(l0));
  plo[1] = movmatrix_trans(h2_as_u32(l1));
  st.l[0] += p[0] + p[2];
  st.l[1] += p[1] + p[3];
}

// O^T += V^T P^T from the row-major value half tile in `buf`.
template <int D>
__device__ __forceinline__ void half_values(SoftState<D> &st, uint32_t buf, int lane,
                                            const uint32_t (&phi)[2], const uint32_t (&plo)[2]) {
  const int mat = lane >> 3, row = lane & 7;
  // matrices (channels cb.., tokens tb..) in A order: (0,0) (8,0) (0,8) (8,8);
  // chunk 2 mc + (mat & 1) of row tb + row, stored at chunk
  // (2 mc ^ (mc >> 2)) ^ ((mat & 1) ^ row)   (tok_major with tok & 7 = row)
  const int tok = (mat >> 1) * 8 + row;
  const uint32_t rbase = buf + tok * (2 * D);
  const int lb = (mat & 1) ^ row;
#pragma unroll
  for (int mc = 0; mc < D / 16; ++mc) {
    uint32_t a[4];
    ldsm_x4_trans(rbase + ((((2 * mc) ^ (mc >> 2)) ^ lb) << 4), a);
    mma_16816(st.o[mc], a, phi[0], phi[1]);
    mma_16816(st.o[mc], a, plo[0], plo[1]);
  }
}

template <int BITS, int G, bool SINKS, int D>
__global__ void __launch_bounds__(kThreads, D == 256 ? 2 : 4)
    decode_attention_kernel(const __grid_constant__ AttnParams p) {
  using F = StageFmt<BITS, G, D>;
  constexpr int W = 32 / BITS;
  extern __shared__ __align__(128) unsigned char smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;

  const int64_t item = blockIdx.x;
  const int split = static_cast<int>(item % p.n_split);
  const int64_t pair = item / p.n_split;
  const int job = static_cast<int>(pair / p.bh);
  const int64_t bhi = pair - static_cast<int64_t>(job) * p.bh;
  const AttnJob &J = p.jobs[job];
  const int64_t b = bhi / p.h_kv, kvh = bhi - b * p.h_kv;
  const int64_t h_q = static_cast<int64_t>(p.h_kv) * p.r;

  SoftState<D> st;
  st.m[0] = st.m[1] = -INFINITY;
  st.l[0] = st.l[1] = 0.0f;
#pragma unroll
  for (int mc = 0; mc < D / 16; ++mc)
#pragma unroll
    for (int i = 0; i < 4; ++i) st.o[mc][i] = 0.0f;

  // ---- the block's tiles: its store range, then (last split) the residual
  // tiles; warp w takes list positions w, w + 4, ... (store tiles first)
  const int st0 = split * p.tiles_per_split;
  const int n_store = max(0, min(st0 + p.tiles_per_split, p.tiles_store) - st0);
  const int n_my = n_store > warp ? (n_store - warp + kWarps - 1) / kWarps : 0;
  unsigned char *ring = smem + warp * F::NS * F::kBytes;
  const uint32_t buf = smem_addr(smem + F::kBufs + warp * F::kBuf);
  const uint32_t bar0 = smem_addr(smem + F::kBars) + warp * F::NS * 8;
  if (lane == 0) {
#pragma unroll
    for (int sidx = 0; sidx < F::NS; ++sidx) mbar_init(bar0 + 8 * sidx, 1);
    fence_mbar_init();
  }
  __syncwarp();

  const uint64_t pol = policy_evict_first();
  const uint32_t *kc_bh = J.k_codes + bhi * (p.cap / W) * D;
  const float *ks_bh = J.k_scale + bhi * (p.cap / G) * D;
  const float *kz_bh = J.k_zero + bhi * (p.cap / G) * D;
  const uint32_t *vc_bh = J.v_codes + bhi * p.cap * (D / W);
  const float *vs_bh = J.v_scale + bhi * p.cap * (D / G);
  const float *vz_bh = J.v_zero + bhi * p.cap * (D / G);
  auto issue = [&](int i) {
    const int64_t tile = st0 + warp + static_cast<int64_t>(kWarps) * i;
    const int sidx = i % F::NS;
    const uint32_t dst = smem_addr(ring + sidx * F::kBytes);
    const uint32_t bar = bar0 + 8 * sidx;
    const int64_t tok = tile * kTile;
    // a store that ends half way through its last tile (G = 16): that tile's
    // first 16 tokens only, the first half of each piece
    const int sh = G < 32 && p.tail_half && tile == p.tiles_store - 1 ? 1 : 0;
    fence_proxy_async_smem();
    mbar_arrive_expect_tx(bar, F::kBytes >> sh);
    bulk_load(dst, kc_bh + (tok / W) * D, F::kKc >> sh, bar, pol);
    bulk_load(dst + F::oKs, ks_bh + (tok / G) * D, F::kKs >> sh, bar, pol);
    bulk_load(dst + F::oKz, kz_bh + (tok / G) * D, F::kKs >> sh, bar, pol);
    bulk_load(dst + F::oVc, vc_bh + tok * (D / W), F::kVc >> sh, bar, pol);
    bulk_load(dst + F::oVs, vs_bh + tok * (D / G), F::kVs >> sh, bar, pol);
    bulk_load(dst + F::oVz, vz_bh + tok * (D / G), F::kVs >> sh, bar, pol);
  };
  int issued = 0;
  if (lane == 0)
    for (; issued < min(F::NS, n_my); ++issued) issue(issued);
  issued = __shfl_sync(0xffffffffu, issued, 0);

  // query heads kvh*r .. kvh*r + r-1 as B fragments (k = channels, n = heads)
  // in shared memory, one copy per block (loaded while the first copies fly)
  uint2 *qsm = reinterpret_cast<uint2 *>(smem + F::kQsm);
  for (int idx = threadIdx.x; idx < (D / 16) * 32; idx += kThreads) {
    const int kk = idx >> 5, ql = idx & 31, qg = ql >> 2, qt = ql & 3;
    const __half *q = static_cast<const __half *>(J.q) + (b * h_q + kvh * p.r + qg) * D;
    const int c0 = 16 * kk + 2 * qt;
    qsm[idx] = qg < p.r ? make_uint2(*reinterpret_cast<const uint32_t *>(q + c0),
                                     *reinterpret_cast<const uint32_t *>(q + c0 + 8))
                        : make_uint2(0u, 0u);
  }
  __syncthreads();

  // KIVI-Sink: this sequence's sink positions (ascending) and this bh's rows;
  // `sc` is the warp's cursor into the list (its tiles come in order)
  const int64_t *spos = nullptr;
  const __half *srow_k = nullptr, *srow_v = nullptr;
  int scnt = 0, sc = 0;
  if (SINKS) {
    spos = J.sink_pos + b * p.sink_cap;
    scnt = min(J.sink_count[b], p.sink_cap);
    srow_k = static_cast<const __half *>(J.sink_k) + bhi * p.sink_cap * D;
    srow_v = static_cast<const __half *>(J.sink_v) + bhi * p.sink_cap * D;
  }

  int done = 0;
  bool failed = false;
#pragma unroll 1
  for (; done < n_my; ++done) {
    const int sidx = done % F::NS;
    // warp-uniform decision: a lane whose wait timed out fails the whole warp
    if (!__all_sync(0xffffffffu, mbar_wait_bounded(bar0 + 8 * sidx, (done / F::NS) & 1,
                                                   kWaitLimitNs))) {
      failed = true;
      break;
    }
    const unsigned char *stg = ring + sidx * F::kBytes;
    const int n_hb = G < 32 && p.tail_half && st0 + warp + kWarps * done == p.tiles_store - 1
                         ? 1 : 2;                  // halves of this tile
    constexpr bool KLUT = BITS == 2 && G >= 32;    // key tables shared by both halves
    uint32_t klo[D / 32], khi[D / 32];
    if (KLUT) {
      const float *ks = reinterpret_cast<const float *>(stg + F::oKs);
      const float *kz = reinterpret_cast<const float *>(stg + F::oKz);
#pragma unroll
      for (int i = 0; i < D / 32; ++i) lut2(ks[lane + 32 * i], kz[lane + 32 * i], klo[i], khi[i]);
    }
#pragma unroll 1
    for (int hb = 0; hb < n_hb; ++hb) {
      float s[4];
      uint32_t phi[2], plo[2];
      // key scale / zero row of the half's group
      const int krow = G < 32 ? hb * D : 0;
      // sinks of this half: list entries [sc, se)
      const int64_t tok0 = static_cast<int64_t>(st0 + warp + kWarps * done) * kTile + kHalf * hb;
      int se = sc;
      if (SINKS) {
        while (sc < scnt && spos[sc] < tok0) ++sc;   // other warps' tiles
        se = sc;
        while (se < scnt && spos[se] < tok0 + kHalf) ++se;
      }
      if (KLUT)
        expand_keys2_lut<D>(reinterpret_cast<const uint32_t *>(stg), klo, khi, hb, buf, lane);
      else
        expand_keys<BITS, D>(reinterpret_cast<const uint32_t *>(stg),
                          reinterpret_cast<const float *>(stg + F::oKs) + krow,
                          reinterpret_cast<const float *>(stg + F::oKz) + krow, hb, buf, lane);
      __syncwarp();
      if (SINKS && se > sc) {                      // the sinks' exact key columns
        for (int j = sc; j < se; ++j)
          sink_key_column<BITS, D>(buf, srow_k + static_cast<int64_t>(j) * D,
                                static_cast<int>(spos[j] - tok0), lane);
        __syncwarp();
      }
      half_scores<true, D>(buf, qsm, lane, s);
      half_softmax(st, s, p.scale_log2, kHalf, g, phi, plo);
      __syncwarp();                                // key half tile read by every lane
      if constexpr (BITS == 2 && G >= 32)
        expand_values2_32<G, D>(reinterpret_cast<const uint32_t *>(stg + F::oVc),
                             reinterpret_cast<const float *>(stg + F::oVs),
                             reinterpret_cast<const float *>(stg + F::oVz), hb, buf, lane);
      else
        expand_values<BITS, G, D>(reinterpret_cast<const uint32_t *>(stg + F::oVc),
                               reinterpret_cast<const float *>(stg + F::oVs),
                               reinterpret_cast<const float *>(stg + F::oVz), hb, buf, lane);
      __syncwarp();                                // value half tile written
      if (SINKS && se > sc) {                      // the sinks' exact value rows
        for (int j = sc; j < se; ++j)
          sink_value_row<BITS, D>(buf, srow_v + static_cast<int64_t>(j) * D,
                               static_cast<int>(spos[j] - tok0), lane);
        __syncwarp();
      }
      sc = se;
      if (hb == n_hb - 1 && issued < n_my) {       // stage consumed: refill it
        if (lane == 0) issue(issued);
        ++issued;
      }
      half_values(st, buf, lane, phi, plo);
      __syncwarp();                                // value half tile read by every lane
    }
  }
  if (failed) {
    // record the timeout and wait (bounded) for this warp's copies still in flight
    if (lane == 0) atomicOr(p.fault, 1u);
#pragma unroll 1
    for (int i = done; i < issued; ++i)
      mbar_wait_bounded(bar0 + 8 * (i % F::NS), (i / F::NS) & 1, kWaitLimitNs);
  }

  // ---- residual tiles (last split): fp16 rows read directly, 16 tokens at a time
  if (split == p.n_split - 1 && !failed) {
    const __half *kr = static_cast<const __half *>(J.k_res) + bhi * p.r_cap * D;
    const __half *vr = static_cast<const __half *>(J.v_res) + bhi * p.r_cap * D;
    // first list position >= n_store that belongs to this warp
    const int first = n_store + ((warp - n_store) % kWarps + kWarps) % kWarps;
#pragma unroll 1
    for (int j = first - n_store; j < p.tiles_res; j += kWarps) {
#pragma unroll 1
      for (int hb = 0; hb < 2; ++hb) {
        const int tok0 = j * kTile + hb * kHalf;
        const int64_t left = p.n_res - tok0;
        if (left <= 0) break;
        const int valid = left < kHalf ? static_cast<int>(left) : kHalf;
        float s[4];
        uint32_t phi[2], plo[2];
        load_residual<false, D>(kr, p.r_cap, p.res_head, tok0, valid, buf, lane);
        __syncwarp();
        half_scores<false, D>(buf, qsm, lane, s);
        half_softmax(st, s, p.scale_log2, valid, g, phi, plo);
        __syncwarp();
        load_residual<BITS == 2, D>(vr, p.r_cap, p.res_head, tok0, valid, buf, lane);
        __syncwarp();
        half_values(st, buf, lane, phi, plo);
        __syncwarp();
      }
    }
  }

  // ---- combine the 4 warps (the stage area is free once every warp is here)
#pragma unroll
  for (int j = 0; j < 2; ++j)
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) st.l[j] += __shfl_xor_sync(0xffffffffu, st.l[j], off);
  __syncthreads();
  float *red_m = reinterpret_cast<float *>(smem);            // [warp][8]
  float *red_l = red_m + kWarps * 8;                         // [warp][8]
  float *red_o = red_l + kWarps * 8;                         // [warp][8][D + 4]
  if (g == 0) {
    red_m[warp * 8 + 2 * t] = st.m[0];
    red_m[warp * 8 + 2 * t + 1] = st.m[1];
    red_l[warp * 8 + 2 * t] = st.l[0];
    red_l[warp * 8 + 2 * t + 1] = st.l[1];
  }
  // accumulator row g of channel block mc is channel 16 mc + g, or with the
  // 2-bit path's chunk order 16 mc + perm8(g) (rows g + 8: + 8)
  const int cg = BITS == 2 ? perm8(g) : g;
#pragma unroll
  for (int mc = 0; mc < D / 16; ++mc) {
    float *o0 = red_o + (warp * 8 + 2 * t) * F::kRowO + 16 * mc + cg;
    float *o1 = o0 + F::kRowO;
    o0[0] = st.o[mc][0];
    o1[0] = st.o[mc][1];
    o0[8] = st.o[mc][2];
    o1[8] = st.o[mc][3];
  }
  __syncthreads();
  const int nr = p.r * D;
#pragma unroll 1
  for (int idx = threadIdx.x; idx < nr; idx += kThreads) {
    const int h = idx / D, c = idx - h * D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, red_m[w * 8 + h]);
    float L = 0.0f, O = 0.0f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float mw = red_m[w * 8 + h];
      if (mw == -INFINITY) continue;
      const float f = exp2f(mw - M);
      L += red_l[w * 8 + h] * f;
      O += red_o[(w * 8 + h) * F::kRowO + c] * f;
    }
    if (p.n_split == 1) {
      J.out[(b * h_q + kvh * p.r + h) * D + c] = O / L;
    } else {
      const int64_t base = item * p.r + h;   // partial (item, head)
      p.ws[base * D + c] = O;
      if (c == 0) {
        float *ml = p.ws + static_cast<int64_t>(gridDim.x) * p.r * D;
        ml[2 * base] = M;
        ml[2 * base + 1] = L;
      }
    }
  }
}

template <int BITS, int G, bool SINKS, int D>
cudaError_t attention_launch_k(const AttnParams &p, cudaStream_t stream) {
  using F = StageFmt<BITS, G, D>;
  auto kern = decode_attention_kernel<BITS, G, SINKS, D>;
  // the shared-memory opt-in is a per-device function attribute: set once per device
  constexpr int kMaxDevices = 64;
  static std::atomic<bool> configured[kMaxDevices];
  int dev = 0;
  cudaError_t e0 = cudaGetDevice(&dev);
  if (e0 != cudaSuccess) return e0;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (!configured[dev].load(std::memory_order_acquire)) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, F::kSmem);
    if (e != cudaSuccess) return e;
    configured[dev].store(true, std::memory_order_release);
  }
  AttnParams q = p;
  cudaError_t e = fault_word_address(&q.fault);
  if (e != cudaSuccess) return e;
  const int64_t items = static_cast<int64_t>(p.n_jobs) * p.bh * p.n_split;
  kern<<<static_cast<unsigned>(items), kThreads, F::kSmem, stream>>>(q);
  e = cudaGetLastError();
  if (e != cudaSuccess || p.n_split == 1) return e;
  return launch_attention_combine(q, stream);
}

template <int BITS, int G, int D>
cudaError_t attention_launch(const AttnParams &p, cudaStream_t stream) {
  if constexpr (D % G != 0) {   // value groups must tile the head
    return cudaErrorInvalidValue;
  } else {
    return p.sink_cap > 0 ? attention_launch_k<BITS, G, true, D>(p, stream)
                          : attention_launch_k<BITS, G, false, D>(p, stream);
  }
}

// The kernels of head_dim D for the call's (bits, G).
template <int D>
cudaError_t attention_dispatch(const AttnParams &p, int group, int bits, cudaStream_t stream) {
  switch (bits * 1000 + group) {
    case 2016: return attention_launch<2, 16, D>(p, stream);
    case 4016: return attention_launch<4, 16, D>(p, stream);
    case 8016: return attention_launch<8, 16, D>(p, stream);
    case 2032: return attention_launch<2, 32, D>(p, stream);
    case 2064: return attention_launch<2, 64, D>(p, stream);
    case 2128: return attention_launch<2, 128, D>(p, stream);
    case 4032: return attention_launch<4, 32, D>(p, stream);
    case 4064: return attention_launch<4, 64, D>(p, stream);
    case 4128: return attention_launch<4, 128, D>(p, stream);
    case 8032: return attention_launch<8, 32, D>(p, stream);
    case 8064: return attention_launch<8, 64, D>(p, stream);
    case 8128: return attention_launch<8, 128, D>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}
}  // namespace

}  // namespace kivi_impl
