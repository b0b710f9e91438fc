// kivi_attention.cu -- decode attention that reads the packed KIVI store.
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
//   O^T += V^T P^T  A = value tile (16 channels x 16 tokens, ldmatrix), B =
//                   P^T from the score accumulators through movmatrix
// P is scaled by 2^12 and split into fp16 high and low parts (two MMAs), so
// the probabilities keep ~22 bits; the scale cancels against the softmax
// denominator accumulated in fp32 from the same values.  The 4 warps' states
// are combined through shared memory; with several splits the partial
// (max, sum, unnormalised output) go to the caller's workspace and a second
// kernel combines them.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "kivi_device.cuh"
#include "kivi_expand.cuh"
#include "kivi_launch.h"

namespace kivi_impl {

// bit 0: a pipeline wait of the decode-attention kernel timed out; bit 1: a
// sink store overflowed (kivi_sink.cu, through fault_word_address)
__device__ unsigned int g_fault_word;

// Split-K workspace of the allocation-free decode-attention entry point: a
// fixed file-scope device array (kAttnScratchFloats floats), so that call
// needs no caller workspace and allocates nothing.  Every partial a call
// reads was written earlier in the same call, so nothing in it needs
// clearing; two calls that overlap on the device share it and race.
constexpr int64_t kAttnScratchFloats = int64_t{1} << 24;   // 64 MiB
static __device__ __align__(256) float g_attn_scratch[kAttnScratchFloats];

namespace {

using namespace kivi_dev;

constexpr int kD = 128;            // head_dim
constexpr int kWarps = 4;
constexpr int kThreads = 32 * kWarps;
constexpr int kTile = 32;          // tokens per tile (one pipeline stage)
constexpr int kHalf = 16;          // tokens expanded and attended at a time
constexpr float kPScale = 4096.0f; // P * 2^12 stays a normal fp16 down to P = 2^-26
constexpr uint64_t kWaitLimitNs = 200000000ull;  // 0.2 s per pipeline wait

// Shared-memory stage of one store tile (byte offsets).
template <int BITS, int G>
struct StageFmt {
  static constexpr int KR = G < 32 ? kTile / G : 1; // key groups per tile
  static constexpr int kKc = BITS * kD * 4;        // key codes: 32/W rows x D words
  static constexpr int kKs = KR * kD * 4;          // key scale (or zero) rows of the groups
  static constexpr int kVc = BITS * kD * 4;        // value codes: 32 rows x D/W words
  static constexpr int kVs = kTile * (kD / G) * 4; // value scales (or zeros) of 32 tokens
  static constexpr int oKs = kKc, oKz = oKs + kKs, oVc = oKz + kKs, oVs = oVc + kVc,
                       oVz = oVs + kVs;
  static constexpr int kBytes = oVz + kVs;
  static constexpr int NS = 2;                     // stages per warp
  static constexpr int kBuf = kHalf * kD * 2;      // fp16 half tile per warp (4 KB)
  static constexpr int kRing = kWarps * NS * kBytes;
  static constexpr int kBufs = kRing;              // [warp] fp16 half tiles
  static constexpr int kBars = kBufs + kWarps * kBuf;
  static constexpr int kQsm = kBars + kWarps * NS * 8;   // [8][32] query fragments
  static constexpr int kSmem = kQsm + 8 * 32 * 8;
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
__device__ __forceinline__ uint32_t tok_major(int tok, int chunk) {
  return static_cast<uint32_t>(tok * 256 + (((chunk ^ (chunk >> 3)) ^ (tok & 7)) << 4));
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
template <int BITS>
__device__ __forceinline__ void expand_keys(const uint32_t *kc, const float *ks, const float *kz,
                                            int hb, uint32_t buf, int lane) {
  constexpr int W = 32 / BITS;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int c = lane + 32 * i;
    if constexpr (BITS == 2) {   // tokens of each chunk in perm8 order
      uint32_t lo, hi;
      lut2(ks[c], kz[c], lo, hi);
      uint4 c0, c1;
      lookup16(kc[hb * kD + c], lo, hi, c0, c1);
      sts128(buf + ch_major(c, 0), c0);
      sts128(buf + ch_major(c, 1), c1);
    } else {
      uint64_t s2, ns2, z2;
      scale_consts(ks[c], kz[c], s2, ns2, z2);
      uint32_t w[16 / W];
#pragma unroll
      for (int k = 0; k < 16 / W; ++k) w[k] = kc[(hb * (16 / W) + k) * kD + c];
      float m[16];
      magics16<BITS>(w, m);
      sts128(buf + ch_major(c, 0), deq8(m, s2, ns2, z2));
      sts128(buf + ch_major(c, 1), deq8(m + 8, s2, ns2, z2));
    }
  }
}

// 2-bit keys with tables built once per tile (G >= 32: one scale and zero per
// channel for the whole tile): lo/hi of channels lane + 32 i.
__device__ __forceinline__ void expand_keys2_lut(const uint32_t *kc, const uint32_t (&lo)[4],
                                                 const uint32_t (&hi)[4], int hb, uint32_t buf,
                                                 int lane) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int c = lane + 32 * i;
    uint4 c0, c1;
    lookup16(kc[hb * kD + c], lo[i], hi[i], c0, c1);
    sts128(buf + ch_major(c, 0), c0);
    sts128(buf + ch_major(c, 1), c1);
  }
}

// Values of tokens 16 hb .. of a store tile -> row-major fp16 half tile.
// Unit = 16 channels of one token (the 16/W consecutive words of channels
// 16 cu ..); consecutive lanes take consecutive units, so their word loads
// are consecutive too.
template <int BITS, int G>
__device__ __forceinline__ void expand_values(const uint32_t *vc, const float *vs, const float *vz,
                                              int hb, uint32_t buf, int lane) {
  constexpr int W = 32 / BITS;
  constexpr int RW = kD / W;          // words per token
  constexpr int NG = kD / G;
  constexpr int WU = 16 / W;          // words per unit
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int u = lane + 32 * k;
    const int tok = u >> 3, cu = u & 7;           // token of the half, 16-channel unit
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
      sts128(buf + tok_major(row, 2 * cu), c0);
      sts128(buf + tok_major(row, 2 * cu + 1), c1);
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
    sts128(buf + tok_major(tok, 2 * cu), deq8(m, s2, ns2, z2));
    sts128(buf + tok_major(tok, 2 * cu + 1), deq8(m + 8, s2, ns2, z2));
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
template <int BITS>
__device__ __forceinline__ void sink_key_column(uint32_t buf, const __half *row, int tt, int lane) {
  const int chunk = tt >> 3;
  const int pos = BITS == 2 ? perm8_inv(tt & 7) : (tt & 7);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int c = lane + 32 * i;
    sts16(buf + ch_major(c, chunk) + 2 * pos, __half_as_ushort(row[c]));
  }
}
template <int BITS>
__device__ __forceinline__ void sink_value_row(uint32_t buf, const __half *row, int tt, int lane) {
  if (lane < kD / 8) {
    uint4 v = *reinterpret_cast<const uint4 *>(row + 8 * lane);
    int r = tt;
    if (BITS == 2) {   // rows and chunk channels in perm8 order: (0,4) (1,5) (2,6) (3,7)
      r = (tt & 8) | perm8_inv(tt & 7);
      v = make_uint4(__byte_perm(v.x, v.z, 0x5410u), __byte_perm(v.x, v.z, 0x7632u),
                     __byte_perm(v.y, v.w, 0x5410u), __byte_perm(v.y, v.w, 0x7632u));
    }
    sts128(buf + tok_major(r, lane), v);
  }
}

// 2-bit values with G >= 32: unit = 32 channels of one token (one group, so
// one table, and two code words); lane takes units lane and lane + 32 (token
// u / 4, channels 32 (u % 4) ..).  Rows and channel chunks in perm8 order as
// in expand_values; each 8-lane phase of a 16-byte store covers two token
// rows whose permuted indices differ by 2, whose chunk sets are
// complementary under the swizzle, so the stores are conflict-free.
template <int G>
__device__ __forceinline__ void expand_values2_32(const uint32_t *vc, const float *vs,
                                                  const float *vz, int hb, uint32_t buf, int lane) {
  constexpr int RW = kD / 16;         // words per token
  constexpr int NG = kD / G;
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int u = lane + 32 * k;
    const int tok = u >> 2, cq = u & 3;
    const int trow = 16 * hb + tok;
    const int grp = (32 * cq) / G;
    uint32_t lo, hi;
    lut2(vs[trow * NG + grp], vz[trow * NG + grp], lo, hi);
    const uint2 w = *reinterpret_cast<const uint2 *>(vc + trow * RW + 2 * cq);
    const int row = (tok & 8) | perm8_inv(tok & 7);
    uint4 c0, c1;
    lookup16(w.x, lo, hi, c0, c1);
    sts128(buf + tok_major(row, 4 * cq), c0);
    sts128(buf + tok_major(row, 4 * cq + 1), c1);
    lookup16(w.y, lo, hi, c0, c1);
    sts128(buf + tok_major(row, 4 * cq + 2), c0);
    sts128(buf + tok_major(row, 4 * cq + 3), c1);
  }
}

// Residual half tile (fp16 ring rows tok0 .. tok0 + 15) -> row-major fp16
// half tile; rows past `valid` (counted from tok0) are zero.  Two lanes per
// token (lanes l and l + 16), eight chunks each.
template <bool PERM>
__device__ __forceinline__ void load_residual(const __half *base, int64_t r_cap, int64_t head,
                                              int tok0, int valid, uint32_t buf, int lane) {
  const int tok = lane & 15, c0 = (lane >> 4) * 8;
  const bool ok = tok < valid;
  const uint4 *src = nullptr;
  if (ok) {
    const int64_t rr = (head + tok0 + tok) % r_cap;
    src = reinterpret_cast<const uint4 *>(base + rr * kD);
  }
#pragma unroll
  for (int ch = 0; ch < 8; ++ch) {
    uint4 v = ok ? src[c0 + ch] : make_uint4(0u, 0u, 0u, 0u);
    if (PERM) {   // channels of the chunk in perm8 order: (0,4) (1,5) (2,6) (3,7)
      v = make_uint4(__byte_perm(v.x, v.z, 0x5410u), __byte_perm(v.x, v.z, 0x7632u),
                     __byte_perm(v.y, v.w, 0x5410u), __byte_perm(v.y, v.w, 0x7632u));
    }
    sts128(buf + tok_major(tok, c0 + ch), v);
  }
}

// Per-thread online-softmax state for heads 2t, 2t+1 (t = lane % 4).
struct SoftState {
  float m[2];
  float l[2];
  float o[8][4];  // O^T accumulators: channel block mc, (ch g, h 2t), (g, 2t+1), (g+8, 2t), (g+8, 2t+1)
};

// Scores of 16 tokens x 8 heads from the key half tile in `buf` (transposed
// layout for store tiles, row-major for residual tiles).
template <bool KEYS_T>
__device__ __forceinline__ void half_scores(uint32_t buf, const uint2 *qsm, int lane,
                                            float (&s)[4]) {
  float s2[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) s[i] = s2[i] = 0.0f;
  const int mat = lane >> 3, row = lane & 7;
#pragma unroll 4
  for (int kk = 0; kk < 8; ++kk) {
    const uint2 qb = qsm[kk * 32 + lane];
    // matrices (tokens tb.., channels cb..) in A order: (0,0) (8,0) (0,8) (8,8)
    const int tb = (mat & 1) * 8, cb = 16 * kk + (mat >> 1) * 8;
    uint32_t a[4];
    if (KEYS_T)
      ldsm_x4_trans(buf + ch_major(cb + row, tb >> 3), a);
    else
      ldsm_x4(buf + tok_major(tb + row, cb >> 3), a);
    mma_16816((kk & 1) ? s2 : s, a, qb.x, qb.y);
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) s[i] += s2[i];
}

// Online softmax update with 16 tokens' scores (the first `valid` real);
// returns the P^T fragments (x 2^12, fp16 high and low parts).
__device__ __forceinline__ void half_softmax(SoftState &st, float (&s)[4], float scale_log2,
                                             int valid, int g, uint32_t (&phi)[2],
                                             uint32_t (&plo)[2]) {
  float mt[2] = {-INFINITY, -INFINITY};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int tok = g + (i >= 2 ? 8 : 0);
    const float v = tok < valid ? s[i] * scale_log2 : -INFINITY;
    s[i] = v;
    mt[i & 1] = fmaxf(mt[i & 1], v);
  }
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    mt[0] = fmaxf(mt[0], __shfl_xor_sync(0xffffffffu, mt[0], off));
    mt[1] = fmaxf(mt[1], __shfl_xor_sync(0xffffffffu, mt[1], off));
  }
  float mn[2], alpha[2];
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    mn[j] = fmaxf(st.m[j], mt[j]);
    alpha[j] = mn[j] == -INFINITY ? 1.0f : exp2f(st.m[j] - mn[j]);
    st.m[j] = mn[j];
  }
  float p[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float m = mn[i & 1];
    p[i] = m == -INFINITY ? 0.0f : exp2f(s[i] - m) * kPScale;
  }
  const __half2 h0 = __floats2half2_rn(p[0], p[1]);   // token g: heads 2t, 2t+1
  const __half2 h1 = __floats2half2_rn(p[2], p[3]);   // token g+8
  const __half2 l0 = __floats2half2_rn(p[0] - __low2float(h0), p[1] - __high2float(h0));
  const __half2 l1 = __floats2half2_rn(p[2] - __low2float(h1), p[3] - __high2float(h1));
  phi[0] = movmatrix_trans(h2_as_u32(h0));
  phi[1] = movmatrix_trans(h2_as_u32(h1));
  plo[0] = movmatrix_trans(h2_as_u32(l0));
  plo[1] = movmatrix_trans(h2_as_u32(l1));
  st.l[0] = st.l[0] * alpha[0] + (p[0] + p[2]);
  st.l[1] = st.l[1] * alpha[1] + (p[1] + p[3]);
  // once the running maximum settles most steps leave it unchanged (alpha 1)
  if (__any_sync(0xffffffffu, alpha[0] != 1.0f || alpha[1] != 1.0f)) {
#pragma unroll
    for (int mc = 0; mc < 8; ++mc) {
      st.o[mc][0] *= alpha[0];
      st.o[mc][1] *= alpha[1];
      st.o[mc][2] *= alpha[0];
      st.o[mc][3] *= alpha[1];
    }
  }
}

// O^T += V^T P^T from the row-major value half tile in `buf`.
__device__ __forceinline__ void half_values(SoftState &st, uint32_t buf, int lane,
                                            const uint32_t (&phi)[2], const uint32_t (&plo)[2]) {
  const int mat = lane >> 3, row = lane & 7;
  // matrices (channels cb.., tokens tb..) in A order: (0,0) (8,0) (0,8) (8,8);
  // chunk 2 mc + (mat & 1) of row tb + row, stored at chunk
  // (2 mc ^ (mc >> 2)) ^ ((mat & 1) ^ row)   (tok_major with tok & 7 = row)
  const int tok = (mat >> 1) * 8 + row;
  const uint32_t rbase = buf + tok * 256;
  const int lb = (mat & 1) ^ row;
#pragma unroll
  for (int mc = 0; mc < 8; ++mc) {
    uint32_t a[4];
    ldsm_x4_trans(rbase + ((((2 * mc) ^ (mc >> 2)) ^ lb) << 4), a);
    mma_16816(st.o[mc], a, phi[0], phi[1]);
    mma_16816(st.o[mc], a, plo[0], plo[1]);
  }
}

template <int BITS, int G, bool SINKS>
__global__ void __launch_bounds__(kThreads, 4) decode_attention_kernel(const __grid_constant__ AttnParams p) {
  using F = StageFmt<BITS, G>;
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

  SoftState st;
  st.m[0] = st.m[1] = -INFINITY;
  st.l[0] = st.l[1] = 0.0f;
#pragma unroll
  for (int mc = 0; mc < 8; ++mc)
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
  const uint32_t *kc_bh = J.k_codes + bhi * (p.cap / W) * kD;
  const float *ks_bh = J.k_scale + bhi * (p.cap / G) * kD;
  const float *kz_bh = J.k_zero + bhi * (p.cap / G) * kD;
  const uint32_t *vc_bh = J.v_codes + bhi * p.cap * (kD / W);
  const float *vs_bh = J.v_scale + bhi * p.cap * (kD / G);
  const float *vz_bh = J.v_zero + bhi * p.cap * (kD / G);
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
    bulk_load(dst, kc_bh + (tok / W) * kD, F::kKc >> sh, bar, pol);
    bulk_load(dst + F::oKs, ks_bh + (tok / G) * kD, F::kKs >> sh, bar, pol);
    bulk_load(dst + F::oKz, kz_bh + (tok / G) * kD, F::kKs >> sh, bar, pol);
    bulk_load(dst + F::oVc, vc_bh + tok * (kD / W), F::kVc >> sh, bar, pol);
    bulk_load(dst + F::oVs, vs_bh + tok * (kD / G), F::kVs >> sh, bar, pol);
    bulk_load(dst + F::oVz, vz_bh + tok * (kD / G), F::kVs >> sh, bar, pol);
  };
  int issued = 0;
  if (lane == 0)
    for (; issued < min(F::NS, n_my); ++issued) issue(issued);
  issued = __shfl_sync(0xffffffffu, issued, 0);

  // query heads kvh*r .. kvh*r + r-1 as B fragments (k = channels, n = heads)
  // in shared memory, one copy per block (loaded while the first copies fly)
  uint2 *qsm = reinterpret_cast<uint2 *>(smem + F::kQsm);
  for (int idx = threadIdx.x; idx < 8 * 32; idx += kThreads) {
    const int kk = idx >> 5, ql = idx & 31, qg = ql >> 2, qt = ql & 3;
    const __half *q = static_cast<const __half *>(J.q) + (b * h_q + kvh * p.r + qg) * kD;
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
    srow_k = static_cast<const __half *>(J.sink_k) + bhi * p.sink_cap * kD;
    srow_v = static_cast<const __half *>(J.sink_v) + bhi * p.sink_cap * kD;
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
    uint32_t klo[4], khi[4];
    if (KLUT) {
      const float *ks = reinterpret_cast<const float *>(stg + F::oKs);
      const float *kz = reinterpret_cast<const float *>(stg + F::oKz);
#pragma unroll
      for (int i = 0; i < 4; ++i) lut2(ks[lane + 32 * i], kz[lane + 32 * i], klo[i], khi[i]);
    }
#pragma unroll 1
    for (int hb = 0; hb < n_hb; ++hb) {
      float s[4];
      uint32_t phi[2], plo[2];
      // key scale / zero row of the half's group
      const int krow = G < 32 ? hb * kD : 0;
      // sinks of this half: list entries [sc, se)
      const int64_t tok0 = static_cast<int64_t>(st0 + warp + kWarps * done) * kTile + kHalf * hb;
      int se = sc;
      if (SINKS) {
        while (sc < scnt && spos[sc] < tok0) ++sc;   // other warps' tiles
        se = sc;
        while (se < scnt && spos[se] < tok0 + kHalf) ++se;
      }
      if (KLUT)
        expand_keys2_lut(reinterpret_cast<const uint32_t *>(stg), klo, khi, hb, buf, lane);
      else
        expand_keys<BITS>(reinterpret_cast<const uint32_t *>(stg),
                          reinterpret_cast<const float *>(stg + F::oKs) + krow,
                          reinterpret_cast<const float *>(stg + F::oKz) + krow, hb, buf, lane);
      __syncwarp();
      if (SINKS && se > sc) {                      // the sinks' exact key columns
        for (int j = sc; j < se; ++j)
          sink_key_column<BITS>(buf, srow_k + static_cast<int64_t>(j) * kD,
                                static_cast<int>(spos[j] - tok0), lane);
        __syncwarp();
      }
      half_scores<true>(buf, qsm, lane, s);
      half_softmax(st, s, p.scale_log2, kHalf, g, phi, plo);
      __syncwarp();                                // key half tile read by every lane
      if constexpr (BITS == 2 && G >= 32)
        expand_values2_32<G>(reinterpret_cast<const uint32_t *>(stg + F::oVc),
                             reinterpret_cast<const float *>(stg + F::oVs),
                             reinterpret_cast<const float *>(stg + F::oVz), hb, buf, lane);
      else
        expand_values<BITS, G>(reinterpret_cast<const uint32_t *>(stg + F::oVc),
                               reinterpret_cast<const float *>(stg + F::oVs),
                               reinterpret_cast<const float *>(stg + F::oVz), hb, buf, lane);
      __syncwarp();                                // value half tile written
      if (SINKS && se > sc) {                      // the sinks' exact value rows
        for (int j = sc; j < se; ++j)
          sink_value_row<BITS>(buf, srow_v + static_cast<int64_t>(j) * kD,
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
    if (lane == 0) atomicOr(&g_fault_word, 1u);
#pragma unroll 1
    for (int i = done; i < issued; ++i)
      mbar_wait_bounded(bar0 + 8 * (i % F::NS), (i / F::NS) & 1, kWaitLimitNs);
  }

  // ---- residual tiles (last split): fp16 rows read directly, 16 tokens at a time
  if (split == p.n_split - 1 && !failed) {
    const __half *kr = static_cast<const __half *>(J.k_res) + bhi * p.r_cap * kD;
    const __half *vr = static_cast<const __half *>(J.v_res) + bhi * p.r_cap * kD;
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
        load_residual<false>(kr, p.r_cap, p.res_head, tok0, valid, buf, lane);
        __syncwarp();
        half_scores<false>(buf, qsm, lane, s);
        half_softmax(st, s, p.scale_log2, valid, g, phi, plo);
        __syncwarp();
        load_residual<BITS == 2>(vr, p.r_cap, p.res_head, tok0, valid, buf, lane);
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
  float *red_o = red_l + kWarps * 8;                         // [warp][8][D]
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
  for (int mc = 0; mc < 8; ++mc) {
    float *o0 = red_o + (warp * 8 + 2 * t) * kD + 16 * mc + cg;
    float *o1 = o0 + kD;
    o0[0] = st.o[mc][0];
    o1[0] = st.o[mc][1];
    o0[8] = st.o[mc][2];
    o1[8] = st.o[mc][3];
  }
  __syncthreads();
  const int nr = p.r * kD;
#pragma unroll 1
  for (int idx = threadIdx.x; idx < nr; idx += kThreads) {
    const int h = idx / kD, c = idx - h * kD;
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
      O += red_o[(w * 8 + h) * kD + c] * f;
    }
    if (p.n_split == 1) {
      J.out[(b * h_q + kvh * p.r + h) * kD + c] = O / L;
    } else {
      const int64_t base = item * p.r + h;   // partial (item, head)
      p.ws[base * kD + c] = O;
      if (c == 0) {
        float *ml = p.ws + static_cast<int64_t>(gridDim.x) * p.r * kD;
        ml[2 * base] = M;
        ml[2 * base + 1] = L;
      }
    }
  }
}

// Combine the splits of one (layer, bh, head): thread = channel.
__global__ void __launch_bounds__(kD) attention_combine_kernel(const __grid_constant__ AttnParams p) {
  const int64_t blk = blockIdx.x;             // (job * bh + bhi) * r + h
  const int h = static_cast<int>(blk % p.r);
  const int64_t pair = blk / p.r;
  const int job = static_cast<int>(pair / p.bh);
  const int64_t bhi = pair - static_cast<int64_t>(job) * p.bh;
  const int64_t b = bhi / p.h_kv, kvh = bhi - b * p.h_kv;
  const int c = threadIdx.x;
  const int64_t items = static_cast<int64_t>(p.n_jobs) * p.bh * p.n_split;
  const float *ml = p.ws + items * p.r * kD;
  float M = -INFINITY;
  for (int s = 0; s < p.n_split; ++s) M = fmaxf(M, ml[2 * ((pair * p.n_split + s) * p.r + h)]);
  float L = 0.0f, O = 0.0f;
  for (int s = 0; s < p.n_split; ++s) {
    const int64_t base = (pair * p.n_split + s) * p.r + h;
    const float ms = ml[2 * base];
    if (ms == -INFINITY) continue;
    const float f = exp2f(ms - M);
    L += ml[2 * base + 1] * f;
    O += p.ws[base * kD + c] * f;
  }
  const int64_t h_q = static_cast<int64_t>(p.h_kv) * p.r;
  p.jobs[job].out[(b * h_q + kvh * p.r + h) * kD + c] = O / L;
}


template <int BITS, int G, bool SINKS>
cudaError_t attention_launch_k(const AttnParams &p, cudaStream_t stream) {
  using F = StageFmt<BITS, G>;
  auto kern = decode_attention_kernel<BITS, G, SINKS>;
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
  const int64_t items = static_cast<int64_t>(p.n_jobs) * p.bh * p.n_split;
  kern<<<static_cast<unsigned>(items), kThreads, F::kSmem, stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || p.n_split == 1) return e;
  return launch_attention_combine(p, stream);
}

template <int BITS, int G>
cudaError_t attention_launch(const AttnParams &p, cudaStream_t stream) {
  return p.sink_cap > 0 ? attention_launch_k<BITS, G, true>(p, stream)
                        : attention_launch_k<BITS, G, false>(p, stream);
}
}  // namespace

cudaError_t launch_attention_combine(const AttnParams &p, cudaStream_t stream) {
  const int64_t blocks = static_cast<int64_t>(p.n_jobs) * p.bh * p.r;
  attention_combine_kernel<<<static_cast<unsigned>(blocks), kD, 0, stream>>>(p);
  return cudaGetLastError();
}

// The kernel the environment variable KIVI_ATTENTION_KERNEL selects: the
// register-MMA kernel of this file unless it reads "tcgen05", which selects
// the tensor-memory kernel (kivi_attention_tc.cu) for the calls that kernel
// takes.  Read at every call, so a process can switch between calls.
static bool tensor_memory_kernel_selected() {
  const char *v = std::getenv("KIVI_ATTENTION_KERNEL");
  return v && std::strcmp(v, "tcgen05") == 0;
}

cudaError_t launch_decode_attention(const AttnParams &p, int group, int bits, cudaStream_t stream) {
  if (tensor_memory_kernel_selected()) {
    bool handled = false;
    const cudaError_t e = launch_decode_attention_tc(p, group, bits, stream, &handled);
    if (handled) return e;
  }
  switch (bits * 1000 + group) {
    case 2016: return attention_launch<2, 16>(p, stream);
    case 4016: return attention_launch<4, 16>(p, stream);
    case 8016: return attention_launch<8, 16>(p, stream);
    case 2032: return attention_launch<2, 32>(p, stream);
    case 2064: return attention_launch<2, 64>(p, stream);
    case 2128: return attention_launch<2, 128>(p, stream);
    case 4032: return attention_launch<4, 32>(p, stream);
    case 4064: return attention_launch<4, 64>(p, stream);
    case 4128: return attention_launch<4, 128>(p, stream);
    case 8032: return attention_launch<8, 32>(p, stream);
    case 8064: return attention_launch<8, 64>(p, stream);
    case 8128: return attention_launch<8, 128>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

int attention_splits(int64_t items, int64_t tiles_store, int group, int bits) {
  (void)group;
  (void)bits;
  if (items <= 0) return 1;
  const int64_t target = static_cast<int64_t>(current_sm_count()) * 4 * 2;   // two waves of 4 CTAs per SM
  const int64_t want = (target + items - 1) / items;
  const int64_t most = std::max<int64_t>(1, std::min<int64_t>(64, tiles_store / (2 * kWarps)));
  return static_cast<int>(std::max<int64_t>(1, std::min(want, most)));
}

// Addresses of this file's device symbols as host code must pass them to
// kernels (the symbol's name in host code is a host-side stand-in, not a
// device address).  The lookup runs once per device and context: entries
// are keyed by the device and the unique id of the context current on it,
// so a device that was reset (a new context, its modules loaded again) gets
// a fresh lookup, and a mutex serialises concurrent host threads.  The
// first call on a device (and the first after a reset) makes the runtime
// calls of the lookup, so it should come before any stream capture.
namespace {

using CtxGetCurrentFn = int (*)(void **);                      // cuCtxGetCurrent
using CtxGetIdFn = int (*)(void *, unsigned long long *);      // cuCtxGetId

// Unique id of the context current on the calling thread (0 if none or if
// the driver does not provide the query).
unsigned long long current_context_id() {
  static std::once_flag once;
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  std::call_once(once, [] {
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(f);
  });
  if (!get_current || !get_id) return 0;
  void *ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != 0 || ctx == nullptr || get_id(ctx, &id) != 0) return 0;
  return id;
}

struct SymbolSlot {
  unsigned long long ctx_id;
  void *addr;
};

// The device address of `symbol` on the current device.
cudaError_t symbol_address(const void *symbol, SymbolSlot (&slots)[64], void **out) {
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  const unsigned long long id = current_context_id();
  if (id != 0 && slots[dev].ctx_id == id && slots[dev].addr != nullptr) {
    *out = slots[dev].addr;
    return cudaSuccess;
  }
  void *a = nullptr;
  e = cudaGetSymbolAddress(&a, symbol);   // creates the context if there is none yet
  if (e != cudaSuccess) return e;
  slots[dev] = {current_context_id(), a};
  *out = a;
  return cudaSuccess;
}

SymbolSlot g_scratch_slots[64];
SymbolSlot g_fault_slots[64];

}  // namespace

cudaError_t attention_scratch(float **ptr, int64_t *max_floats) {
  void *a = nullptr;
  const cudaError_t e = symbol_address(reinterpret_cast<const void *>(&g_attn_scratch),
                                       g_scratch_slots, &a);
  if (e != cudaSuccess) return e;
  *ptr = static_cast<float *>(a);
  *max_floats = kAttnScratchFloats;
  return cudaSuccess;
}

int64_t attention_scratch_floats() { return kAttnScratchFloats; }

cudaError_t fault_word_address(unsigned int **ptr) {
  void *a = nullptr;
  const cudaError_t e = symbol_address(reinterpret_cast<const void *>(&g_fault_word),
                                       g_fault_slots, &a);
  if (e != cudaSuccess) return e;
  *ptr = static_cast<unsigned int *>(a);
  return cudaSuccess;
}

// One warp waits (bounded) on a phase that nothing completes: the wait gives
// up after limit_ns and the timeout is recorded as bit 2 of the fault word.
__global__ void __launch_bounds__(32) wait_timeout_selftest_kernel(uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = smem_addr(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);      // one arrival expected; none ever happens
    fence_mbar_init();
  }
  __syncwarp();
  const bool done = __all_sync(0xffffffffu, mbar_wait_bounded(b, 0, limit_ns));
  if (!done && threadIdx.x == 0) atomicOr(&g_fault_word, 4u);
}

cudaError_t launch_wait_timeout_selftest(uint64_t limit_ns, cudaStream_t stream) {
  wait_timeout_selftest_kernel<<<1, 32, 0, stream>>>(limit_ns);
  return cudaGetLastError();
}

cudaError_t read_and_clear_fault(uint32_t *fault) {
  unsigned int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_fault_word, sizeof(v));
  if (e != cudaSuccess) return e;
  const unsigned int zero = 0;
  e = cudaMemcpyToSymbol(g_fault_word, &zero, sizeof(zero));
  *fault = v;
  return e;
}

}  // namespace kivi_impl
