// kivi_tc_common.cuh -- building blocks of the tcgen05 decode-attention
// kernel (kivi_attention_ws.cu): the staged tile's layout, the fp16 operand layouts and shared-memory matrix descriptors of
// tcgen05.mma (no swizzle), the instruction descriptors, the MMA, commit,
// fence and tensor-memory load wrappers, and the expansion of a staged tile's
// codes into the fp16 key and value operands (the arithmetic of the
// dequantize kernels, bit-identical).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "kivi_device.cuh"
#include "kivi_expand.cuh"
#include "kivi_launch.h"

namespace kivi_impl {
namespace tcc {

using namespace kivi_dev;

constexpr int kD = 128;                  // head_dim
constexpr int kTile = 128;               // tokens per tile (MMA M of the scores)
constexpr int kPiece = 32;               // tokens per store piece (the split granule)
constexpr int kN = 16;                   // MMA N
constexpr int kMaxR = 8;                 // query heads per KV head
constexpr float kLog2PScale = 8.0f;      // P = 2^(s - m + 8)
constexpr float kTau = 7.0f;             // s <= m + 7 keeps P <= 2^15
constexpr uint64_t kWaitLimitNs = 200000000ull;

// One staged 128-token store tile of a (layer, bh): its key codes, key
// scale and zero rows, value codes, value scales and zeros, as contiguous
// pieces (byte offsets), and the size of one fp16 operand tile.
template <int BITS, int G>
struct TcStage {
  static constexpr int W = 32 / BITS;
  static constexpr int kKc = kTile / W * kD * 4;      // key code rows of a tile
  static constexpr int kKs = kTile / G * kD * 4;      // key scale (or zero) rows
  static constexpr int kVc = kTile * (kD / W) * 4;    // value codes
  static constexpr int kVs = kTile * (kD / G) * 4;    // value scales (or zeros)
  static constexpr int oKs = kKc, oKz = oKs + kKs, oVc = oKz + kKs, oVs = oVc + kVc,
                       oVz = oVs + kVs;
  static constexpr int kStage = oVz + kVs;
  static constexpr int kOp = kTile * kD * 2;          // one fp16 operand tile
};

// ---- operand layouts (no swizzle; core matrix = 8 rows x 16 bytes) --------
// MN-major A of the scores (store keys: m = token slot, k = channel): the
// 16-byte row (8 token slots from 8 s8) of channel c.
__device__ __forceinline__ uint32_t kt_row(int c, int s8) {
  return static_cast<uint32_t>((c >> 3) * 2048 + s8 * 128 + (c & 7) * 16);
}
// Token-major rows [token][channel]: K-major A of the scores (residual keys)
// and MN-major A of the output (values, m = channel, k = token): the 16-byte
// chunk of channels 8 j .. 8 j + 7 of token slot s.
__device__ __forceinline__ uint32_t tm_chunk(int s, int j) {
  return static_cast<uint32_t>((s >> 3) * 2048 + j * 128 + (s & 7) * 16);
}
// K-major B [n][k] (Q: k = channel): element (n, k).
__device__ __forceinline__ uint32_t b_elem(int n, int k) {
  return static_cast<uint32_t>((n >> 3) * 2048 + (k >> 3) * 128 + (n & 7) * 16 + (k & 7) * 2);
}
// MN-major B (P: n = head row, k = token slot): the 16-byte row of slot k
// holds n = 0..7 (high parts), the next core matrix (+128) n = 8..15 (low
// parts); k-groups of 8 slots are 256 bytes apart.
__device__ __forceinline__ uint32_t p_row(int k) {
  return static_cast<uint32_t>((k >> 3) * 256 + (k & 7) * 16);
}

// 2^x by the hardware's approximate base-2 exponential (results below the
// normal range flush to zero)
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Shared-memory matrix descriptor: start, leading and stride byte offsets
// (16-byte units), descriptor version 1, no swizzle.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return static_cast<uint64_t>((addr >> 4) & 0x3FFFu) |
         (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (uint64_t{1} << 46);
}
// Instruction descriptor: f32 accumulator, f16 A and B, B K-major, N = 16,
// M = 128; A MN-major or K-major.
constexpr uint32_t kIdescMN = (1u << 4) | (1u << 15) | ((kN >> 3) << 17) | ((kTile >> 4) << 24);
constexpr uint32_t kIdescK = (1u << 4) | ((kN >> 3) << 17) | ((kTile >> 4) << 24);
// the output MMA: A (values) MN-major, B (P) MN-major
constexpr uint32_t kIdescO = kIdescMN | (1u << 16);

__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Eight consecutive 32-bit accumulator columns of this warp's 32 lanes.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float (&v)[8]) {
  uint32_t r[8];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                 "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

// Keys of a staged tile -> MN-major operand tile.  Unit = (channel c, one
// 32-token piece): thread t takes c = t % 128 and pieces t / 128 and
// 2 + t / 128, so each unit builds its group's scale constants once, and 8
// consecutive lanes write 8 consecutive 16-byte rows of a core matrix.
template <int BITS, int G>
__device__ __forceinline__ void expand_keys_tc(const unsigned char *stg, uint32_t tile, int tid) {
  using F = TcStage<BITS, G>;
  constexpr int W = F::W;
  const uint32_t *kc = reinterpret_cast<const uint32_t *>(stg);
  const float *ks = reinterpret_cast<const float *>(stg + F::oKs);
  const float *kz = reinterpret_cast<const float *>(stg + F::oKz);
  const int c = tid & 127;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int pc = 2 * i + (tid >> 7);        // 32-token piece of the tile
    const int grp = (kPiece * pc) / G;
    if constexpr (BITS == 2) {   // token slots in the table lookups' order
      uint32_t lo, hi;
      lut2(ks[grp * kD + c], kz[grp * kD + c], lo, hi);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int tb = 2 * pc + h;             // 16-token block: one code word
        uint4 c0, c1;
        lookup16(kc[tb * kD + c], lo, hi, c0, c1);
        sts128(tile + kt_row(c, 2 * tb), c0);
        sts128(tile + kt_row(c, 2 * tb + 1), c1);
      }
    } else {
      uint64_t s2, ns2, z2;
      scale_consts(ks[grp * kD + c], kz[grp * kD + c], s2, ns2, z2);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int tb = 2 * pc + h;
        uint32_t w[16 / W];
#pragma unroll
        for (int k = 0; k < 16 / W; ++k) w[k] = kc[(tb * (16 / W) + k) * kD + c];
        float m[16];
        magics16<BITS>(w, m);
        sts128(tile + kt_row(c, 2 * tb), deq8(m, s2, ns2, z2));
        sts128(tile + kt_row(c, 2 * tb + 1), deq8(m + 8, s2, ns2, z2));
      }
    }
  }
}

// Values of a staged tile -> token-major operand tile.  Unit = (token tok,
// 64-channel half h): thread t takes tok = t % 128 and h = t / 128, so a
// unit's codes are one to four 16-byte loads and 8 consecutive lanes write
// the same chunk of 8 consecutive token rows.  Tokens at or past `valid` are
// written as zeros (their probabilities are zero, and 0 * NaN of a stale
// stage would not be).  2-bit: token rows in the keys' slot order, channels
// of each chunk in the lookup order.
template <int BITS, int G>
__device__ __forceinline__ void expand_values_tc(const unsigned char *stg, uint32_t tile, int tid,
                                                 int valid) {
  using F = TcStage<BITS, G>;
  constexpr int W = F::W;
  constexpr int RW = kD / W;          // words per token
  constexpr int NG = kD / G;
  constexpr int WH = 64 / W;          // words per 64-channel half
  const uint32_t *vc = reinterpret_cast<const uint32_t *>(stg + F::oVc);
  const float *vs = reinterpret_cast<const float *>(stg + F::oVs);
  const float *vz = reinterpret_cast<const float *>(stg + F::oVz);
  const int tok = tid & 127, h = tid >> 7;
  const int slot = BITS == 2 ? ((tok & ~7) | perm8_inv(tok & 7)) : tok;
  if (tok >= valid) {
#pragma unroll
    for (int k = 0; k < 8; ++k) sts128(tile + tm_chunk(slot, 8 * h + k), make_uint4(0u, 0u, 0u, 0u));
    return;
  }
  // the half's groups: two at G = 32, one otherwise
  constexpr int NGH = G == 32 ? 2 : 1;
  const int g0 = (64 * h) / G;
  float sg[NGH], zg[NGH];
#pragma unroll
  for (int k = 0; k < NGH; ++k) {
    sg[k] = vs[tok * NG + g0 + k];
    zg[k] = vz[tok * NG + g0 + k];
  }
  if constexpr (BITS == 2) {   // the half's 4 words in one load
    const uint4 v = *reinterpret_cast<const uint4 *>(vc + tok * RW + h * WH);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < NGH; ++k) {
      uint32_t lo, hi;
      lut2(sg[k], zg[k], lo, hi);
#pragma unroll
      for (int cb = k * (4 / NGH); cb < (k + 1) * (4 / NGH); ++cb) {   // 16-channel blocks
        uint4 c0, c1;
        lookup16(w[cb], lo, hi, c0, c1);
        sts128(tile + tm_chunk(slot, 8 * h + 2 * cb), c0);
        sts128(tile + tm_chunk(slot, 8 * h + 2 * cb + 1), c1);
      }
    }
  } else {
#pragma unroll
    for (int k = 0; k < NGH; ++k) {
      uint64_t s2, ns2, z2;
      scale_consts(sg[k], zg[k], s2, ns2, z2);
#pragma unroll
      for (int cb = k * (4 / NGH); cb < (k + 1) * (4 / NGH); ++cb) {   // a block's words
        uint32_t w[16 / W];
        if constexpr (BITS == 8) {
          const uint4 v = *reinterpret_cast<const uint4 *>(vc + tok * RW + h * WH + cb * 4);
          w[0] = v.x;
          w[1] = v.y;
          w[2] = v.z;
          w[3] = v.w;
        } else {
          const uint2 v = *reinterpret_cast<const uint2 *>(vc + tok * RW + h * WH + cb * 2);
          w[0] = v.x;
          w[1] = v.y;
        }
        float m[16];
        magics16<BITS>(w, m);
        sts128(tile + tm_chunk(slot, 8 * h + 2 * cb), deq8(m, s2, ns2, z2));
        sts128(tile + tm_chunk(slot, 8 * h + 2 * cb + 1), deq8(m + 8, s2, ns2, z2));
      }
    }
  }
}

// fp16 residual rows tok0 .. tok0 + 127 of a ring -> token-major operand
// tile; rows past `valid` are zero.  Thread t takes token t % 128 and chunks
// 2 i + t / 128.  PERM: channels of each chunk in the 2-bit lookup order.
template <bool PERM>
__device__ __forceinline__ void load_residual_tc(const __half *base, int64_t r_cap, int64_t head,
                                                 int64_t tok0, int valid, uint32_t tile, int tid) {
  const int tok = tid & 127;
  const bool ok = tok < valid;
  const uint4 *src = nullptr;
  if (ok) src = reinterpret_cast<const uint4 *>(base + ((head + tok0 + tok) % r_cap) * kD);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int j = 2 * i + (tid >> 7);
    uint4 v = ok ? src[j] : make_uint4(0u, 0u, 0u, 0u);
    if (PERM)
      v = make_uint4(__byte_perm(v.x, v.z, 0x5410u), __byte_perm(v.x, v.z, 0x7632u),
                     __byte_perm(v.y, v.w, 0x5410u), __byte_perm(v.y, v.w, 0x7632u));
    sts128(tile + tm_chunk(tok, j), v);
  }
}

}  // namespace tcc
}  // namespace kivi_impl
