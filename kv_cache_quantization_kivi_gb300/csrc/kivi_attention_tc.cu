// kivi_attention_tc.cu -- decode attention over the packed KIVI store on the
// fifth-generation tensor cores (tcgen05 matrix multiply with the
// accumulators in tensor memory).
//
// What it computes is that of decode_attention_kernel (kivi_attention_kernel.cuh):
// for every layer, sequence and query head, softmax(scale * q K^T) V over the
// cache's store tokens (dequantized on chip, bit-identical to the dequantize
// kernels' fp16 reconstructions) followed by its fp16 residual tokens, query
// head h reading KV head h / r (the fused-kernel post's closing section:
// attention that reads the packed codes).  It serves head_dim 128 with
// G >= 32 and no sink store; the register-MMA kernel keeps the other cases.
//
// One CTA of 8 warps per (layer, bh, split).  The split's store range is
// walked in tiles of 128 tokens (four 32-token pieces; each piece's key and
// value codes, scales and zeros are contiguous runs) staged into a
// shared-memory ring by bulk copies, then the residual in 128-token tiles.
// Per tile i:
//   keys    expanded into the fp16 key operand -- MN-major (token
//           contiguous) for store tiles, a lane writing one channel's 8
//           tokens as one 16-byte core-matrix row; K-major for residual rows
//           -- then one thread issues S^T = K Q^T (8 tcgen05.mma, M = 128
//           tokens, N = 16: the r <= 8 query heads, padded; K = 16 channels)
//           into tensor-memory columns 0..15;
//   values  expanded into the fp16 value operand (token-major rows, which is
//           V^T MN-major) while that MMA runs;
//   softmax the scores come back with tcgen05.ld (lane = token; a warp's
//           quarter of the lanes, 4 heads per thread), P = 2^(s - m) * 2^8 is
//           split into fp16 high and low parts written as one N = 16 operand
//           (heads 0..7 high, 8..15 low; MN-major, so a thread stores its 4
//           heads' parts as two 8-byte words), so the values are read once;
//   output  O^T += V^T P^T (8 tcgen05.mma, M = 128 channels) accumulates in
//           tensor-memory columns 16..31 across tiles, running under the
//           next tile's key expansion.
// The softmax reference m of a head moves only when a score exceeds it by
// more than 2^7 (one vote on the tile's barrier): then the tile maximum is
// taken across the warps, the accumulated output is read back, rescaled into
// registers and the accumulation restarts.  Every tile's P is therefore at
// most 2^15 (a finite fp16) and the per-thread sums of P need no per-tile
// exchange; they are reduced once at the end.  (The result is that of any
// reference: o and l are both relative to it.)
// Expanded 2-bit tiles keep the token order (0,4)(1,5)(2,6)(3,7) of the
// table lookups inside each 8-token chunk for keys and values alike, and the
// value channels the same order inside each 8-channel chunk (residual rows
// are permuted to match); the output undoes the channel order.
//
// Every wait is bounded (0.2 s of the global timer); a timeout sets bit 0 of
// the device fault word, the CTA stops taking tiles, waits (bounded) for its
// copies and matrix multiplies in flight and frees its tensor memory.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>

#include "kivi_device.cuh"
#include "kivi_expand.cuh"
#include "kivi_launch.h"

namespace kivi_impl {
namespace {

using namespace kivi_dev;

constexpr int kD = 128;                  // head_dim
constexpr int kWarps = 8;
constexpr int kThreads = 32 * kWarps;
constexpr int kTile = 128;               // tokens per tile (MMA M of the scores)
constexpr int kPiece = 32;               // tokens per store piece (the split granule)
constexpr int kN = 16;                   // MMA N
constexpr int kMaxR = 8;                 // query heads per KV head
constexpr float kLog2PScale = 8.0f;      // P = 2^(s - m + 8)
constexpr float kTau = 7.0f;             // s <= m + 7 keeps P <= 2^15
constexpr uint64_t kWaitLimitNs = 200000000ull;
constexpr uint32_t kTmemCols = 32;       // scores: columns 0..15, output: 16..31

// Shared memory (byte offsets from the dynamic base): the staged code ring,
// the fp16 key and value operands, Q and P (B operands), the cross-warp
// exchange and the mbarriers.  NS: ring stages, as many as keep two CTAs on
// an SM (at most 4) when two stages fit that way, else as many as one CTA
// holds (at most 6).
template <int BITS, int G>
struct TcFmt {
  static constexpr int W = 32 / BITS;
  static constexpr int kKc = kTile / W * kD * 4;      // key code rows of a tile
  static constexpr int kKs = kTile / G * kD * 4;      // key scale (or zero) rows
  static constexpr int kVc = kTile * (kD / W) * 4;    // value codes
  static constexpr int kVs = kTile * (kD / G) * 4;    // value scales (or zeros)
  static constexpr int oKs = kKc, oKz = oKs + kKs, oVc = oKz + kKs, oVs = oVc + kVc,
                       oVz = oVs + kVs;
  static constexpr int kStage = oVz + kVs;
  static constexpr int kOp = kTile * kD * 2;          // one fp16 operand tile
  static constexpr int kRed = 2 * kWarps * 4 * 4;     // maxima and sums
  static constexpr int kBars = 128;
  static constexpr int kFixed = 2 * kOp + kN * kD * 2 + kN * kTile * 2 + kRed + kBars;
  static constexpr int kTwo = (113 * 1024 - kFixed) / kStage;
  static constexpr int kOne = (227 * 1024 - kFixed) / kStage;
  static constexpr int NS = kTwo >= 2 ? (kTwo > 4 ? 4 : kTwo) : (kOne > 6 ? 6 : kOne);
  static constexpr int oK = NS * kStage;
  static constexpr int oV = oK + kOp;
  static constexpr int oQ = oV + kOp;                 // Q [16][128] fp16
  static constexpr int oP = oQ + kN * kD * 2;         // P [16][128] fp16
  static constexpr int oRed = oP + kN * kTile * 2;    // [2][8 warps][4 heads] floats
  static constexpr int oBar = oRed + kRed;            // NS + 2 mbarriers, TMEM address
  static constexpr int kSmem = oBar + kBars;
  static_assert(NS >= 2 && kSmem <= 227 * 1024, "ring does not fit");
  static_assert(NS + 2 <= 15, "mbarrier area");
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
// Four consecutive 32-bit accumulator columns of this warp's 32 lanes.
__device__ __forceinline__ void tmem_ld4(uint32_t taddr, float (&v)[4]) {
  uint32_t r[4];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 4; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}
__device__ __forceinline__ void sts64(uint32_t addr, uint32_t a, uint32_t b) {
  asm volatile("st.shared.v2.b32 [%0], {%1,%2};" ::"r"(addr), "r"(a), "r"(b) : "memory");
}

// Keys of a staged tile -> MN-major operand tile.  Unit = (channel c, one
// 32-token piece): thread t takes c = t % 128 and pieces t / 128 and
// 2 + t / 128, so each unit builds its group's scale constants once, and 8
// consecutive lanes write 8 consecutive 16-byte rows of a core matrix.
template <int BITS, int G>
__device__ __forceinline__ void expand_keys_tc(const unsigned char *stg, uint32_t tile, int tid) {
  using F = TcFmt<BITS, G>;
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
  using F = TcFmt<BITS, G>;
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

template <int BITS, int G>
__global__ void __launch_bounds__(kThreads, 2) decode_attention_tc_kernel(const __grid_constant__ AttnParams p) {
  using F = TcFmt<BITS, G>;
  constexpr int W = F::W;
  constexpr int NS = F::NS;
  extern __shared__ __align__(1024) unsigned char smem[];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quarter = warp & 3;            // tensor-memory lanes 32 quarter .. + 31
  const int hc0 = (warp >> 2) * 4;         // this thread's 4 heads
  const int64_t item = blockIdx.x;
  const int split = static_cast<int>(item % p.n_split);
  const int64_t pair = item / p.n_split;
  const int job = static_cast<int>(pair / p.bh);
  const int64_t bhi = pair - static_cast<int64_t>(job) * p.bh;
  const AttnJob &J = p.jobs[job];
  const int64_t b = bhi / p.h_kv, kvh = bhi - b * p.h_kv;
  const int64_t h_q = static_cast<int64_t>(p.h_kv) * p.r;

  // this split's store pieces [pc0, pc0 + n_pc), in tiles of four pieces
  const int pc0 = split * p.tiles_per_split;
  const int n_pc = max(0, min(pc0 + p.tiles_per_split, p.tiles_store) - pc0);
  const int n_st = (n_pc + 3) / 4;
  const int n_rt = split == p.n_split - 1 ? static_cast<int>((p.n_res + kTile - 1) / kTile) : 0;
  const int n_tiles = n_st + n_rt;

  const uint32_t base = smem_addr(smem);
  const uint32_t kbuf = base + F::oK, vbuf = base + F::oV;
  const uint32_t qb = base + F::oQ, pb = base + F::oP;
  float *red_m = reinterpret_cast<float *>(smem + F::oRed);        // [8][4]
  float *red_l = red_m + kWarps * 4;                               // [8][4]
  const uint32_t full_bar = base + F::oBar;                        // [NS]
  const uint32_t s_bar = full_bar + 8 * NS, o_bar = s_bar + 8;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + F::oBar + 8 * (NS + 2));

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) mbar_init(full_bar + 8 * s, 1);
    mbar_init(s_bar, 1);
    mbar_init(o_bar, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    __syncwarp();
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }

  const uint64_t pol = policy_evict_first();
  const uint32_t *kc_bh = J.k_codes + bhi * (p.cap / W) * kD;
  const float *ks_bh = J.k_scale + bhi * (p.cap / G) * kD;
  const float *kz_bh = J.k_zero + bhi * (p.cap / G) * kD;
  const uint32_t *vc_bh = J.v_codes + bhi * p.cap * (kD / W);
  const float *vs_bh = J.v_scale + bhi * p.cap * (kD / G);
  const float *vz_bh = J.v_zero + bhi * p.cap * (kD / G);
  // store tile t: pieces pc0 + 4 t .., tokens from (pc0 + 4 t) * 32, into stage t % NS
  auto issue = [&](int t) {
    const int np = min(4, n_pc - 4 * t);
    const int64_t tok = static_cast<int64_t>(pc0 + 4 * t) * kPiece;
    const int ntok = np * kPiece;
    const uint32_t dst = base + static_cast<uint32_t>((t % NS) * F::kStage);
    const uint32_t bar = full_bar + 8 * (t % NS);
    const uint32_t kcb = ntok / W * kD * 4, ksb = (ntok + G - 1) / G * kD * 4;
    const uint32_t vcb = ntok * (kD / W) * 4, vsb = ntok * (kD / G) * 4;
    mbar_arrive_expect_tx(bar, kcb + 2 * ksb + vcb + 2 * vsb);
    bulk_load(dst, kc_bh + (tok / W) * kD, kcb, bar, pol);
    bulk_load(dst + F::oKs, ks_bh + (tok / G) * kD, ksb, bar, pol);
    bulk_load(dst + F::oKz, kz_bh + (tok / G) * kD, ksb, bar, pol);
    bulk_load(dst + F::oVc, vc_bh + tok * (kD / W), vcb, bar, pol);
    bulk_load(dst + F::oVs, vs_bh + tok * (kD / G), vsb, bar, pol);
    bulk_load(dst + F::oVz, vz_bh + tok * (kD / G), vsb, bar, pol);
  };
  int issued = 0, s_issued = 0, o_issued = 0;      // (thread 0's counts)
  if (tid == 0) {
    fence_proxy_async_smem();
    for (; issued < min(NS, n_st); ++issued) issue(issued);
  }

  // Q of this KV head's r query heads as the B operand (rows >= r zero)
  for (int idx = tid; idx < kN * (kD / 8); idx += kThreads) {
    const int n = (idx & 7) + 8 * (idx >> 7), kcn = (idx >> 3) & 15;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (n < p.r)
      v = reinterpret_cast<const uint4 *>(static_cast<const __half *>(J.q) +
                                          (b * h_q + kvh * p.r + n) * kD)[kcn];
    sts128(qb + b_elem(n, 8 * kcn), v);
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t t_lane = tmem + (static_cast<uint32_t>(32 * quarter) << 16);

  // per-thread softmax state of heads hc0 .. hc0 + 3: reference m, partial
  // sum of this thread's tokens; output of channel slot 32 quarter + lane
  // folded out of tensor memory at each rescale
  float m_ref[4], l_acc[4], o_acc[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    m_ref[j] = -INFINITY;
    l_acc[j] = 0.0f;
    o_acc[j] = 0.0f;
  }
  bool o_live = false;     // tensor memory holds output accumulated since the last fold
  bool failed = false;
  const __half *kr = static_cast<const __half *>(J.k_res) + bhi * p.r_cap * kD;
  const __half *vr = static_cast<const __half *>(J.v_res) + bhi * p.r_cap * kD;
  const int slot = 32 * quarter + lane;    // this thread's token slot (scores), channel slot (output)

  int it = 0;
#pragma unroll 1
  for (; it < n_tiles; ++it) {
    const bool store = it < n_st;
    const unsigned char *stg = smem + (it % NS) * F::kStage;
    int valid;             // real token slots (the first `valid`; whole pieces for store tiles)
    int64_t rtok0 = 0;     // residual: first residual token of the tile
    bool ok = true;
    // ---- keys (the previous score MMA has completed: waited below)
    if (store) {
      valid = min(4, n_pc - 4 * it) * kPiece;
      ok = mbar_wait_bounded(full_bar + 8 * (it % NS), (it / NS) & 1, kWaitLimitNs);
      if (ok) expand_keys_tc<BITS, G>(stg, kbuf, tid);
    } else {
      rtok0 = static_cast<int64_t>(it - n_st) * kTile;
      valid = static_cast<int>(p.n_res - rtok0 < kTile ? p.n_res - rtok0 : kTile);
      load_residual_tc<false>(kr, p.r_cap, p.res_head, rtok0, valid, kbuf, tid);
    }
    fence_proxy_async_smem();
    tc_fence_before();
    if (__syncthreads_or(!ok)) { failed = true; break; }
    tc_fence_after();
    if (tid == 0) {        // S^T[token][head] = K Q^T over 8 steps of 16 channels
#pragma unroll
      for (int s = 0; s < kD / 16; ++s) {
        const uint64_t a = store ? smem_desc(kbuf + s * 4096, 2048, 128)
                                 : smem_desc(kbuf + s * 256, 128, 2048);
        mma_f16(tmem, a, smem_desc(qb + s * 256, 128, 2048), store ? kIdescMN : kIdescK,
                s > 0);
      }
      mma_commit(s_bar);
      ++s_issued;
    }
    // ---- values, while the score MMA runs (the previous output MMA, the
    // last reader of the value and P operands, must have completed)
    if (it > 0) ok = mbar_wait_bounded(o_bar, (it - 1) & 1, kWaitLimitNs);
    if (ok) {
      if (store)
        expand_values_tc<BITS, G>(stg, vbuf, tid, valid);
      else
        load_residual_tc<BITS == 2>(vr, p.r_cap, p.res_head, rtok0, valid, vbuf, tid);
    }
    // ---- scores (warp-uniform: tcgen05.ld is a whole-warp instruction)
    const bool ok_s = __all_sync(0xffffffffu, mbar_wait_bounded(s_bar, it & 1, kWaitLimitNs));
    tc_fence_after();
    float sc[4];
    if (ok_s) tmem_ld4(t_lane + hc0, sc);
    const bool real = slot < valid;
    bool vote = false;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      sc[j] = real && ok_s ? sc[j] * p.scale_log2 : -INFINITY;
      vote |= sc[j] > m_ref[j] + kTau;
    }
    float pf[4];
    auto write_p = [&]() {
      uint32_t hi2[2], lo2[2];
#pragma unroll
      for (int j = 0; j < 4; j += 2) {
        pf[j] = sc[j] == -INFINITY ? 0.0f : exp2f(sc[j] - m_ref[j] + kLog2PScale);
        pf[j + 1] = sc[j + 1] == -INFINITY ? 0.0f : exp2f(sc[j + 1] - m_ref[j + 1] + kLog2PScale);
        const __half2 hi = __floats2half2_rn(pf[j], pf[j + 1]);
        const float2 hf = __half22float2(hi);
        const __half2 lo = __floats2half2_rn(pf[j] - hf.x, pf[j + 1] - hf.y);
        hi2[j / 2] = h2_as_u32(hi);
        lo2[j / 2] = h2_as_u32(lo);
      }
      const uint32_t row = pb + p_row(slot) + 2 * hc0;
      sts64(row, hi2[0], hi2[1]);
      sts64(row + 128, lo2[0], lo2[1]);
    };
    write_p();
    fence_proxy_async_smem();
    tc_fence_before();
    if (__syncthreads_or(vote || !ok || !ok_s)) {
      if (__syncthreads_or(!ok || !ok_s)) { failed = true; break; }
      tc_fence_after();
      // move the reference to the maximum over the tile and the old reference
      float mt[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) mt[j] = sc[j];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1)
#pragma unroll
        for (int j = 0; j < 4; ++j) mt[j] = fmaxf(mt[j], __shfl_xor_sync(0xffffffffu, mt[j], off));
      if (lane == 0)
#pragma unroll
        for (int j = 0; j < 4; ++j) red_m[warp * 4 + j] = mt[j];
      __syncthreads();
      float alpha[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float m_t = m_ref[j];
#pragma unroll
        for (int q = 0; q < 4; ++q) m_t = fmaxf(m_t, red_m[((warp & 4) + q) * 4 + j]);
        alpha[j] = m_ref[j] == -INFINITY ? 0.0f : exp2f(m_ref[j] - m_t);
        m_ref[j] = m_t;
      }
      // fold the output accumulated so far (its MMAs have completed) and
      // restart the accumulation
      if (o_live) {
        float hi[4], lo[4];
        tmem_ld4(t_lane + 16 + hc0, hi);
        tmem_ld4(t_lane + 24 + hc0, lo);
#pragma unroll
        for (int j = 0; j < 4; ++j) o_acc[j] = (o_acc[j] + hi[j] + lo[j]) * alpha[j];
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) o_acc[j] *= alpha[j];
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) l_acc[j] *= alpha[j];
      o_live = false;
      write_p();
      fence_proxy_async_smem();
      tc_fence_before();
      __syncthreads();
    }
    tc_fence_after();
#pragma unroll
    for (int j = 0; j < 4; ++j) l_acc[j] += pf[j];
    if (tid == 0) {        // O^T[channel][n] += V^T P^T over 8 steps of 16 tokens
#pragma unroll
      for (int s = 0; s < kTile / 16; ++s)
        mma_f16(tmem + 16, smem_desc(vbuf + s * 4096, 2048, 128),
                smem_desc(pb + s * 512, 256, 128), kIdescO, s > 0 || o_live);
      mma_commit(o_bar);
      ++o_issued;
      // this tile's stage has been read (keys and values): refill it
      if (store && issued < n_st) {
        fence_proxy_async_smem();
        issue(issued);
        ++issued;
      }
    }
    o_live = true;
  }

  if (!failed && n_tiles > 0) {
    // the last output MMA, then the fold
    const bool ok = __all_sync(0xffffffffu,
                               mbar_wait_bounded(o_bar, (n_tiles - 1) & 1, kWaitLimitNs));
    tc_fence_after();
    if (ok) {
      float hi[4], lo[4];
      tmem_ld4(t_lane + 16 + hc0, hi);
      tmem_ld4(t_lane + 24 + hc0, lo);
#pragma unroll
      for (int j = 0; j < 4; ++j) o_acc[j] += hi[j] + lo[j];
    }
    failed = __syncthreads_or(!ok);
  }
  if (failed) {
    // record the timeout; wait (bounded) for the copies and matrix
    // multiplies still in flight (tiles before `it` were consumed)
    if (tid == 0) {
      atomicOr(p.fault, 1u);
      for (int t = it; t < issued; ++t)
        mbar_wait_bounded(full_bar + 8 * (t % NS), (t / NS) & 1, kWaitLimitNs);
      if (s_issued > 0) mbar_wait_bounded(s_bar, (s_issued - 1) & 1, kWaitLimitNs);
      if (o_issued > 0) mbar_wait_bounded(o_bar, (o_issued - 1) & 1, kWaitLimitNs);
    }
  } else {
    // sums of P per head over the 4 warps of its lanes
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
#pragma unroll
      for (int j = 0; j < 4; ++j) l_acc[j] += __shfl_xor_sync(0xffffffffu, l_acc[j], off);
    if (lane == 0)
#pragma unroll
      for (int j = 0; j < 4; ++j) red_l[warp * 4 + j] = l_acc[j];
    __syncthreads();
    // output of channel slot `slot`, heads hc0 .. hc0 + 3 (2-bit: slot m
    // holds channel (m & ~7) | perm8(m & 7))
    const int ch = BITS == 2 ? ((slot & ~7) | perm8(slot & 7)) : slot;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int h = hc0 + j;
      if (h >= p.r) continue;
      float l_t = 0.0f;
#pragma unroll
      for (int q = 0; q < 4; ++q) l_t += red_l[((warp & 4) + q) * 4 + j];
      if (p.n_split == 1) {
        J.out[(b * h_q + kvh * p.r + h) * kD + ch] = o_acc[j] / l_t;
      } else {
        const int64_t pbase = item * p.r + h;     // partial (item, head)
        p.ws[pbase * kD + ch] = o_acc[j];
        if (slot == 0) {
          float *ml = p.ws + static_cast<int64_t>(gridDim.x) * p.r * kD;
          ml[2 * pbase] = m_ref[j];
          ml[2 * pbase + 1] = l_t;
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols)
                 : "memory");
  }
}

template <int BITS, int G>
cudaError_t tc_launch(const AttnParams &p, cudaStream_t stream) {
  using F = TcFmt<BITS, G>;
  auto kern = decode_attention_tc_kernel<BITS, G>;
  constexpr int kMaxDevices = 64;
  static std::atomic<bool> configured[kMaxDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (!configured[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, F::kSmem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    configured[dev].store(true, std::memory_order_release);
  }
  // splits start on whole 128-token tiles (four 32-token pieces), so every
  // tile's key groups (G <= 128) start inside it; trailing splits may be empty
  AttnParams q = p;
  const int tps = (p.tiles_store + p.n_split - 1) / p.n_split;
  q.tiles_per_split = (tps + 3) / 4 * 4;
  e = fault_word_address(&q.fault);
  if (e != cudaSuccess) return e;
  const int64_t items = static_cast<int64_t>(p.n_jobs) * p.bh * p.n_split;
  kern<<<static_cast<unsigned>(items), kThreads, F::kSmem, stream>>>(q);
  e = cudaGetLastError();
  if (e != cudaSuccess || p.n_split == 1) return e;
  return launch_attention_combine(q, stream);
}

}  // namespace

cudaError_t launch_decode_attention_tc(const AttnParams &p, int group, int bits,
                                       cudaStream_t stream, bool *handled) {
  *handled = false;
  if (p.d != kD || p.sink_cap > 0 || p.r > kMaxR || group < 32) return cudaSuccess;
  *handled = true;
  switch (bits * 1000 + group) {
    case 2032: return tc_launch<2, 32>(p, stream);
    case 2064: return tc_launch<2, 64>(p, stream);
    case 2128: return tc_launch<2, 128>(p, stream);
    case 4032: return tc_launch<4, 32>(p, stream);
    case 4064: return tc_launch<4, 64>(p, stream);
    case 4128: return tc_launch<4, 128>(p, stream);
    case 8032: return tc_launch<8, 32>(p, stream);
    case 8064: return tc_launch<8, 64>(p, stream);
    case 8128: return tc_launch<8, 128>(p, stream);
    default: *handled = false; return cudaSuccess;
  }
}

}  // namespace kivi_impl
