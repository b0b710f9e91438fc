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
// tokens each) are dealt to the warps round-robin; each warp streams its
// tiles' key codes, key scale/zero row, value codes and value scales/zeros
// (six contiguous pieces) into a private shared-memory ring with bulk
// asynchronous copies completed on per-stage mbarriers, so no CTA barrier
// is needed until the end.  Per tile:
//   S^T = K Q^T     m16n8k16 tensor-core MMAs: A = the dequantized key tile
//                   (16 tokens x 16 channels), B = the query heads
//   online softmax  per head column, base-2 exponent with the scale folded in
//   O^T += V^T P^T  A = the dequantized value tile (16 channels x 16 tokens),
//                   B = P^T from the score accumulators through movmatrix
// P is scaled by 2^12 and split into fp16 high and low parts (two MMAs), so
// the probabilities keep ~22 bits; the scale cancels against the softmax
// denominator accumulated in fp32 from the same values.  The 4 warps' states
// are combined through shared memory; with several splits the partial
// (max, sum, unnormalised output) go to the caller's workspace and a second
// kernel combines them.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>

#include "kivi_device.cuh"
#include "kivi_launch.h"

namespace kivi_impl {

// bit 0: a pipeline wait of the decode-attention kernel timed out
__device__ unsigned int g_fault_word;

namespace {

using namespace kivi_dev;

constexpr int kD = 128;            // head_dim
constexpr int kWarps = 4;
constexpr int kThreads = 32 * kWarps;
constexpr int kTile = 32;          // tokens per tile
constexpr float kPScale = 4096.0f; // P * 2^12 stays a normal fp16 down to P = 2^-26
constexpr uint64_t kWaitLimitNs = 200000000ull;  // 0.2 s per pipeline wait

// Shared-memory stage of one store tile (byte offsets).
template <int BITS, int G>
struct StageFmt {
  static constexpr int kKc = BITS * kD * 4;        // key codes: 32/W rows x D words
  static constexpr int kKs = kD * 4;               // key scale (or zero) row of the group
  static constexpr int kVc = BITS * kD * 4;        // value codes: 32 rows x D/W words
  static constexpr int kVs = kTile * (kD / G) * 4; // value scales (or zeros) of 32 tokens
  static constexpr int oKs = kKc, oKz = oKs + kKs, oVc = oKz + kKs, oVs = oVc + kVc,
                       oVz = oVs + kVs;
  static constexpr int kBytes = oVz + kVs;
  static constexpr int NS = BITS == 2 ? 3 : 2;     // stages per warp
  static constexpr int kSmem = kWarps * NS * kBytes + kWarps * NS * 8;
};

// 2^23 + q as a float, from the code at bit `pos` of w.
template <int BITS>
__device__ __forceinline__ float code_magic(uint32_t w, int pos) {
  if (BITS == 8) return __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7650u + (pos >> 3)));
  return __uint_as_float(((w >> pos) & ((1u << BITS) - 1u)) | 0x4B000000u);
}

// fp16 reconstructions of two codes (as 2^23 + q floats) with per-element
// (scale, -2^23 scale, zero): fp16(RN(RN(q scale) + zero)) -- the product
// formed inside an FMA with an exact addend (nothing for the compiler to
// contract), then a separately rounded add.
__device__ __forceinline__ uint32_t deq2(float m0, float m1, uint64_t s2, uint64_t ns2,
                                         uint64_t z2) {
  const uint64_t r = f2_add(f2_fma(f2_pack(m0, m1), s2, ns2), z2);
  return h2_as_u32(__floats2half2_rn(__uint_as_float(static_cast<uint32_t>(r)),
                                     __uint_as_float(static_cast<uint32_t>(r >> 32))));
}

__device__ __forceinline__ uint64_t neg2p23(float s0, float s1) {
  return f2_pack(__fmul_rn(s0, -8388608.0f), __fmul_rn(s1, -8388608.0f));
}

// Per-thread online-softmax state for heads 2t, 2t+1 (t = lane % 4).
struct SoftState {
  float m[2];
  float l[2];
  float o[8][4];  // O^T accumulators: channel block mc, (ch g, h 2t), (g, 2t+1), (g+8, 2t), (g+8, 2t+1)
};

// Key fragments of a store tile in shared memory.
template <int BITS, int G>
struct StoreKeys {
  const uint32_t *kc;
  const float *ks, *kz;
  int g, t;
  uint64_t s2a, ns2a, z2a, s2b, ns2b, z2b;
  __device__ __forceinline__ void prepare(int kk) {
    const int c0 = 16 * kk + 2 * t;
    const float2 sa = *reinterpret_cast<const float2 *>(ks + c0);
    const float2 sb = *reinterpret_cast<const float2 *>(ks + c0 + 8);
    const float2 za = *reinterpret_cast<const float2 *>(kz + c0);
    const float2 zb = *reinterpret_cast<const float2 *>(kz + c0 + 8);
    s2a = f2_pack(sa.x, sa.y);
    ns2a = neg2p23(sa.x, sa.y);
    z2a = f2_pack(za.x, za.y);
    s2b = f2_pack(sb.x, sb.y);
    ns2b = neg2p23(sb.x, sb.y);
    z2b = f2_pack(zb.x, zb.y);
  }
  // A fragment: tokens 16 mb + {g, g+8} x channels 16 kk + {2t, 2t+1, 2t+8, 2t+9}
  __device__ __forceinline__ void frag(int mb, int kk, uint32_t (&a)[4]) const {
    constexpr int W = 32 / BITS;
    const int c0 = 16 * kk + 2 * t;
    const int tau0 = 16 * mb + g, tau1 = tau0 + 8;
    const int r0 = tau0 / W, r1 = tau1 / W;
    const int p0 = (tau0 % W) * BITS, p1 = (tau1 % W) * BITS;
    const uint2 w0a = *reinterpret_cast<const uint2 *>(kc + r0 * kD + c0);
    const uint2 w0b = *reinterpret_cast<const uint2 *>(kc + r0 * kD + c0 + 8);
    uint2 w1a = w0a, w1b = w0b;
    if (r1 != r0) {
      w1a = *reinterpret_cast<const uint2 *>(kc + r1 * kD + c0);
      w1b = *reinterpret_cast<const uint2 *>(kc + r1 * kD + c0 + 8);
    }
    a[0] = deq2(code_magic<BITS>(w0a.x, p0), code_magic<BITS>(w0a.y, p0), s2a, ns2a, z2a);
    a[1] = deq2(code_magic<BITS>(w1a.x, p1), code_magic<BITS>(w1a.y, p1), s2a, ns2a, z2a);
    a[2] = deq2(code_magic<BITS>(w0b.x, p0), code_magic<BITS>(w0b.y, p0), s2b, ns2b, z2b);
    a[3] = deq2(code_magic<BITS>(w1b.x, p1), code_magic<BITS>(w1b.y, p1), s2b, ns2b, z2b);
  }
};

// Value fragments of a store tile in shared memory.
template <int BITS, int G>
struct StoreValues {
  const uint32_t *vc;
  const float *vs, *vz;
  int g, t;
  uint64_t s2a, ns2a, z2a, s2b, ns2b, z2b;   // tokens (2t, 2t+1) and (2t+8, 2t+9)
  int cur;                                    // (mb, group) of the loaded scales, -1: none
  __device__ __forceinline__ void prepare(int mb, int mc) {
    const int grp = 16 * mc / G;
    if (mb * 16 + grp == cur) return;
    cur = mb * 16 + grp;
    constexpr int NG = kD / G;
    const int ta = 16 * mb + 2 * t, tb = ta + 8;
    const float sa0 = vs[ta * NG + grp], sa1 = vs[(ta + 1) * NG + grp];
    const float sb0 = vs[tb * NG + grp], sb1 = vs[(tb + 1) * NG + grp];
    const float za0 = vz[ta * NG + grp], za1 = vz[(ta + 1) * NG + grp];
    const float zb0 = vz[tb * NG + grp], zb1 = vz[(tb + 1) * NG + grp];
    s2a = f2_pack(sa0, sa1);
    ns2a = neg2p23(sa0, sa1);
    z2a = f2_pack(za0, za1);
    s2b = f2_pack(sb0, sb1);
    ns2b = neg2p23(sb0, sb1);
    z2b = f2_pack(zb0, zb1);
  }
  // A fragment of V^T: channels 16 mc + {g, g+8} x tokens 16 mb + {2t, 2t+1, 2t+8, 2t+9}
  __device__ __forceinline__ void frag(int mb, int mc, uint32_t (&a)[4]) const {
    constexpr int W = 32 / BITS;
    constexpr int RW = kD / W;                 // words per token row
    const int c = 16 * mc + g, c8 = c + 8;
    const int wi = c / W, wi8 = c8 / W;
    const int pc = (c % W) * BITS, pc8 = (c8 % W) * BITS;
    const int ta = 16 * mb + 2 * t, tb = ta + 8;
    const uint32_t *row_a0 = vc + ta * RW, *row_a1 = row_a0 + RW;
    const uint32_t *row_b0 = vc + tb * RW, *row_b1 = row_b0 + RW;
    a[0] = deq2(code_magic<BITS>(row_a0[wi], pc), code_magic<BITS>(row_a1[wi], pc), s2a, ns2a, z2a);
    a[1] = deq2(code_magic<BITS>(row_a0[wi8], pc8), code_magic<BITS>(row_a1[wi8], pc8), s2a, ns2a,
                z2a);
    a[2] = deq2(code_magic<BITS>(row_b0[wi], pc), code_magic<BITS>(row_b1[wi], pc), s2b, ns2b, z2b);
    a[3] = deq2(code_magic<BITS>(row_b0[wi8], pc8), code_magic<BITS>(row_b1[wi8], pc8), s2b, ns2b,
                z2b);
  }
};

// Key / value fragments of a residual tile, read from the fp16 ring.
struct ResidualKV {
  const __half *kr, *vr;   // this bh slice of the rings
  int64_t r_cap, head;
  int tok0, valid;         // first logical residual token of the tile, valid tokens in it
  int g, t;
  __device__ __forceinline__ const __half *row(const __half *base, int tau) const {
    int64_t rr = head + tok0 + tau;
    rr %= r_cap;
    return base + rr * kD;
  }
  __device__ __forceinline__ uint32_t ld2(const __half *base, int tau, int c) const {
    if (tau >= valid) return 0u;
    return *reinterpret_cast<const uint32_t *>(row(base, tau) + c);
  }
  __device__ __forceinline__ uint32_t pair_tok(const __half *base, int tau, int c) const {
    // (x[tau][c], x[tau+1][c]) as a half2
    const unsigned short lo =
        tau < valid ? *reinterpret_cast<const unsigned short *>(row(base, tau) + c) : 0;
    const unsigned short hi =
        tau + 1 < valid ? *reinterpret_cast<const unsigned short *>(row(base, tau + 1) + c) : 0;
    return static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
  }
  __device__ __forceinline__ void prepare(int) {}
  __device__ __forceinline__ void prepare(int, int) {}
  __device__ __forceinline__ void kfrag(int mb, int kk, uint32_t (&a)[4]) const {
    const int c0 = 16 * kk + 2 * t;
    const int tau0 = 16 * mb + g, tau1 = tau0 + 8;
    a[0] = ld2(kr, tau0, c0);
    a[1] = ld2(kr, tau1, c0);
    a[2] = ld2(kr, tau0, c0 + 8);
    a[3] = ld2(kr, tau1, c0 + 8);
  }
  __device__ __forceinline__ void vfrag(int mb, int mc, uint32_t (&a)[4]) const {
    const int c = 16 * mc + g;
    const int ta = 16 * mb + 2 * t, tb = ta + 8;
    a[0] = pair_tok(vr, ta, c);
    a[1] = pair_tok(vr, ta, c + 8);
    a[2] = pair_tok(vr, tb, c);
    a[3] = pair_tok(vr, tb, c + 8);
  }
};

// Adapters so that attend_tile sees one interface.
template <typename K>
struct KeyAdapter {
  K &k;
  __device__ __forceinline__ void prepare(int kk) { k.prepare(kk); }
  __device__ __forceinline__ void frag(int mb, int kk, uint32_t (&a)[4]) const { k.frag(mb, kk, a); }
};
template <typename V>
struct ValueAdapter {
  V &v;
  __device__ __forceinline__ void prepare(int mb, int mc) { v.prepare(mb, mc); }
  __device__ __forceinline__ void frag(int mb, int mc, uint32_t (&a)[4]) const { v.frag(mb, mc, a); }
};
struct ResKeyAdapter {
  const ResidualKV &r;
  __device__ __forceinline__ void prepare(int) {}
  __device__ __forceinline__ void frag(int mb, int kk, uint32_t (&a)[4]) const { r.kfrag(mb, kk, a); }
};
struct ResValueAdapter {
  const ResidualKV &r;
  __device__ __forceinline__ void prepare(int, int) {}
  __device__ __forceinline__ void frag(int mb, int mc, uint32_t (&a)[4]) const { r.vfrag(mb, mc, a); }
};

// One tile of 32 tokens (the first `valid` of them real).
template <typename KA, typename VA>
__device__ __forceinline__ void attend_tile(SoftState &st, const uint32_t (&qf)[8][2],
                                            float scale_log2, int valid, KA ka, VA va, int g) {
  float s[2][4];
#pragma unroll
  for (int mb = 0; mb < 2; ++mb)
#pragma unroll
    for (int i = 0; i < 4; ++i) s[mb][i] = 0.0f;
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    ka.prepare(kk);
#pragma unroll
    for (int mb = 0; mb < 2; ++mb) {
      uint32_t a[4];
      ka.frag(mb, kk, a);
      mma_16816(s[mb], a, qf[kk][0], qf[kk][1]);
    }
  }
  // scale (log2 units), mask, tile maximum per head column
  float mt[2] = {-INFINITY, -INFINITY};
#pragma unroll
  for (int mb = 0; mb < 2; ++mb)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int tok = 16 * mb + g + (i >= 2 ? 8 : 0);
      const float v = tok < valid ? s[mb][i] * scale_log2 : -INFINITY;
      s[mb][i] = v;
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
  // probabilities (x 2^12) as fp16 high + low parts, transposed into B fragments
  uint32_t phi[2][2], plo[2][2];
  float lsum[2] = {0.0f, 0.0f};
#pragma unroll
  for (int mb = 0; mb < 2; ++mb) {
    float p[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float m = mn[i & 1];
      p[i] = m == -INFINITY ? 0.0f : exp2f(s[mb][i] - m) * kPScale;
      lsum[i & 1] += p[i];
    }
    const __half2 h0 = __floats2half2_rn(p[0], p[1]);   // token g: heads 2t, 2t+1
    const __half2 h1 = __floats2half2_rn(p[2], p[3]);   // token g+8
    const __half2 l0 = __floats2half2_rn(p[0] - __low2float(h0), p[1] - __high2float(h0));
    const __half2 l1 = __floats2half2_rn(p[2] - __low2float(h1), p[3] - __high2float(h1));
    phi[mb][0] = movmatrix_trans(h2_as_u32(h0));
    phi[mb][1] = movmatrix_trans(h2_as_u32(h1));
    plo[mb][0] = movmatrix_trans(h2_as_u32(l0));
    plo[mb][1] = movmatrix_trans(h2_as_u32(l1));
  }
#pragma unroll
  for (int j = 0; j < 2; ++j) st.l[j] = st.l[j] * alpha[j] + lsum[j];
#pragma unroll
  for (int mc = 0; mc < 8; ++mc) {
    st.o[mc][0] *= alpha[0];
    st.o[mc][1] *= alpha[1];
    st.o[mc][2] *= alpha[0];
    st.o[mc][3] *= alpha[1];
  }
#pragma unroll
  for (int mb = 0; mb < 2; ++mb)
#pragma unroll
    for (int mc = 0; mc < 8; ++mc) {
      va.prepare(mb, mc);
      uint32_t a[4];
      va.frag(mb, mc, a);
      mma_16816(st.o[mc], a, phi[mb][0], phi[mb][1]);
      mma_16816(st.o[mc], a, plo[mb][0], plo[mb][1]);
    }
}

template <int BITS, int G>
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

  // query heads kvh*r .. kvh*r + r-1 as B fragments (k = channels, n = heads)
  uint32_t qf[8][2];
  {
    const __half *q = static_cast<const __half *>(J.q) + (b * h_q + kvh * p.r + g) * kD;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const int c0 = 16 * kk + 2 * t;
      qf[kk][0] = g < p.r ? *reinterpret_cast<const uint32_t *>(q + c0) : 0u;
      qf[kk][1] = g < p.r ? *reinterpret_cast<const uint32_t *>(q + c0 + 8) : 0u;
    }
  }
  SoftState st;
  st.m[0] = st.m[1] = -INFINITY;
  st.l[0] = st.l[1] = 0.0f;
#pragma unroll
  for (int mc = 0; mc < 8; ++mc)
#pragma unroll
    for (int i = 0; i < 4; ++i) st.o[mc][i] = 0.0f;

  // ---- store tiles through the warp's shared-memory ring
  const int st0 = split * p.tiles_per_split;
  const int st1 = min(st0 + p.tiles_per_split, p.tiles_store);
  const int n_my = st1 - st0 > warp ? (st1 - st0 - warp + kWarps - 1) / kWarps : 0;
  unsigned char *ring = smem + warp * F::NS * F::kBytes;
  const uint32_t bar0 = smem_addr(smem + kWarps * F::NS * F::kBytes) + warp * F::NS * 8;
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
    fence_proxy_async_smem();
    mbar_arrive_expect_tx(bar, F::kBytes);
    bulk_load(dst, kc_bh + (tok / W) * kD, F::kKc, bar, pol);
    bulk_load(dst + F::oKs, ks_bh + (tok / G) * kD, F::kKs, bar, pol);
    bulk_load(dst + F::oKz, kz_bh + (tok / G) * kD, F::kKs, bar, pol);
    bulk_load(dst + F::oVc, vc_bh + tok * (kD / W), F::kVc, bar, pol);
    bulk_load(dst + F::oVs, vs_bh + tok * (kD / G), F::kVs, bar, pol);
    bulk_load(dst + F::oVz, vz_bh + tok * (kD / G), F::kVs, bar, pol);
  };
  int issued = 0;
  if (lane == 0)
    for (; issued < min(F::NS, n_my); ++issued) issue(issued);
  issued = __shfl_sync(0xffffffffu, issued, 0);

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
    StoreKeys<BITS, G> kf{reinterpret_cast<const uint32_t *>(stg),
                          reinterpret_cast<const float *>(stg + F::oKs),
                          reinterpret_cast<const float *>(stg + F::oKz), g, t};
    StoreValues<BITS, G> vf{reinterpret_cast<const uint32_t *>(stg + F::oVc),
                            reinterpret_cast<const float *>(stg + F::oVs),
                            reinterpret_cast<const float *>(stg + F::oVz), g, t};
    vf.cur = -1;
    attend_tile(st, qf, p.scale_log2, kTile, KeyAdapter<StoreKeys<BITS, G>>{kf},
                ValueAdapter<StoreValues<BITS, G>>{vf}, g);
    __syncwarp();
    if (issued < n_my) {
      if (lane == 0) issue(issued);
      ++issued;
    }
  }
  if (failed) {
    // record the timeout and wait (bounded) for this warp's copies still in flight
    if (lane == 0) atomicOr(&g_fault_word, 1u);
#pragma unroll 1
    for (int i = done; i < issued; ++i)
      mbar_wait_bounded(bar0 + 8 * (i % F::NS), (i / F::NS) & 1, kWaitLimitNs);
  }

  // ---- residual tiles (last split): fp16 rows read directly
  if (split == p.n_split - 1 && !failed) {
    const __half *kr = static_cast<const __half *>(J.k_res) + bhi * p.r_cap * kD;
    const __half *vr = static_cast<const __half *>(J.v_res) + bhi * p.r_cap * kD;
#pragma unroll 1
    for (int j = warp; j < p.tiles_res; j += kWarps) {
      const int tok0 = j * kTile;
      const int64_t left = p.n_res - tok0;
      const int valid = left < kTile ? static_cast<int>(left) : kTile;
      ResidualKV rk{kr, vr, p.r_cap, p.res_head, tok0, valid, g, t};
      attend_tile(st, qf, p.scale_log2, valid, ResKeyAdapter{rk}, ResValueAdapter{rk}, g);
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
#pragma unroll
  for (int mc = 0; mc < 8; ++mc) {
    float *o0 = red_o + (warp * 8 + 2 * t) * kD + 16 * mc + g;
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

int g_num_sms = 0;
int num_sms() {
  if (g_num_sms == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    g_num_sms = n > 0 ? n : 1;
  }
  return g_num_sms;
}

template <int BITS, int G>
cudaError_t attention_launch(const AttnParams &p, cudaStream_t stream) {
  using F = StageFmt<BITS, G>;
  auto kern = decode_attention_kernel<BITS, G>;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, F::kSmem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const int64_t items = static_cast<int64_t>(p.n_jobs) * p.bh * p.n_split;
  kern<<<static_cast<unsigned>(items), kThreads, F::kSmem, stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || p.n_split == 1) return e;
  const int64_t blocks = static_cast<int64_t>(p.n_jobs) * p.bh * p.r;
  attention_combine_kernel<<<static_cast<unsigned>(blocks), kD, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_attention(const AttnParams &p, int group, int bits, cudaStream_t stream) {
  switch (bits * 1000 + group) {
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
  const int64_t target = static_cast<int64_t>(num_sms()) * 4 * 2;   // two waves of 4 CTAs per SM
  const int64_t want = (target + items - 1) / items;
  const int64_t most = std::max<int64_t>(1, std::min<int64_t>(64, tiles_store / (2 * kWarps)));
  return static_cast<int>(std::max<int64_t>(1, std::min(want, most)));
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
