// kivi_values.cu -- per-token value quantization and value dequantization.
//
// Values are grouped along the contiguous head_dim axis: one (scale, zero)
// per token per group of G channels (VeloxQuant-MLX KIVI fused-kernel post,
// "The layout problem that shapes everything").  One thread owns 32
// consecutive channels of one token (four 16-byte loads); a group of G >= 32
// channels is a sub-warp of G/32 lanes, reduced with __shfl_xor_sync on the
// packed half2 {min, -max} (one shuffle per step carries both extremes), and
// at G = 16 a thread holds two whole groups.
// Codes are packed along channels in registers and written with one 8- or
// 16-byte store per word group.
//
// The grid is persistent (a multiple of the SM count times the resident
// blocks per SM) and every warp walks the units in warp-aligned steps, so
// the lanes of a group are always together and inactive tail lanes still
// take part in the shuffles.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "kivi_device.cuh"
#include "kivi_expand.cuh"
#include "kivi_launch.h"

namespace kivi_impl {
namespace {

using namespace kivi_dev;

struct RowRef {
  int job;
  uint32_t b;
  uint32_t r;
  uint32_t k;  // 32-channel chunk within the row
};

// unit = ((job * bh + b) * rows + r) * chunks + k   (all < 2^31, host-checked);
// DC > 0: head_dim DC known at compile time, chunks = DC / 32
template <int DC = 0, typename P>
__device__ __forceinline__ RowRef decode_unit(uint32_t u, const P &p) {
  RowRef t;
  uint32_t row;
  if constexpr (DC > 0 && ((DC / 32) & (DC / 32 - 1)) == 0) {   // a power of two
    constexpr uint32_t CH = DC / 32;
    row = u / CH;
    t.k = u % CH;
  } else {
    row = p.div_chunks.div(u);
    t.k = u - row * p.div_chunks.d;
  }
  const uint32_t jb = p.div_rows.div(row);
  t.r = row - jb * p.div_rows.d;
  const uint32_t job = p.div_bh.div(jb);
  t.b = jb - job * p.div_bh.d;
  t.job = static_cast<int>(job);
  return t;
}

// Coalesced store of a warp's 32 units of 64 bytes (32 fp16 each): each lane
// parks its unit in a per-warp shared-memory block, and each 16-byte store
// instruction of the warp then writes 512 consecutive bytes: lane l stores
// chunk l + 32 i of the block, whose destination is that of unit (l + 32 i)
// / 4, taken from the owning lane by a shuffle.  Chunk c of unit u sits at
// slot 4 u + (c ^ ((u >> 1) & 3)): in every 8-lane phase the writes (8 units,
// one chunk each) and the reads (2 units, 4 chunks each) then touch 8
// distinct 16-byte bank groups (a padded stride serves only one of the two
// patterns).  All 32 lanes must call it; `valid` marks lanes whose unit
// exists (their `out` and `dst` are used).
constexpr int kUnitWords = 16;   // 64 bytes per unit, no padding
constexpr int kBlockThreads = 256;

__device__ __forceinline__ uint32_t unit_slot(uint32_t u, uint32_t c) {
  return u * kUnitWords + 4u * (c ^ ((u >> 1) & 3u));
}

__device__ __forceinline__ void warp_store_units(uint32_t *blk, uint32_t lane, bool valid,
                                                 const uint32_t (&out)[16], __half *dst,
                                                 uint32_t base, uint32_t total) {
  if (valid) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
      *reinterpret_cast<uint4 *>(blk + unit_slot(lane, i)) =
          make_uint4(out[4 * i], out[4 * i + 1], out[4 * i + 2], out[4 * i + 3]);
  }
  __syncwarp();
  const unsigned long long dbits = reinterpret_cast<unsigned long long>(dst);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t j = lane + 32u * i;      // chunk of the warp block
    const uint32_t owner = j >> 2;          // unit (lane) that produced it
    const unsigned long long d = __shfl_sync(0xffffffffu, dbits, owner);
#ifdef KIVI_DEBUG_BOUNDS
    const bool owner_valid = __shfl_sync(0xffffffffu, valid ? 1 : 0, owner) != 0;
#else
    constexpr bool owner_valid = true;      // valid == (the lane's unit exists)
#endif
    if (base + owner < total && owner_valid) {
      const uint4 v = *reinterpret_cast<const uint4 *>(blk + unit_slot(owner, j & 3u));
      st_stream(reinterpret_cast<__half *>(d) + 8 * (j & 3), v);
    }
  }
  __syncwarp();
}

// PF: the next unit's four loads are issued before the current unit is
// quantized (one more unit of loads in flight per thread, at three resident
// blocks per SM instead of four): faster on large flushes, slower on small
// ones (see value_quant_launch).
template <int BITS, int G, int DC, int MODE, bool PF>
__global__ void __launch_bounds__(kBlockThreads, PF ? 3 : 4)
    value_quant_kernel(const __grid_constant__ QuantParams p) {
  // a launch whose inputs do not depend on the previous grid in the stream
  // (defer_wait) starts at once and waits for it only before it ends
  if (!p.defer_wait) kivi_dev::grid_dependency_wait();
  kivi_dev::grid_launch_dependents();
  constexpr bool RECON = MODE == kQuantRecon;
  constexpr bool SINK = MODE == kQuantSink;
  constexpr int L = G < 32 ? 1 : G / 32;  // lanes per group
  constexpr int SUB = G < 32 ? 32 / G : 1; // groups per thread
  constexpr int W = CodeFmt<BITS>::W;
  constexpr uint32_t Q = CodeFmt<BITS>::Q;
  const float qf = static_cast<float>(Q);

  const int D = DC > 0 ? DC : p.d;          // head_dim, compile-time when DC > 0
  const uint32_t total = static_cast<uint32_t>(p.n_jobs) * static_cast<uint32_t>(p.bh) *
                         static_cast<uint32_t>(p.rows) * p.div_chunks.d;
  const uint32_t lane = threadIdx.x & 31u;
  const uint32_t stride = gridDim.x * blockDim.x;
  __shared__ __align__(16) uint32_t stage[RECON ? kBlockThreads / 32 : 1]
                                         [RECON ? 32 * kUnitWords : 4];
  uint32_t *blk = stage[RECON ? (threadIdx.x >> 5) : 0];

  // the unit of the warp step starting at b0: its row reference and its 64
  // input bytes (zero for a lane past the end)
  RowRef tn;
  uint4 vn[4];
  bool an = false;
  auto fetch = [&](uint32_t b0) {
    const uint32_t u = b0 + lane;
    an = u < total;
    tn = decode_unit<DC>(an ? u : b0, p);
    int64_t phys = tn.r;
    if (p.ring > 0) {
      phys += p.head;
      if (phys >= p.ring) phys -= p.ring;  // head < ring and r < ring
    }
    const __half *src = static_cast<const __half *>(p.jobs[tn.job].x) + tn.b * p.x_bh_stride +
                        phys * D + tn.k * 32;
    // debug builds: the unit's input lies inside its bh slice
    const bool x_ok =
        KIVI_BOUND(p.fault, !an || (tn.b < p.bh && phys * D + tn.k * 32 + 32 <= p.x_bh_stride));
#pragma unroll
    for (int i = 0; i < 4; ++i) vn[i] = make_uint4(0u, 0u, 0u, 0u);
    if (an && x_ok) {
#pragma unroll
      for (int i = 0; i < 4; ++i) vn[i] = ld_stream(src + 8 * i);
    }
  };
  const uint32_t base0 = (blockIdx.x * blockDim.x + threadIdx.x) & ~31u;
  if (PF && base0 < total) fetch(base0);
#pragma unroll 1
  for (uint32_t base = base0; base < total; base += stride) {
    if (!PF) fetch(base);
    const bool active = an;
    const RowRef t = tn;
    const uint4 v[4] = {vn[0], vn[1], vn[2], vn[3]};
    if (PF && base + stride < total) fetch(base + stride);
    const QuantJob &job = p.jobs[t.job];
    __half2 h[16];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      h[4 * i + 0] = u32_as_h2(v[i].x);
      h[4 * i + 1] = u32_as_h2(v[i].y);
      h[4 * i + 2] = u32_as_h2(v[i].z);
      h[4 * i + 3] = u32_as_h2(v[i].w);
    }

    // min / max of each group's channels (tree in half2 over the group's
    // 8 / SUB slots of four channels, then the two halves)
    __half2 mn2[8], mx2[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      mn2[i] = __hmin2(h[2 * i], h[2 * i + 1]);
      mx2[i] = __hmax2(h[2 * i], h[2 * i + 1]);
    }
    // {min, -max}: a single element-wise min combines both extremes
    __half2 ext[SUB];
#pragma unroll
    for (int sg = 0; sg < SUB; ++sg) {
      const int i0 = sg * (8 / SUB);
#pragma unroll
      for (int w = 4 / SUB; w >= 1; w >>= 1) {
#pragma unroll
        for (int i = 0; i < w; ++i) {
          mn2[i0 + i] = __hmin2(mn2[i0 + i], mn2[i0 + i + w]);
          mx2[i0 + i] = __hmax2(mx2[i0 + i], mx2[i0 + i + w]);
        }
      }
      const __half mn = __hmin(__low2half(mn2[i0]), __high2half(mn2[i0]));
      const __half mx = __hmax(__low2half(mx2[i0]), __high2half(mx2[i0]));
      ext[sg] = __halves2half2(mn, __hneg(mx));
    }
    if (L > 1) {
#pragma unroll
      for (int off = 1; off < L; off <<= 1) {
        const uint32_t other = __shfl_xor_sync(0xffffffffu, h2_as_u32(ext[0]), off);
        ext[0] = __hmin2(ext[0], u32_as_h2(other));
      }
    }
    __half *ydst = RECON ? static_cast<__half *>(job.y) + t.b * p.y_bh_stride +
                               (p.y_row0 + static_cast<int64_t>(t.r)) * D + t.k * 32
                         : nullptr;
    const bool y_ok = KIVI_BOUND(
        p.fault, !RECON || !active ||
                     (p.y_row0 + static_cast<int64_t>(t.r)) * D + t.k * 32 + 32 <= p.y_bh_stride);
    if (!RECON && !active) continue;
    uint32_t out[16];  // reconstruction of the 32 channels (RECON)
    if (active) {
      float gmn[SUB], gmx[SUB];
#pragma unroll
      for (int sg = 0; sg < SUB; ++sg) {
        gmn[sg] = __low2float(ext[sg]);
        gmx[sg] = -__high2float(ext[sg]);
      }
      const int64_t out_row = p.out0 + t.r;
      const bool codes_out =
          (!RECON || job.codes != nullptr) &&
          KIVI_BOUND(p.fault, out_row * (D / W) + t.k * BITS + BITS <= p.codes_bh_stride &&
                                  out_row * (D / G) + t.k * SUB / L + SUB <= p.sz_bh_stride);
      // (scale, zero) of this thread's first group: row out_row, entry k SUB / L
      const int64_t so = t.b * p.sz_bh_stride + out_row * (D / G) + t.k * SUB / L;
      // sink mode: a sink token's row is not quantized (codes, scales, zeros 0)
      if (SINK && ((job.mask[static_cast<int64_t>(t.b / p.heads) * p.mask_words + (t.r >> 5)] >>
                    (t.r & 31)) & 1u)) {
        if (!codes_out) continue;
        if (t.k % L == 0) {
#pragma unroll
          for (int sg = 0; sg < SUB; ++sg) {
            __stcs(job.scale + so + sg, 0.0f);
            __stcs(job.zero + so + sg, 0.0f);
          }
        }
        uint32_t *dst = job.codes + t.b * p.codes_bh_stride + out_row * (D / W) + t.k * BITS;
        if (BITS == 2) {
          st_stream(dst, make_uint2(0u, 0u));
        } else {
#pragma unroll
          for (int i = 0; i < BITS; i += 4) st_stream(dst + i, make_uint4(0u, 0u, 0u, 0u));
        }
        continue;
      }
      GroupD2 gq[SUB];
      float gsc[SUB], gze[SUB];
      uint64_t sc2[SUB], nsc2[SUB], ze2[SUB];
#pragma unroll
      for (int sg = 0; sg < SUB; ++sg) {
        const GroupQ g = make_group_szr(gmn[sg], gmx[sg], qf);
        gq[sg] = make_group_d2(g, g);
        gsc[sg] = g.scale;
        gze[sg] = g.zero;
        sc2[sg] = nsc2[sg] = ze2[sg] = 0;
        if (RECON) {
          sc2[sg] = f2_pack(g.scale, g.scale);
          nsc2[sg] = neg_scale_2p23_pair(g.scale, g.scale);
          ze2[sg] = f2_pack(g.zero, g.zero);
        }
        if (t.k % L == 0 && codes_out) {
          __stcs(job.scale + so + sg, g.scale);
          __stcs(job.zero + so + sg, g.zero);
        }
      }

      // Pack along channels: word wi holds channels [wi*W, wi*W + W) of this
      // thread's 32 (all in group sg = wi W / G when SUB = 2, as W <= 16).  A
      // half-word (H = 16/BITS channels) accumulates its H/2 channel pairs
      // with packed FMAs by powers of two, which leaves even channels in the
      // low and odd channels in the high element; one more FMA interleaves
      // them.
      constexpr int H = 16 / BITS;
      uint32_t w[BITS];
#pragma unroll
      for (int wi = 0; wi < BITS; ++wi) {
        const int sg = SUB == 1 ? 0 : (wi * W) / G;
        uint64_t acc[2];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int p0 = (wi * W + hh * H) / 2;   // first channel pair of the half
          uint32_t neg_acc = 0xFFFFFFFFu;
          uint64_t n[H / 2];
#pragma unroll
          for (int j = 0; j < H / 2; ++j)
            n[j] = codes2_diff_nobranch<BITS>(h2_as_u32(h[p0 + j]), gq[sg], neg_acc);
          if (!(neg_acc >> 31)) {  // rare: redo this half pair by pair, exactly where needed
#pragma unroll
            for (int j = 0; j < H / 2; ++j)
              n[j] = codes2_diff<BITS>(h2_as_u32(h[p0 + j]), gq[sg], gsc[sg], gze[sg], gsc[sg],
                                       gze[sg], qf);
          }
          acc[hh] = n[0];
#pragma unroll
          for (int j = 1; j < H / 2; ++j)
            acc[hh] = f2_fma(n[j], f2_const(static_cast<float>(1u << (2 * BITS * j))), acc[hh]);
          if (RECON) {
#pragma unroll
            for (int j = 0; j < H / 2; ++j)
              out[p0 + j] = recon_pair(n[j], sc2[sg], nsc2[sg], ze2[sg]);
          }
        }
        // even channels (low) + odd channels (high) shifted by one code
        float half[2];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
          half[hh] = __fmaf_rn(__uint_as_float(f2_hi_bits(acc[hh])), static_cast<float>(1u << BITS),
                               __uint_as_float(f2_lo_bits(acc[hh])));
        w[wi] = join_halves(half[0], half[1]);
      }

      if (codes_out) {
        uint32_t *dst = job.codes + t.b * p.codes_bh_stride + out_row * (D / W) + t.k * BITS;
        if (BITS == 2) {
          st_stream(dst, make_uint2(w[0], w[1 % BITS]));
        } else {
#pragma unroll
          for (int i = 0; i < BITS; i += 4)
            st_stream(dst + i, make_uint4(w[i % BITS], w[(i + 1) % BITS], w[(i + 2) % BITS],
                                          w[(i + 3) % BITS]));
        }
      }
    }  // active
    if (RECON) warp_store_units(blk, lane, active && y_ok, out, ydst, base, total);
  }
  if (p.defer_wait) kivi_dev::grid_dependency_wait();
}

// Dequantize: a thread reconstructs the 32 channels of one (row, chunk) unit
// (codes, scale and zero read with 8/16-byte and 4-byte loads) and the warp
// writes its 32 units with warp_store_units.
template <int BITS, int G, int DC>
__global__ void __launch_bounds__(kBlockThreads)
    value_dequant_kernel(const __grid_constant__ DequantParams p) {
  // a launch whose inputs do not depend on the previous grid in the stream
  // (defer_wait) starts at once and waits for it only before it ends
  if (!p.defer_wait) kivi_dev::grid_dependency_wait();
  kivi_dev::grid_launch_dependents();
  constexpr int L = G < 32 ? 1 : G / 32;  // lanes per group
  constexpr int SUB = G < 32 ? 32 / G : 1; // groups per thread
  constexpr int W = CodeFmt<BITS>::W;
  const int D = DC > 0 ? DC : p.d;
  const uint32_t total = static_cast<uint32_t>(p.n_jobs) * static_cast<uint32_t>(p.bh) *
                         static_cast<uint32_t>(p.rows) * p.div_chunks.d;
  const uint32_t lane = threadIdx.x & 31u;
  const uint32_t stride = gridDim.x * blockDim.x;
  __shared__ __align__(16) uint32_t stage[kBlockThreads / 32][32 * kUnitWords];
  uint32_t *blk = stage[threadIdx.x >> 5];

#pragma unroll 1
  for (uint32_t base = (blockIdx.x * blockDim.x + threadIdx.x) & ~31u; base < total;
       base += stride) {
    const uint32_t u = base + lane;
    const bool active = u < total;
    const RowRef t = decode_unit(active ? u : base, p);
    const DequantJob &J = p.jobs[t.job];
    __half *y = static_cast<__half *>(J.y) + t.b * p.y_bh_stride + static_cast<int64_t>(t.r) * D +
                t.k * 32;
    uint32_t out[16];
    // debug builds: the unit's reads and its output row lie inside its bh slice
    const bool ok = KIVI_BOUND(
        p.fault, !active || (t.b < p.bh &&
                             static_cast<int64_t>(t.r) * (D / W) + t.k * BITS + BITS <=
                                 p.codes_bh_stride &&
                             static_cast<int64_t>(t.r) * (D / G) + t.k * SUB / L + SUB <=
                                 p.sz_bh_stride &&
                             static_cast<int64_t>(t.r) * D + t.k * 32 + 32 <= p.y_bh_stride));
    if (active && ok) {
      const uint32_t *src = J.codes + t.b * p.codes_bh_stride +
                            static_cast<int64_t>(t.r) * (D / W) + t.k * BITS;
      uint32_t w[BITS];
      if (BITS == 2) {
        const uint2 a = __ldcs(reinterpret_cast<const uint2 *>(src));
        w[0] = a.x;
        w[1 % BITS] = a.y;
      } else {
#pragma unroll
        for (int i = 0; i < BITS; i += 4) {
          const uint4 a = ld_stream(src + i);
          w[i % BITS] = a.x;
          w[(i + 1) % BITS] = a.y;
          w[(i + 2) % BITS] = a.z;
          w[(i + 3) % BITS] = a.w;
        }
      }
      const int64_t so =
          t.b * p.sz_bh_stride + static_cast<int64_t>(t.r) * (D / G) + t.k * SUB / L;
      float sc[SUB], ze[SUB], nsc[SUB];
#pragma unroll
      for (int sg = 0; sg < SUB; ++sg) {
        sc[sg] = __ldcs(J.scale + so + sg);
        ze[sg] = __ldcs(J.zero + so + sg);
        nsc[sg] = __fmul_rn(sc[sg], -8388608.0f);  // -2^23 * scale, exact
      }
      if constexpr (BITS == 2) {
        // The four possible fp16 reconstructions of a group (codes 0..3, the
        // same arithmetic as below) as an 8-byte table in two registers;
        // code q is bytes 2q, 2q + 1, and a byte permute picks two codes'
        // values at once.  Four codes (one byte of a word) are spread one to
        // a byte, and q * 0x22 + 0x10 gives the nibble pair (2q, 2q + 1):
        // the permute selectors of channels (4k, 4k + 1) in the low half and
        // (4k + 2, 4k + 3) in the high half.
        uint32_t lo[SUB], hi[SUB];
#pragma unroll
        for (int sg = 0; sg < SUB; ++sg) {
          lo[sg] = h2_as_u32(__floats2half2_rn(recon_f32(0u, sc[sg], nsc[sg], ze[sg]),
                                               recon_f32(1u, sc[sg], nsc[sg], ze[sg])));
          hi[sg] = h2_as_u32(__floats2half2_rn(recon_f32(2u, sc[sg], nsc[sg], ze[sg]),
                                               recon_f32(3u, sc[sg], nsc[sg], ze[sg])));
        }
#pragma unroll
        for (int i = 0; i < 2; ++i) {              // word i: channels 16 i .. 16 i + 15
          const int sg = SUB == 1 ? 0 : i;         // at G = 16 a word is one group
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint32_t bt = (w[i] >> (8 * k)) & 0xFFu;
            uint32_t x = (bt | (bt << 12)) & 0x000F000Fu;
            x = (x | (x << 6)) & 0x03030303u;      // code 4k + j in byte j
            const uint32_t sel = x * 0x22u + 0x10101010u;
            out[8 * i + 2 * k] = __byte_perm(lo[sg], hi[sg], sel);
            out[8 * i + 2 * k + 1] = __byte_perm(lo[sg], hi[sg], sel >> 16);
          }
        }
      } else if constexpr (BITS == 4) {
        // 16 channels at a time (one group at G = 16): the codes spread
        // under the exponent of 2^23 by byte permutes, then the same
        // reconstruction on packed pairs (kivi_expand.cuh) -- 12-16% faster
        // than the per-element form below at 4 bits, 0.3-0.6% slower at 8
#pragma unroll
        for (int cb = 0; cb < 2; ++cb) {
          const int sg = SUB == 1 ? 0 : cb;
          uint64_t s2, ns2, z2;
          scale_consts(sc[sg], ze[sg], s2, ns2, z2);
          float m[16];
          magics16<BITS>(w + cb * (16 / W), m);
          const uint4 a = deq8(m, s2, ns2, z2), b = deq8(m + 8, s2, ns2, z2);
          out[8 * cb + 0] = a.x;
          out[8 * cb + 1] = a.y;
          out[8 * cb + 2] = a.z;
          out[8 * cb + 3] = a.w;
          out[8 * cb + 4] = b.x;
          out[8 * cb + 5] = b.y;
          out[8 * cb + 6] = b.z;
          out[8 * cb + 7] = b.w;
        }
      } else {
        constexpr uint32_t Q = CodeFmt<BITS>::Q;
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const int sg = SUB == 1 ? 0 : e / G;     // channels e, e + 1 share a group
          const uint32_t q0 = (w[e / W] >> ((e % W) * BITS)) & Q;
          const uint32_t q1 = (w[(e + 1) / W] >> (((e + 1) % W) * BITS)) & Q;
          const float r0 = recon_f32(q0, sc[sg], nsc[sg], ze[sg]);
          const float r1 = recon_f32(q1, sc[sg], nsc[sg], ze[sg]);
          out[e >> 1] = h2_as_u32(__floats2half2_rn(r0, r1));
        }
      }
    }
    warp_store_units(blk, lane, active && ok, out, y, base, total);
  }
  if (p.defer_wait) kivi_dev::grid_dependency_wait();
}


template <typename K>
cudaError_t persistent_grid(K kern, int threads, int64_t units, int64_t *grid) {
  int per_sm = 0;
  cudaError_t err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, 0);
  if (err != cudaSuccess) return err;
  if (per_sm < 1) per_sm = 1;
  const int64_t blocks = (units + threads - 1) / threads;
  *grid = std::max<int64_t>(1, std::min<int64_t>(blocks, static_cast<int64_t>(current_sm_count()) * per_sm));
  return cudaSuccess;
}

template <typename P>
P with_dividers(const P &p) {
  P q = p;
  q.div_chunks = FastDiv::make(static_cast<uint32_t>(p.d / 32));
  q.div_rows = FastDiv::make(static_cast<uint32_t>(p.rows));
  q.div_bh = FastDiv::make(static_cast<uint32_t>(p.bh));
  return q;
}

template <int BITS, int G, int DC, int MODE, bool PF>
cudaError_t value_quant_launch_pf(const QuantParams &p, cudaStream_t stream) {
  const int threads = kBlockThreads;
  auto kern = value_quant_kernel<BITS, G, DC, MODE, PF>;
  const int64_t units = static_cast<int64_t>(p.n_jobs) * p.bh * p.rows * (p.d / 32);
  int64_t grid = 0;
  cudaError_t err = persistent_grid(kern, threads, units, &grid);
  if (err != cudaSuccess) return err;
  // Three waves of resident blocks, by measurement over bits x G and the
  // model-shaped stores: 1-3% faster than one wave (which leaves each block
  // a long fixed stride) and than one block per 256 units, except for the
  // fused reconstruction at G = 16, where the flat grid is 12% faster.
  const int64_t flat = flat_grid(units, threads);
  grid = (MODE == kQuantRecon && G == 16) ? flat : std::min<int64_t>(flat, 3 * grid);
  QuantParams q = with_dividers(p);
  err = debug_fault_word(&q.fault);
  if (err != cudaSuccess) return err;
  return launch_dependent(kern, grid, threads, stream, q);
}

// Plain quantization at head_dim 128 of at least 3 x 2^20 units takes the
// prefetching kernel: measured 3-4% faster on a 28-layer x 4-head x 32 K-token
// flush (14.6 M units) and on the store sweep (8.4 M), 1% on a 28-layer x
// 8-head x 4 K-token flush (3.6 M); a 32-token decode flush of 32 layers x
// 512 heads (2.1 M units) measured 3.5% slower with it.
constexpr int64_t kPrefetchUnits = int64_t{3} << 20;

template <int BITS, int G, int DC, int MODE>
cudaError_t value_quant_launch(const QuantParams &p, cudaStream_t stream) {
  if constexpr (MODE == kQuantPlain && DC == 128) {
    const int64_t units = static_cast<int64_t>(p.n_jobs) * p.bh * p.rows * (p.d / 32);
    if (units >= kPrefetchUnits) return value_quant_launch_pf<BITS, G, DC, MODE, true>(p, stream);
  }
  return value_quant_launch_pf<BITS, G, DC, MODE, false>(p, stream);
}

// The dequantize kernels take one block per kBlockThreads units rather than a
// persistent grid: with every block's loads issued once and retired, the reads
// of the packed store spread over the memory partitions better than a fixed
// grid striding the same pattern (measured +6-10% on the value and key
// dequantize of 28-layer and 64-head stores).  The loop stays grid-stride, so
// the clamp to the launch limit keeps it correct at any size.
template <int BITS, int G, int DC>
cudaError_t value_dequant_launch(const DequantParams &p, cudaStream_t stream) {
  const int threads = kBlockThreads;
  auto kern = value_dequant_kernel<BITS, G, DC>;
  const int64_t units = static_cast<int64_t>(p.n_jobs) * p.bh * p.rows * (p.d / 32);
  const int64_t grid = flat_grid(units, threads);
  DequantParams q = with_dividers(p);
  const cudaError_t e = debug_fault_word(&q.fault);
  if (e != cudaSuccess) return e;
  return launch_dependent(kern, grid, threads, stream, q);
}

}  // namespace

#include "kivi_dispatch.h"

cudaError_t launch_value_quant(const QuantParams &p, int group, int bits, int mode,
                               cudaStream_t stream) {
  KIVI_DISPATCH_MODE(value_quant_launch, p, group, bits, mode, stream);
}

cudaError_t launch_value_dequant(const DequantParams &p, int group, int bits,
                                 cudaStream_t stream) {
  KIVI_DISPATCH(value_dequant_launch, p, group, bits, stream);
}

}  // namespace kivi_impl
