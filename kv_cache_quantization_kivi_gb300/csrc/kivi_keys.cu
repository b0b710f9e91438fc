// kivi_keys.cu -- per-channel key quantization and key dequantization.
//
// Keys are grouped along the token axis: one (scale, zero) per channel per
// group of G tokens (VeloxQuant-MLX KIVI fused-kernel post, "The layout
// problem that shapes everything": the group runs along the strided axis,
// consecutive group elements are d apart).
//
// Quantize: as in the post's "Kernel A", a thread owns whole columns of a
// group, so the reduction over tokens happens in registers and a warp's loads
// are coalesced along d; no transpose is materialised and no shared memory or
// barrier is needed.  Here a thread owns a channel pair (half2) and
// min(G, 32) tokens (a whole group at G = 16); for G = 64 and 128 the G/32
// threads of a column are adjacent lanes that combine their extremes with
// two-step shuffles.  The arithmetic is the
// difference-first fast path of kivi_device.cuh with the exact-division
// fallback; codes are packed along tokens in registers and stored as 8-byte
// words pairs.  The plain quantize at head_dim 128 takes the staged kernel
// instead (kivi_staged.cu: whole tiles streamed into shared memory by a
// producer warp) at G = 128 and at 2-bit G = 64 (see launch_key_quant).
//
// Dequantize: one thread per (layer, bh, group, 8 channels); 16-byte loads of
// codes, scales and zeros, 16-byte streaming stores.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdlib>
#include <cstring>

#include "kivi_device.cuh"
#include "kivi_launch.h"

namespace kivi_impl {
namespace {

using namespace kivi_dev;

// Work unit of the quantize kernel: u = ((job * bh + b) * ng + g) * (C * T)
// + col * T + split, with C = d/2 channel pairs, TPT = min(G, 32) tokens per
// thread and T = G/TPT token splits.  Thread u owns channels (2 col, 2 col +
// 1) and tokens [TPT split, TPT split + TPT) of group g.  Consecutive lanes take consecutive splits, then columns,
// so every warp load reads T rows x (32/T) columns x 4 bytes: whole 32-byte
// sectors, and the T threads of one column are adjacent lanes that combine
// their partial extremes with __shfl_xor_sync.
struct KeyUnit {
  int job;
  int b, g;
  int col, split;
};

template <int T>
__device__ __forceinline__ KeyUnit decode_key_unit(uint32_t u, const QuantParams &p) {
  KeyUnit k;
  k.split = static_cast<int>(u & (T - 1));
  const uint32_t cu = u / T;
  const uint32_t tile = p.div_chunks.div(cu);            // divide by C
  k.col = static_cast<int>(cu - tile * p.div_chunks.d);
  const uint32_t jb = p.div_rows.div(tile);              // divide by ng
  k.g = static_cast<int>(tile - jb * p.div_rows.d);
  const uint32_t job = p.div_bh.div(jb);                 // divide by bh
  k.b = static_cast<int>(jb - job * p.div_bh.d);
  k.job = static_cast<int>(job);
  return k;
}

// Rare paths, kept out of line so that they do not weigh on the register
// allocation of the main loop.

// Token t (0 .. TPT-1) of a split with `rows_here` valid rows, padded by repeating
// the group's last row (which is row rows_here - 1 of the split, or lies in
// an earlier split when rows_here <= 0).
__device__ __forceinline__ int padded_row(int t, int rows_here) {
  return t < rows_here ? t : rows_here - 1;
}

// Partial (min, max) of a split of TPT tokens of a ragged group.
template <int TPT>
__device__ __noinline__ uint2 key_partial_ragged(const __half2 *src, int rows_here, int D) {
  __half2 mn = __ldcs(src + static_cast<int64_t>(padded_row(0, rows_here)) * (D / 2));
  __half2 mx = mn;
#pragma unroll 1
  for (int t = 1; t < TPT; ++t) {
    const __half2 h = __ldcs(src + static_cast<int64_t>(padded_row(t, rows_here)) * (D / 2));
    mn = __hmin2(mn, h);
    mx = __hmax2(mx, h);
  }
  return make_uint2(h2_as_u32(mn), h2_as_u32(mx));
}

// Exact codes of one thread's TPT tokens x 2 channels (rows padded as above),
// computed from global memory with the literal division, and stored.
template <int BITS, int TPT>
__device__ __noinline__ void key_exact_store(const __half2 *src, int rows_here, int D,
                                             uint32_t ext_mn, uint32_t ext_mx, uint32_t *cdst,
                                             __half *ycol) {
  constexpr int W = CodeFmt<BITS>::W;
  const float qf = static_cast<float>(CodeFmt<BITS>::Q);
  const float2 mnf = __half22float2(u32_as_h2(ext_mn));
  const float2 mxf = __half22float2(u32_as_h2(ext_mx));
  const GroupQ g0 = make_group(mnf.x, mxf.x, qf);
  const GroupQ g1 = make_group(mnf.y, mxf.y, qf);
#pragma unroll 1
  for (int wr = 0; wr < TPT / W; ++wr) {
    uint32_t a0 = 0u, a1 = 0u;
#pragma unroll 1
    for (int k = 0; k < W; ++k) {
      const int t = wr * W + k;
      const int r = padded_row(t, rows_here);
      const float2 xf = __half22float2(__ldcs(src + static_cast<int64_t>(r) * (D / 2)));
      const uint32_t q0 = exact_code(xf.x, g0, qf), q1 = exact_code(xf.y, g1, qf);
      a0 |= q0 << (k * BITS);
      a1 |= q1 << (k * BITS);
      if (ycol != nullptr && t < rows_here)  // reconstruction of real tokens only
        __stcs(reinterpret_cast<unsigned int *>(ycol + static_cast<int64_t>(t) * D),
               recon_pair(f2_pack(static_cast<float>(q0), static_cast<float>(q1)),
                          f2_pack(g0.scale, g1.scale), neg_scale_2p23_pair(g0.scale, g1.scale),
                          f2_pack(g0.zero, g1.zero)));
    }
    if (cdst != nullptr) st_stream(cdst + static_cast<int64_t>(wr) * D, make_uint2(a0, a1));
  }
}

constexpr int kKeyThreads = 256;

// Fused reconstruction at head_dim 128 with G = 64 or 128 (T = 2 or 4 token
// splits per group): the units are ordered split-major within a group,
// u = tile * 64 T + split * 64 + col, so a warp holds 32 consecutive channel
// pairs of one split and every warp load reads, and every store writes,
// whole 128-byte rows (a lane order with the splits adjacent leaves rows of
// 128 / T bytes per warp, and isolated 32-byte row pieces halve the write
// bandwidth of the fused reconstruction).  A block's 256 units are whole groups (64 T divides 256);
// the T partial extremes of a column meet in shared memory across one block
// barrier, double-buffered by iteration parity so that one barrier per
// iteration suffices.
template <int T>
__device__ __forceinline__ KeyUnit decode_key_unit_xch(uint32_t u, const QuantParams &p) {
  KeyUnit k;
  constexpr int kShift = T == 2 ? 7 : 8;       // log2(64 T)
  const uint32_t tile = u >> kShift;
  const uint32_t rem = u & ((1u << kShift) - 1u);
  k.split = static_cast<int>(rem >> 6);
  k.col = static_cast<int>(rem & 63u);
  const uint32_t jb = p.div_rows.div(tile);    // divide by ng
  k.g = static_cast<int>(tile - jb * p.div_rows.d);
  const uint32_t job = p.div_bh.div(jb);       // divide by bh
  k.b = static_cast<int>(jb - job * p.div_bh.d);
  k.job = static_cast<int>(job);
  return k;
}

// Register budget: 64 per thread (4 blocks per SM) at 2 bits; 85 (3 blocks)
// at 4 and 8 bits, whose branch-free halves (below) keep more values live.
template <int BITS>
__host__ __device__ constexpr int key_min_blocks() { return BITS >= 4 ? 3 : 4; }

template <int BITS, int G, int DC, int MODE>
__global__ void __launch_bounds__(kKeyThreads, key_min_blocks<BITS>()) key_quant_kernel(const __grid_constant__ QuantParams p) {
  // a launch whose inputs do not depend on the previous grid in the stream
  // (defer_wait) starts at once and waits for it only before it ends
  if (!p.defer_wait) kivi_dev::grid_dependency_wait();
  kivi_dev::grid_launch_dependents();
  constexpr bool RECON = MODE == kQuantRecon;
  constexpr bool SINK = MODE == kQuantSink;
  constexpr int TPT = G < 32 ? G : 32;      // tokens per thread
  constexpr int T = G / TPT;                 // token splits per group
  constexpr int W = CodeFmt<BITS>::W;        // codes per word
  constexpr int WPT = TPT / W;               // words per channel per thread
  constexpr uint32_t Q = CodeFmt<BITS>::Q;
  // split-major units with the shared-memory exchange: with the fused
  // reconstruction (whose row pieces would otherwise be 128 / T bytes) and
  // the plain 2-bit quantize (+1% at G = 64, +3% at G = 128); the plain 4-
  // and 8-bit quantize keep the shuffle order, measured 5-9% faster
  constexpr bool XCH = (RECON || (MODE == kQuantPlain && BITS == 2)) && DC == 128 && T > 1;
  const float qf = static_cast<float>(Q);
  __shared__ uint2 xch[XCH ? 2 : 1][XCH ? kKeyThreads : 1];
  int parity = 0;

  const int D = DC > 0 ? DC : p.d;           // head_dim, compile-time when DC > 0
  const uint32_t total = static_cast<uint32_t>(p.n_jobs) * p.div_bh.d * p.div_rows.d *
                         p.div_chunks.d * T;

  // Block-uniform loop (every thread of a block runs the same iterations, so
  // the exchange barrier is reached by all of them).
#pragma unroll 1
  for (uint32_t blk = blockIdx.x * kKeyThreads; blk < total; blk += gridDim.x * kKeyThreads) {
    const uint32_t base = blk + (threadIdx.x & ~31u);
    const uint32_t u = blk + threadIdx.x;
    const bool active = u < total;
    // inactive lanes decode a valid unit (their warp's first, else the block's)
    const uint32_t ud = active ? u : base < total ? base : blk;
    const KeyUnit k = XCH ? decode_key_unit_xch<T>(ud, p) : decode_key_unit<T>(ud, p);
    const QuantJob &job = p.jobs[k.job];
    int64_t row0 = static_cast<int64_t>(k.g) * G;  // first stored row of the group
    const int rows_here = static_cast<int>(p.rows - row0) - k.split * TPT;  // valid rows of the split
    if (p.ring > 0) {
      row0 += p.head;
      if (row0 >= p.ring) row0 -= p.ring;    // head < ring and g*G < ring
    }
    // column (2 col, 2 col + 1) of the first row of this thread's split
    const __half2 *src = reinterpret_cast<const __half2 *>(
                             static_cast<const __half *>(job.x) +
                             static_cast<int64_t>(k.b) * p.x_bh_stride + row0 * D) +
                         k.col + static_cast<int64_t>(k.split) * TPT * (D / 2);
    const bool full = active && rows_here >= TPT;
    // debug builds: every row this thread reads (padded rows included) lies
    // inside its bh slice
    [[maybe_unused]] const int64_t r_first = row0 + static_cast<int64_t>(k.split) * TPT;
    const bool x_ok = KIVI_BOUND(
        p.fault, !active || (k.b < p.bh && r_first + min(0, rows_here - 1) >= 0 &&
                             (r_first + (rows_here >= 1 ? min(rows_here, TPT) : rows_here)) * D <=
                                 p.x_bh_stride));

    // sink mode: bit t = token t of this split is a sink (left out of the
    // group's min / max, code 0); the flush only moves whole groups.  Mask
    // bit r of a sequence is logical row r.
    uint32_t sink_bits = 0u;
    if (SINK && full) {
      const int64_t lr = static_cast<int64_t>(k.g) * G + k.split * TPT;   // first logical row
      sink_bits = job.mask[static_cast<int64_t>(k.b / p.heads) * p.mask_words + (lr >> 5)] >>
                  (lr & 31);
    }

    // TPT tokens of this thread's channel pair; min / max in four chains
    __half2 h[TPT];
    __half2 gmn, gmx;
    if (full && x_ok) {
#pragma unroll
      for (int t = 0; t < TPT; ++t) h[t] = __ldcs(src + t * (D / 2));
      if (SINK && sink_bits != 0u) {   // a group holding sinks (rare)
        const __half2 pinf = u32_as_h2(0x7C007C00u), ninf = u32_as_h2(0xFC00FC00u);
        __half2 mn[4] = {pinf, pinf, pinf, pinf};
        __half2 mx[4] = {ninf, ninf, ninf, ninf};
#pragma unroll
        for (int t = 0; t < TPT; ++t) {
          const uint32_t m = 0u - ((sink_bits >> t) & 1u);   // all ones for a sink
          const uint32_t x = h2_as_u32(h[t]);
          mn[t & 3] = __hmin2(mn[t & 3], u32_as_h2((x & ~m) | (0x7C007C00u & m)));
          mx[t & 3] = __hmax2(mx[t & 3], u32_as_h2((x & ~m) | (0xFC00FC00u & m)));
        }
        gmn = __hmin2(__hmin2(mn[0], mn[1]), __hmin2(mn[2], mn[3]));
        gmx = __hmax2(__hmax2(mx[0], mx[1]), __hmax2(mx[2], mx[3]));
      } else {
        __half2 mn[4] = {h[0], h[1], h[2], h[3]};
        __half2 mx[4] = {h[0], h[1], h[2], h[3]};
#pragma unroll
        for (int t = 4; t < TPT; ++t) {
          mn[t & 3] = __hmin2(mn[t & 3], h[t]);
          mx[t & 3] = __hmax2(mx[t & 3], h[t]);
        }
        gmn = __hmin2(__hmin2(mn[0], mn[1]), __hmin2(mn[2], mn[3]));
        gmx = __hmax2(__hmax2(mx[0], mx[1]), __hmax2(mx[2], mx[3]));
      }
    } else if (active && x_ok) {  // ragged last group: padded by repeating the last row
      const uint2 e = key_partial_ragged<TPT>(src, rows_here, D);
      gmn = u32_as_h2(e.x);
      gmx = u32_as_h2(e.y);
    } else {
      gmn = gmx = __float2half2_rn(0.0f);
    }
    if (XCH) {
      // the T partials of this column: units split * 64 + col of this group
      xch[parity][threadIdx.x] = make_uint2(h2_as_u32(gmn), h2_as_u32(gmx));
      __syncthreads();
      const int g0 = static_cast<int>(threadIdx.x) & ~(64 * T - 1);
#pragma unroll
      for (int sp = 0; sp < T; ++sp) {
        const uint2 e = xch[parity][g0 + sp * 64 + k.col];
        gmn = __hmin2(gmn, u32_as_h2(e.x));
        gmx = __hmax2(gmx, u32_as_h2(e.y));
      }
      parity ^= 1;
    } else if (T > 1) {
      // partners of inactive lanes are inactive too (whole groups per lane set)
#pragma unroll
      for (int off = 1; off < T; off <<= 1) {
        gmn = __hmin2(gmn, u32_as_h2(__shfl_xor_sync(0xffffffffu, h2_as_u32(gmn), off)));
        gmx = __hmax2(gmx, u32_as_h2(__shfl_xor_sync(0xffffffffu, h2_as_u32(gmx), off)));
      }
    }

    if (SINK && sink_bits != 0u) {
      // a group of sinks only (no finite extreme) gets scale 0 and zero 0
      const float2 a = __half22float2(gmn), bx = __half22float2(gmx);
      gmn = __floats2half2_rn(a.x > bx.x ? 0.0f : a.x, a.y > bx.y ? 0.0f : a.y);
      gmx = __floats2half2_rn(a.x > bx.x ? 0.0f : bx.x, a.y > bx.y ? 0.0f : bx.y);
      // a sink takes the group minimum's place, whose code is 0 by the
      // definition (x - zero = 0), and the fast path yields exactly 0 for it
      const uint32_t gm = h2_as_u32(gmn);
#pragma unroll
      for (int t = 0; t < TPT; ++t) {
        const uint32_t m = 0u - ((sink_bits >> t) & 1u);   // all ones for a sink
        h[t] = u32_as_h2((h2_as_u32(h[t]) & ~m) | (gm & m));
      }
    }

    if (active) {
      const int64_t out_g = p.out0 + k.g;
      // debug builds: the code words, scale / zero and reconstruction rows this
      // thread writes lie inside its bh slice
      const bool codes_out =
          (!RECON || job.codes != nullptr) &&
          KIVI_BOUND(p.fault, (out_g * (G / W) + k.split * WPT + WPT - 1) * D + 2 * k.col + 2 <=
                                  p.codes_bh_stride &&
                              out_g * D + 2 * k.col + 2 <= p.sz_bh_stride);
      const bool y_ok = KIVI_BOUND(
          p.fault, !RECON || rows_here <= 0 ||
                       (p.y_row0 + static_cast<int64_t>(k.g) * G + k.split * TPT +
                        min(rows_here, TPT) - 1) * D + 2 * k.col + 2 <= p.y_bh_stride);
      uint32_t *cdst = codes_out ? job.codes + static_cast<int64_t>(k.b) * p.codes_bh_stride +
                                       (out_g * (G / W) + k.split * WPT) * D + 2 * k.col
                                 : nullptr;
      // reconstruction: column (2 col, 2 col + 1) of the first token of the split
      __half *ycol = RECON && y_ok ? static_cast<__half *>(job.y) +
                                 static_cast<int64_t>(k.b) * p.y_bh_stride +
                                 (p.y_row0 + static_cast<int64_t>(k.g) * G + k.split * TPT) * D +
                                 2 * k.col
                           : nullptr;
      GroupD2 gq;
      float s0, z0, s1, z1;
      uint64_t sc2 = 0, nsc2 = 0, ze2 = 0;
      const float2 mnf = __half22float2(gmn);
      const float2 mxf = __half22float2(gmx);
      {
        const GroupQ g0 = make_group_szr(mnf.x, mxf.x, qf);
        const GroupQ g1 = make_group_szr(mnf.y, mxf.y, qf);
        gq = make_group_d2(g0, g1);
        s0 = g0.scale;
        z0 = g0.zero;
        s1 = g1.scale;
        z1 = g1.zero;
        if (RECON) {
          sc2 = f2_pack(g0.scale, g1.scale);
          nsc2 = neg_scale_2p23_pair(g0.scale, g1.scale);
          ze2 = f2_pack(g0.zero, g1.zero);
        }
        if (k.split == 0 && codes_out) {
          const int64_t o = static_cast<int64_t>(k.b) * p.sz_bh_stride + out_g * D + 2 * k.col;
          __stcs(reinterpret_cast<float2 *>(job.scale + o), make_float2(g0.scale, g1.scale));
          __stcs(reinterpret_cast<float2 *>(job.zero + o), make_float2(g0.zero, g1.zero));
        }
      }
      if (!full) {
        // ragged group: literal division, rows read again from memory
        if (x_ok)
          key_exact_store<BITS, TPT>(src, rows_here, D, h2_as_u32(gmn), h2_as_u32(gmx), cdst,
                                     ycol);
      } else {
        // Quantize and pack along tokens: WPT words per channel, word wi holds
        // tokens [wi*W, wi*W + W) of this thread's TPT (token wi*W + j at bits
        // [j*BITS, (j+1)*BITS)).  Each half-word (H = 16/BITS tokens)
        // accumulates the code pairs of both channels with packed FMAs by
        // powers of two.
        constexpr int H = 16 / BITS;
#pragma unroll
        for (int wi = 0; wi < WPT; ++wi) {
          // 2 bits: a pair the fast path declines is recomputed on the spot (a
          // branch per pair, almost never taken).  4 and 8 bits: the H <= 4
          // pairs of a half run without branches, their acceptance tests AND-ed,
          // and the half is redone from registers when a pair is declined; with
          // the larger register budget this was 3-4% faster there and slower
          // at 2 bits (measured).
          constexpr bool BF = BITS >= 4;
          uint64_t half[2];
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const int t0 = wi * W + hh * H;
            uint64_t n[H];
            if constexpr (BF) {
              uint32_t ok = 0xFFFFFFFFu;
#pragma unroll
              for (int j = 0; j < H; ++j)
                n[j] = codes2_diff_nobranch<BITS>(h2_as_u32(h[t0 + j]), gq, ok);
              if (!(ok >> 31)) {   // rare: redo this half pair by pair from registers
#pragma unroll
                for (int j = 0; j < H; ++j)
                  n[j] = codes2_diff<BITS>(h2_as_u32(h[t0 + j]), gq, s0, z0, s1, z1, qf);
              }
            }
#pragma unroll
            for (int j = 0; j < H; ++j) {
              if constexpr (!BF)
                n[j] = codes2_diff<BITS>(h2_as_u32(h[t0 + j]), gq, s0, z0, s1, z1, qf);
              half[hh] = j == 0 ? n[j]
                                : f2_fma(n[j], f2_const(static_cast<float>(1u << (BITS * j))),
                                         half[hh]);
              if (RECON && y_ok)
                __stcs(reinterpret_cast<unsigned int *>(ycol + static_cast<int64_t>(t0 + j) * D),
                       recon_pair(n[j], sc2, nsc2, ze2));
            }
          }
          if (codes_out)
            st_stream(cdst + static_cast<int64_t>(wi) * D, join_halves2(half[0], half[1]));
        }
      }
    }

  }
  if (p.defer_wait) kivi_dev::grid_dependency_wait();
}

// One thread: channels [8*chunk, 8*chunk + 8) of group g of one bh slice.
// unit = ((job * bh + b) * ng + g) * (d/8) + chunk  (< 2^31, host-checked);
// p.div_chunks, p.div_rows and p.div_bh divide by d/8, ng and bh.
template <int BITS, int G, int DC>
__global__ void __launch_bounds__(256) key_dequant_kernel(const __grid_constant__ DequantParams p) {
  // a launch whose inputs do not depend on the previous grid in the stream
  // (defer_wait) starts at once and waits for it only before it ends
  if (!p.defer_wait) kivi_dev::grid_dependency_wait();
  kivi_dev::grid_launch_dependents();
  constexpr int W = CodeFmt<BITS>::W;
  constexpr uint32_t Q = CodeFmt<BITS>::Q;
  const int D = DC > 0 ? DC : p.d;
  // a unit is 8 channels x one TPU-token split of a group: groups above 32
  // tokens are split so that every G gives a thread the work of G = 32 (the
  // group's scale and zero are read once per split, the repeats from cache)
  constexpr int TPU = G < 32 ? G : 32;
  constexpr int S = G / TPU;                  // splits per group
  const uint32_t total = static_cast<uint32_t>(p.n_jobs) * p.div_bh.d * p.div_rows.d * S *
                         p.div_chunks.d;
  const uint32_t stride = gridDim.x * blockDim.x;
#pragma unroll 1
  for (uint32_t u = blockIdx.x * blockDim.x + threadIdx.x; u < total; u += stride) {
    const uint32_t gs_all = p.div_chunks.div(u);
    const int ch = static_cast<int>(u - gs_all * p.div_chunks.d);
    const int split = static_cast<int>(gs_all % S);
    const uint32_t bg_all = gs_all / S;
    const uint32_t jb = p.div_rows.div(bg_all);
    const int64_t g = bg_all - jb * p.div_rows.d;
    const uint32_t job = p.div_bh.div(jb);
    const int64_t b = jb - job * p.div_bh.d;
    const DequantJob &J = p.jobs[job];

    // debug builds: the unit's reads and writes stay inside its bh slice
    if (!KIVI_BOUND(p.fault,
                    b < p.bh && g * D + ch * 8 + 8 <= p.sz_bh_stride &&
                        (g * (G / W) + split * (TPU / W) + TPU / W - 1) * D + ch * 8 + 8 <=
                            p.codes_bh_stride &&
                        (min(p.rows, g * G + split * TPU + TPU) - 1) * D + ch * 8 + 8 <=
                            p.y_bh_stride))
      continue;
    const int64_t so = b * p.sz_bh_stride + g * D + ch * 8;
    const uint4 s_a = ld_stream(J.scale + so), s_b = ld_stream(J.scale + so + 4);
    const uint4 z_a = ld_stream(J.zero + so), z_b = ld_stream(J.zero + so + 4);
    float sc[8] = {__uint_as_float(s_a.x), __uint_as_float(s_a.y), __uint_as_float(s_a.z),
                   __uint_as_float(s_a.w), __uint_as_float(s_b.x), __uint_as_float(s_b.y),
                   __uint_as_float(s_b.z), __uint_as_float(s_b.w)};
    float ze[8] = {__uint_as_float(z_a.x), __uint_as_float(z_a.y), __uint_as_float(z_a.z),
                   __uint_as_float(z_a.w), __uint_as_float(z_b.x), __uint_as_float(z_b.y),
                   __uint_as_float(z_b.z), __uint_as_float(z_b.w)};
    float nsc[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) nsc[c] = __fmul_rn(sc[c], -8388608.0f);  // -2^23 * scale, exact

    const uint32_t *cw =
        J.codes + b * p.codes_bh_stride + (g * (G / W) + split * (TPU / W)) * D + ch * 8;
    __half *y = static_cast<__half *>(J.y) + b * p.y_bh_stride + ch * 8;
    const int64_t t0 = g * G + split * TPU;
    if constexpr (BITS == 2) {
      // Each channel's four fp16 reconstructions (codes 0..3, the same
      // arithmetic as below) as an 8-byte table in two registers; one byte
      // permute fetches a channel's values for two consecutive tokens (its
      // selector from the two codes, q * 0x22 + 0x10 per byte after spreading
      // four codes one to a byte), and a 2 x 2 transpose of halves (two more
      // permutes) turns channel pairs of tokens into token rows of channel
      // pairs.
      uint32_t lo[8], hi[8];
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        lo[c] = h2_as_u32(__floats2half2_rn(recon_f32(0u, sc[c], nsc[c], ze[c]),
                                            recon_f32(1u, sc[c], nsc[c], ze[c])));
        hi[c] = h2_as_u32(__floats2half2_rn(recon_f32(2u, sc[c], nsc[c], ze[c]),
                                            recon_f32(3u, sc[c], nsc[c], ze[c])));
      }
#pragma unroll 1
      for (int wr = 0; wr < TPU / W; ++wr) {
        const uint4 ca = ld_stream(cw + static_cast<int64_t>(wr) * D);
        const uint4 cb = ld_stream(cw + static_cast<int64_t>(wr) * D + 4);
        const uint32_t words[8] = {ca.x, ca.y, ca.z, ca.w, cb.x, cb.y, cb.z, cb.w};
#pragma unroll
        for (int kb = 0; kb < 4; ++kb) {         // tokens 4 kb .. 4 kb + 3 of the word row
          uint32_t a01[8], a23[8];              // channel c: (token 0, 1) and (token 2, 3)
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint32_t bt = (words[c] >> (8 * kb)) & 0xFFu;
            uint32_t x = (bt | (bt << 12)) & 0x000F000Fu;
            x = (x | (x << 6)) & 0x03030303u;   // code of token j in byte j
            const uint32_t sel = x * 0x22u + 0x10101010u;
            a01[c] = __byte_perm(lo[c], hi[c], sel);
            a23[c] = __byte_perm(lo[c], hi[c], sel >> 16);
          }
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int64_t t = t0 + wr * W + 4 * kb + j;
            if (t >= p.rows) break;
            const uint32_t *src = j < 2 ? a01 : a23;
            const uint32_t pick = (j & 1) ? 0x7632u : 0x5410u;   // high or low halves
            uint32_t out[4];
#pragma unroll
            for (int cp = 0; cp < 4; ++cp) out[cp] = __byte_perm(src[2 * cp], src[2 * cp + 1], pick);
            st_stream(y + t * D, make_uint4(out[0], out[1], out[2], out[3]));
          }
        }
      }
    } else {
#pragma unroll 1
      for (int wr = 0; wr < TPU / W; ++wr) {
        const uint4 ca = ld_stream(cw + static_cast<int64_t>(wr) * D);
        const uint4 cb = ld_stream(cw + static_cast<int64_t>(wr) * D + 4);
        const uint32_t words[8] = {ca.x, ca.y, ca.z, ca.w, cb.x, cb.y, cb.z, cb.w};
#pragma unroll
        for (int k = 0; k < W; ++k) {
          const int64_t t = t0 + wr * W + k;
          if (t >= p.rows) break;
          uint32_t out[4];
#pragma unroll
          for (int c = 0; c < 8; c += 2) {
            const uint32_t q0 = (words[c] >> (k * BITS)) & Q;
            const uint32_t q1 = (words[c + 1] >> (k * BITS)) & Q;
            const float r0 = recon_f32(q0, sc[c], nsc[c], ze[c]);
            const float r1 = recon_f32(q1, sc[c + 1], nsc[c + 1], ze[c + 1]);
            out[c >> 1] = h2_as_u32(__floats2half2_rn(r0, r1));
          }
          st_stream(y + t * D, make_uint4(out[0], out[1], out[2], out[3]));
        }
      }
    }
  }
  if (p.defer_wait) kivi_dev::grid_dependency_wait();
}


template <int BITS, int G, int DC, int MODE>
cudaError_t key_quant_launch(const QuantParams &p, cudaStream_t stream) {
  const int threads = kKeyThreads;
  auto kern = key_quant_kernel<BITS, G, DC, MODE>;
  const int64_t ng = (p.rows + G - 1) / G;
  const int64_t units = static_cast<int64_t>(p.n_jobs) * p.bh * ng * (p.d / 2) * (G < 32 ? 1 : G / 32);
  // Grid shape by measurement over bits x G on stores larger than L2: one
  // block per 256 units (flat) is 6-17% faster for the fused reconstruction
  // and ~3.5% faster for 2-bit codes with G <= 64; two waves of resident
  // blocks are 3-11% faster for the plain 4- and 8-bit quantize, whose
  // kernels hold more registers and fit fewer blocks per SM (one wave is
  // ~1% slower, three or more waves lose again at 8 bits).
  constexpr bool kFlat = MODE == kQuantRecon || (BITS == 2 && G <= 64);
  int64_t grid = flat_grid(units, threads);
  if (!kFlat) {
    int per_sm = 0;
    cudaError_t err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, 0);
    if (err != cudaSuccess) return err;
    if (per_sm < 1) per_sm = 1;
    grid = std::min<int64_t>(grid, 2 * static_cast<int64_t>(current_sm_count()) * per_sm);
  }
  QuantParams q = p;
  q.div_chunks = FastDiv::make(static_cast<uint32_t>(p.d / 2));
  q.div_rows = FastDiv::make(static_cast<uint32_t>(ng));
  q.div_bh = FastDiv::make(static_cast<uint32_t>(p.bh));
  cudaError_t e = debug_fault_word(&q.fault);
  if (e != cudaSuccess) return e;
  return launch_dependent(kern, grid, threads, stream, q);
}

template <int BITS, int G, int DC>
cudaError_t key_dequant_launch(const DequantParams &p, cudaStream_t stream) {
  const int threads = 256;
  auto kern = key_dequant_kernel<BITS, G, DC>;
  const int64_t ng = (p.rows + G - 1) / G;
  const int64_t units = static_cast<int64_t>(p.n_jobs) * p.bh * ng * (G < 32 ? 1 : G / 32) * (p.d / 8);
  // one block per 256 units, not a persistent grid (see flat_grid)
  const int64_t grid = flat_grid(units, threads);
  DequantParams q = p;
  q.div_chunks = FastDiv::make(static_cast<uint32_t>(p.d / 8));
  q.div_rows = FastDiv::make(static_cast<uint32_t>(ng));
  q.div_bh = FastDiv::make(static_cast<uint32_t>(p.bh));
  const cudaError_t e = debug_fault_word(&q.fault);
  if (e != cudaSuccess) return e;
  return launch_dependent(kern, grid, threads, stream, q);
}

}  // namespace

#include "kivi_dispatch.h"

// Which key quantizer a plain quantize takes.  By measurement of whole flush
// + dequantize steps on a GB300, each pair on one box: the staged kernel
// (kivi_staged.cu) at G = 128, and at G = 64 with 2-bit codes (store sweep
// cells 2/64 +1.5%, 2/128 +3%, 4/128 and 8/128 level), the register kernel
// everywhere else (4-bit G = 64 flush of 28 layers x 4 heads x 32 K tokens
// +0.6%, 2-bit G = 32 prefill flush +3.3% and decode flush +4%, the G = 32
// and 4/8-bit G = 64 sweep cells +0.6-1.2%).  The staged kernel is the
// faster one alone at every G >= 32 but holds every SM's shared memory and
// most of its registers, so the kernels around it cannot overlap it; the
// register kernel's cost grows with G (G / 32 lanes per column exchanging
// extremes), so the staged one gains where G is large and the codes narrow.
// KIVI_KEY_QUANTIZER=staged or =register in the environment (read at every
// call) takes that kernel wherever it applies.
static bool staged_key_quantizer(int group, int bits) {
  const char *v = std::getenv("KIVI_KEY_QUANTIZER");
  if (v && std::strcmp(v, "staged") == 0) return true;
  if (v && std::strcmp(v, "register") == 0) return false;
  return group == 128 || (bits == 2 && group >= 64);
}

cudaError_t launch_key_quant(const QuantParams &p, int group, int bits, int mode,
                             cudaStream_t stream) {
  if (staged_key_quantizer(group, bits)) {
    bool handled = false;
    const cudaError_t e = launch_key_quant_staged(p, group, bits, mode, stream, &handled);
    if (handled) return e;
  }
  KIVI_DISPATCH_MODE(key_quant_launch, p, group, bits, mode, stream);
}

cudaError_t launch_key_dequant(const DequantParams &p, int group, int bits,
                               cudaStream_t stream) {
  KIVI_DISPATCH(key_dequant_launch, p, group, bits, stream);
}

}  // namespace kivi_impl
