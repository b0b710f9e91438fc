// kivi_staged.cu -- the staged per-channel key quantizer: whole key tiles
// streamed into a shared-memory ring by bulk asynchronous copies.
//
// Keys are grouped along the token axis (VeloxQuant-MLX KIVI fused-kernel
// post, "The layout problem that shapes everything"): a group of G tokens
// of every channel is one contiguous G x d block of the [bh][s][d] tensor
// (also in the residual ring, whose head and capacity are multiples of G).
// So a whole tile -- one (layer, bh, group), G rows of 256 bytes at
// head_dim 128 -- arrives with one bulk copy (the non-tensor form of the
// tensor memory accelerator), completed on a per-stage mbarrier.
//
// Warp roles (one CTA per SM, persistent over the tiles):
//   producer  one lane of the last warp walks the CTA's tiles and issues
//             each tile's copy into the next free stage of the ring
//   consumers 8 warps in groups of P = G / 32; the P warps of a group own
//             every stage s with s % (8 / P) == their group, each warp 32
//             rows of the tile (lane l: channels 4l .. 4l+3, conflict-free
//             8-byte shared-memory reads of whole 256-byte rows).
// A stage is released (its `empty` mbarrier, P arrivals) after its group
// has read it; the only other synchronisation is, for G > 32, one named
// barrier of the group's P warps per tile to exchange partial extremes.
// There is no CTA-wide barrier after set-up: the copies of later tiles are
// in flight while earlier ones are quantized.
//
// Per tile a consumer warp takes min / max of its 32 rows in half2 (exact:
// binary16 -> binary32 is monotone), combines the group's partials, forms
// the four channels' (scale, zero) with the same arithmetic as the
// register-only kernel (kivi_device.cuh), re-reads its rows from shared
// memory to quantize them (the difference-first fast path of kivi_device.cuh,
// straight from the binary16 values, with the exact fallback), packs the
// codes along tokens and writes whole 512-byte code rows per warp; the
// fused form also writes each row's fp16 reconstruction.
//
// Every mbarrier wait is bounded (0.2 s of the global timer); a wait that
// gives up sets bit 3 of the device fault word and the remaining waits of
// that warp are skipped, so the kernel always ends.  The producer waits,
// before it exits, for every copy it issued, so no copy is in flight when
// the CTA ends.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>

#include "kivi_device.cuh"
#include "kivi_launch.h"

namespace kivi_impl {
namespace {

using namespace kivi_dev;

constexpr int kD = 128;                  // head_dim of the staged kernel
constexpr int kRowBytes = kD * 2;        // one fp16 row
constexpr int kWarpRows = 32;            // rows of a tile one consumer warp takes
#ifndef KIVI_STAGED_WARPS
#define KIVI_STAGED_WARPS 16
#endif
constexpr int kConsumerWarps = KIVI_STAGED_WARPS;
constexpr int kRingBytes = 192 * 1024;   // shared-memory ring
constexpr uint64_t kWaitLimitNs = 200000000ull;   // 0.2 s

template <int G>
struct KeyStaged {
  static constexpr int P = G / kWarpRows;           // consumer warps per tile (a unit)
  static constexpr int U = kConsumerWarps / P;      // units
  static constexpr int kTile = G * kRowBytes;       // bytes per stage
  static constexpr int S = kRingBytes / kTile;      // ring stages (24, 12, 6)
  static constexpr int kSmem = S * kTile;           // dynamic shared memory
  static constexpr int kThreads = 32 * (kConsumerWarps + 1);
};

__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}

// Waits (bounded) until the producer has published tile j for stage slot
// *slot; false on timeout.
__device__ __forceinline__ bool wait_stage_tile(const volatile uint32_t *slot, uint32_t j,
                                                uint64_t limit_ns) {
  if (*slot == j) return true;
  const uint64_t t0 = global_timer_ns();
#pragma unroll 1
  while (*slot != j) {
    __nanosleep(64);
    if (global_timer_ns() - t0 > limit_ns) return false;
  }
  return true;
}

__device__ __forceinline__ void named_barrier(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

struct Tile {
  int job;
  uint32_t b, g;
};

// tile t = (job * bh + b) * ng + g
__device__ __forceinline__ Tile decode_tile(uint32_t t, const QuantParams &p) {
  Tile k;
  const uint32_t jb = p.div_rows.div(t);    // divide by ng
  k.g = t - jb * p.div_rows.d;
  const uint32_t job = p.div_bh.div(jb);    // divide by bh
  k.b = jb - job * p.div_bh.d;
  k.job = static_cast<int>(job);
  return k;
}

// Codes of H consecutive rows (one half-word per channel pair) accumulated
// as integer-valued float pairs, and the fused form's reconstruction of each
// row.  The rows go in chunks of up to four: a chunk's fast path runs
// without a branch (the acceptance tests AND-ed), so its rows' arithmetic
// interleaves; a chunk whose test failed somewhere (mostly exact .5 ties) is
// redone pair by pair, each declined pair by the literal division.  FULL:
// rows_here >= G (no edge padding), known per tile.
template <int BITS, bool RECON, bool FULL>
__device__ __forceinline__ void key_half(uint32_t row_addr, int row_first, int rows_here,
                                         const GroupD2 &q01, const GroupD2 &q23,
                                         const float4 &sc, const float4 &ze, float qf,
                                         uint64_t &h01, uint64_t &h23, __half *ydst, int y_first) {
  constexpr int H = 16 / BITS;
  constexpr int HS = H < 4 ? H : 4;   // rows per chunk
  uint64_t sc01 = 0, sc23 = 0, nsc01 = 0, nsc23 = 0, ze01 = 0, ze23 = 0;
  if constexpr (RECON) {
    sc01 = f2_pack(sc.x, sc.y);
    sc23 = f2_pack(sc.z, sc.w);
    nsc01 = neg_scale_2p23_pair(sc.x, sc.y);
    nsc23 = neg_scale_2p23_pair(sc.z, sc.w);
    ze01 = f2_pack(ze.x, ze.y);
    ze23 = f2_pack(ze.z, ze.w);
  }
#pragma unroll
  for (int c0 = 0; c0 < H; c0 += HS) {
    uint64_t n01[HS], n23[HS];
    uint32_t okm = 0xFFFFFFFFu;
#pragma unroll
    for (int jj = 0; jj < HS; ++jj) {
      const int rr = FULL ? row_first + c0 + jj : min(row_first + c0 + jj, rows_here - 1);
      const uint2 v = lds64(row_addr + rr * kRowBytes);
      n01[jj] = codes2_diff_nobranch<BITS>(v.x, q01, okm);
      n23[jj] = codes2_diff_nobranch<BITS>(v.y, q23, okm);
    }
    if (!(okm >> 31)) {
#pragma unroll
      for (int jj = 0; jj < HS; ++jj) {
        const int rr = FULL ? row_first + c0 + jj : min(row_first + c0 + jj, rows_here - 1);
        const uint2 v = lds64(row_addr + rr * kRowBytes);
        n01[jj] = codes2_diff<BITS>(v.x, q01, sc.x, ze.x, sc.y, ze.y, qf);
        n23[jj] = codes2_diff<BITS>(v.y, q23, sc.z, ze.z, sc.w, ze.w, qf);
      }
    }
#pragma unroll
    for (int jj = 0; jj < HS; ++jj) {
      const int j = c0 + jj;   // row within the half-word
      const uint64_t m = f2_const(static_cast<float>(1u << (BITS * j)));
      h01 = j == 0 ? n01[jj] : f2_fma(n01[jj], m, h01);
      h23 = j == 0 ? n23[jj] : f2_fma(n23[jj], m, h23);
      if constexpr (RECON) {
        if ((FULL || row_first + j < rows_here) && ydst != nullptr)
          __stcs(reinterpret_cast<uint2 *>(ydst + static_cast<int64_t>(y_first + j) * kD),
                 make_uint2(recon_pair(n01[jj], sc01, nsc01, ze01),
                            recon_pair(n23[jj], sc23, nsc23, ze23)));
      }
    }
  }
}

// Pass 2 of a warp's 32 rows: codes packed along tokens (word wr holds rows
// wr W .. wr W + W - 1, row j at bits [j b, j b + b) LSB first), one 16-byte
// store of four channels' words per lane and word row.
template <int BITS, bool RECON, bool FULL>
__device__ __forceinline__ void key_rows(uint32_t base, int r0, int rows_here, const GroupD2 &q01,
                                         const GroupD2 &q23, const float4 &sc, const float4 &ze,
                                         float qf, uint32_t *cdst, __half *ydst) {
  constexpr int W = CodeFmt<BITS>::W;
  constexpr int H = 16 / BITS;
#pragma unroll 1
  for (int wr = 0; wr < kWarpRows / W; ++wr) {
    uint64_t h01[2], h23[2];
#pragma unroll
    for (int hh = 0; hh < 2; ++hh)
      key_half<BITS, RECON, FULL>(base, r0 + wr * W + hh * H, rows_here, q01, q23, sc, ze, qf,
                                  h01[hh], h23[hh], ydst, wr * W + hh * H);
    if (cdst != nullptr) {
      const uint2 w01 = join_halves2(h01[0], h01[1]);
      const uint2 w23 = join_halves2(h23[0], h23[1]);
      st_stream(cdst + static_cast<int64_t>(wr) * kD, make_uint4(w01.x, w01.y, w23.x, w23.y));
    }
  }
}

template <int BITS, int G, int MODE>
__global__ void __launch_bounds__(KeyStaged<G>::kThreads, 1)
    key_quant_staged_kernel(const __grid_constant__ QuantParams p) {
  using C = KeyStaged<G>;
  constexpr int P = C::P, U = C::U, S = C::S;
  constexpr bool RECON = MODE == kQuantRecon;
  constexpr int W = CodeFmt<BITS>::W;   // codes per word
  const float qf = static_cast<float>(CodeFmt<BITS>::Q);

  extern __shared__ __align__(128) uint8_t ring[];
  __shared__ __align__(8) uint64_t full_bar[S];
  __shared__ __align__(8) uint64_t empty_bar[S];
  __shared__ __align__(16) uint4 xch[P > 1 ? U * 2 * P * 32 : 1];
  __shared__ uint32_t claim_ctr;
  __shared__ uint32_t claim_slot[P > 1 ? U * 2 : 1];
  // the local tile a stage holds (or is being filled with); published by the
  // producer before it issues the copy
  __shared__ uint32_t stage_tile[S];

  // a launch whose inputs do not depend on the previous grid in the stream
  // (defer_wait) starts at once and waits for it only before it ends.  The
  // next grid in the stream is released only when this one ends (no early
  // trigger): launched early, its blocks cannot share an SM with these CTAs
  // (every SM's shared memory and most of its registers), and a 28-layer x
  // 4-head x 32 K-token flush + dequantize step measured 3.8% slower so.
  if (!p.defer_wait) grid_dependency_wait();
  const int warp = static_cast<int>(threadIdx.x >> 5);
  const int lane = static_cast<int>(threadIdx.x & 31u);
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_addr(&full_bar[s]), 1);
      mbar_init(smem_addr(&empty_bar[s]), P);
      stage_tile[s] = 0xFFFFFFFFu;
    }
    fence_mbar_init();
    claim_ctr = 0;
  }
  __syncthreads();

  const uint32_t ng = p.div_rows.d;
  const uint32_t total = static_cast<uint32_t>(p.n_jobs) * p.div_bh.d * ng;
  const uint32_t mine = total > blockIdx.x ? (total - blockIdx.x + gridDim.x - 1) / gridDim.x : 0u;
  const uint32_t ring0 = smem_addr(ring);

  if (warp == kConsumerWarps) {
    // ---------------- producer: local tile j = global tile blockIdx.x + j * gridDim.x
    if (lane != 0) {
      if (p.defer_wait) grid_dependency_wait();
      return;
    }
    const uint64_t pol = policy_evict_first();
    uint32_t j = 0;
    for (; j < mine; ++j) {
      const int s = static_cast<int>(j % S);
      const uint32_t use = j / S;
      if (!mbar_wait_bounded(smem_addr(&empty_bar[s]), (use & 1u) ^ 1u, kWaitLimitNs)) {
        atomicOr(p.fault, 8u);
        break;
      }
      const Tile k = decode_tile(blockIdx.x + j * gridDim.x, p);
      const QuantJob &job = p.jobs[k.job];
      const int64_t lr0 = static_cast<int64_t>(k.g) * G;          // first logical row
      const int rows_here = static_cast<int>(min(static_cast<int64_t>(G), p.rows - lr0));
      int64_t row0 = lr0;
      if (p.ring > 0) {
        row0 += p.head;
        if (row0 >= p.ring) row0 -= p.ring;   // head < ring and lr0 < ring
      }
      const void *src = static_cast<const __half *>(job.x) +
                        static_cast<int64_t>(k.b) * p.x_bh_stride + row0 * kD;
      const uint32_t bytes = static_cast<uint32_t>(rows_here) * kRowBytes;
      *reinterpret_cast<volatile uint32_t *>(&stage_tile[s]) = j;
      // debug builds: the tile lies inside its bh slice (else the stage's phase
      // completes without a copy)
      if (KIVI_BOUND(p.fault, k.b < p.bh && rows_here > 0 && rows_here <= G &&
                                  (row0 + rows_here) * kD <= p.x_bh_stride)) {
        mbar_arrive_expect_tx(smem_addr(&full_bar[s]), bytes);
        bulk_load(ring0 + static_cast<uint32_t>(s) * C::kTile, src, bytes,
                  smem_addr(&full_bar[s]), pol);
      } else {
        mbar_arrive(smem_addr(&full_bar[s]));
      }
    }
    // every issued copy has landed before the CTA may end
    for (int s = 0; s < S && static_cast<uint32_t>(s) < j; ++s) {
      const uint32_t last = static_cast<uint32_t>(s) + ((j - 1u - s) / S) * S;
      mbar_wait_bounded(smem_addr(&full_bar[s]), (last / S) & 1u, kWaitLimitNs);
    }
    if (p.defer_wait) grid_dependency_wait();
    return;
  }

  // ---------------- consumers: units of P warps claim local tiles in order
  const int unit = warp / P;
  const int pw = warp % P;             // this warp's rows: 32 pw .. 32 pw + 31 of the tile
  const int r0 = pw * kWarpRows;
  bool ok = true;
  uint32_t j;
  if constexpr (P == 1) {
    uint32_t c = 0;
    if (lane == 0) c = atomicAdd(&claim_ctr, 1u);
    j = __shfl_sync(0xffffffffu, c, 0);
  } else {
    if (pw == 0 && lane == 0) claim_slot[unit * 2] = atomicAdd(&claim_ctr, 1u);
    named_barrier(1 + unit, 32 * P);
    j = claim_slot[unit * 2];
  }
#pragma unroll 1
  for (uint32_t use_u = 0; j < mine; ++use_u) {
    const int s = static_cast<int>(j % S);
    // Units claim tiles ahead of the ring (possibly laps ahead of a copy still
    // in flight in the same stage), so a parity alone cannot name the phase:
    // first the producer's record that this stage now takes tile j (issued
    // after the stage's previous tile was released), then that copy's phase.
    if (ok && !wait_stage_tile(&stage_tile[s], j, kWaitLimitNs)) ok = false;
    if (ok && !mbar_wait_bounded(smem_addr(&full_bar[s]), (j / S) & 1u, kWaitLimitNs)) ok = false;
    if (!ok && lane == 0) atomicOr(p.fault, 8u);
    const Tile k = decode_tile(blockIdx.x + j * gridDim.x, p);
    const QuantJob &job = p.jobs[k.job];
    const int64_t lr0 = static_cast<int64_t>(k.g) * G;
    const int rows_here = static_cast<int>(min(static_cast<int64_t>(G), p.rows - lr0));
    const bool full = rows_here >= G;
    // this lane's 8 bytes (channels 4 lane .. 4 lane + 3) of tile row 0
    const uint32_t base = ring0 + static_cast<uint32_t>(s) * C::kTile + 8u * lane;

    // pass 1: extremes of this warp's 32 rows (ragged tiles: rows past the
    // end repeat the last row, the post's edge padding)
    __half2 mn0a, mn0b, mx0a, mx0b, mn1a, mn1b, mx1a, mx1b;
    {
      const uint2 v = lds64(base + (full ? r0 : min(r0, rows_here - 1)) * kRowBytes);
      mn0a = mn0b = mx0a = mx0b = u32_as_h2(v.x);
      mn1a = mn1b = mx1a = mx1b = u32_as_h2(v.y);
    }
    if (full) {
#pragma unroll
      for (int i = 1; i < kWarpRows; i += 2) {
        const uint2 v = lds64(base + (r0 + i) * kRowBytes);
        mn0a = __hmin2(mn0a, u32_as_h2(v.x));
        mx0a = __hmax2(mx0a, u32_as_h2(v.x));
        mn1a = __hmin2(mn1a, u32_as_h2(v.y));
        mx1a = __hmax2(mx1a, u32_as_h2(v.y));
        if (i + 1 < kWarpRows) {
          const uint2 w = lds64(base + (r0 + i + 1) * kRowBytes);
          mn0b = __hmin2(mn0b, u32_as_h2(w.x));
          mx0b = __hmax2(mx0b, u32_as_h2(w.x));
          mn1b = __hmin2(mn1b, u32_as_h2(w.y));
          mx1b = __hmax2(mx1b, u32_as_h2(w.y));
        }
      }
    } else {
#pragma unroll 1
      for (int i = 1; i < kWarpRows; ++i) {
        const uint2 v = lds64(base + min(r0 + i, rows_here - 1) * kRowBytes);
        mn0a = __hmin2(mn0a, u32_as_h2(v.x));
        mx0a = __hmax2(mx0a, u32_as_h2(v.x));
        mn1a = __hmin2(mn1a, u32_as_h2(v.y));
        mx1a = __hmax2(mx1a, u32_as_h2(v.y));
      }
    }
    __half2 mn0 = __hmin2(mn0a, mn0b), mx0 = __hmax2(mx0a, mx0b);
    __half2 mn1 = __hmin2(mn1a, mn1b), mx1 = __hmax2(mx1a, mx1b);
    uint32_t j_next;
    if constexpr (P > 1) {
      // the unit's P partials meet in shared memory, double-buffered by the
      // unit's tile parity (a buffer is rewritten two tiles later, after every
      // warp of the unit has passed the barrier in between); the unit's next
      // tile is claimed here and read after the same barrier
      const uint32_t par = use_u & 1u;
      uint4 *xb = xch + ((unit * 2 + par) * P) * 32;
      xb[pw * 32 + lane] = make_uint4(h2_as_u32(mn0), h2_as_u32(mx0), h2_as_u32(mn1),
                                      h2_as_u32(mx1));
      if (pw == 0 && lane == 0) claim_slot[unit * 2 + (par ^ 1u)] = atomicAdd(&claim_ctr, 1u);
      named_barrier(1 + unit, 32 * P);
      j_next = claim_slot[unit * 2 + (par ^ 1u)];
#pragma unroll
      for (int pp = 0; pp < P; ++pp) {
        const uint4 e = xb[pp * 32 + lane];
        mn0 = __hmin2(mn0, u32_as_h2(e.x));
        mx0 = __hmax2(mx0, u32_as_h2(e.y));
        mn1 = __hmin2(mn1, u32_as_h2(e.z));
        mx1 = __hmax2(mx1, u32_as_h2(e.w));
      }
    } else {
      uint32_t c = 0;
      if (lane == 0) c = atomicAdd(&claim_ctr, 1u);
      j_next = __shfl_sync(0xffffffffu, c, 0);
    }

    // group parameters of the lane's four channels
    const float2 a0 = __half22float2(mn0), b0 = __half22float2(mx0);
    const float2 a1 = __half22float2(mn1), b1 = __half22float2(mx1);
    const GroupQ g0 = make_group_szr(a0.x, b0.x, qf), g1 = make_group_szr(a0.y, b0.y, qf);
    const GroupQ g2 = make_group_szr(a1.x, b1.x, qf), g3 = make_group_szr(a1.y, b1.y, qf);
    const GroupD2 q01 = make_group_d2(g0, g1), q23 = make_group_d2(g2, g3);
    const float4 sc = make_float4(g0.scale, g1.scale, g2.scale, g3.scale);
    const float4 ze = make_float4(g0.zero, g1.zero, g2.zero, g3.zero);
    const int64_t out_g = p.out0 + k.g;
    // debug builds: the code words, scales, zeros and reconstruction rows this
    // lane writes lie inside its bh slice
    const bool codes_out =
        (!RECON || job.codes != nullptr) &&
        KIVI_BOUND(p.fault, (out_g * (G / W) + pw * (kWarpRows / W) + kWarpRows / W - 1) * kD +
                                    4 * lane + 4 <= p.codes_bh_stride &&
                                out_g * kD + 4 * lane + 4 <= p.sz_bh_stride);
    const bool y_ok = KIVI_BOUND(
        p.fault, !RECON || rows_here <= r0 ||
                     (p.y_row0 + lr0 + min(rows_here, r0 + kWarpRows) - 1) * kD + 4 * lane + 4 <=
                         p.y_bh_stride);
    if (pw == 0 && codes_out) {
      const int64_t o = static_cast<int64_t>(k.b) * p.sz_bh_stride + out_g * kD + 4 * lane;
      __stcs(reinterpret_cast<float4 *>(job.scale + o), sc);
      __stcs(reinterpret_cast<float4 *>(job.zero + o), ze);
    }
    uint32_t *cdst = codes_out ? job.codes + static_cast<int64_t>(k.b) * p.codes_bh_stride +
                                     (out_g * (G / W) + pw * (kWarpRows / W)) * kD + 4 * lane
                               : nullptr;
    __half *ydst = RECON && y_ok ? static_cast<__half *>(job.y) + static_cast<int64_t>(k.b) * p.y_bh_stride +
                               (p.y_row0 + lr0 + r0) * kD + 4 * lane
                         : nullptr;

    // pass 2: the warp's rows quantized and packed
    if (full)
      key_rows<BITS, RECON, true>(base, r0, rows_here, q01, q23, sc, ze, qf, cdst, ydst);
    else
      key_rows<BITS, RECON, false>(base, r0, rows_here, q01, q23, sc, ze, qf, cdst, ydst);
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_addr(&empty_bar[s]));
    j = j_next;
  }
  if (p.defer_wait) grid_dependency_wait();
}

template <int BITS, int G, int MODE>
cudaError_t key_staged_launch(const QuantParams &p, cudaStream_t stream) {
  using C = KeyStaged<G>;
  auto kern = key_quant_staged_kernel<BITS, G, MODE>;
  constexpr int kMaxDevices = 64;
  static std::atomic<bool> configured[kMaxDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (!configured[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return e;
    configured[dev].store(true, std::memory_order_release);
  }
  const int64_t ng = (p.rows + G - 1) / G;
  const int64_t tiles = static_cast<int64_t>(p.n_jobs) * p.bh * ng;
  const int64_t grid = std::max<int64_t>(1, std::min<int64_t>(tiles, current_sm_count()));
  QuantParams q = p;
  q.div_rows = FastDiv::make(static_cast<uint32_t>(ng));
  q.div_bh = FastDiv::make(static_cast<uint32_t>(p.bh));
  e = fault_word_address(&q.fault);
  if (e != cudaSuccess) return e;
  return launch_dependent(kern, grid, C::kThreads, stream, q, C::kSmem);
}

template <int BITS, int MODE>
cudaError_t key_staged_by_group(const QuantParams &p, int group, cudaStream_t stream) {
  switch (group) {
    case 32: return key_staged_launch<BITS, 32, MODE>(p, stream);
    case 64: return key_staged_launch<BITS, 64, MODE>(p, stream);
    default: return key_staged_launch<BITS, 128, MODE>(p, stream);
  }
}

template <int MODE>
cudaError_t key_staged_by_bits(const QuantParams &p, int group, int bits, cudaStream_t stream) {
  switch (bits) {
    case 2: return key_staged_by_group<2, MODE>(p, group, stream);
    case 4: return key_staged_by_group<4, MODE>(p, group, stream);
    default: return key_staged_by_group<8, MODE>(p, group, stream);
  }
}

}  // namespace

cudaError_t launch_key_quant_staged(const QuantParams &p, int group, int bits, int mode,
                                    cudaStream_t stream, bool *handled) {
  *handled = false;
  if (p.d != kD || (group != 32 && group != 64 && group != 128)) return cudaSuccess;
  if (bits != 2 && bits != 4 && bits != 8) return cudaSuccess;
  // the fused form (kQuantRecon) stays on the register kernel: measured faster there
  if (mode != kQuantPlain) return cudaSuccess;
  if (p.sz_bh_stride % 4 != 0) return cudaSuccess;   // 16-byte scale / zero rows
  *handled = true;
  return key_staged_by_bits<kQuantPlain>(p, group, bits, stream);
}

}  // namespace kivi_impl
