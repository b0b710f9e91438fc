// kivi_attention_ws.cu -- decode attention over the packed KIVI store on the
// fifth-generation tensor cores, warp-specialised and persistent.
//
// What it computes is that of decode_attention_kernel (kivi_attention_kernel.cuh):
// for every layer,
// sequence and query head, softmax(scale * q K^T) V over the cache's store
// tokens (dequantized on chip, bit-identical to the dequantize kernels' fp16
// reconstructions) followed by its fp16 residual tokens, query head h reading
// KV head h / r (the fused-kernel post's closing section: attention that
// reads the packed codes).  It serves head_dim 128 with G >= 32 and no sink
// store, with the operand layouts, descriptors and expansion of
// kivi_tc_common.cuh.
//
// One CTA per SM walks work items (layer, bh, split) blockIdx.x,
// blockIdx.x + gridDim.x, ..., and each item's 128-token tiles (store tiles,
// then residual tiles), with the roles in separate warps that meet only on
// mbarriers:
//   warp 0      copies each store tile's codes, scales and zeros into a ring
//               of NS stages (bulk copies; `full` / `empty` barriers);
//   warps 6-21  two groups of 8: group e expands the tiles g with g % 2 = e,
//               keys into fp16 key operand e and values into value operand
//               e (residual tiles: the fp16 rows), arriving on `kfull` /
//               `vfull`; an operand is refilled once the MMA that read it
//               two tiles earlier has completed (`sfull` / `odone`); the
//               first tile of an item also writes the item's query operand;
//   warp 1      one thread issues S^T = K Q^T of tile g into score buffer
//               g % 4 of tensor memory (columns 16 (g % 4) .. + 15; M = 128
//               tokens, N = 16), once the softmax has read that buffer's
//               previous tile (`sfree`), and commits to `sfull`;
//   warp 22     one thread issues O^T += V^T P^T of tile g into columns
//               64 .. 79 and commits to `odone`; the score and output
//               streams do not wait on each other;
//   warps 2-5   read the scores back (lane = token, 8 heads per thread),
//               update the softmax and write P (fp16 high and low parts as
//               one N = 16 operand, double-buffered) for the output MMA
//               (`pfull`); at the end of an item they fold the output out of
//               tensor memory and write it (or the split's partial).
// The softmax reference of a head moves only when a score exceeds it by
// more than 2^7 (one vote of the four softmax warps on a named barrier);
// then the tile maximum is exchanged, the output accumulated so far is read
// back and rescaled into registers, and the next output MMA starts a new
// accumulation -- otherwise no exchange is needed.  P = 2^(s - m + 8) <=
// 2^15 stays a finite fp16; o and l are relative to the same reference.
//
// Every mbarrier wait is bounded (0.2 s of the global timer).  A timeout
// sets bit 0 of the device fault word and a shared abort flag; every role
// then leaves its loop (the softmax warps together, by a vote on their
// named barrier), the copy and MMA threads wait (bounded) for their
// operations in flight, and the CTA frees its tensor memory.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>

#include "kivi_tc_common.cuh"

namespace kivi_impl {
namespace {

using namespace tcc;

constexpr int kProdWarp = 0;
constexpr int kSWarp = 1;                   // issues the score MMAs
constexpr int kSoftWarp0 = 2;               // softmax warps 2..5
constexpr int kSoftWarps = 4;
constexpr int kExpWarp0 = 6;                // expansion warps 6..21: two groups of 8
constexpr int kExpWarps = 8;                // warps of a group (one tile's expansion)
constexpr int kOWarp = kExpWarp0 + 2 * kExpWarps;   // issues the output MMAs
constexpr int kWsWarps = kOWarp + 1;
constexpr int kWsThreads = 32 * kWsWarps;
constexpr int kSBufs = 4;                   // score buffers in tensor memory
constexpr uint32_t kWsTmemCols = 128;       // scores of four tiles: 0..63; output: 64..79
constexpr uint32_t kColO = 64;
constexpr int kMaxStages = 8;

// Shared memory (byte offsets): the key, value, query and P operands (two
// of each), the staged ring, the softmax exchange and the mbarriers.
template <int BITS, int G>
struct WsFmt {
  using S = TcStage<BITS, G>;
  static constexpr int kOp = S::kOp;               // 32 KB fp16 operand
  static constexpr int kQ = kN * kD * 2;           // query operand [16][128] fp16
  static constexpr int kP = kN * kTile * 2;        // P operand [16][128] fp16
  static constexpr int oK = 0;
  static constexpr int oV = oK + 2 * kOp;
  static constexpr int oQ = oV + 2 * kOp;
  static constexpr int oP = oQ + 2 * kQ;
  static constexpr int oRing = oP + 2 * kP;
  // maxima and sums [4 warps][8 heads], accumulate flags [2], abort flag
  static constexpr int kRed = (2 * kSoftWarps * 8 + 4) * 4;
  // full, empty [kMaxStages]; kfull, vfull, pfull, odone [2]; sfull, sfree
  // [kSBufs]; TMEM address
  static constexpr int kBars = 8 * (2 * kMaxStages + 8 + 2 * kSBufs) + 16;
  static constexpr int kFixed = oRing + kRed + kBars;
  static constexpr int kAvail = (227 * 1024 - kFixed) / S::kStage;
  static constexpr int NS = kAvail > kMaxStages ? kMaxStages : kAvail;
  static constexpr int oRed = oRing + NS * S::kStage;
  static constexpr int oBar = oRed + kRed;
  static constexpr int kSmem = oBar + kBars;
  static_assert(NS >= 2 && kSmem <= 227 * 1024, "ring does not fit");
};

// The softmax warps' named barrier (id 1, 128 threads): a barrier that also
// returns whether `v` held on any of their threads.
__device__ __forceinline__ bool soft_any(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, 1, 128, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v))
      : "memory");
  return r != 0;
}
__device__ __forceinline__ void soft_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// A bounded wait (as mbar_wait_bounded) whose polls let the hardware
// suspend the thread for up to kSuspendNs until the phase completes, so a
// waiting role takes few issue slots from the expansion warps.
constexpr uint32_t kSuspendNs = 2000;
__device__ __forceinline__ bool try_wait_hint(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(kSuspendNs)
      : "memory");
  return ok != 0u;
}
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity) {
  if (try_wait_hint(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
#pragma unroll 1
  while (true) {
    if (try_wait_hint(bar, parity)) return true;
    if (global_timer_ns() - t0 > kWaitLimitNs) return false;
  }
}

// A work item's place and tiles.
struct Item {
  int job;
  int64_t bhi, b, kvh;
  int pc0, n_pc;     // store pieces [pc0, pc0 + n_pc)
  int n_st, n_rt;    // store tiles (four pieces each) and residual tiles
};
// (32-bit divisions: layers x bh x splits < 2^31, host-checked)
__device__ __forceinline__ Item item_of(const AttnParams &p, int64_t item) {
  Item it;
  const uint32_t u = static_cast<uint32_t>(item), ns = static_cast<uint32_t>(p.n_split);
  const uint32_t bh = static_cast<uint32_t>(p.bh), hkv = static_cast<uint32_t>(p.h_kv);
  const uint32_t pair = u / ns;
  const int split = static_cast<int>(u - pair * ns);
  const uint32_t job = pair / bh;
  const uint32_t bhi = pair - job * bh;
  const uint32_t b = bhi / hkv;
  it.job = static_cast<int>(job);
  it.bhi = bhi;
  it.b = b;
  it.kvh = bhi - b * hkv;
  it.pc0 = split * p.tiles_per_split;
  it.n_pc = max(0, min(it.pc0 + p.tiles_per_split, p.tiles_store) - it.pc0);
  it.n_st = (it.n_pc + 3) / 4;
  it.n_rt = split == p.n_split - 1 ? static_cast<int>((p.n_res + kTile - 1) / kTile) : 0;
  return it;
}
// Real tokens of tile t of an item (whole pieces for store tiles).
__device__ __forceinline__ int tile_valid(const AttnParams &p, const Item &it, int t) {
  if (t < it.n_st) return min(4, it.n_pc - 4 * t) * kPiece;
  const int64_t rtok0 = static_cast<int64_t>(t - it.n_st) * kTile;
  return static_cast<int>(p.n_res - rtok0 < kTile ? p.n_res - rtok0 : kTile);
}

template <int BITS, int G>
__global__ void __launch_bounds__(kWsThreads, 1) decode_attention_ws_kernel(const __grid_constant__ AttnParams p) {
  using F = WsFmt<BITS, G>;
  using S = TcStage<BITS, G>;
  constexpr int W = S::W;
  constexpr int NS = F::NS;
  extern __shared__ __align__(1024) unsigned char smem[];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t base = smem_addr(smem);
  float *red_m = reinterpret_cast<float *>(smem + F::oRed);            // [4][8]
  float *red_l = red_m + kSoftWarps * 8;                               // [4][8]
  volatile int *acc_flag = reinterpret_cast<volatile int *>(red_l + kSoftWarps * 8);  // [2]
  volatile int *abort_flag = acc_flag + 2;
  const uint32_t bar0 = base + F::oBar;
  auto full = [&](int s) { return bar0 + 8 * s; };
  auto empty = [&](int s) { return bar0 + 8 * (kMaxStages + s); };
  const uint32_t kfull0 = bar0 + 8 * (2 * kMaxStages);
  auto kfull = [&](int b) { return kfull0 + 8 * b; };
  auto vfull = [&](int b) { return kfull0 + 16 + 8 * b; };
  auto pfull = [&](int b) { return kfull0 + 32 + 8 * b; };
  auto odone = [&](int b) { return kfull0 + 48 + 8 * b; };
  auto sfull = [&](int sb) { return kfull0 + 64 + 8 * sb; };
  auto sfree = [&](int sb) { return kfull0 + 64 + 8 * kSBufs + 8 * sb; };
  uint32_t *tmem_slot =
      reinterpret_cast<uint32_t *>(smem + F::oBar + 8 * (2 * kMaxStages + 8 + 2 * kSBufs));
  auto kop = [&](int b) { return base + F::oK + b * F::kOp; };
  auto vop = [&](int b) { return base + F::oV + b * F::kOp; };
  auto qop = [&](int b) { return base + F::oQ + b * F::kQ; };
  auto pop_ = [&](int b) { return base + F::oP + b * F::kP; };
  auto stage = [&](int s) { return smem + F::oRing + s * S::kStage; };

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), kExpWarps);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(kfull(b), kExpWarps);
      mbar_init(vfull(b), kExpWarps);
      mbar_init(pfull(b), kSoftWarps);
      mbar_init(odone(b), 1);
    }
    for (int sb = 0; sb < kSBufs; ++sb) {
      mbar_init(sfull(sb), 1);
      mbar_init(sfree(sb), kSoftWarps);
    }
    acc_flag[0] = acc_flag[1] = 0;
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kProdWarp) {
    __syncwarp();
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(tmem_slot)),
                 "r"(kWsTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int64_t n_items = static_cast<int64_t>(p.n_jobs) * p.bh * p.n_split;
  const int64_t h_q = static_cast<int64_t>(p.h_kv) * p.r;
  auto fail = [&]() {
    *abort_flag = 1;
    atomicOr(p.fault, 1u);
  };

  if (warp == kProdWarp) {
    // ---------------- copies of the store tiles into the ring
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      int gs = 0;
      bool stop = false;
      for (int64_t item = blockIdx.x; item < n_items && !stop; item += gridDim.x) {
        const Item it = item_of(p, item);
        const AttnJob &J = p.jobs[it.job];
        const uint32_t *kc_bh = J.k_codes + it.bhi * (p.cap / W) * kD;
        const float *ks_bh = J.k_scale + it.bhi * (p.cap / G) * kD;
        const float *kz_bh = J.k_zero + it.bhi * (p.cap / G) * kD;
        const uint32_t *vc_bh = J.v_codes + it.bhi * p.cap * (kD / W);
        const float *vs_bh = J.v_scale + it.bhi * p.cap * (kD / G);
        const float *vz_bh = J.v_zero + it.bhi * p.cap * (kD / G);
        for (int t = 0; t < it.n_st; ++t, ++gs) {
          const int s = gs % NS;
          if (*abort_flag ||
              (gs >= NS && !wait_phase(empty(s), ((gs / NS) - 1) & 1))) {
            fail();
            stop = true;
            break;
          }
          const int np = min(4, it.n_pc - 4 * t);
          const int64_t tok = static_cast<int64_t>(it.pc0 + 4 * t) * kPiece;
          const int ntok = np * kPiece;
          const uint32_t dst = smem_addr(stage(s));
          const uint32_t kcb = ntok / W * kD * 4, ksb = (ntok + G - 1) / G * kD * 4;
          const uint32_t vcb = ntok * (kD / W) * 4, vsb = ntok * (kD / G) * 4;
          fence_proxy_async_smem();
          mbar_arrive_expect_tx(full(s), kcb + 2 * ksb + vcb + 2 * vsb);
          bulk_load(dst, kc_bh + (tok / W) * kD, kcb, full(s), pol);
          bulk_load(dst + S::oKs, ks_bh + (tok / G) * kD, ksb, full(s), pol);
          bulk_load(dst + S::oKz, kz_bh + (tok / G) * kD, ksb, full(s), pol);
          bulk_load(dst + S::oVc, vc_bh + tok * (kD / W), vcb, full(s), pol);
          bulk_load(dst + S::oVs, vs_bh + tok * (kD / G), vsb, full(s), pol);
          bulk_load(dst + S::oVz, vz_bh + tok * (kD / G), vsb, full(s), pol);
        }
      }
      // the copies still landing (stages issued but perhaps not consumed)
      for (int t = max(0, gs - NS); t < gs; ++t)
        wait_phase(full(t % NS), (t / NS) & 1);
    }
  } else if (warp == kSWarp) {
    // ---------------- the score MMAs (one thread): tile g into score buffer g % 4
    if (lane == 0) {
      int g = 0, q_ix = 0;
      bool stop = false;
      for (int64_t item = blockIdx.x; item < n_items && !stop; item += gridDim.x) {
        const Item it = item_of(p, item);
        const int n_tiles = it.n_st + it.n_rt;
        if (n_tiles == 0) continue;
        const int qb = q_ix & 1;
        ++q_ix;
        for (int t = 0; t < n_tiles; ++t, ++g) {
          const int b = g & 1, sb = g % kSBufs;
          const bool store = t < it.n_st;
          // the key operand is full; the softmax has read score buffer sb's last tile
          if (*abort_flag || !wait_phase(kfull(b), (g >> 1) & 1) ||
              (g >= kSBufs &&
               !wait_phase(sfree(sb), ((g - kSBufs) / kSBufs) & 1))) {
            fail();
            stop = true;
            break;
          }
          tc_fence_after();
          // S^T[token][head] = K Q^T over 8 steps of 16 channels
#pragma unroll
          for (int s = 0; s < kD / 16; ++s) {
            const uint64_t a = store ? smem_desc(kop(b) + s * 4096, 2048, 128)
                                     : smem_desc(kop(b) + s * 256, 128, 2048);
            mma_f16(tmem + 16 * sb, a, smem_desc(qop(qb) + s * 256, 128, 2048),
                    store ? kIdescMN : kIdescK, s > 0 ? 1u : 0u);
          }
          mma_commit(sfull(sb));
        }
      }
      // the last commit (bounded): nothing in flight at exit
      if (g > 0) wait_phase(sfull((g - 1) % kSBufs), ((g - 1) / kSBufs) & 1);
    }
  } else if (warp == kOWarp) {
    // ---------------- the output MMAs (one thread): O^T += V^T P^T of tile g
    if (lane == 0) {
      int g = 0;
      bool stop = false;
      for (int64_t item = blockIdx.x; item < n_items && !stop; item += gridDim.x) {
        const Item it = item_of(p, item);
        const int n_tiles = it.n_st + it.n_rt;
        for (int t = 0; t < n_tiles; ++t, ++g) {
          const int b = g & 1;
          if (*abort_flag || !wait_phase(vfull(b), (g >> 1) & 1) ||
              !wait_phase(pfull(b), (g >> 1) & 1)) {
            fail();
            stop = true;
            break;
          }
          tc_fence_after();
          const uint32_t acc = acc_flag[b] ? 1u : 0u;
#pragma unroll
          for (int s = 0; s < kTile / 16; ++s)
            mma_f16(tmem + kColO, smem_desc(vop(b) + s * 4096, 2048, 128),
                    smem_desc(pop_(b) + s * 512, 256, 128), kIdescO, s > 0 ? 1u : acc);
          mma_commit(odone(b));
        }
      }
      if (g > 0) wait_phase(odone((g - 1) & 1), ((g - 1) >> 1) & 1);
    }
  } else if (warp >= kExpWarp0) {
    // ---------------- expansion of the operands: group e (256 threads)
    // takes the tiles g with g % 2 == e, i.e. the operands of index e
    const int etid = (tid - 32 * kExpWarp0) & 255;
    const int egroup = (warp - kExpWarp0) / kExpWarps;
    int g = 0, gs = 0, q_ix = 0;
    bool stop = false;
    for (int64_t item = blockIdx.x; item < n_items && !stop; item += gridDim.x) {
      const Item it = item_of(p, item);
      const int n_tiles = it.n_st + it.n_rt;
      if (n_tiles == 0) continue;
      const AttnJob &J = p.jobs[it.job];
      const int qb = q_ix & 1;
      ++q_ix;
      const __half *kr = static_cast<const __half *>(J.k_res) + it.bhi * p.r_cap * kD;
      const __half *vr = static_cast<const __half *>(J.v_res) + it.bhi * p.r_cap * kD;
      for (int t = 0; t < n_tiles; ++t, ++g) {
        const int b = g & 1;
        const bool store = t < it.n_st;
        if (b != egroup) {             // the other group's tile
          if (store) ++gs;
          continue;
        }
        const int valid = tile_valid(p, it, t);
        const int s = gs % NS;
        // key operand b (and the query operand of two items back) are free
        // once the score MMA of tile g - 2 has completed; the stage is full
        bool ok = !*abort_flag;
        if (ok && g >= 2)
          ok = wait_phase(sfull((g - 2) % kSBufs), ((g - 2) / kSBufs) & 1);
        if (ok && store) ok = wait_phase(full(s), (gs / NS) & 1);
        if (!__all_sync(0xffffffffu, ok)) {
          if (lane == 0) fail();
          stop = true;
          break;
        }
        if (t == 0) {   // this item's r query heads as the B operand (rows >= r zero)
          for (int idx = etid; idx < kN * (kD / 8); idx += 32 * kExpWarps) {
            const int n = (idx & 7) + 8 * (idx >> 7), kcn = (idx >> 3) & 15;
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (n < p.r)
              v = reinterpret_cast<const uint4 *>(static_cast<const __half *>(J.q) +
                                                  (it.b * h_q + it.kvh * p.r + n) * kD)[kcn];
            sts128(qop(qb) + b_elem(n, 8 * kcn), v);
          }
        }
        if (store) {
          expand_keys_tc<BITS, G>(stage(s), kop(b), etid);
        } else {
          const int64_t rtok0 = static_cast<int64_t>(t - it.n_st) * kTile;
          load_residual_tc<false>(kr, p.r_cap, p.res_head, rtok0, valid, kop(b), etid);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(kfull(b));
        // value operand b is free once the output MMA of tile g - 2 has completed
        ok = !*abort_flag;
        if (ok && g >= 2) ok = wait_phase(odone(b), ((g - 2) >> 1) & 1);
        if (!__all_sync(0xffffffffu, ok)) {
          if (lane == 0) fail();
          stop = true;
          break;
        }
        if (store) {
          expand_values_tc<BITS, G>(stage(s), vop(b), etid, valid);
        } else {
          const int64_t rtok0 = static_cast<int64_t>(t - it.n_st) * kTile;
          load_residual_tc<BITS == 2>(vr, p.r_cap, p.res_head, rtok0, valid, vop(b), etid);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(vfull(b));
          if (store) mbar_arrive(empty(s));
        }
        if (store) ++gs;
      }
    }
  } else {
    // ---------------- softmax, output (warps 2..5; 128 threads)
    const int sw = warp - kSoftWarp0;            // 0..3
    const int r = p.r;
    const int quarter = warp & 3;                // tensor-memory lanes 32 quarter ..
    const int slot = 32 * quarter + lane;        // token slot (scores), channel slot (output)
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(32 * quarter) << 16);
    int g = 0;
    bool stop = false;
    for (int64_t item = blockIdx.x; item < n_items && !stop; item += gridDim.x) {
      const Item it = item_of(p, item);
      const int n_tiles = it.n_st + it.n_rt;
      const AttnJob &J = p.jobs[it.job];
      float m_ref[8], l_acc[8], o_acc[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        m_ref[j] = -INFINITY;
        l_acc[j] = 0.0f;
        o_acc[j] = 0.0f;
      }
      bool o_live = false;   // tensor memory holds output accumulated since the last fold
      for (int t = 0; t < n_tiles; ++t, ++g) {
        const int b = g & 1;
        const int valid = tile_valid(p, it, t);
        bool ok = !*abort_flag;
        const int sb = g % kSBufs;
        if (ok)
          ok = __all_sync(0xffffffffu, wait_phase(sfull(sb), (g / kSBufs) & 1));
        // P operand b is free once the output MMA of tile g - 2 has completed
        if (ok && g >= 2)
          ok = __all_sync(0xffffffffu, wait_phase(odone(b), ((g - 2) >> 1) & 1));
        tc_fence_after();
        float sc[8];
        if (ok) tmem_ld8(t_lane + 16 * sb, sc);
        // score buffer sb read: the next score MMA into it may start
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(sfree(sb));
        const bool real = slot < valid && ok;
        bool vote = false;
#pragma unroll
        for (int j = 0; j < 8; ++j) {   // heads past r: zero query rows, P = 0
          sc[j] = real && j < r ? sc[j] * p.scale_log2 : -INFINITY;
          vote |= sc[j] > m_ref[j] + kTau;
        }
        if (soft_any(!ok)) {
          if (sw == 0 && lane == 0) fail();
          stop = true;
          break;
        }
        if (soft_any(vote)) {
          // move the reference to the maximum over the tile and the old reference
          float mt[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) mt[j] = sc[j];
#pragma unroll
          for (int off = 16; off > 0; off >>= 1)
#pragma unroll
            for (int j = 0; j < 8; ++j) mt[j] = fmaxf(mt[j], __shfl_xor_sync(0xffffffffu, mt[j], off));
          if (lane == 0)
#pragma unroll
            for (int j = 0; j < 8; ++j) red_m[sw * 8 + j] = mt[j];
          soft_sync();
          float alpha[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            float m_t = m_ref[j];
#pragma unroll
            for (int q = 0; q < kSoftWarps; ++q) m_t = fmaxf(m_t, red_m[q * 8 + j]);
            alpha[j] = m_ref[j] == -INFINITY ? 0.0f : exp2f(m_ref[j] - m_t);
            m_ref[j] = m_t;
          }
          // fold the output accumulated so far (its last MMA, tile g - 1)
          bool ok_o = true;
          if (o_live)
            ok_o = __all_sync(0xffffffffu, wait_phase(odone((g - 1) & 1), ((g - 1) >> 1) & 1));
          if (soft_any(!ok_o)) {
            if (sw == 0 && lane == 0) fail();
            stop = true;
            break;
          }
          tc_fence_after();
          if (o_live) {
            float hi[8], lo[8];
            tmem_ld8(t_lane + kColO, hi);
            tmem_ld8(t_lane + kColO + 8, lo);
#pragma unroll
            for (int j = 0; j < 8; ++j) o_acc[j] = (o_acc[j] + hi[j] + lo[j]) * alpha[j];
          } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) o_acc[j] *= alpha[j];
          }
#pragma unroll
          for (int j = 0; j < 8; ++j) l_acc[j] *= alpha[j];
          o_live = false;
        }
        // P = 2^(s - m + 8): fp16 high parts (heads 0..7) and low parts (8..15)
        uint32_t hi2[4], lo2[4];
        float pf[8];
#pragma unroll
        for (int j = 0; j < 8; j += 2) {
          if (j < r) {   // (r is uniform: pairs past it skip the exponentials)
            pf[j] = sc[j] == -INFINITY ? 0.0f : ex2_approx(sc[j] - m_ref[j] + kLog2PScale);
            pf[j + 1] = sc[j + 1] == -INFINITY ? 0.0f : ex2_approx(sc[j + 1] - m_ref[j + 1] + kLog2PScale);
            const __half2 hh = __floats2half2_rn(pf[j], pf[j + 1]);
            const float2 hf = __half22float2(hh);
            const __half2 ll = __floats2half2_rn(pf[j] - hf.x, pf[j + 1] - hf.y);
            hi2[j / 2] = h2_as_u32(hh);
            lo2[j / 2] = h2_as_u32(ll);
          } else {
            pf[j] = pf[j + 1] = 0.0f;
            hi2[j / 2] = lo2[j / 2] = 0u;
          }
        }
        const uint32_t row = pop_(b) + p_row(slot);
        sts128(row, make_uint4(hi2[0], hi2[1], hi2[2], hi2[3]));
        sts128(row + 128, make_uint4(lo2[0], lo2[1], lo2[2], lo2[3]));
        if (sw == 0 && lane == 0) acc_flag[b] = o_live ? 1 : 0;
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(pfull(b));
#pragma unroll
        for (int j = 0; j < 8; ++j) l_acc[j] += pf[j];
        o_live = true;
      }
      if (stop) break;
      // ---- the item's result: fold the last output, sum P over the tokens
      bool ok = true;
      if (n_tiles > 0)
        ok = __all_sync(0xffffffffu, wait_phase(odone((g - 1) & 1), ((g - 1) >> 1) & 1));
      if (soft_any(!ok)) {
        if (sw == 0 && lane == 0) fail();
        stop = true;
        break;
      }
      tc_fence_after();
      if (n_tiles > 0) {
        float hi[8], lo[8];
        tmem_ld8(t_lane + kColO, hi);
        tmem_ld8(t_lane + kColO + 8, lo);
#pragma unroll
        for (int j = 0; j < 8; ++j) o_acc[j] += hi[j] + lo[j];
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1)
#pragma unroll
        for (int j = 0; j < 8; ++j) l_acc[j] += __shfl_xor_sync(0xffffffffu, l_acc[j], off);
      if (lane == 0)
#pragma unroll
        for (int j = 0; j < 8; ++j) red_l[sw * 8 + j] = l_acc[j];
      soft_sync();
      // output of channel slot `slot` (2-bit: slot m holds channel (m & ~7) | perm8(m & 7))
      const int ch = BITS == 2 ? ((slot & ~7) | perm8(slot & 7)) : slot;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (j >= p.r) continue;
        float l_t = 0.0f;
#pragma unroll
        for (int q = 0; q < kSoftWarps; ++q) l_t += red_l[q * 8 + j];
        if (p.n_split == 1) {
          J.out[(it.b * h_q + it.kvh * p.r + j) * kD + ch] = o_acc[j] / l_t;
        } else {
          const int64_t pbase = item * p.r + j;     // partial (item, head)
          p.ws[pbase * kD + ch] = o_acc[j];
          if (slot == 0) {
            float *ml = p.ws + n_items * p.r * kD;
            ml[2 * pbase] = m_ref[j];
            ml[2 * pbase + 1] = l_t;
          }
        }
      }
      soft_sync();   // red_l read by every softmax thread before it is written again
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kProdWarp) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kWsTmemCols)
                 : "memory");
  }
}

template <int BITS, int G>
cudaError_t ws_launch(const AttnParams &p, cudaStream_t stream) {
  using F = WsFmt<BITS, G>;
  auto kern = decode_attention_ws_kernel<BITS, G>;
  constexpr int kMaxDevices = 64;
  static std::atomic<bool> configured[kMaxDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (!configured[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, F::kSmem);
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
  const int64_t grid = std::min<int64_t>(items, current_sm_count());
  if (grid > 0) {
    kern<<<static_cast<unsigned>(grid), kWsThreads, F::kSmem, stream>>>(q);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (p.n_split == 1) return cudaSuccess;
  return launch_attention_combine(q, stream);
}

}  // namespace

cudaError_t launch_decode_attention_ws(const AttnParams &p, int group, int bits,
                                       cudaStream_t stream, bool *handled) {
  *handled = false;
  if (p.d != kD || p.sink_cap > 0 || p.r > kMaxR || group < 32) return cudaSuccess;
  *handled = true;
  switch (bits * 1000 + group) {
    case 2032: return ws_launch<2, 32>(p, stream);
    case 2064: return ws_launch<2, 64>(p, stream);
    case 2128: return ws_launch<2, 128>(p, stream);
    case 4032: return ws_launch<4, 32>(p, stream);
    case 4064: return ws_launch<4, 64>(p, stream);
    case 4128: return ws_launch<4, 128>(p, stream);
    case 8032: return ws_launch<8, 32>(p, stream);
    case 8064: return ws_launch<8, 64>(p, stream);
    case 8128: return ws_launch<8, 128>(p, stream);
    default: *handled = false; return cudaSuccess;
  }
}

}  // namespace kivi_impl
