// kivi_sink.cu -- KIVI-Sink: tokens with anomalously high key L2-norm kept
// fp16 and left out of the quantization-parameter calibration (VeloxQuant-MLX
// project description, section "KVSink-adapted sink protection": the mean of
// the key norms over the KV heads ranks the token positions, a running top-k
// is kept, and a flushed token in it is stored fp16 instead of quantized).
//
//   sink_score_tile_kernel  block per 32 new tokens of a (layer, sequence):
//                        rows staged in shared memory, the scores
//                        (sink_score_kernel, thread per token: > 64 heads)
//   sink_select_kernel   block per (layer, sequence): the new scores merged
//                        into the running top-k
//   sink_prepare_kernel  block per (layer, sequence), before the flush's
//                        quantize kernels: which of the tokens being flushed
//                        are in the top-k (one bit each, read by their sink
//                        mode), and the flushed sinks' positions and fp16
//                        key / value rows into the sink store, in position
//                        order
//   sink_restore_kernel  the sink rows put back into dequantized tensors
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "kivi_device.cuh"
#include "kivi_launch.h"

namespace kivi_impl {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

// a ranks before b: larger score, then smaller position
__device__ __forceinline__ bool ranks_before(float sa, int64_t pa, float sb, int64_t pb) {
  return sa > sb || (sa == sb && pa < pb);
}

// Score of one token: (sum over heads of the key row's L2 norm) / heads, in
// binary32 -- squared norm by fused multiply-adds in channel order, correctly
// rounded square root, norms added in head order, one correctly rounded
// division.
// The row is read 8 sixteen-byte pieces at a time (the loads of a batch are
// in flight together; the accumulation order stays the channel order).
__device__ float token_score(const __half *k_seq, int64_t head_stride, int heads, int64_t d) {
  constexpr int kBatch = 8;
  float sum = 0.0f;
  for (int h = 0; h < heads; ++h) {
    const uint4 *row = reinterpret_cast<const uint4 *>(k_seq + h * head_stride);
    float acc = 0.0f;
    for (int64_t c0 = 0; c0 < d / 8; c0 += kBatch) {
      uint4 v[kBatch];
#pragma unroll
      for (int b = 0; b < kBatch; ++b)
        v[b] = c0 + b < d / 8 ? row[c0 + b] : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
        if (c0 + b >= d / 8) break;
        const uint32_t w[4] = {v[b].x, v[b].y, v[b].z, v[b].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 f = __half22float2(kivi_dev::u32_as_h2(w[i]));
          acc = __fmaf_rn(f.x, f.x, acc);
          acc = __fmaf_rn(f.y, f.y, acc);
        }
      }
    }
    sum = __fadd_rn(sum, __fsqrt_rn(acc));
  }
  return __fdiv_rn(sum, static_cast<float>(heads));
}

// Scores of 32 consecutive new tokens of one (layer, sequence) per block.
// A warp stages 32 rows of one head through shared memory, 64 channels at a
// time, with coalesced loads (8 lanes per 128-byte row segment), and each
// lane then runs its own row's fused multiply-adds in channel order from
// shared memory; the roots of the heads' squared norms are added in head
// order and divided by the head count -- the arithmetic of token_score.
// (Reading a whole row per lane straight from global memory touches 32
// lines per warp load for 16 bytes each and caps the read near 4.5 TB/s.)
constexpr int kScoreTile = 32;                    // tokens per block
constexpr int kScoreChunk = 64;                   // channels staged per pass
constexpr int kScoreRow = kScoreChunk * 2 + 16;   // padded row: conflict-free 16-byte reads
constexpr int kScoreMaxHeads = 64;

__global__ void __launch_bounds__(kThreads, 3) sink_score_tile_kernel(const __grid_constant__ SinkParams p) {
  kivi_dev::grid_dependency_wait();
  kivi_dev::grid_launch_dependents();
  __shared__ __align__(16) unsigned char stage[kWarps][kScoreTile * kScoreRow];
  __shared__ float norm[kScoreMaxHeads * kScoreTile];
  // grid = layers x sequences x tiles (< 2^31 blocks, host-checked)
  const uint32_t tiles = static_cast<uint32_t>((p.n + kScoreTile - 1) / kScoreTile);
  const uint32_t js = blockIdx.x / tiles;
  const int64_t tile = blockIdx.x - js * tiles;
  const int job = static_cast<int>(js / static_cast<uint32_t>(p.batch));
  const int64_t seq = js - static_cast<uint32_t>(job) * static_cast<uint32_t>(p.batch);
  const SinkJob &J = p.jobs[job];
  const int64_t i_base = tile * kScoreTile;
  const int ntok = static_cast<int>(p.n - i_base < kScoreTile ? p.n - i_base : kScoreTile);
  const int heads = static_cast<int>(p.heads);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  unsigned char *st = stage[warp];
  const int pc = lane & 7;                        // this lane's 16-byte piece when loading
  // the ring row of the tile's first token; this lane loads rows (lane >> 3) + 4 m
  const int64_t row0 = (p.res_head + p.i0 + i_base) % p.r_cap;
  const int64_t r_lane = row0 + (lane >> 3);
  // The warp's work is the sequence of items (head h = warp + 8 k, chunk c);
  // the loads of item i + 1 are issued before item i is accumulated.
  const int chunks = static_cast<int>((p.d + kScoreChunk - 1) / kScoreChunk);
  const int my_heads = heads > warp ? (heads - warp + kWarps - 1) / kWarps : 0;
  const int items = my_heads * chunks;
  uint4 v[kScoreTile / 4];
  auto load = [&](int item) {
    const int h = warp + kWarps * (item / chunks);
    const int64_t c0 = static_cast<int64_t>(item % chunks) * kScoreChunk;
    const int pieces = static_cast<int>(p.d - c0 < kScoreChunk ? p.d - c0 : kScoreChunk) / 8;
    const __half *kc = static_cast<const __half *>(J.k_res) +
                       (seq * p.heads + h) * p.r_cap * p.d + c0 + 8 * pc;
#pragma unroll
    for (int m = 0; m < kScoreTile / 4; ++m) {
      const int r = (lane >> 3) + 4 * m;
      if (r < ntok && pc < pieces) {
        int64_t row = r_lane + 4 * m;
        if (row >= p.r_cap) row -= p.r_cap;       // r < n <= r_cap: one wrap at most
        v[m] = *reinterpret_cast<const uint4 *>(kc + row * p.d);
      }
    }
  };
  if (items > 0) load(0);
  float acc = 0.0f;
  for (int it = 0; it < items; ++it) {
    const int c = it % chunks;
    const int64_t c0 = static_cast<int64_t>(c) * kScoreChunk;
    const int pieces = static_cast<int>(p.d - c0 < kScoreChunk ? p.d - c0 : kScoreChunk) / 8;
#pragma unroll
    for (int m = 0; m < kScoreTile / 4; ++m) {
      const int r = (lane >> 3) + 4 * m;
      if (r < ntok && pc < pieces)
        *reinterpret_cast<uint4 *>(st + r * kScoreRow + 16 * pc) = v[m];
    }
    __syncwarp();
    if (it + 1 < items) load(it + 1);             // in flight during the accumulation
    if (lane < ntok) {
      for (int q = 0; q < pieces; ++q) {
        const uint4 w4 = *reinterpret_cast<const uint4 *>(st + lane * kScoreRow + 16 * q);
        const uint32_t w[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 f = __half22float2(kivi_dev::u32_as_h2(w[i]));
          acc = __fmaf_rn(f.x, f.x, acc);
          acc = __fmaf_rn(f.y, f.y, acc);
        }
      }
    }
    __syncwarp();
    if (c == chunks - 1) {                        // the head's last chunk
      const int h = warp + kWarps * (it / chunks);
      if (lane < ntok) norm[h * kScoreTile + lane] = __fsqrt_rn(acc);
      acc = 0.0f;
    }
  }
  __syncthreads();
  if (static_cast<int>(threadIdx.x) < ntok) {
    float sum = 0.0f;
    for (int h = 0; h < heads; ++h) sum = __fadd_rn(sum, norm[h * kScoreTile + threadIdx.x]);
    J.scores[seq * p.r_cap + i_base + threadIdx.x] = __fdiv_rn(sum, static_cast<float>(heads));
  }
}

// thread = (job, sequence, new token): its score into the scores scratch
// (more than 64 heads per sequence)
__global__ void __launch_bounds__(kThreads) sink_score_kernel(const __grid_constant__ SinkParams p) {
  kivi_dev::grid_dependency_wait();
  kivi_dev::grid_launch_dependents();
  const int64_t u = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
  if (u >= static_cast<int64_t>(p.n_jobs) * p.batch * p.n) return;
  const int64_t i = u % p.n, js = u / p.n;
  const int job = static_cast<int>(js / p.batch);
  const int64_t seq = js - static_cast<int64_t>(job) * p.batch;
  const SinkJob &J = p.jobs[job];
  const int64_t li = p.i0 + i;                                   // logical residual token
  const int64_t row = (p.res_head + li) % p.r_cap;
  const __half *k_seq = static_cast<const __half *>(J.k_res) + seq * p.heads * p.r_cap * p.d;
  J.scores[seq * p.r_cap + i] =
      token_score(k_seq + row * p.d, p.r_cap * p.d, static_cast<int>(p.heads), p.d);
}

// Sorted (best first) list of up to LK candidates kept by one thread;
// has() / hs() / hq(): the best candidate not yet taken; pop() takes it.
template <int LK>
struct LocalTop {
  float s[LK];
  int64_t q[LK];
  int n, head;
  __device__ __forceinline__ void init() { n = head = 0; }
  __device__ __forceinline__ void offer(float sc, int64_t pos, int k) {
    if (n == k && !ranks_before(sc, pos, s[n - 1], q[n - 1])) return;
    int i = n < k ? n++ : n - 1;                  // slot freed at the end
#pragma unroll 1
    while (i > 0 && ranks_before(sc, pos, s[i - 1], q[i - 1])) {
      s[i] = s[i - 1];
      q[i] = q[i - 1];
      --i;
    }
    s[i] = sc;
    q[i] = pos;
  }
  __device__ __forceinline__ bool has() const { return head < n; }
  __device__ __forceinline__ float hs() const { return s[head]; }
  __device__ __forceinline__ int64_t hq() const { return q[head]; }
  __device__ __forceinline__ void pop() { ++head; }
};

// The same for k <= 8, held in registers: every index is static (an unrolled
// insertion network), empty slots are sentinels that every real candidate
// ranks before (scores are finite and non-negative), and the list keeps its
// best 8 (a superset of the best k).
struct RegTop8 {
  static constexpr int LK = 8;
  static constexpr int64_t kNone = INT64_MAX;
  float s[LK];
  int64_t q[LK];
  __device__ __forceinline__ void init() {
#pragma unroll
    for (int i = 0; i < LK; ++i) {
      s[i] = -INFINITY;
      q[i] = kNone;
    }
  }
  __device__ __forceinline__ void offer(float sc, int64_t pos, int) {
    if (!ranks_before(sc, pos, s[LK - 1], q[LK - 1])) return;
#pragma unroll
    for (int i = LK - 1; i > 0; --i) {   // slot i from the old slots i-1 and i
      const bool here = ranks_before(sc, pos, s[i], q[i]);
      const bool above = ranks_before(sc, pos, s[i - 1], q[i - 1]);
      s[i] = here ? (above ? s[i - 1] : sc) : s[i];
      q[i] = here ? (above ? q[i - 1] : pos) : q[i];
    }
    if (ranks_before(sc, pos, s[0], q[0])) {
      s[0] = sc;
      q[0] = pos;
    }
  }
  __device__ __forceinline__ bool has() const { return q[0] != kNone; }
  __device__ __forceinline__ float hs() const { return s[0]; }
  __device__ __forceinline__ int64_t hq() const { return q[0]; }
  __device__ __forceinline__ void pop() {
#pragma unroll
    for (int i = 0; i < LK - 1; ++i) {
      s[i] = s[i + 1];
      q[i] = q[i + 1];
    }
    s[LK - 1] = -INFINITY;
    q[LK - 1] = kNone;
  }
};

// A list head as a ranking key: sb = the score's bits + 1 (scores are
// finite and non-negative, so their bit patterns order as unsigned
// integers; 0 = no candidate) and the position.
struct HeadKey {
  uint32_t sb;
  int64_t pos;
};

// The best key over the 32 lanes of a warp (largest score, then smallest
// position), by three warp reductions: the largest score, then among the
// lanes holding it the smallest high and low position words (positions are
// non-negative).
__device__ __forceinline__ HeadKey warp_best(uint32_t sb, int64_t pos) {
  const uint32_t best = __reduce_max_sync(0xffffffffu, sb);
  const uint32_t hi = static_cast<uint32_t>(static_cast<uint64_t>(pos) >> 32);
  const uint32_t lo = static_cast<uint32_t>(static_cast<uint64_t>(pos));
  const bool in = sb == best;
  const uint32_t bhi = __reduce_min_sync(0xffffffffu, in ? hi : 0xFFFFFFFFu);
  const uint32_t blo = __reduce_min_sync(0xffffffffu, in && hi == bhi ? lo : 0xFFFFFFFFu);
  return {best, static_cast<int64_t>((static_cast<uint64_t>(bhi) << 32) | blo)};
}

// block = (job, sequence): the new scores and the kept top-k merged.  Each
// of the NT threads keeps the best k of its strided share; k rounds of a
// block-wide argmax over the threads' list heads (warp reductions within
// each warp, then across the warps' winners in warp 0) give the k best
// overall.
template <typename List, int NT>
__global__ void __launch_bounds__(NT) sink_select_kernel(const __grid_constant__ SinkParams p) {
  kivi_dev::grid_dependency_wait();
  kivi_dev::grid_launch_dependents();
  constexpr int NW = NT / 32;
  const int job = static_cast<int>(blockIdx.x / p.batch);
  const int64_t seq = blockIdx.x - static_cast<int64_t>(job) * p.batch;
  const SinkJob &J = p.jobs[job];
  __shared__ float new_s[kMaxSinkTop];
  __shared__ int64_t new_p[kMaxSinkTop];
  __shared__ uint32_t red_sb[NW];
  __shared__ int64_t red_p[NW];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int k = p.k_top;
  List lt;
  lt.init();
  const int tn = J.top_count[seq];
  for (int e = tid; e < tn; e += NT)
    lt.offer(J.top_score[seq * p.k_top + e], J.top_pos[seq * p.k_top + e], k);
  // the thread's strided share of the new scores, loaded kBatch at a time
  // (independent loads in flight together) and then offered in order
  constexpr int kBatch = 8;
  const float *sc = J.scores + seq * p.r_cap;
  for (int64_t i0 = tid; i0 < p.n; i0 += kBatch * NT) {
    float v[kBatch];
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int64_t i = i0 + static_cast<int64_t>(b) * NT;
      v[b] = i < p.n ? sc[i] : 0.0f;
    }
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int64_t i = i0 + static_cast<int64_t>(b) * NT;
      if (i < p.n) lt.offer(v[b], p.s_q + p.i0 + i, k);
    }
  }
  const int64_t avail = tn + p.n;
  const int keep = avail < k ? static_cast<int>(avail) : k;
  for (int j = 0; j < keep; ++j) {
    const bool have = lt.has();
    const uint32_t sb = have ? __float_as_uint(lt.hs()) + 1u : 0u;
    const int64_t hp = have ? lt.hq() : INT64_MAX;
    const HeadKey wk = warp_best(sb, hp);
    if (lane == 0) {
      red_sb[warp] = wk.sb;
      red_p[warp] = wk.pos;
    }
    __syncthreads();
    if (warp == 0) {
      const HeadKey bk = warp_best(lane < NW ? red_sb[lane] : 0u, lane < NW ? red_p[lane] : INT64_MAX);
      if (lane == 0) {
        new_s[j] = __uint_as_float(bk.sb - 1u);
        new_p[j] = bk.pos;
      }
    }
    __syncthreads();
    // the one thread whose list head is the winner (positions are unique)
    // takes it off; warp 0 writes the next round's entry only after the
    // next barrier
    if (have && sb == __float_as_uint(new_s[j]) + 1u && hp == new_p[j]) lt.pop();
  }
  if (tid < keep) {
    J.top_score[seq * p.k_top + tid] = new_s[tid];
    J.top_pos[seq * p.k_top + tid] = new_p[tid];
  }
  if (tid == 0) J.top_count[seq] = keep;
}

// block = (job, sequence), before the flush's quantize kernels: the
// flushed top-k positions in ascending order; one mask bit per flushed token
// (in the top-k or not), read by the quantize kernels' sink mode; the sinks'
// positions and fp16 key / value rows of every head appended to the sink
// store (the quantize kernels read neither the store nor its count).  An
// overflowing store keeps what fits (the earliest flushed sinks) and sets
// bit 1 of the device fault word; the mask flags only the sinks it kept, so
// the flushed top-k tokens that did not fit are quantized as plain tokens
// rather than lost.
__global__ void __launch_bounds__(kThreads) sink_prepare_kernel(const __grid_constant__ SinkParams p) {
  kivi_dev::grid_dependency_wait();
  kivi_dev::grid_launch_dependents();
  const int job = static_cast<int>(blockIdx.x / p.batch);
  const int64_t seq = blockIdx.x - static_cast<int64_t>(job) * p.batch;
  const SinkJob &J = p.jobs[job];
  __shared__ int64_t pos[kMaxSinkTop];
  __shared__ int slot0, m;
  if (threadIdx.x == 0) {
    int cnt = 0;
    const int tn = J.top_count[seq];
    for (int e = 0; e < tn; ++e) {
      const int64_t q = J.top_pos[seq * p.k_top + e];
      if (q < p.s_q || q >= p.s_q + p.n) continue;
      int i = cnt++;
      while (i > 0 && pos[i - 1] > q) {
        pos[i] = pos[i - 1];
        --i;
      }
      pos[i] = q;
    }
    const int have = J.sink_count[seq];
    if (have + cnt > p.sink_cap) {   // the store is full: record it, keep what fits
      atomicOr(p.fault, 2u);
      cnt = max(0, p.sink_cap - have);
    }
    for (int i = 0; i < cnt; ++i) J.sink_pos[seq * p.sink_cap + have + i] = pos[i];
    J.sink_count[seq] = have + cnt;
    slot0 = have;
    m = cnt;
  }
  __syncthreads();
  const int64_t words = (p.n + 31) / 32;
  for (int64_t w = threadIdx.x; w < words; w += kThreads) {
    const int64_t lo = p.s_q + 32 * w;
    uint32_t bits = 0u;
    for (int e = 0; e < m; ++e)   // the stored sinks only
      if (pos[e] >= lo && pos[e] < lo + 32) bits |= 1u << (pos[e] - lo);
    J.mask[seq * p.mask_words + w] = bits;
  }
  const int64_t chunks = p.d / 8;                       // 16-byte pieces per row
  const int64_t total = static_cast<int64_t>(m) * p.heads * chunks;
  for (int64_t idx = threadIdx.x; idx < total; idx += kThreads) {
    const int64_t c = idx % chunks;
    const int64_t hj = idx / chunks;
    const int64_t h = hj % p.heads, j = hj / p.heads;
    const int64_t bb = seq * p.heads + h;
    const int64_t row = (p.res_head + (pos[j] - p.s_q)) % p.r_cap;
    const int64_t dst = (bb * p.sink_cap + slot0 + j) * p.d + 8 * c;
    const int64_t src = (bb * p.r_cap + row) * p.d + 8 * c;
    *reinterpret_cast<uint4 *>(static_cast<__half *>(J.sink_k) + dst) =
        *reinterpret_cast<const uint4 *>(static_cast<const __half *>(J.k_res) + src);
    *reinterpret_cast<uint4 *>(static_cast<__half *>(J.sink_v) + dst) =
        *reinterpret_cast<const uint4 *>(static_cast<const __half *>(J.v_res) + src);
  }
}

// thread = (job, sequence, sink slot, head, 16-byte piece)
__global__ void __launch_bounds__(kThreads) sink_restore_kernel(const __grid_constant__ SinkParams p) {
  kivi_dev::grid_dependency_wait();
  kivi_dev::grid_launch_dependents();
  const int64_t chunks = p.d / 8;
  const int64_t per_seq = static_cast<int64_t>(p.sink_cap) * p.heads * chunks;
  const int64_t u = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
  if (u >= static_cast<int64_t>(p.n_jobs) * p.batch * per_seq) return;
  const int64_t js = u / per_seq, r = u % per_seq;
  const int job = static_cast<int>(js / p.batch);
  const int64_t seq = js - static_cast<int64_t>(job) * p.batch;
  const SinkJob &J = p.jobs[job];
  const int64_t c = r % chunks, hj = r / chunks;
  const int64_t h = hj % p.heads, j = hj / p.heads;
  // the count, the slot's position and its rows are read together (slot j <
  // sink_cap lies inside every array whether or not it is in use), so the
  // thread waits for one round trip instead of three
  const int64_t bb = seq * p.heads + h;
  const int64_t src = (bb * p.sink_cap + j) * p.d + 8 * c;
  const int cnt = J.sink_count[seq];
  const int64_t t = J.sink_pos[seq * p.sink_cap + j];
  const uint4 kv = *reinterpret_cast<const uint4 *>(static_cast<const __half *>(J.sink_k) + src);
  const uint4 vv = *reinterpret_cast<const uint4 *>(static_cast<const __half *>(J.sink_v) + src);
  if (j >= cnt || t < 0 || t >= p.out_rows) return;
  const int64_t dst = (bb * p.out_rows + t) * p.d + 8 * c;
  *reinterpret_cast<uint4 *>(static_cast<__half *>(J.k_out) + dst) = kv;
  *reinterpret_cast<uint4 *>(static_cast<__half *>(J.v_out) + dst) = vv;
}

unsigned blocks_for(int64_t threads) {
  return static_cast<unsigned>((threads + kThreads - 1) / kThreads);
}

}  // namespace

cudaError_t launch_sink_update(const SinkParams &p, cudaStream_t stream) {
  cudaError_t e;
  if (p.heads <= kScoreMaxHeads) {
    const int64_t tiles = (p.n + kScoreTile - 1) / kScoreTile;
    e = launch_dependent(sink_score_tile_kernel, p.n_jobs * p.batch * tiles, kThreads, stream, p);
  } else {
    e = launch_dependent(sink_score_kernel,
                         static_cast<int64_t>(blocks_for(static_cast<int64_t>(p.n_jobs) * p.batch * p.n)),
                         kThreads, stream, p);
  }
  if (e != cudaSuccess) return e;
  const int64_t blocks = static_cast<int64_t>(p.n_jobs) * p.batch;
  // 1024 threads: a short share of the scores per thread (the offers are the
  // serial part); the list heads meet in two shuffle stages per round
  constexpr int kSelectThreads = 1024;
  if (p.k_top <= 8)
    return launch_dependent(sink_select_kernel<RegTop8, kSelectThreads>, blocks, kSelectThreads,
                            stream, p);
  return launch_dependent(sink_select_kernel<LocalTop<kMaxSinkTop>, kSelectThreads>, blocks,
                          kSelectThreads, stream, p);
}

cudaError_t launch_sink_prepare(const SinkParams &p, cudaStream_t stream) {
  return launch_dependent(sink_prepare_kernel, static_cast<int64_t>(p.n_jobs) * p.batch, kThreads,
                          stream, p);
}

cudaError_t launch_sink_restore(const SinkParams &p, cudaStream_t stream) {
  const int64_t threads =
      static_cast<int64_t>(p.n_jobs) * p.batch * p.sink_cap * p.heads * (p.d / 8);
  if (threads == 0) return cudaSuccess;
  return launch_dependent(sink_restore_kernel, static_cast<int64_t>(blocks_for(threads)), kThreads,
                          stream, p);
}

}  // namespace kivi_impl
