// kivi_keys.cu -- per-channel key quantization and key dequantization.
//
// Keys are grouped along the token axis: one (scale, zero) per channel per
// group of G tokens (VeloxQuant-MLX KIVI fused-kernel post, "The layout
// problem that shapes everything": the group runs along the strided axis,
// consecutive group elements are d apart).  In the row-contiguous [bh][s][d]
// layout the G rows of one group are one contiguous block of G*d fp16 values,
// so a whole group tile is fetched with a single bulk asynchronous copy into
// shared memory -- no transpose is ever materialised.
//
// Quantize kernel (persistent, one tile = one (layer, bh, token group)):
//   * thread 0 keeps NS tiles in flight: mbarrier.arrive.expect_tx +
//     cp.async.bulk per stage, L2 evict-first;
//   * thread (col, split) owns channel pair (2col, 2col+1) and the 32 tokens
//     [32 split, 32 split + 32) of the group: it reads them from shared
//     memory as half2 (a warp reads 128 consecutive bytes of one row: no bank
//     conflicts), reduces min/max in half2 registers, exchanges the partial
//     extremes of the G/32 splits through a small shared buffer, then
//     quantizes its 64 values and packs its codes along tokens;
//   * one __syncthreads per tile both publishes the partial extremes and
//     frees the stage for the next bulk copy.
// Dequantize kernel: one thread per (layer, bh, group, 8 channels); 16-byte
// loads of codes, scales and zeros, 16-byte streaming stores.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "kivi_device.cuh"
#include "kivi_launch.h"

namespace kivi_impl {
namespace {

using namespace kivi_dev;

// Fault record of the quantize kernel: the first timed-out wait stores
// (1 << 31) | (block index & 0x7FFFFFFF).
__device__ unsigned int g_key_fault = 0u;

constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s

template <int G>
struct KeyTileCfg;
template <>
struct KeyTileCfg<32> { static constexpr int NS = 4; };
template <>
struct KeyTileCfg<64> { static constexpr int NS = 3; };
template <>
struct KeyTileCfg<128> { static constexpr int NS = 2; };

__host__ __device__ constexpr int key_threads(int g, int d) { return (d / 2) * (g / 32); }

template <int G>
__host__ __device__ constexpr size_t key_smem_bytes(int d) {
  // stages | mbarriers | partial extremes [2][G/32][d/2] (uint2)
  return static_cast<size_t>(KeyTileCfg<G>::NS) * G * d * 2 +
         KeyTileCfg<G>::NS * sizeof(uint64_t) + 2ull * (G / 32) * (d / 2) * sizeof(uint2);
}

struct TileRef {
  int job;
  int64_t b;
  int64_t g;
  int rows_valid;
};

__device__ __forceinline__ TileRef decode_tile(const QuantParams &p, int64_t tile, int64_t ng,
                                               int group) {
  TileRef t;
  const int64_t per_job = p.bh * ng;
  t.job = static_cast<int>(tile / per_job);
  const int64_t rem = tile - t.job * per_job;
  t.b = rem / ng;
  t.g = rem - t.b * ng;
  const int64_t left = p.rows - t.g * group;
  t.rows_valid = static_cast<int>(left < group ? left : group);
  return t;
}

template <int BITS, int G>
__global__ void __launch_bounds__(512) key_quant_kernel(const __grid_constant__ QuantParams p) {
  constexpr int NS = KeyTileCfg<G>::NS;
  constexpr int T = G / 32;                  // token splits per group
  constexpr int W = CodeFmt<BITS>::W;        // codes per word
  constexpr uint32_t Q = CodeFmt<BITS>::Q;
  constexpr uint32_t MAGIC_SUM = CodeFmt<BITS>::magic_sum();
  const float qf = static_cast<float>(Q);

  const int D = p.d;
  const int C = D >> 1;                      // half2 columns
  const int tid = threadIdx.x;
  const int col = tid % C;
  const int split = tid / C;

  extern __shared__ __align__(128) unsigned char smem[];
  const int stage_bytes = G * D * 2;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + static_cast<size_t>(NS) * stage_bytes);
  uint2 *red = reinterpret_cast<uint2 *>(bars + NS);

  const int64_t ng = (p.rows + G - 1) / G;
  const int64_t n_tiles = static_cast<int64_t>(p.n_jobs) * p.bh * ng;
  if (static_cast<int64_t>(blockIdx.x) >= n_tiles) return;
  const int64_t my_tiles = (n_tiles - blockIdx.x + gridDim.x - 1) / gridDim.x;

  uint64_t policy = 0;
  if (tid == 0) {
    for (int s = 0; s < NS; ++s) mbar_init(smem_addr(&bars[s]), 1u);
    fence_mbar_init();
    policy = policy_evict_first();
  }
  __syncthreads();

  auto issue = [&](int64_t i) {  // thread 0 only
    const int64_t tile = blockIdx.x + i * static_cast<int64_t>(gridDim.x);
    const TileRef t = decode_tile(p, tile, ng, G);
    int64_t row0 = t.g * G;
    if (p.ring > 0) row0 = (p.head + row0) % p.ring;
    const __half *src = static_cast<const __half *>(p.jobs[t.job].x) + t.b * p.x_bh_stride +
                        row0 * D;
    const int s = static_cast<int>(i % NS);
    const uint32_t bytes = static_cast<uint32_t>(t.rows_valid) * D * 2u;
    const uint32_t bar = smem_addr(&bars[s]);
    mbar_arrive_expect_tx(bar, bytes);
    bulk_load(smem_addr(smem + static_cast<size_t>(s) * stage_bytes), src, bytes, bar, policy);
  };

  if (tid == 0) {
    const int64_t pre = my_tiles < NS ? my_tiles : NS;
    for (int64_t i = 0; i < pre; ++i) issue(i);
  }

  int64_t i = 0;
  bool faulted = false;
#pragma unroll 1
  for (; i < my_tiles; ++i) {
    const int s = static_cast<int>(i % NS);
    const uint32_t parity = static_cast<uint32_t>((i / NS) & 1);
    const bool ok = mbar_wait_bounded(smem_addr(&bars[s]), parity, kWaitLimitNs);

    const int64_t tile = blockIdx.x + i * static_cast<int64_t>(gridDim.x);
    const TileRef t = decode_tile(p, tile, ng, G);
    const __half2 *tile_h2 =
        reinterpret_cast<const __half2 *>(smem + static_cast<size_t>(s) * stage_bytes);

    // 32 tokens of this thread's channel pair; rows past the end of a ragged
    // group repeat the last row (edge padding).
    __half2 h[32];
#pragma unroll
    for (int k = 0; k < 32; ++k) {
      int r = split * 32 + k;
      r = r < t.rows_valid ? r : t.rows_valid - 1;
      h[k] = tile_h2[r * C + col];
    }
    __half2 mn = h[0], mx = h[0];
#pragma unroll
    for (int k = 1; k < 32; ++k) {
      mn = __hmin2(mn, h[k]);
      mx = __hmax2(mx, h[k]);
    }
    uint2 *red_buf = red + (i & 1) * (T * C);
    if (T > 1) red_buf[split * C + col] = make_uint2(h2_as_u32(mn), h2_as_u32(mx));

    // Publishes the partial extremes, certifies that every thread has read
    // this stage, and agrees on a timed-out wait.
    if (__syncthreads_or(!ok)) {
      faulted = true;
      break;
    }
    if (tid == 0 && i + NS < my_tiles) issue(i + NS);

    if (T > 1) {
#pragma unroll
      for (int j = 0; j < T; ++j) {
        if (j == split) continue;
        const uint2 o = red_buf[j * C + col];
        mn = __hmin2(mn, u32_as_h2(o.x));
        mx = __hmax2(mx, u32_as_h2(o.y));
      }
    }
    const float2 mnf = __half22float2(mn);
    const float2 mxf = __half22float2(mx);
    const GroupQ g0 = make_group(mnf.x, mxf.x, qf);
    const GroupQ g1 = make_group(mnf.y, mxf.y, qf);

    // Quantize and pack along tokens: BITS words per channel, word wi holds
    // tokens [wi*W, wi*W + W) of this thread's 32.
    uint32_t w0[BITS], w1[BITS];
    bool bad = false;
#pragma unroll
    for (int wi = 0; wi < BITS; ++wi) {
      uint32_t a0 = 0u, a1 = 0u;
#pragma unroll
      for (int k = 0; k < W; ++k) {
        const float2 xf = __half22float2(h[wi * W + k]);
        a0 += fast_code_bits(xf.x, g0, bad) << (k * BITS);
        a1 += fast_code_bits(xf.y, g1, bad) << (k * BITS);
      }
      // each raw term is (0x4B400000 + q) << slot; removing the constant part
      // of all W terms leaves the packed codes
      w0[wi] = a0 - MAGIC_SUM;
      w1[wi] = a1 - MAGIC_SUM;
    }
    if (bad) {  // rare: some element needs the exact division
#pragma unroll
      for (int wi = 0; wi < BITS; ++wi) {
        uint32_t a0 = 0u, a1 = 0u;
#pragma unroll
        for (int k = 0; k < W; ++k) {
          const float2 xf = __half22float2(h[wi * W + k]);
          a0 |= exact_code(xf.x, g0, qf) << (k * BITS);
          a1 |= exact_code(xf.y, g1, qf) << (k * BITS);
        }
        w0[wi] = a0;
        w1[wi] = a1;
      }
    }

    const QuantJob &job = p.jobs[t.job];
    const int64_t out_g = p.out0 + t.g;
    uint32_t *cdst = job.codes + t.b * p.codes_bh_stride +
                     (out_g * (G / W) + split * BITS) * D + 2 * col;
#pragma unroll
    for (int wi = 0; wi < BITS; ++wi)
      st_stream(cdst + static_cast<int64_t>(wi) * D, make_uint2(w0[wi], w1[wi]));
    if (split == 0) {
      const int64_t o = t.b * p.sz_bh_stride + out_g * D + 2 * col;
      __stcs(reinterpret_cast<float2 *>(job.scale + o), make_float2(g0.scale, g1.scale));
      __stcs(reinterpret_cast<float2 *>(job.zero + o), make_float2(g0.zero, g1.zero));
    }
  }

  if (faulted && tid == 0) {
    atomicCAS(&g_key_fault, 0u, 0x80000000u | (blockIdx.x & 0x7FFFFFFFu));
    // Let every copy still in flight land before the CTA exits.
    const int64_t end = (i + NS < my_tiles) ? i + NS : my_tiles;
    for (int64_t k = i; k < end; ++k) {
      (void)mbar_wait_bounded(smem_addr(&bars[k % NS]), static_cast<uint32_t>((k / NS) & 1),
                              kWaitLimitNs);
    }
  }
}

// One thread: channels [8*chunk, 8*chunk + 8) of group g of one bh slice.
template <int BITS, int G>
__global__ void __launch_bounds__(256) key_dequant_kernel(const __grid_constant__ DequantParams p) {
  constexpr int W = CodeFmt<BITS>::W;
  constexpr uint32_t Q = CodeFmt<BITS>::Q;
  const int D = p.d;
  const int chunks = D >> 3;
  const int64_t ng = (p.rows + G - 1) / G;
  const int64_t per_job = p.bh * ng * chunks;
  const int64_t total = per_job * p.n_jobs;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
#pragma unroll 1
  for (int64_t u = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; u < total;
       u += stride) {
    const int job = static_cast<int>(u / per_job);
    int64_t rem = u - job * per_job;
    const int64_t bg = rem / chunks;
    const int ch = static_cast<int>(rem - bg * chunks);
    const int64_t b = bg / ng;
    const int64_t g = bg - b * ng;
    const DequantJob &J = p.jobs[job];

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

    const uint32_t *cw = J.codes + b * p.codes_bh_stride + g * (G / W) * D + ch * 8;
    __half *y = static_cast<__half *>(J.y) + b * p.y_bh_stride + ch * 8;
    const int64_t t0 = g * G;
#pragma unroll 1
    for (int wr = 0; wr < G / W; ++wr) {
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
cudaError_t key_quant_launch(const QuantParams &p, cudaStream_t stream) {
  const int threads = key_threads(G, p.d);
  const size_t smem = key_smem_bytes<G>(p.d);
  auto kern = key_quant_kernel<BITS, G>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  int per_sm = 0;
  err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, smem);
  if (err != cudaSuccess) return err;
  if (per_sm < 1) per_sm = 1;
  const int64_t ng = (p.rows + G - 1) / G;
  const int64_t tiles = static_cast<int64_t>(p.n_jobs) * p.bh * ng;
  const int64_t grid = std::min<int64_t>(tiles, static_cast<int64_t>(num_sms()) * per_sm);
  kern<<<static_cast<unsigned>(grid), threads, smem, stream>>>(p);
  return cudaGetLastError();
}

template <int BITS, int G>
cudaError_t key_dequant_launch(const DequantParams &p, cudaStream_t stream) {
  const int threads = 256;
  auto kern = key_dequant_kernel<BITS, G>;
  int per_sm = 0;
  cudaError_t err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, 0);
  if (err != cudaSuccess) return err;
  if (per_sm < 1) per_sm = 1;
  const int64_t ng = (p.rows + G - 1) / G;
  const int64_t units = static_cast<int64_t>(p.n_jobs) * p.bh * ng * (p.d / 8);
  const int64_t blocks = (units + threads - 1) / threads;
  const int64_t grid = std::min<int64_t>(blocks, static_cast<int64_t>(num_sms()) * per_sm);
  kern<<<static_cast<unsigned>(grid), threads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

#define KIVI_DISPATCH(FN, P, GROUP, BITS, STREAM)                                   \
  do {                                                                              \
    switch ((BITS) * 1000 + (GROUP)) {                                              \
      case 2032: return FN<2, 32>(P, STREAM);                                       \
      case 2064: return FN<2, 64>(P, STREAM);                                       \
      case 2128: return FN<2, 128>(P, STREAM);                                      \
      case 4032: return FN<4, 32>(P, STREAM);                                       \
      case 4064: return FN<4, 64>(P, STREAM);                                       \
      case 4128: return FN<4, 128>(P, STREAM);                                      \
      case 8032: return FN<8, 32>(P, STREAM);                                       \
      case 8064: return FN<8, 64>(P, STREAM);                                       \
      case 8128: return FN<8, 128>(P, STREAM);                                      \
      default: return cudaErrorInvalidValue;                                        \
    }                                                                               \
  } while (0)

cudaError_t launch_key_quant(const QuantParams &p, int group, int bits, cudaStream_t stream) {
  KIVI_DISPATCH(key_quant_launch, p, group, bits, stream);
}

cudaError_t launch_key_dequant(const DequantParams &p, int group, int bits,
                               cudaStream_t stream) {
  KIVI_DISPATCH(key_dequant_launch, p, group, bits, stream);
}

cudaError_t read_and_clear_key_fault(uint32_t *fault) {
  cudaError_t err = cudaDeviceSynchronize();
  if (err != cudaSuccess) return err;
  unsigned int v = 0;
  err = cudaMemcpyFromSymbol(&v, g_key_fault, sizeof(v));
  if (err != cudaSuccess) return err;
  const unsigned int zero = 0;
  err = cudaMemcpyToSymbol(g_key_fault, &zero, sizeof(zero));
  if (err != cudaSuccess) return err;
  *fault = v;
  return cudaSuccess;
}

}  // namespace kivi_impl
