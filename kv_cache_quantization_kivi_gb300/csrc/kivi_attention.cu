// kivi_attention.cu -- decode attention over the packed KIVI store: the
// register-operand kernel at head_dim 128 (kivi_attention_kernel.cuh; 64 and
// 256 in kivi_attention_d64.cu / kivi_attention_d256.cu), the split combine,
// the dispatch between the kernels, and the device words the attention and
// KIVI-Sink kernels share (the fault word, the allocation-free call's
// workspace).
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "kivi_attention_kernel.cuh"
#include "kivi_device.cuh"
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

// Combine the splits of one (layer, bh, head): thread = channel (blockDim.x
// = head_dim).
__global__ void __launch_bounds__(256) attention_combine_kernel(const __grid_constant__ AttnParams p) {
  const int D = p.d;
  const int64_t blk = blockIdx.x;             // (job * bh + bhi) * r + h
  const int h = static_cast<int>(blk % p.r);
  const int64_t pair = blk / p.r;
  const int job = static_cast<int>(pair / p.bh);
  const int64_t bhi = pair - static_cast<int64_t>(job) * p.bh;
  const int64_t b = bhi / p.h_kv, kvh = bhi - b * p.h_kv;
  const int c = threadIdx.x;
  const int64_t items = static_cast<int64_t>(p.n_jobs) * p.bh * p.n_split;
  const float *ml = p.ws + items * p.r * D;
  float M = -INFINITY;
  for (int s = 0; s < p.n_split; ++s) M = fmaxf(M, ml[2 * ((pair * p.n_split + s) * p.r + h)]);
  float L = 0.0f, O = 0.0f;
  for (int s = 0; s < p.n_split; ++s) {
    const int64_t base = (pair * p.n_split + s) * p.r + h;
    const float ms = ml[2 * base];
    if (ms == -INFINITY) continue;
    const float f = exp2f(ms - M);
    L += ml[2 * base + 1] * f;
    O += p.ws[base * D + c] * f;
  }
  const int64_t h_q = static_cast<int64_t>(p.h_kv) * p.r;
  p.jobs[job].out[(b * h_q + kvh * p.r + h) * D + c] = O / L;
}

}  // namespace

cudaError_t launch_attention_combine(const AttnParams &p, cudaStream_t stream) {
  const int64_t blocks = static_cast<int64_t>(p.n_jobs) * p.bh * p.r;
  attention_combine_kernel<<<static_cast<unsigned>(blocks), p.d, 0, stream>>>(p);
  return cudaGetLastError();
}

// The kernel the environment variable KIVI_ATTENTION_KERNEL selects: the
// register-operand kernel unless it reads "tcgen05", which selects the
// warp-specialised tensor-memory kernel (kivi_attention_ws.cu) for the calls
// that kernel takes.  Read at every call, so a process can switch between
// calls.
static bool tensor_memory_kernel_selected() {
  const char *v = std::getenv("KIVI_ATTENTION_KERNEL");
  return v && std::strcmp(v, "tcgen05") == 0;
}

cudaError_t launch_decode_attention(const AttnParams &p, int group, int bits, cudaStream_t stream) {
  if (tensor_memory_kernel_selected()) {
    bool handled = false;
    const cudaError_t e = launch_decode_attention_ws(p, group, bits, stream, &handled);
    if (handled) return e;
  }
  switch (p.d) {
    case 64: return launch_decode_attention_d64(p, group, bits, stream);
    case 128: return attention_dispatch<128>(p, group, bits, stream);
    case 256: return launch_decode_attention_d256(p, group, bits, stream);
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
