// kivi_api.cu -- the extern "C" entry points declared in include/kivi.h:
// host-side validation, parameter blocks, launches and flush bookkeeping.
//
// Every check happens before the first CUDA call, so an invalid call
// launches nothing and touches no memory.  Launch failures are reported as
// KIVI_ERR_CUDA with the cudaError_t kept per host thread.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstring>

#include "../../include/kivi.h"
#include "kivi_launch.h"

namespace kivi_impl {

int current_sm_count() {
  constexpr int kMaxDevices = 64;
  static std::atomic<int> count[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 1;
  int n = count[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
      n = 1;
    count[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

}  // namespace kivi_impl

namespace {

thread_local int t_last_cuda_error = 0;

bool valid_bits(int bits) { return bits == 2 || bits == 4 || bits == 8; }
bool valid_group(int g) { return g == 16 || g == 32 || g == 64 || g == 128; }
bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool bytes16(int64_t n_elems, int64_t elem_bytes) { return (n_elems * elem_bytes) % 16 == 0; }
bool bytes_mult(int64_t n_elems, int64_t elem_bytes, int64_t m) {
  return (n_elems * elem_bytes) % m == 0;
}
// Value code rows are written and read in pieces of 4*bits bytes per 32
// channels (8 bytes at 2 bits, 16 bytes otherwise).
int64_t value_code_align(int bits) { return bits == 2 ? 8 : 16; }

constexpr int64_t kMaxUnits = (int64_t{1} << 31) - 1;

bool valid_key_dim(int64_t d) { return d >= 8 && d <= 256 && d % 8 == 0; }
// values are processed in 32-channel pieces (two 16-channel groups at G = 16)
bool valid_value_dim(int64_t d, int group) {
  return d >= 32 && d <= 256 && d % group == 0 && d % 32 == 0;
}

int64_t groups_of(int64_t s, int group) { return s / group + (s % group != 0); }

// a * b for a, b >= 0, saturated at INT64_MAX (sizes are validated with it
// before any product that could overflow is formed).
int64_t sat_mul(int64_t a, int64_t b) {
  return a != 0 && b > INT64_MAX / a ? INT64_MAX : a * b;
}

kivi_status cuda_status(cudaError_t err) {
  if (err == cudaSuccess) return KIVI_OK;
  t_last_cuda_error = static_cast<int>(err);
  return KIVI_ERR_CUDA;
}

struct KeyGeom {
  int64_t code_words;  // per bh slice
  int64_t sz;          // per bh slice
};

KeyGeom key_geom(int64_t s, int64_t d, int group, int bits) {
  const int64_t ng = groups_of(s, group);
  return {ng * group / (32 / bits) * d, ng * d};
}

// Threads of the key kernels: one per (bh, group, min(G, 32)-token split)
// and channel pair (quantize) or 8 channels (dequantize); of the value
// kernels: one per 32 channels of a row.
int64_t key_quant_units(int64_t bh, int64_t s, int64_t d, int group) {
  return sat_mul(sat_mul(bh, groups_of(s, group)), (d / 2) * (group < 32 ? 1 : group / 32));
}
int64_t key_dequant_units(int64_t bh, int64_t s, int64_t d, int group) {
  return sat_mul(sat_mul(bh, groups_of(s, group)), (d / 8) * (group < 32 ? 1 : group / 32));
}
int64_t value_units(int64_t bh, int64_t s, int64_t d) { return sat_mul(sat_mul(bh, s), d / 32); }

}  // namespace

extern "C" {

int kivi_abi_version(void) { return KIVI_ABI_VERSION; }

const char *kivi_status_string(kivi_status status) {
  switch (status) {
    case KIVI_OK: return "ok";
    case KIVI_ERR_INVAL: return "invalid argument";
    case KIVI_ERR_ALIGN: return "pointer or stride not 16-byte aligned";
    case KIVI_ERR_CAPACITY: return "store capacity exceeded";
    case KIVI_ERR_CUDA: return "CUDA runtime error";
  }
  return "unknown status";
}

int kivi_last_cuda_error(void) { return t_last_cuda_error; }

int64_t kivi_flush_size(int64_t n_res, int residual, int group) {
  if (n_res < 0 || residual < 0 || group <= 0) return -1;
  if (n_res < static_cast<int64_t>(residual) + group) return 0;
  return (n_res - residual) / group * group;
}

int64_t kivi_key_code_words(int64_t s, int64_t d, int group, int bits) {
  if (!valid_bits(bits) || !valid_group(group) || s < 0 || d < 0) return -1;
  return key_geom(s, d, group, bits).code_words;
}

int64_t kivi_value_code_words(int64_t s, int64_t d, int group, int bits) {
  if (!valid_bits(bits) || !valid_group(group) || s < 0 || d < 0) return -1;
  return s * (d / (32 / bits));
}

// ---------------------------------------------------------------------------
// full-tensor calls
// ---------------------------------------------------------------------------

kivi_status kivi_quantize_keys(const void *x, int64_t bh, int64_t s, int64_t d,
                               int64_t x_bh_stride, int group, int bits, uint32_t *codes,
                               int64_t codes_bh_stride, float *scale, float *zero,
                               int64_t sz_bh_stride, kivi_stream_t stream) {
  if (!valid_bits(bits) || !valid_group(group) || bh < 0 || s < 0 || !valid_key_dim(d))
    return KIVI_ERR_INVAL;
  if (bh == 0 || s == 0) return KIVI_OK;
  if (key_quant_units(bh, s, d, group) > kMaxUnits) return KIVI_ERR_INVAL;  // also bounds s * d
  if (!x || !codes || !scale || !zero) return KIVI_ERR_INVAL;
  const KeyGeom kg = key_geom(s, d, group, bits);
  if (x_bh_stride < s * d || codes_bh_stride < kg.code_words || sz_bh_stride < kg.sz)
    return KIVI_ERR_INVAL;
  if (!aligned16(x) || !aligned16(codes) || !aligned16(scale) || !aligned16(zero) ||
      !bytes16(x_bh_stride, 2) || !bytes16(codes_bh_stride, 4) || !bytes_mult(sz_bh_stride, 4, 8))
    return KIVI_ERR_ALIGN;

  kivi_impl::QuantParams p;
  std::memset(&p, 0, sizeof(p));
  p.n_jobs = 1;
  p.d = static_cast<int32_t>(d);
  p.bh = bh;
  p.rows = s;
  p.x_bh_stride = x_bh_stride;
  p.codes_bh_stride = codes_bh_stride;
  p.sz_bh_stride = sz_bh_stride;
  p.jobs[0] = {x, codes, scale, zero, nullptr, nullptr};
  return cuda_status(kivi_impl::launch_key_quant(p, group, bits, kivi_impl::kQuantPlain, stream));
}

kivi_status kivi_quantize_values(const void *x, int64_t bh, int64_t s, int64_t d,
                                 int64_t x_bh_stride, int group, int bits, uint32_t *codes,
                                 int64_t codes_bh_stride, float *scale, float *zero,
                                 int64_t sz_bh_stride, kivi_stream_t stream) {
  if (!valid_bits(bits) || !valid_group(group) || bh < 0 || s < 0 || !valid_value_dim(d, group))
    return KIVI_ERR_INVAL;
  if (bh == 0 || s == 0) return KIVI_OK;
  if (value_units(bh, s, d) > kMaxUnits) return KIVI_ERR_INVAL;  // also bounds s * d
  if (!x || !codes || !scale || !zero) return KIVI_ERR_INVAL;
  if (x_bh_stride < s * d || codes_bh_stride < s * (d / (32 / bits)) ||
      sz_bh_stride < s * (d / group))
    return KIVI_ERR_INVAL;
  if (!aligned16(x) || !aligned16(codes) || !aligned16(scale) || !aligned16(zero) ||
      !bytes16(x_bh_stride, 2) || !bytes_mult(codes_bh_stride, 4, value_code_align(bits)))
    return KIVI_ERR_ALIGN;

  kivi_impl::QuantParams p;
  std::memset(&p, 0, sizeof(p));
  p.n_jobs = 1;
  p.d = static_cast<int32_t>(d);
  p.bh = bh;
  p.rows = s;
  p.x_bh_stride = x_bh_stride;
  p.codes_bh_stride = codes_bh_stride;
  p.sz_bh_stride = sz_bh_stride;
  p.jobs[0] = {x, codes, scale, zero, nullptr, nullptr};
  return cuda_status(kivi_impl::launch_value_quant(p, group, bits, kivi_impl::kQuantPlain, stream));
}

// Fused quantize + dequantize: the same kernels with the reconstruction
// written as each code is made.  codes/scale/zero are all given or all NULL.
kivi_status kivi_fakequant_keys(const void *x, int64_t bh, int64_t s, int64_t d,
                                int64_t x_bh_stride, int group, int bits, void *y,
                                int64_t y_bh_stride, uint32_t *codes, int64_t codes_bh_stride,
                                float *scale, float *zero, int64_t sz_bh_stride,
                                kivi_stream_t stream) {
  if (!valid_bits(bits) || !valid_group(group) || bh < 0 || s < 0 || !valid_key_dim(d))
    return KIVI_ERR_INVAL;
  if (bh == 0 || s == 0) return KIVI_OK;
  if (key_quant_units(bh, s, d, group) > kMaxUnits) return KIVI_ERR_INVAL;  // also bounds s * d
  const bool store = codes != nullptr;
  if (!x || !y || (scale != nullptr) != store || (zero != nullptr) != store)
    return KIVI_ERR_INVAL;
  const KeyGeom kg = key_geom(s, d, group, bits);
  if (x_bh_stride < s * d || y_bh_stride < s * d) return KIVI_ERR_INVAL;
  if (store && (codes_bh_stride < kg.code_words || sz_bh_stride < kg.sz)) return KIVI_ERR_INVAL;
  if (!aligned16(x) || !aligned16(y) || !bytes16(x_bh_stride, 2) || !bytes16(y_bh_stride, 2))
    return KIVI_ERR_ALIGN;
  if (store && (!aligned16(codes) || !aligned16(scale) || !aligned16(zero) ||
                !bytes16(codes_bh_stride, 4) || !bytes_mult(sz_bh_stride, 4, 8)))
    return KIVI_ERR_ALIGN;

  kivi_impl::QuantParams p;
  std::memset(&p, 0, sizeof(p));
  p.n_jobs = 1;
  p.d = static_cast<int32_t>(d);
  p.bh = bh;
  p.rows = s;
  p.x_bh_stride = x_bh_stride;
  p.codes_bh_stride = store ? codes_bh_stride : 0;
  p.sz_bh_stride = store ? sz_bh_stride : 0;
  p.y_bh_stride = y_bh_stride;
  p.jobs[0] = {x, codes, scale, zero, y, nullptr};
  return cuda_status(kivi_impl::launch_key_quant(p, group, bits, kivi_impl::kQuantRecon, stream));
}

kivi_status kivi_fakequant_values(const void *x, int64_t bh, int64_t s, int64_t d,
                                  int64_t x_bh_stride, int group, int bits, void *y,
                                  int64_t y_bh_stride, uint32_t *codes, int64_t codes_bh_stride,
                                  float *scale, float *zero, int64_t sz_bh_stride,
                                  kivi_stream_t stream) {
  if (!valid_bits(bits) || !valid_group(group) || bh < 0 || s < 0 || !valid_value_dim(d, group))
    return KIVI_ERR_INVAL;
  if (bh == 0 || s == 0) return KIVI_OK;
  if (value_units(bh, s, d) > kMaxUnits) return KIVI_ERR_INVAL;  // also bounds s * d
  const bool store = codes != nullptr;
  if (!x || !y || (scale != nullptr) != store || (zero != nullptr) != store)
    return KIVI_ERR_INVAL;
  if (x_bh_stride < s * d || y_bh_stride < s * d) return KIVI_ERR_INVAL;
  if (store && (codes_bh_stride < s * (d / (32 / bits)) || sz_bh_stride < s * (d / group)))
    return KIVI_ERR_INVAL;
  if (!aligned16(x) || !aligned16(y) || !bytes16(x_bh_stride, 2) || !bytes16(y_bh_stride, 2))
    return KIVI_ERR_ALIGN;
  if (store && (!aligned16(codes) || !aligned16(scale) || !aligned16(zero) ||
                !bytes_mult(codes_bh_stride, 4, value_code_align(bits))))
    return KIVI_ERR_ALIGN;

  kivi_impl::QuantParams p;
  std::memset(&p, 0, sizeof(p));
  p.n_jobs = 1;
  p.d = static_cast<int32_t>(d);
  p.bh = bh;
  p.rows = s;
  p.x_bh_stride = x_bh_stride;
  p.codes_bh_stride = store ? codes_bh_stride : 0;
  p.sz_bh_stride = store ? sz_bh_stride : 0;
  p.y_bh_stride = y_bh_stride;
  p.jobs[0] = {x, codes, scale, zero, y, nullptr};
  return cuda_status(kivi_impl::launch_value_quant(p, group, bits, kivi_impl::kQuantRecon, stream));
}

kivi_status kivi_dequantize_keys(const uint32_t *codes, int64_t codes_bh_stride,
                                 const float *scale, const float *zero, int64_t sz_bh_stride,
                                 int64_t bh, int64_t s, int64_t d, int group, int bits, void *y,
                                 int64_t y_bh_stride, kivi_stream_t stream) {
  if (!valid_bits(bits) || !valid_group(group) || bh < 0 || s < 0 || !valid_key_dim(d))
    return KIVI_ERR_INVAL;
  if (bh == 0 || s == 0) return KIVI_OK;
  if (key_dequant_units(bh, s, d, group) > kMaxUnits) return KIVI_ERR_INVAL;  // also bounds s * d
  if (!codes || !scale || !zero || !y) return KIVI_ERR_INVAL;
  const KeyGeom kg = key_geom(s, d, group, bits);
  if (codes_bh_stride < kg.code_words || sz_bh_stride < kg.sz || y_bh_stride < s * d)
    return KIVI_ERR_INVAL;
  if (!aligned16(codes) || !aligned16(scale) || !aligned16(zero) || !aligned16(y) ||
      !bytes16(codes_bh_stride, 4) || !bytes16(sz_bh_stride, 4) || !bytes16(y_bh_stride, 2))
    return KIVI_ERR_ALIGN;

  kivi_impl::DequantParams p;
  std::memset(&p, 0, sizeof(p));
  p.n_jobs = 1;
  p.d = static_cast<int32_t>(d);
  p.bh = bh;
  p.rows = s;
  p.codes_bh_stride = codes_bh_stride;
  p.sz_bh_stride = sz_bh_stride;
  p.y_bh_stride = y_bh_stride;
  p.jobs[0] = {codes, scale, zero, y};
  return cuda_status(kivi_impl::launch_key_dequant(p, group, bits, stream));
}

kivi_status kivi_dequantize_values(const uint32_t *codes, int64_t codes_bh_stride,
                                   const float *scale, const float *zero, int64_t sz_bh_stride,
                                   int64_t bh, int64_t s, int64_t d, int group, int bits,
                                   void *y, int64_t y_bh_stride, kivi_stream_t stream) {
  if (!valid_bits(bits) || !valid_group(group) || bh < 0 || s < 0 || !valid_value_dim(d, group))
    return KIVI_ERR_INVAL;
  if (bh == 0 || s == 0) return KIVI_OK;
  if (value_units(bh, s, d) > kMaxUnits) return KIVI_ERR_INVAL;  // also bounds s * d
  if (!codes || !scale || !zero || !y) return KIVI_ERR_INVAL;
  if (codes_bh_stride < s * (d / (32 / bits)) || sz_bh_stride < s * (d / group) ||
      y_bh_stride < s * d)
    return KIVI_ERR_INVAL;
  if (!aligned16(codes) || !aligned16(scale) || !aligned16(zero) || !aligned16(y) ||
      !bytes_mult(codes_bh_stride, 4, value_code_align(bits)) || !bytes16(y_bh_stride, 2))
    return KIVI_ERR_ALIGN;

  kivi_impl::DequantParams p;
  std::memset(&p, 0, sizeof(p));
  p.n_jobs = 1;
  p.d = static_cast<int32_t>(d);
  p.bh = bh;
  p.rows = s;
  p.codes_bh_stride = codes_bh_stride;
  p.sz_bh_stride = sz_bh_stride;
  p.y_bh_stride = y_bh_stride;
  p.jobs[0] = {codes, scale, zero, y};
  return cuda_status(kivi_impl::launch_value_dequant(p, group, bits, stream));
}

// ---------------------------------------------------------------------------
// cache: flush and batched dequantization
// ---------------------------------------------------------------------------

// allow_no_store: a layer's key (or value) store pointers may all be NULL
// (fake-quant flush that keeps only the reconstruction).
static kivi_status check_cache(const kivi_layer *layers, int n_layers, const kivi_cache *c,
                               bool allow_no_store = false) {
  if (!layers || !c || n_layers < 1 || n_layers > KIVI_MAX_LAYERS) return KIVI_ERR_INVAL;
  if (!valid_bits(c->bits) || !valid_group(c->group) || c->residual < 0 || c->reserved != 0)
    return KIVI_ERR_INVAL;
  const int64_t G = c->group;
  if (c->bh < 0 || !valid_key_dim(c->d) || !valid_value_dim(c->d, c->group)) return KIVI_ERR_INVAL;
  if (c->r_cap <= 0 || c->r_cap % G != 0 || c->cap < 0 || c->cap % G != 0) return KIVI_ERR_INVAL;
  if (c->s_q < 0 || c->s_q % G != 0 || c->s_q > c->cap) return KIVI_ERR_INVAL;
  if (c->res_head < 0 || c->res_head >= c->r_cap || c->res_head % G != 0) return KIVI_ERR_INVAL;
  if (c->n_res < 0 || c->n_res > c->r_cap) return KIVI_ERR_INVAL;
  if (sat_mul(value_units(c->bh, c->cap, c->d), n_layers) > kMaxUnits ||
      value_units(c->bh, c->r_cap, c->d) > kMaxUnits)
    return KIVI_ERR_INVAL;
  for (int l = 0; l < n_layers; ++l) {
    const kivi_layer &L = layers[l];
    const void *ptrs[8] = {L.k_res, L.v_res, L.k_codes, L.k_scale,
                           L.k_zero, L.v_codes, L.v_scale, L.v_zero};
    if (!L.k_res || !L.v_res) return KIVI_ERR_INVAL;
    for (int t = 0; t < 2; ++t) {  // key store, value store
      const int nn = (ptrs[2 + 3 * t] != nullptr) + (ptrs[3 + 3 * t] != nullptr) +
                     (ptrs[4 + 3 * t] != nullptr);
      if (nn != 3 && !(allow_no_store && nn == 0)) return KIVI_ERR_INVAL;
    }
    for (const void *q : ptrs) {
      if (!aligned16(q)) return KIVI_ERR_ALIGN;  // NULL is aligned
    }
  }
  return KIVI_OK;
}

static cudaError_t record(void *const *events, int i, cudaStream_t s) {
  if (!events || !events[i]) return cudaSuccess;
  return cudaEventRecord(static_cast<cudaEvent_t>(events[i]), s);
}

static kivi_status check_append(const kivi_layer *layers, int n_layers, const kivi_cache *cache,
                                const void *const *k_new, const void *const *v_new,
                                int64_t new_bh_stride, int64_t n, bool allow_no_store) {
  const kivi_status st = check_cache(layers, n_layers, cache, allow_no_store);
  if (st != KIVI_OK) return st;
  if (n < 0 || !k_new || !v_new) return KIVI_ERR_INVAL;
  if (cache->n_res + n > cache->r_cap) return KIVI_ERR_CAPACITY;
  const int64_t d = cache->d;
  if (n > 0 && cache->bh > 0) {
    if (new_bh_stride < n * d) return KIVI_ERR_INVAL;
    if (sat_mul(sat_mul(sat_mul(n_layers, cache->bh), n), d / 8) > kMaxUnits)
      return KIVI_ERR_INVAL;
    for (int l = 0; l < n_layers; ++l) {
      if (!k_new[l] || !v_new[l]) return KIVI_ERR_INVAL;
      if (!aligned16(k_new[l]) || !aligned16(v_new[l])) return KIVI_ERR_ALIGN;
    }
    if (!bytes16(new_bh_stride, 2)) return KIVI_ERR_ALIGN;
  }
  return KIVI_OK;
}

// The append's launch (arguments already checked) and the state update.
static kivi_status append_impl(const kivi_layer *layers, int n_layers, kivi_cache *cache,
                               const void *const *k_new, const void *const *v_new,
                               int64_t new_bh_stride, int64_t n, kivi_stream_t stream) {
  const int64_t d = cache->d;
  if (n > 0 && cache->bh > 0) {
    kivi_impl::AppendParams p;
    std::memset(&p, 0, sizeof(p));
    p.n_jobs = n_layers;
    p.d = static_cast<int32_t>(d);
    p.bh = cache->bh;
    p.n = n;
    p.r_cap = cache->r_cap;
    p.row0 = (cache->res_head + cache->n_res) % cache->r_cap;
    p.new_bh_stride = new_bh_stride;
    for (int l = 0; l < n_layers; ++l)
      p.jobs[l] = {k_new[l], v_new[l], const_cast<void *>(layers[l].k_res),
                   const_cast<void *>(layers[l].v_res)};
    const kivi_status r = cuda_status(kivi_impl::launch_append(p, stream));
    if (r != KIVI_OK) return r;
  }
  cache->n_res += n;
  return KIVI_OK;
}

kivi_status kivi_append(const kivi_layer *layers, int n_layers, kivi_cache *cache,
                        const void *const *k_new, const void *const *v_new,
                        int64_t new_bh_stride, int64_t n, kivi_stream_t stream) {
  const kivi_status st =
      check_append(layers, n_layers, cache, k_new, v_new, new_bh_stride, n, true);
  if (st != KIVI_OK) return st;
  return append_impl(layers, n_layers, cache, k_new, v_new, new_bh_stride, n, stream);
}

kivi_status kivi_flush(const kivi_layer *layers, int n_layers, kivi_cache *cache,
                       int64_t *n_flushed, kivi_stream_t stream) {
  return kivi_flush_timed(layers, n_layers, cache, n_flushed, stream, nullptr);
}

// defer_key: the key launch's inputs do not depend on the previous launch in
// the stream (the flushed rows were not written by it), so it may defer its
// dependency wait (QuantParams::defer_wait); the value launch never depends
// on the key launch and always defers.
static kivi_status flush_impl(const kivi_layer *layers, int n_layers, kivi_cache *cache,
                              void *const *k_hat, void *const *v_hat, int64_t *n_flushed,
                              kivi_stream_t stream, void *const *events,
                              bool defer_key = false) {
  const bool recon = k_hat != nullptr;
  const kivi_status st = check_cache(layers, n_layers, cache, recon);
  if (st != KIVI_OK) return st;
  if (recon) {
    for (int l = 0; l < n_layers; ++l) {
      if (!k_hat[l] || !v_hat[l]) return KIVI_ERR_INVAL;
      if (!aligned16(k_hat[l]) || !aligned16(v_hat[l])) return KIVI_ERR_ALIGN;
    }
  }
  const int64_t G = cache->group;
  const int W = 32 / cache->bits;
  const int64_t n = kivi_flush_size(cache->n_res, cache->residual, cache->group);
  if (n > 0 && cache->s_q + n > cache->cap) return KIVI_ERR_CAPACITY;
  if (n == 0 || cache->bh == 0) {
    if (n_flushed) *n_flushed = 0;
    if (n > 0) {  // bh == 0: nothing to move, but the state advances
      cache->s_q += n;
      cache->res_head = (cache->res_head + n) % cache->r_cap;
      cache->n_res -= n;
      if (n_flushed) *n_flushed = n;
    }
    return KIVI_OK;
  }

  const int64_t d = cache->d;
  kivi_impl::QuantParams kp;
  std::memset(&kp, 0, sizeof(kp));
  kp.n_jobs = n_layers;
  kp.d = static_cast<int32_t>(d);
  kp.bh = cache->bh;
  kp.rows = n;
  kp.x_bh_stride = cache->r_cap * d;
  kp.ring = cache->r_cap;
  kp.head = cache->res_head;
  kp.y_bh_stride = cache->cap * d;  // reconstruction [bh][cap][d], rows s_q ..
  kp.y_row0 = cache->s_q;

  kivi_impl::QuantParams vp = kp;
  kp.codes_bh_stride = cache->cap / W * d;
  kp.sz_bh_stride = cache->cap / G * d;
  kp.out0 = cache->s_q / G;
  kp.defer_wait = defer_key ? 1 : 0;
  vp.codes_bh_stride = cache->cap * (d / W);
  vp.sz_bh_stride = cache->cap * (d / G);
  vp.out0 = cache->s_q;
  vp.defer_wait = 1;
  for (int l = 0; l < n_layers; ++l) {
    const kivi_layer &L = layers[l];
    kp.jobs[l] = {L.k_res, L.k_codes, L.k_scale, L.k_zero, recon ? k_hat[l] : nullptr, nullptr};
    vp.jobs[l] = {L.v_res, L.v_codes, L.v_scale, L.v_zero, recon ? v_hat[l] : nullptr, nullptr};
  }
  cudaStream_t s = stream;
  kivi_status r = cuda_status(record(events, 0, s));
  if (r != KIVI_OK) return r;
  const int mode = recon ? kivi_impl::kQuantRecon : kivi_impl::kQuantPlain;
  r = cuda_status(kivi_impl::launch_key_quant(kp, cache->group, cache->bits, mode, s));
  if (r != KIVI_OK) return r;
  r = cuda_status(record(events, 1, s));
  if (r != KIVI_OK) return r;
  r = cuda_status(kivi_impl::launch_value_quant(vp, cache->group, cache->bits, mode, s));
  if (r != KIVI_OK) return r;
  r = cuda_status(record(events, 2, s));
  if (r != KIVI_OK) return r;

  cache->s_q += n;
  cache->res_head = (cache->res_head + n) % cache->r_cap;
  cache->n_res -= n;
  if (n_flushed) *n_flushed = n;
  return KIVI_OK;
}

kivi_status kivi_flush_timed(const kivi_layer *layers, int n_layers, kivi_cache *cache,
                             int64_t *n_flushed, kivi_stream_t stream, void *const events[3]) {
  return flush_impl(layers, n_layers, cache, nullptr, nullptr, n_flushed, stream, events);
}

kivi_status kivi_flush_fakequant(const kivi_layer *layers, int n_layers, kivi_cache *cache,
                                 void *const *k_hat, void *const *v_hat, int64_t *n_flushed,
                                 kivi_stream_t stream, void *const events[3]) {
  if (!k_hat || !v_hat) return KIVI_ERR_INVAL;
  return flush_impl(layers, n_layers, cache, k_hat, v_hat, n_flushed, stream, events);
}

kivi_status kivi_append_flush(const kivi_layer *layers, int n_layers, kivi_cache *cache,
                              const void *const *k_new, const void *const *v_new,
                              int64_t new_bh_stride, int64_t n, int64_t *n_flushed,
                              kivi_stream_t stream, void *const events[4]) {
  // every check of both steps before the first launch
  kivi_status st = check_append(layers, n_layers, cache, k_new, v_new, new_bh_stride, n, false);
  if (st != KIVI_OK) return st;
  const int64_t n_res_before = cache->n_res;
  const int64_t n_flush = kivi_flush_size(n_res_before + n, cache->residual, cache->group);
  if (n_flush > 0 && cache->s_q + n_flush > cache->cap) return KIVI_ERR_CAPACITY;
  cudaStream_t s = stream;
  kivi_status r = cuda_status(record(events, 0, s));
  if (r != KIVI_OK) return r;
  r = append_impl(layers, n_layers, cache, k_new, v_new, new_bh_stride, n, stream);
  if (r != KIVI_OK) return r;
  // the flushed rows are residual tokens 0 .. n_flush - 1; when they were all
  // in the ring before the append, the quantizers do not read what it wrote
  return flush_impl(layers, n_layers, cache, nullptr, nullptr, n_flushed, stream,
                    events ? events + 1 : nullptr, n_flush <= n_res_before);
}

kivi_status kivi_dequantize_cache(const kivi_layer *layers, int n_layers, const kivi_cache *cache,
                                  void *const *k_out, void *const *v_out, kivi_stream_t stream) {
  return kivi_dequantize_cache_timed(layers, n_layers, cache, k_out, v_out, stream, nullptr);
}

kivi_status kivi_dequantize_cache_timed(const kivi_layer *layers, int n_layers,
                                        const kivi_cache *cache, void *const *k_out,
                                        void *const *v_out, kivi_stream_t stream,
                                        void *const events[3]) {
  const kivi_status st = check_cache(layers, n_layers, cache);
  if (st != KIVI_OK) return st;
  if (!k_out || !v_out) return KIVI_ERR_INVAL;
  if (cache->s_q == 0 || cache->bh == 0) return KIVI_OK;
  for (int l = 0; l < n_layers; ++l) {
    if (!k_out[l] || !v_out[l]) return KIVI_ERR_INVAL;
    if (!aligned16(k_out[l]) || !aligned16(v_out[l])) return KIVI_ERR_ALIGN;
  }
  const int64_t G = cache->group;
  const int W = 32 / cache->bits;
  const int64_t d = cache->d;
  kivi_impl::DequantParams kp;
  std::memset(&kp, 0, sizeof(kp));
  kp.n_jobs = n_layers;
  kp.d = static_cast<int32_t>(d);
  kp.bh = cache->bh;
  kp.rows = cache->s_q;
  kp.y_bh_stride = cache->s_q * d;
  kivi_impl::DequantParams vp = kp;
  kp.codes_bh_stride = cache->cap / W * d;
  kp.sz_bh_stride = cache->cap / G * d;
  vp.codes_bh_stride = cache->cap * (d / W);
  vp.sz_bh_stride = cache->cap * (d / G);
  vp.defer_wait = 1;   // the value store does not depend on the key launch
  for (int l = 0; l < n_layers; ++l) {
    const kivi_layer &L = layers[l];
    kp.jobs[l] = {L.k_codes, L.k_scale, L.k_zero, k_out[l]};
    vp.jobs[l] = {L.v_codes, L.v_scale, L.v_zero, v_out[l]};
  }
  cudaStream_t s = stream;
  kivi_status r = cuda_status(record(events, 0, s));
  if (r != KIVI_OK) return r;
  r = cuda_status(kivi_impl::launch_key_dequant(kp, cache->group, cache->bits, s));
  if (r != KIVI_OK) return r;
  r = cuda_status(record(events, 1, s));
  if (r != KIVI_OK) return r;
  r = cuda_status(kivi_impl::launch_value_dequant(vp, cache->group, cache->bits, s));
  if (r != KIVI_OK) return r;
  return cuda_status(record(events, 2, s));
}

// ---------------------------------------------------------------------------
// decode attention over the packed cache
// ---------------------------------------------------------------------------

static constexpr int kAttnTile = 32;
static constexpr int kAttnMaxSplit = 64;

struct AttnGeom {
  int64_t h_kv, r, tiles_store, tiles_res;
};

// head dims of the decode-attention kernels (the value groups must tile the head)
static bool attn_dim(const kivi_cache *c) {
  return (c->d == 64 || c->d == 128 || c->d == 256) && c->d % c->group == 0;
}

static kivi_status attn_geom(const kivi_cache *c, int64_t batch, int32_t h_q, AttnGeom *g) {
  if (!attn_dim(c) || batch < 1 || c->bh % batch != 0) return KIVI_ERR_INVAL;
  g->h_kv = c->bh / batch;
  if (g->h_kv < 1 || h_q < 1 || h_q % g->h_kv != 0) return KIVI_ERR_INVAL;
  g->r = h_q / g->h_kv;
  if (g->r > 8) return KIVI_ERR_INVAL;
  g->tiles_store = (c->s_q + kAttnTile - 1) / kAttnTile;   // the last one half at G = 16
  g->tiles_res = (c->n_res + kAttnTile - 1) / kAttnTile;
  return KIVI_OK;
}

int32_t kivi_decode_attention_splits(const kivi_cache *cache, int n_layers, int64_t batch) {
  if (!cache || n_layers < 1 || batch < 1 || cache->bh < 0) return 1;
  const int64_t items = sat_mul(n_layers, cache->bh);
  const int64_t tiles = cache->s_q > 0 ? (cache->s_q + kAttnTile - 1) / kAttnTile : 0;
  return kivi_impl::attention_splits(items, tiles, cache->group, cache->bits);
}

int64_t kivi_decode_attention_workspace(const kivi_cache *cache, int n_layers, int64_t batch,
                                        int32_t h_q, int32_t n_split) {
  AttnGeom g;
  if (!cache || n_layers < 1 || n_split < 1 || n_split > kAttnMaxSplit) return -1;
  if (attn_geom(cache, batch, h_q, &g) != KIVI_OK) return -1;
  if (n_split == 1) return 0;
  return sat_mul(sat_mul(sat_mul(n_layers, cache->bh), n_split), g.r * (cache->d + 2));
}

// Validation and parameter block of a decode-attention call; the workspace
// (n_split > 1) is checked by the caller of this function.
static kivi_status attn_prepare(const kivi_layer *layers, int n_layers, const kivi_cache *cache,
                                int64_t batch, int32_t h_q, float sm_scale, const void *const *q,
                                float *const *out, int32_t n_split, kivi_impl::AttnParams *p) {
  const kivi_status st = check_cache(layers, n_layers, cache);
  if (st != KIVI_OK) return st;
  AttnGeom g;
  if (attn_geom(cache, batch, h_q, &g) != KIVI_OK) return KIVI_ERR_INVAL;
  if (!q || !out || !(sm_scale == sm_scale) || sm_scale > 3.0e38f || sm_scale < -3.0e38f)
    return KIVI_ERR_INVAL;
  if (n_split < 1 || n_split > kAttnMaxSplit) return KIVI_ERR_INVAL;
  if (cache->s_q + cache->n_res < 1 && cache->bh > 0) return KIVI_ERR_INVAL;  // nothing to attend
  for (int l = 0; l < n_layers; ++l) {
    if (!q[l] || !out[l]) return KIVI_ERR_INVAL;
    if (!aligned16(q[l]) || !aligned16(out[l])) return KIVI_ERR_ALIGN;
  }
  if (sat_mul(sat_mul(n_layers, cache->bh), n_split) > kMaxUnits) return KIVI_ERR_INVAL;

  std::memset(p, 0, sizeof(*p));
  p->n_jobs = n_layers;
  p->d = static_cast<int32_t>(cache->d);
  p->r = static_cast<int32_t>(g.r);
  p->h_kv = static_cast<int32_t>(g.h_kv);
  p->n_split = n_split;
  p->tiles_store = static_cast<int32_t>(g.tiles_store);
  p->tiles_res = static_cast<int32_t>(g.tiles_res);
  p->tiles_per_split = static_cast<int32_t>((g.tiles_store + n_split - 1) / n_split);
  p->tail_half = cache->s_q % kAttnTile != 0;
  p->bh = cache->bh;
  p->cap = cache->cap;
  p->r_cap = cache->r_cap;
  p->res_head = cache->res_head;
  p->n_res = cache->n_res;
  p->scale_log2 = static_cast<float>(static_cast<double>(sm_scale) * 1.4426950408889634);
  for (int l = 0; l < n_layers; ++l) {
    const kivi_layer &L = layers[l];
    p->jobs[l] = {L.k_codes, L.k_scale, L.k_zero, L.v_codes, L.v_scale, L.v_zero,
                  L.k_res, L.v_res, q[l], out[l], nullptr, nullptr, nullptr, nullptr};
  }
  return KIVI_OK;
}

kivi_status kivi_decode_attention(const kivi_layer *layers, int n_layers, const kivi_cache *cache,
                                  int64_t batch, int32_t h_q, float sm_scale,
                                  const void *const *q, float *const *out, int32_t n_split,
                                  float *workspace, int64_t workspace_floats,
                                  kivi_stream_t stream) {
  kivi_impl::AttnParams p;
  const kivi_status st =
      attn_prepare(layers, n_layers, cache, batch, h_q, sm_scale, q, out, n_split, &p);
  if (st != KIVI_OK) return st;
  if (n_split > 1) {
    const int64_t need = kivi_decode_attention_workspace(cache, n_layers, batch, h_q, n_split);
    if (!workspace || workspace_floats < need) return KIVI_ERR_INVAL;
    if (!aligned16(workspace)) return KIVI_ERR_ALIGN;
    p.ws = workspace;
  }
  if (cache->bh == 0) return KIVI_OK;
  return cuda_status(kivi_impl::launch_decode_attention(p, cache->group, cache->bits, stream));
}

kivi_status kivi_decode_attention_noalloc(const kivi_layer *layers, int n_layers,
                                          const kivi_cache *cache, int64_t batch, int32_t h_q,
                                          float sm_scale, const void *const *q,
                                          float *const *out, int32_t n_split,
                                          kivi_stream_t stream) {
  kivi_impl::AttnParams p;
  const kivi_status st =
      attn_prepare(layers, n_layers, cache, batch, h_q, sm_scale, q, out, n_split, &p);
  if (st != KIVI_OK) return st;
  if (n_split > 1) {
    const int64_t need = kivi_decode_attention_workspace(cache, n_layers, batch, h_q, n_split);
    if (need > kivi_impl::attention_scratch_floats()) return KIVI_ERR_CAPACITY;
  }
  if (cache->bh == 0) return KIVI_OK;
  if (n_split > 1) {   // every check is done: the first CUDA call
    int64_t max_floats = 0;
    const kivi_status s2 = cuda_status(kivi_impl::attention_scratch(&p.ws, &max_floats));
    if (s2 != KIVI_OK) return s2;
  }
  return cuda_status(kivi_impl::launch_decode_attention(p, cache->group, cache->bits, stream));
}

// ---------------------------------------------------------------------------
// KIVI-Sink
// ---------------------------------------------------------------------------

static kivi_status check_sinks(const kivi_sink_layer *sinks, int n_layers, const kivi_cache *c,
                               const kivi_sink_cfg *cfg) {
  if (!sinks || !cfg) return KIVI_ERR_INVAL;
  if (cfg->batch < 1 || c->bh % cfg->batch != 0 || cfg->k_top < 0 ||
      cfg->k_top > kivi_impl::kMaxSinkTop || cfg->sink_cap < 0 || cfg->reserved != 0)
    return KIVI_ERR_INVAL;
  // launch sizes of the sink kernels: the update's score blocks (32 tokens)
  // and tokens over all layers and sequences, the restore's 16-byte pieces
  if (sat_mul(sat_mul(n_layers, cfg->batch), c->r_cap) > kMaxUnits ||
      sat_mul(sat_mul(sat_mul(n_layers, c->bh), cfg->sink_cap), c->d / 8) > kMaxUnits)
    return KIVI_ERR_INVAL;
  for (int l = 0; l < n_layers; ++l) {
    const kivi_sink_layer &S = sinks[l];
    const void *ptrs[9] = {S.top_pos, S.top_score, S.top_count, S.sink_pos,
                           S.sink_count, S.sink_k, S.sink_v, S.mask, S.scores};
    for (const void *q : ptrs)
      if (!q) return KIVI_ERR_INVAL;
    if (!aligned16(S.sink_k) || !aligned16(S.sink_v)) return KIVI_ERR_ALIGN;
  }
  return KIVI_OK;
}

static void sink_params(const kivi_layer *layers, const kivi_sink_layer *sinks, int n_layers,
                        const kivi_cache *c, const kivi_sink_cfg *cfg,
                        kivi_impl::SinkParams *p) {
  std::memset(p, 0, sizeof(*p));
  p->n_jobs = n_layers;
  p->k_top = cfg->k_top;
  p->sink_cap = cfg->sink_cap;
  p->batch = cfg->batch;
  p->heads = c->bh / cfg->batch;
  p->d = c->d;
  p->r_cap = c->r_cap;
  p->res_head = c->res_head;
  p->s_q = c->s_q;
  p->mask_words = (c->r_cap + 31) / 32;
  for (int l = 0; l < n_layers; ++l) {
    const kivi_sink_layer &S = sinks[l];
    kivi_impl::SinkJob &J = p->jobs[l];
    J.k_res = layers ? layers[l].k_res : nullptr;
    J.v_res = layers ? layers[l].v_res : nullptr;
    J.top_pos = S.top_pos;
    J.top_score = S.top_score;
    J.top_count = S.top_count;
    J.sink_pos = S.sink_pos;
    J.sink_count = S.sink_count;
    J.sink_k = S.sink_k;
    J.sink_v = S.sink_v;
    J.mask = S.mask;
    J.scores = S.scores;
  }
}

kivi_status kivi_sink_update(const kivi_layer *layers, const kivi_sink_layer *sinks, int n_layers,
                             const kivi_cache *cache, const kivi_sink_cfg *cfg, int64_t i0,
                             int64_t n, kivi_stream_t stream) {
  kivi_status st = check_cache(layers, n_layers, cache);
  if (st != KIVI_OK) return st;
  st = check_sinks(sinks, n_layers, cache, cfg);
  if (st != KIVI_OK) return st;
  if (i0 < 0 || n < 0 || i0 + n > cache->n_res) return KIVI_ERR_INVAL;
  if (n == 0 || cache->bh == 0 || cfg->k_top == 0) return KIVI_OK;
  kivi_impl::SinkParams p;
  sink_params(layers, sinks, n_layers, cache, cfg, &p);
  p.i0 = i0;
  p.n = n;
  return cuda_status(kivi_impl::launch_sink_update(p, stream));
}

kivi_status kivi_flush_sink(const kivi_layer *layers, const kivi_sink_layer *sinks, int n_layers,
                            kivi_cache *cache, const kivi_sink_cfg *cfg, int64_t *n_flushed,
                            kivi_stream_t stream) {
  kivi_status st = check_cache(layers, n_layers, cache);
  if (st != KIVI_OK) return st;
  st = check_sinks(sinks, n_layers, cache, cfg);
  if (st != KIVI_OK) return st;
  const int64_t G = cache->group;
  const int W = 32 / cache->bits;
  const int64_t n = kivi_flush_size(cache->n_res, cache->residual, cache->group);
  if (n > 0 && cache->s_q + n > cache->cap) return KIVI_ERR_CAPACITY;
  if (n == 0 || cache->bh == 0) {
    if (n_flushed) *n_flushed = 0;
    if (n > 0) {
      cache->s_q += n;
      cache->res_head = (cache->res_head + n) % cache->r_cap;
      cache->n_res -= n;
      if (n_flushed) *n_flushed = n;
    }
    return KIVI_OK;
  }
  kivi_impl::SinkParams sp;
  sink_params(layers, sinks, n_layers, cache, cfg, &sp);
  sp.n = n;

  const int64_t d = cache->d;
  kivi_impl::QuantParams kp;
  std::memset(&kp, 0, sizeof(kp));
  kp.n_jobs = n_layers;
  kp.d = static_cast<int32_t>(d);
  kp.bh = cache->bh;
  kp.rows = n;
  kp.x_bh_stride = cache->r_cap * d;
  kp.ring = cache->r_cap;
  kp.head = cache->res_head;
  kp.heads = cache->bh / cfg->batch;
  kp.mask_words = (cache->r_cap + 31) / 32;
  kivi_impl::QuantParams vp = kp;
  kp.codes_bh_stride = cache->cap / W * d;
  kp.sz_bh_stride = cache->cap / G * d;
  kp.out0 = cache->s_q / G;
  vp.codes_bh_stride = cache->cap * (d / W);
  vp.sz_bh_stride = cache->cap * (d / G);
  vp.out0 = cache->s_q;
  vp.defer_wait = 1;   // reads the mask, complete before the key launch began its work
  for (int l = 0; l < n_layers; ++l) {
    const kivi_layer &L = layers[l];
    kp.jobs[l] = {L.k_res, L.k_codes, L.k_scale, L.k_zero, nullptr, sinks[l].mask};
    vp.jobs[l] = {L.v_res, L.v_codes, L.v_scale, L.v_zero, nullptr, sinks[l].mask};
  }
  cudaStream_t s = stream;
  const int mode = cfg->k_top > 0 ? kivi_impl::kQuantSink : kivi_impl::kQuantPlain;
  kivi_status r = KIVI_OK;
  if (cfg->k_top > 0) {   // mask and sink store first: the quantizers read the mask only
    r = cuda_status(kivi_impl::fault_word_address(&sp.fault));
    if (r != KIVI_OK) return r;
    r = cuda_status(kivi_impl::launch_sink_prepare(sp, s));
    if (r != KIVI_OK) return r;
  }
  r = cuda_status(kivi_impl::launch_key_quant(kp, cache->group, cache->bits, mode, s));
  if (r != KIVI_OK) return r;
  r = cuda_status(kivi_impl::launch_value_quant(vp, cache->group, cache->bits, mode, s));
  if (r != KIVI_OK) return r;
  cache->s_q += n;
  cache->res_head = (cache->res_head + n) % cache->r_cap;
  cache->n_res -= n;
  if (n_flushed) *n_flushed = n;
  return KIVI_OK;
}

kivi_status kivi_sink_restore(const kivi_sink_layer *sinks, int n_layers, const kivi_cache *cache,
                              const kivi_sink_cfg *cfg, void *const *k_out, void *const *v_out,
                              kivi_stream_t stream) {
  if (!cache || n_layers < 1 || n_layers > KIVI_MAX_LAYERS) return KIVI_ERR_INVAL;
  if (!valid_key_dim(cache->d) || cache->bh < 0 || cache->s_q < 0) return KIVI_ERR_INVAL;
  const kivi_status st = check_sinks(sinks, n_layers, cache, cfg);
  if (st != KIVI_OK) return st;
  if (!k_out || !v_out) return KIVI_ERR_INVAL;
  for (int l = 0; l < n_layers; ++l) {
    if (!k_out[l] || !v_out[l]) return KIVI_ERR_INVAL;
    if (!aligned16(k_out[l]) || !aligned16(v_out[l])) return KIVI_ERR_ALIGN;
  }
  if (cache->bh == 0 || cache->s_q == 0 || cfg->sink_cap == 0) return KIVI_OK;
  kivi_impl::SinkParams p;
  sink_params(nullptr, sinks, n_layers, cache, cfg, &p);
  p.out_rows = cache->s_q;
  for (int l = 0; l < n_layers; ++l) {
    p.jobs[l].k_out = k_out[l];
    p.jobs[l].v_out = v_out[l];
  }
  return cuda_status(kivi_impl::launch_sink_restore(p, stream));
}

kivi_status kivi_selftest_wait_timeout(uint32_t limit_us, kivi_stream_t stream) {
  if (limit_us < 1 || limit_us > 1000000) return KIVI_ERR_INVAL;
  return cuda_status(
      kivi_impl::launch_wait_timeout_selftest(uint64_t{limit_us} * 1000u, stream));
}

kivi_status kivi_decode_attention_sinks(const kivi_layer *layers, const kivi_sink_layer *sinks,
                                        int n_layers, const kivi_cache *cache,
                                        const kivi_sink_cfg *cfg, int64_t batch, int32_t h_q,
                                        float sm_scale, const void *const *q, float *const *out,
                                        int32_t n_split, float *workspace,
                                        int64_t workspace_floats, kivi_stream_t stream) {
  kivi_impl::AttnParams p;
  kivi_status st =
      attn_prepare(layers, n_layers, cache, batch, h_q, sm_scale, q, out, n_split, &p);
  if (st != KIVI_OK) return st;
  st = check_sinks(sinks, n_layers, cache, cfg);
  if (st != KIVI_OK) return st;
  if (cfg->batch != batch) return KIVI_ERR_INVAL;
  if (n_split > 1) {
    const int64_t need = kivi_decode_attention_workspace(cache, n_layers, batch, h_q, n_split);
    if (!workspace || workspace_floats < need) return KIVI_ERR_INVAL;
    if (!aligned16(workspace)) return KIVI_ERR_ALIGN;
    p.ws = workspace;
  }
  if (cache->bh == 0) return KIVI_OK;
  if (cfg->sink_cap > 0) {
    p.sink_cap = cfg->sink_cap;
    for (int l = 0; l < n_layers; ++l) {
      p.jobs[l].sink_pos = sinks[l].sink_pos;
      p.jobs[l].sink_count = sinks[l].sink_count;
      p.jobs[l].sink_k = sinks[l].sink_k;
      p.jobs[l].sink_v = sinks[l].sink_v;
    }
  }
  return cuda_status(kivi_impl::launch_decode_attention(p, cache->group, cache->bits, stream));
}

kivi_status kivi_device_fault(uint32_t *fault) {
  if (!fault) return KIVI_ERR_INVAL;
  return cuda_status(kivi_impl::read_and_clear_fault(fault));
}

}  // extern "C"
