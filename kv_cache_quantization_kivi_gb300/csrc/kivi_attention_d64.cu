// kivi_attention_d64.cu -- the register-operand decode-attention kernels
// (kivi_attention_kernel.cuh) at head_dim 64, in a translation unit of their
// own so that the head dims compile in parallel.
#include "kivi_attention_kernel.cuh"

namespace kivi_impl {

cudaError_t launch_decode_attention_d64(const AttnParams &p, int group, int bits,
                                         cudaStream_t stream) {
  return attention_dispatch<64>(p, group, bits, stream);
}

}  // namespace kivi_impl
