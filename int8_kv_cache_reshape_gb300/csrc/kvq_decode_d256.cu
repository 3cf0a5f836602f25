// kvq_decode_d256.cu -- split-KV decode kernels for head_dim 256 (one
// translation unit per head_dim and ALiBi setting keeps the build parallel).
#include "kvq_decode.cuh"

namespace kvq {
int launch_decode_d256(const AttnParams& p, int dtype, int ntiles, void* stream) {
  return launch_decode_d<256, false>(p, dtype, ntiles, static_cast<cudaStream_t>(stream));
}
}  // namespace kvq
