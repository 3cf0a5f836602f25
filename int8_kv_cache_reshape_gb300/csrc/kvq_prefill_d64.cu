// kvq_prefill_d64.cu -- tensor-core prefill kernels for head_dim 64.
#include "kvq_prefill.cuh"

namespace kvq {
int launch_prefill_d64(const AttnParams& p, const PrefillMaps& maps, int dtype, int64_t num_tiles,
                       void* stream) {
  return launch_prefill_d<64>(p, maps, dtype, num_tiles, static_cast<cudaStream_t>(stream));
}
}  // namespace kvq
