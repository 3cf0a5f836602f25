// kvq_prefill_d64_alibi.cu -- tensor-core prefill kernels for head_dim 64, with the ALiBi bias (one
// translation unit per head_dim and ALiBi setting keeps the build parallel).
#include "kvq_prefill.cuh"

namespace kvq {
int launch_prefill_d64_alibi(const AttnParams& p, const PrefillMaps& maps, int dtype, int64_t ctas,
                             void* stream) {
  return launch_prefill_d<64, true>(p, maps, dtype, ctas,
                                       static_cast<cudaStream_t>(stream));
}
}  // namespace kvq
