// kvq_prefill_d256.cu -- tensor-core prefill kernels for head_dim 256 (one
// translation unit per head_dim and ALiBi setting keeps the build parallel).
#include "kvq_prefill.cuh"

namespace kvq {
int launch_prefill_d256(const AttnParams& p, const PrefillMaps& maps, int dtype, int64_t ctas,
                        void* stream) {
  return launch_prefill_d<256, false>(p, maps, dtype, ctas,
                                       static_cast<cudaStream_t>(stream));
}
}  // namespace kvq
