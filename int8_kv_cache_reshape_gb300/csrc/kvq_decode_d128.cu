// kvq_decode_d128.cu -- split-KV decode kernels and the fused decode step for head_dim
// 128 (one translation unit per head_dim and ALiBi setting keeps the
// build parallel).
#include "kvq_decode.cuh"

namespace kvq {
int launch_decode_d128(const AttnParams& p, int dtype, int ntiles, void* stream) {
  return launch_decode_d<128, false>(p, dtype, ntiles, static_cast<cudaStream_t>(stream));
}
int launch_step_d128(const AttnParams& p, const StepParams& sp, int dtype, int64_t* warps,
                     void* stream) {
  return launch_step_d<128, false>(p, sp, dtype, warps, static_cast<cudaStream_t>(stream));
}
}  // namespace kvq
