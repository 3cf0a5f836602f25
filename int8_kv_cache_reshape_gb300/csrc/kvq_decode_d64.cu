// kvq_decode_d64.cu -- split-KV decode kernels and the fused decode step for head_dim
// 64 (one translation unit per head_dim and ALiBi setting keeps the
// build parallel).
#include "kvq_decode.cuh"

namespace kvq {
int launch_decode_d64(const AttnParams& p, int dtype, int ntiles, void* stream) {
  return launch_decode_d<64, false>(p, dtype, ntiles, static_cast<cudaStream_t>(stream));
}
int launch_step_d64(const AttnParams& p, const StepParams& sp, int dtype, int64_t* warps,
                     void* stream) {
  return launch_step_d<64, false>(p, sp, dtype, warps, static_cast<cudaStream_t>(stream));
}
}  // namespace kvq
