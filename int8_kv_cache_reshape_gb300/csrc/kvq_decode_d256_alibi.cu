// kvq_decode_d256_alibi.cu -- split-KV decode kernels and the fused decode step for head_dim
// 256, with the ALiBi bias (one translation unit per head_dim and ALiBi setting keeps the
// build parallel).
#include "kvq_decode.cuh"

namespace kvq {
int launch_decode_d256_alibi(const AttnParams& p, int dtype, int ntiles, void* stream) {
  return launch_decode_d<256, true>(p, dtype, ntiles, static_cast<cudaStream_t>(stream));
}
int launch_step_d256_alibi(const AttnParams& p, const StepParams& sp, int dtype, int64_t* warps,
                     void* stream) {
  return launch_step_d<256, true>(p, sp, dtype, warps, static_cast<cudaStream_t>(stream));
}
}  // namespace kvq
