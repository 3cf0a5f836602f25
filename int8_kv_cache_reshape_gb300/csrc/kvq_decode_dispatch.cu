// kvq_decode_dispatch.cu -- head_dim (and ALiBi) dispatch of the split-KV
// decode and the tensor-core prefill kernels (one translation unit per
// head_dim and ALiBi setting holds the instances).
#include "kvq_internal.h"
#include "kvq_merge.cuh"

namespace kvq {

// The merge runs right after the decode kernel on the stream, launched as its
// programmatic dependent (the decode kernel lets it be scheduled at once; it
// waits for the decode grid before reading): no launch gap between the two.
int launch_merge(const AttnParams& p, int head_dim, int64_t num_merges, void* stream) {
  if (num_merges <= 0) return KVQ_OK;
  void (*kern)(AttnParams);
  switch (head_dim) {
    case 64: kern = merge_splits_kernel<64>; break;
    case 128: kern = merge_splits_kernel<128>; break;
    case 256: kern = merge_splits_kernel<256>; break;
    default: return KVQ_E_UNSUPPORTED;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)num_merges);
  cfg.blockDim = dim3(kMergeThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, p) != cudaSuccess) {
    cudaGetLastError();
    return KVQ_E_CUDA;
  }
  return KVQ_OK;
}

int launch_merge_step(const AttnParams& p, const StepParams& sp, int head_dim, int64_t warps,
                      void* stream) {
  if (sp.num_tiles <= 0) return KVQ_OK;
  void (*kern)(AttnParams, StepParams, int64_t);
  switch (head_dim) {
    case 64: kern = merge_step_kernel<64>; break;
    case 128: kern = merge_step_kernel<128>; break;
    case 256: kern = merge_step_kernel<256>; break;
    default: return KVQ_E_UNSUPPORTED;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)sp.num_tiles);
  cfg.blockDim = dim3(kMergeThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, p, sp, warps) != cudaSuccess) {
    cudaGetLastError();
    return KVQ_E_CUDA;
  }
  return KVQ_OK;
}

#define KVQ_DECLARE(D)                                                                       \
  int launch_decode_d##D(const AttnParams&, int, int, void*);                               \
  int launch_decode_d##D##_alibi(const AttnParams&, int, int, void*);                       \
  int launch_step_d##D(const AttnParams&, const StepParams&, int, int64_t*, void*);         \
  int launch_step_d##D##_alibi(const AttnParams&, const StepParams&, int, int64_t*, void*); \
  int launch_prefill_d##D(const AttnParams&, const PrefillMaps&, int, int64_t, void*);      \
  int launch_prefill_d##D##_alibi(const AttnParams&, const PrefillMaps&, int, int64_t, void*);
KVQ_DECLARE(64)
KVQ_DECLARE(128)
KVQ_DECLARE(256)
#undef KVQ_DECLARE

int launch_decode(const AttnParams& p, int dtype, int head_dim, int ntiles, void* stream) {
  if (p.num_chunks <= 0) return KVQ_OK;
  const bool al = uses_alibi(p);
  switch (head_dim) {
    case 64: return al ? launch_decode_d64_alibi(p, dtype, ntiles, stream)
                       : launch_decode_d64(p, dtype, ntiles, stream);
    case 128: return al ? launch_decode_d128_alibi(p, dtype, ntiles, stream)
                        : launch_decode_d128(p, dtype, ntiles, stream);
    case 256: return al ? launch_decode_d256_alibi(p, dtype, ntiles, stream)
                        : launch_decode_d256(p, dtype, ntiles, stream);
    default: return KVQ_E_UNSUPPORTED;
  }
}

namespace {
int step_dispatch(const AttnParams& p, const StepParams& sp, int dtype, int head_dim, bool al,
                  int64_t* warps, void* stream) {
  switch (head_dim) {
    case 64: return al ? launch_step_d64_alibi(p, sp, dtype, warps, stream)
                       : launch_step_d64(p, sp, dtype, warps, stream);
    case 128: return al ? launch_step_d128_alibi(p, sp, dtype, warps, stream)
                        : launch_step_d128(p, sp, dtype, warps, stream);
    case 256: return al ? launch_step_d256_alibi(p, sp, dtype, warps, stream)
                        : launch_step_d256(p, sp, dtype, warps, stream);
    default: return KVQ_E_UNSUPPORTED;
  }
}
}  // namespace

int step_warps(int dtype, int head_dim, bool alibi, int max_rows, int64_t* warps) {
  AttnParams p{};
  StepParams sp{};
  sp.max_rows = max_rows;
  *warps = 0;
  return step_dispatch(p, sp, dtype, head_dim, alibi, warps, nullptr);
}

int launch_decode_step(const AttnParams& p, const StepParams& sp, int dtype, int head_dim,
                       int64_t warps, void* stream) {
  return step_dispatch(p, sp, dtype, head_dim, uses_alibi(p), &warps, stream);
}

int launch_prefill(const AttnParams& p, const PrefillMaps& maps, int dtype, int head_dim,
                   int64_t ctas, void* stream) {
  if (ctas <= 0) return KVQ_OK;
  const bool al = uses_alibi(p);
  switch (head_dim) {
    case 64: return al ? launch_prefill_d64_alibi(p, maps, dtype, ctas, stream)
                       : launch_prefill_d64(p, maps, dtype, ctas, stream);
    case 128: return al ? launch_prefill_d128_alibi(p, maps, dtype, ctas, stream)
                        : launch_prefill_d128(p, maps, dtype, ctas, stream);
    case 256: return al ? launch_prefill_d256_alibi(p, maps, dtype, ctas, stream)
                        : launch_prefill_d256(p, maps, dtype, ctas, stream);
    default: return KVQ_E_UNSUPPORTED;
  }
}

}  // namespace kvq
