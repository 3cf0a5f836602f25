// kvq_cache.cu -- reshape_and_cache: quantise new K/V rows into the paged
// caches through slot_mapping.
//
// vllm PR 39445 page, Breakdown item 1 (the reshape kernel that writes the
// fp8 cache with scalar e4m3 quantisation) and vllm PR 38378 page,
// Breakdown item 3 (_reshape_cache_per_token_head: per-(token, head) absmax
// scale computed on the fly and stored inline).  The CPU design packs rows
// for AMX tiles; here rows stay in the plain paged layout
// [block][slot][kv_head][row] and each (token, head) row is handled by
// D/8 threads, each with one 16-byte load of K and of V (kvq_cache_row.cuh).
//
// HBM bound: per element 2 bytes read, 1 byte written (+16 bytes of scale
// per row per-token-head).
#include <cuda_runtime.h>

#include "kvq_cache_row.cuh"
#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {
namespace {

constexpr int kThreads = 256;

// One (token, kv_head) row per TPR = D/8 threads; grid-stride over rows.
template <int DT, int D>
__global__ void __launch_bounds__(kThreads)
reshape_and_cache_kernel(const uint16_t* __restrict__ key, const uint16_t* __restrict__ value,
                         int64_t num_tokens, int64_t key_stride, int64_t value_stride,
                         int heads_kv, uint8_t* __restrict__ key_cache,
                         uint8_t* __restrict__ value_cache, int64_t num_slots,
                         const int64_t* __restrict__ slot_mapping, float k_scale,
                         float v_scale) {
  row::write_rows<DT, D>(key, value, num_tokens, key_stride, value_stride, heads_kv, key_cache,
                         value_cache, num_slots, slot_mapping, k_scale, v_scale, kThreads,
                         threadIdx.x, blockIdx.x, gridDim.x);
}

template <int DT, int D>
int launch(const void* key, const void* value, int64_t num_tokens, int64_t key_stride,
           int64_t value_stride, int heads_kv, void* key_cache, void* value_cache,
           int64_t num_slots, const int64_t* slot_mapping, float k_scale, float v_scale,
           cudaStream_t stream) {
  constexpr int kRowsPerBlock = kThreads / (D / 8);
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return KVQ_E_CUDA;
  const int64_t rows = num_tokens * heads_kv;
  int64_t blocks = (rows + kRowsPerBlock - 1) / kRowsPerBlock;
  const int64_t cap = (int64_t)sms * 8;  // 8 resident 256-thread blocks per SM
  if (blocks > cap) blocks = cap;
  reshape_and_cache_kernel<DT, D><<<(unsigned)blocks, kThreads, 0, stream>>>(
      static_cast<const uint16_t*>(key), static_cast<const uint16_t*>(value), num_tokens,
      key_stride, value_stride, heads_kv, static_cast<uint8_t*>(key_cache),
      static_cast<uint8_t*>(value_cache), num_slots, slot_mapping, k_scale, v_scale);
  return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_E_CUDA;
}

template <int DT>
int launch_d(int head_dim, const void* key, const void* value, int64_t num_tokens,
             int64_t key_stride, int64_t value_stride, int heads_kv, void* key_cache,
             void* value_cache, int64_t num_slots, const int64_t* slot_mapping, float k_scale,
             float v_scale, cudaStream_t stream) {
  switch (head_dim) {
    case 64:
      return launch<DT, 64>(key, value, num_tokens, key_stride, value_stride, heads_kv,
                            key_cache, value_cache, num_slots, slot_mapping, k_scale, v_scale,
                            stream);
    case 128:
      return launch<DT, 128>(key, value, num_tokens, key_stride, value_stride, heads_kv,
                             key_cache, value_cache, num_slots, slot_mapping, k_scale, v_scale,
                             stream);
    case 256:
      return launch<DT, 256>(key, value, num_tokens, key_stride, value_stride, heads_kv,
                             key_cache, value_cache, num_slots, slot_mapping, k_scale, v_scale,
                             stream);
    default:
      return KVQ_E_UNSUPPORTED;
  }
}

}  // namespace

int launch_reshape_and_cache(const void* key, const void* value, int64_t num_tokens,
                             int64_t key_stride, int64_t value_stride, int num_heads_kv,
                             int head_dim, void* key_cache, void* value_cache,
                             int64_t num_blocks, int block_size, const int64_t* slot_mapping,
                             int dtype, float k_scale, float v_scale, void* stream) {
  const int64_t slots = num_blocks * (int64_t)block_size;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
#define KVQ_CACHE_CASE(DT)                                                                    \
  case DT:                                                                                    \
    return launch_d<DT>(head_dim, key, value, num_tokens, key_stride, value_stride,           \
                        num_heads_kv, key_cache, value_cache, slots, slot_mapping, k_scale,   \
                        v_scale, s);
  switch (dtype) {
    KVQ_CACHE_CASE(KVQ_AUTO)
    KVQ_CACHE_CASE(KVQ_FP8_E4M3)
    KVQ_CACHE_CASE(KVQ_FP8_E5M2)
    KVQ_CACHE_CASE(KVQ_INT8_PER_TOKEN_HEAD)
    KVQ_CACHE_CASE(KVQ_FP8_PER_TOKEN_HEAD)
    KVQ_CACHE_CASE(KVQ_FP8_E5M2_PER_TOKEN_HEAD)
    default:
      return KVQ_E_UNSUPPORTED;
  }
#undef KVQ_CACHE_CASE
}

}  // namespace kvq
