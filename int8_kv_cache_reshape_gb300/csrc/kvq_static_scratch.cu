// kvq_static_scratch.cu -- attention_with_kv_cache for callers that cannot
// allocate device memory.
//
// Some callers cannot call cudaMalloc at the point where they run attention:
// code inside a memory-pool-managed serving loop, an allocator hook, or a
// host runtime that owns the device heap and forbids other allocations.
// For them this entry point takes no workspace: the split-KV partial rows go
// to a fixed array in the library's own device memory, reserved when the
// library is loaded on a device and held until the process exits.
#include <cuda_runtime.h>

#include <mutex>

#include "kvq_internal.h"

namespace {

// The scratch itself.  Device code can name it; host code must not use the
// symbol's host-side stand-in as an address -- it asks the runtime for the
// device address (once per device, below).
static __device__ __align__(256) unsigned char kvq_static_scratch[KVQ_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch on the current device (set up on the first
// call on each device).  Returns KVQ_OK, KVQ_E_CUDA or KVQ_E_UNSUPPORTED.
int scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return KVQ_E_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return KVQ_E_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_scratch_ptr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, kvq_static_scratch) != cudaSuccess || !ptr) {
      cudaGetLastError();
      return KVQ_E_CUDA;
    }
    g_scratch_ptr[dev] = ptr;
  }
  *out = g_scratch_ptr[dev];
  return KVQ_OK;
}

}  // namespace

extern "C" int kvq_attention_with_kv_cache_static_scratch(
    const kvq_sched_t* sched, int heads_q, int heads_kv, int head_dim, kvq_dtype_t dtype,
    const void* q, const void* key_cache, const void* value_cache,
    const int32_t* query_start_loc, const int32_t* seq_lens, const int32_t* block_table,
    int block_table_stride, int block_size, int64_t num_blocks, float sm_scale, int causal,
    int window, float soft_cap, const float* alibi_slopes, const float* sinks, float k_scale,
    float v_scale, void* out, void* stream) {
  if (!sched) return KVQ_E_INVALID_ARG;
  kvq_sched_info_t info;
  int rc = kvq_sched_get_info(sched, &info);
  if (rc != KVQ_OK) return rc;
  if (info.workspace_bytes > (size_t)KVQ_STATIC_SCRATCH_BYTES) return KVQ_E_WORKSPACE_TOO_SMALL;
  void* scratch = nullptr;
  rc = scratch_address(&scratch);
  if (rc != KVQ_OK) return rc;
  return kvq_attention_with_kv_cache(sched, heads_q, heads_kv, head_dim, dtype, q, key_cache,
                                     value_cache, query_start_loc, seq_lens, block_table,
                                     block_table_stride, block_size, num_blocks, sm_scale,
                                     causal, window, soft_cap, alibi_slopes, sinks, k_scale,
                                     v_scale, out, scratch,
                                     (size_t)KVQ_STATIC_SCRATCH_BYTES, stream);
}
