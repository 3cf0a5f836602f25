// kvq_cache.cu -- reshape_and_cache: quantise new K/V rows into the paged
// caches through slot_mapping.
//
// vllm PR 39445 page, Breakdown item 1 (the reshape kernel that writes the
// fp8 cache with scalar e4m3 quantisation) and vllm PR 38378 page,
// Breakdown item 3 (_reshape_cache_per_token_head: per-(token, head) absmax
// scale computed on the fly and stored inline).  The CPU design packs rows
// for AMX tiles; here rows stay in the plain paged layout
// [block][slot][kv_head][row] and each (token, head) row is handled by
// D/8 threads, each with one 16-byte load of K and of V.
//
// HBM bound: per element 2 bytes read, 1 byte written (+16 bytes of scale
// per row per-token-head).
#include <cuda_runtime.h>

#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {
namespace {

constexpr int kThreads = 256;

template <int DT>
__device__ __forceinline__ void quantise8(const uint4 x, float s, uint32_t& lo, uint32_t& hi) {
  const uint32_t w[4] = {x.x, x.y, x.z, x.w};
  uint32_t code[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float a = __fdiv_rn(dev::bf16_lo(w[i]), s);
    float b = __fdiv_rn(dev::bf16_hi(w[i]), s);
    if constexpr (DT == KVQ_INT8_PER_TOKEN_HEAD) {
      code[i] = dev::enc_int8(a) | (dev::enc_int8(b) << 8);
    } else if constexpr (DT == KVQ_FP8_E5M2) {
      code[i] = dev::enc_e5m2x2(a, b);
    } else {
      code[i] = dev::enc_e4m3x2(a, b);
    }
  }
  lo = code[0] | (code[1] << 16);
  hi = code[2] | (code[3] << 16);
}

__device__ __forceinline__ float absmax8(const uint4 x) {
  const uint32_t w[4] = {x.x, x.y, x.z, x.w};
  float m = 0.0f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    m = fmaxf(m, fabsf(dev::bf16_lo(w[i])));
    m = fmaxf(m, fabsf(dev::bf16_hi(w[i])));
  }
  return m;
}

// Writes one row's share (8 elements) of codes, and for per-token-head the
// scale tail.  TPR threads (a power of two, aligned in the warp) own a row.
template <int DT, int TPR>
__device__ __forceinline__ void write_part(const uint4 x, float tensor_scale, uint8_t* row,
                                           int part, bool active) {
  constexpr int kRowCodes = 8 * TPR;  // head_dim
  if constexpr (DT == KVQ_AUTO) {
    if (active) *reinterpret_cast<uint4*>(row + part * 16) = x;
  } else if constexpr (DT == KVQ_FP8_E4M3 || DT == KVQ_FP8_E5M2) {
    uint32_t lo, hi;
    quantise8<DT>(x, tensor_scale, lo, hi);
    if (active) *reinterpret_cast<uint2*>(row + part * 8) = make_uint2(lo, hi);
  } else {
    float m = absmax8(x);
#pragma unroll
    for (int off = TPR / 2; off > 0; off >>= 1)
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    const float s = __fdiv_rn(m, per_token_head_qmax(DT));
    uint32_t lo = 0, hi = 0;
    if (s != 0.0f) quantise8<code_format(DT)>(x, s, lo, hi);
    if (active) {
      *reinterpret_cast<uint2*>(row + part * 8) = make_uint2(lo, hi);
      if (part == 0)
        *reinterpret_cast<uint4*>(row + kRowCodes) = make_uint4(__float_as_uint(s), 0u, 0u, 0u);
    }
  }
}

// One (token, kv_head) row per TPR = D/8 threads; grid-stride over rows.
template <int DT, int D>
__global__ void __launch_bounds__(kThreads)
reshape_and_cache_kernel(const uint16_t* __restrict__ key, const uint16_t* __restrict__ value,
                         int64_t num_tokens, int64_t key_stride, int64_t value_stride,
                         int heads_kv, uint8_t* __restrict__ key_cache,
                         uint8_t* __restrict__ value_cache, int64_t num_slots,
                         const int64_t* __restrict__ slot_mapping, float k_scale,
                         float v_scale) {
  constexpr int TPR = D / 8;
  constexpr int kRowsPerBlock = kThreads / TPR;
  constexpr int kRow = row_bytes(DT, D);
  const int part = threadIdx.x % TPR;
  const int64_t total_rows = num_tokens * heads_kv;
  for (int64_t r0 = (int64_t)blockIdx.x * kRowsPerBlock; r0 < total_rows;
       r0 += (int64_t)gridDim.x * kRowsPerBlock) {
    const int64_t r = r0 + threadIdx.x / TPR;
    // Rows past the end still take part in the shuffles (per-token-head)
    // with a clamped, in-bounds read; they write nothing.
    const bool in_range = r < total_rows;
    const int64_t rr = in_range ? r : total_rows - 1;
    const int64_t t = rr / heads_kv;
    const int h = (int)(rr - t * heads_kv);
    const int64_t slot = slot_mapping[t];
    const bool active = in_range && slot >= 0 && slot < num_slots;
    const uint4 kx = dev::ldg_stream(key + t * key_stride + (int64_t)h * D + part * 8);
    const uint4 vx = dev::ldg_stream(value + t * value_stride + (int64_t)h * D + part * 8);
    const int64_t dst = (active ? (slot * heads_kv + h) : 0) * (int64_t)kRow;
    write_part<DT, TPR>(kx, k_scale, key_cache + dst, part, active);
    write_part<DT, TPR>(vx, v_scale, value_cache + dst, part, active);
  }
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
