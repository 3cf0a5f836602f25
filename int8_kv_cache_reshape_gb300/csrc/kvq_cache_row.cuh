// kvq_cache_row.cuh -- the cache writer's per-row quantisation, shared by
// the reshape_and_cache kernel and the fused decode step.
//
// vllm PR 39445 page, Breakdown item 1 (the reshape kernel writing the fp8
// cache with scalar e4m3 quantisation) and vllm PR 38378 page, Breakdown
// item 3 (_reshape_cache_per_token_head: per-(token, head) absmax scale
// computed on the fly and stored inline).  A (token, kv_head) row is handled
// by D/8 threads, each with one 16-byte load of K and of V.
#pragma once

#include <cuda_runtime.h>

#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {
namespace row {

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

// The (token, kv_head) rows of K and V, D/8 threads per row, the rows of a
// step of `threads` threads (a multiple of 32) side by side, over
// [first_step, steps) strided by `stride` steps.  Rows past the end still
// take part in the shuffles (per-token-head) with a clamped, in-bounds read;
// they write nothing.
template <int DT, int D>
__device__ __forceinline__ void write_rows(const uint16_t* __restrict__ key,
                                           const uint16_t* __restrict__ value, int64_t num_tokens,
                                           int64_t key_stride, int64_t value_stride, int heads_kv,
                                           uint8_t* __restrict__ key_cache,
                                           uint8_t* __restrict__ value_cache, int64_t num_slots,
                                           const int64_t* __restrict__ slot_mapping,
                                           float k_scale, float v_scale, int threads, int tid,
                                           int64_t first_step, int64_t stride) {
  constexpr int TPR = D / 8;
  constexpr int kRow = row_bytes(DT, D);
  const int rows_per_step = threads / TPR;
  const int part = tid % TPR;
  const int64_t total_rows = num_tokens * heads_kv;
  for (int64_t r0 = first_step * rows_per_step; r0 < total_rows; r0 += stride * rows_per_step) {
    const int64_t r = r0 + tid / TPR;
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

}  // namespace row
}  // namespace kvq
