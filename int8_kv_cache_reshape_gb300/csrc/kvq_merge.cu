// kvq_merge.cu -- merge of KV splits (the reduction after split-KV decode)
// and the head_dim dispatch of the row-tile kernels.
//
// vllm PR 50194 page, Key source snippet (enable_kv_split): the scheduler
// may split one sequence's keys across workers; the partial results are
// combined here.  Each split wrote o_s = (sum_j p_j v_j) / l_s and
// lse_s = m_s + log2(l_s) in log2 units; the merged row is
//   o = sum_s 2^(lse_s - M) o_s / sum_s 2^(lse_s - M),  M = max_s lse_s.
#include <cuda_runtime.h>

#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {

int launch_rowtile_d64(const AttnParams&, int, int, int64_t, int64_t, void*);
int launch_rowtile_d128(const AttnParams&, int, int, int64_t, int64_t, void*);
int launch_rowtile_d256(const AttnParams&, int, int, int64_t, int64_t, void*);

int launch_rowtile(const AttnParams& p, int dtype, int head_dim, int ntiles,
                   int64_t item_offset, int64_t num_items, void* stream) {
  if (num_items <= 0) return KVQ_OK;
  switch (head_dim) {
    case 64: return launch_rowtile_d64(p, dtype, ntiles, item_offset, num_items, stream);
    case 128: return launch_rowtile_d128(p, dtype, ntiles, item_offset, num_items, stream);
    case 256: return launch_rowtile_d256(p, dtype, ntiles, item_offset, num_items, stream);
    default: return KVQ_E_UNSUPPORTED;
  }
}

namespace {

constexpr int kMergeThreads = 128;

// One CTA per merge item; warp w merges rows w, w + 4, ...; each lane owns
// D/32 consecutive dims.
template <int D>
__global__ void __launch_bounds__(kMergeThreads) merge_kernel(const AttnParams p) {
  constexpr int kPer = D / 32;
  const MergeItem m = p.merges[blockIdx.x];
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int G = p.group;
  const int q0 = p.query_start_loc[m.req];
  for (int n = warp; n < m.nrows; n += kMergeThreads / 32) {
    float M = -INFINITY;
    for (int s = lane; s < m.nsplits; s += 32)
      M = fmaxf(M, p.part_lse[m.part + s * m.nrows + n]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    float acc[kPer];
#pragma unroll
    for (int e = 0; e < kPer; ++e) acc[e] = 0.0f;
    float wsum = 0.0f;
    for (int s = 0; s < m.nsplits; ++s) {
      const int row = m.part + s * m.nrows + n;
      const float lse = p.part_lse[row];
      const float w = (lse == -INFINITY || M == -INFINITY) ? 0.0f : exp2f(lse - M);
      wsum += w;
      const float* src = p.part_o + (int64_t)row * D + lane * kPer;
#pragma unroll
      for (int e = 0; e < kPer; e += 2) {
        const float2 v = *reinterpret_cast<const float2*>(src + e);
        acc[e] += w * v.x;
        acc[e + 1] += w * v.y;
      }
    }
    const float inv = wsum > 0.0f ? 1.0f / wsum : 0.0f;
    const int R = m.row0 + n;
    const int tok = q0 + R / G;
    const int head = m.kv_head * G + R % G;
    uint16_t* dst = p.out + ((int64_t)tok * p.heads_q + head) * D + lane * kPer;
#pragma unroll
    for (int e = 0; e < kPer; e += 2)
      *reinterpret_cast<uint32_t*>(dst + e) = dev::pack_bf16x2(acc[e] * inv, acc[e + 1] * inv);
  }
}

}  // namespace

int launch_merge(const AttnParams& p, int head_dim, int64_t num_items, void* stream) {
  if (num_items <= 0) return KVQ_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  switch (head_dim) {
    case 64: merge_kernel<64><<<(unsigned)num_items, kMergeThreads, 0, s>>>(p); break;
    case 128: merge_kernel<128><<<(unsigned)num_items, kMergeThreads, 0, s>>>(p); break;
    case 256: merge_kernel<256><<<(unsigned)num_items, kMergeThreads, 0, s>>>(p); break;
    default: return KVQ_E_UNSUPPORTED;
  }
  return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_E_CUDA;
}

}  // namespace kvq
