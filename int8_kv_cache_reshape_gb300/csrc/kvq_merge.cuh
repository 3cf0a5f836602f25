// kvq_merge.cuh -- merge of the split-KV decode's cut tiles, one CTA per
// tile, after the decode kernels of an attention call.
//
// vllm PR 50194 page, Key source snippet (enable_kv_split: the KV range of a
// tile is split and the partial results combined).  Piece s of a tile left,
// for each of its rows, o_s = (sum_j p_j v_j) / l_s and lse_s = m_s +
// log2(l_s) (log2 units, the weights' 2^6 lift included); the merged row is
//   o = sum_s 2^(lse_s - M) o_s / (sum_s 2^(lse_s - M) + sink),  M = max_s lse_s.
// An attention sink (log2 units, with the same 2^6 lift) is one more term of
// the normaliser.
//
// The pieces of a cut tile all end at the ends of warp segments, i.e. at the
// end of the decode kernel; merged there by the last piece's warp, a tile's
// partial rows were read by one warp with a few loads in flight, while the
// other warps' streaming still loaded the memory system (up to 10-17 us of
// tail).  Here a CTA of 256 threads merges a tile: 16 threads per row find
// its largest lse and the splits' weights 2^(lse_s - M) (kept in shared
// memory for up to kMergeWSplits splits) and normaliser; then each thread
// takes (row, 4-dim) items, consecutive threads on consecutive dims of a
// partial row, with eight splits' loads in flight.
#pragma once

#include <cuda_runtime.h>

#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {

constexpr int kMergeThreads = 256;
constexpr int kMergeWSplits = 64;  // splits whose weights stay in shared memory

// Merge of one cut tile m (nr = m.nrows rows, ns splits; its request's
// first query token q0) by a CTA of kMergeThreads threads; base(s): the
// partial row of split s's row 0 (its row n at base(s) + n).  With PRE, a
// thread's first item's partials of the first kMergePre splits are loaded
// together with the rows' lse values, so the merge is one round trip to L2
// after the decode grid completes (host plans, where base(s) is one
// multiply-add; the fused step's split rows take 64-bit divisions to find,
// and there the early loads measured slower).
constexpr int kMergePre = 8;
template <int D, bool PRE, class Base>
__device__ __forceinline__ void merge_tile(const AttnParams& p, const MergeItem& m, int q0, int ns,
                                           Base base) {
  const int G = p.group;
  const int nr = m.nrows;
  const int tid = threadIdx.x;
  const float log2e = 1.4426950408889634f;
  const bool w_smem = ns <= kMergeWSplits;
  constexpr int kQuads = D / 4;
  __shared__ float row_max[kTileMaxRows], row_inv[kTileMaxRows];
  __shared__ float wts[kTileMaxRows * kMergeWSplits];
  float4 pre[kMergePre];
  if constexpr (PRE) {
    const bool have = tid < nr * kQuads;
    const int n = tid / kQuads, d = (tid % kQuads) * 4;
#pragma unroll
    for (int s = 0; s < kMergePre; ++s)
      pre[s] = have && s < ns
                   ? __ldcg(reinterpret_cast<const float4*>(p.part_o + ((int64_t)base(s) + n) * D + d))
                   : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  }
  {
    const int n = tid >> 4, sub = tid & 15;
    const bool live = n < nr;
    float M = -INFINITY;
    if (live)
      for (int s = sub; s < ns; s += 16) M = fmaxf(M, __ldcg(p.part_lse + base(s) + n));
#pragma unroll
    for (int off = 8; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    const float sink = p.sinks && live ? fmaf(p.sinks[m.kv_head * G + (m.row0 + n) % G], log2e, 6.0f)
                                       : -INFINITY;
    M = fmaxf(M, sink);
    float sum = 0.0f;
    if (live && M != -INFINITY)
      for (int s = sub; s < ns; s += 16) {
        const float l = __ldcg(p.part_lse + base(s) + n);
        const float w = l == -INFINITY ? 0.0f : exp2f(l - M);
        if (w_smem) wts[n * kMergeWSplits + s] = w;
        sum += w;
      }
#pragma unroll
    for (int off = 8; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
    if (live && sub == 0) {
      if (sink != -INFINITY) sum += exp2f(sink - M);
      row_max[n] = M;
      row_inv[n] = sum > 0.0f ? 1.0f / sum : 0.0f;
    }
  }
  __syncthreads();
  if constexpr (KVQ_CHECKED) {
    // the tile's rows must lie in out (host plans: total_q_tokens is set)
    if (p.total_q_tokens > 0 && (q0 < 0 || q0 + (m.row0 + nr - 1) / G >= p.total_q_tokens)) {
      if (tid == 0) atomicExch(p.error_flag, 2);
      return;
    }
  }
  for (int it = tid; it < nr * kQuads; it += kMergeThreads) {
    const int n = it / kQuads, d = (it % kQuads) * 4;
    const float M = row_max[n], inv = row_inv[n];
    float a0 = 0.0f, a1 = 0.0f, a2 = 0.0f, a3 = 0.0f;
    int s0 = 0;
    if (PRE && it == tid && M != -INFINITY) {
      // the first item: its first splits' partials are in registers
#pragma unroll
      for (int s = 0; s < kMergePre; ++s) {
        if (s < ns) {
          float w;
          if (w_smem) {
            w = wts[n * kMergeWSplits + s];
          } else {
            const float l = __ldcg(p.part_lse + base(s) + n);
            w = l == -INFINITY ? 0.0f : exp2f(l - M);
          }
          a0 += w * pre[s].x;
          a1 += w * pre[s].y;
          a2 += w * pre[s].z;
          a3 += w * pre[s].w;
        }
      }
      s0 = kMergePre;
    }
    if (M != -INFINITY) {
#pragma unroll 8
      for (int s = s0; s < ns; ++s) {
        const int64_t r = (int64_t)base(s) + n;
        float w;
        if (w_smem) {
          w = wts[n * kMergeWSplits + s];
        } else {
          const float l = __ldcg(p.part_lse + r);
          w = l == -INFINITY ? 0.0f : exp2f(l - M);
        }
        const float4 v = __ldcg(reinterpret_cast<const float4*>(p.part_o + r * D + d));
        a0 += w * v.x;
        a1 += w * v.y;
        a2 += w * v.z;
        a3 += w * v.w;
      }
    }
    const int R = m.row0 + n;
    uint16_t* dst = p.out + ((int64_t)(q0 + R / G) * p.heads_q + m.kv_head * G + R % G) * D + d;
    *reinterpret_cast<uint2*>(dst) =
        make_uint2(dev::pack_bf16x2(a0 * inv, a1 * inv), dev::pack_bf16x2(a2 * inv, a3 * inv));
  }
}

// Host-planned calls: merge item blockIdx.x of the schedule (split s's rows
// at m.part + s * nrows).
template <int D>
__global__ void __launch_bounds__(kMergeThreads) merge_splits_kernel(const AttnParams p) {
  // Launched as a programmatic dependent of the decode kernel: this CTA may
  // be resident before the decode grid ends; the partials are read only once
  // that grid has completed and its writes are visible.  (The merge item and
  // the request's first token come from the host plan and the caller's
  // inputs, written before the decode kernel started.)
  const MergeItem m = p.merges[blockIdx.x];
  const int q0 = p.query_start_loc[m.req];
  asm volatile("griddepcontrol.wait;" ::: "memory");
  merge_tile<D, true>(p, m, q0, m.nsplits, [&](int s) { return m.part + s * m.nrows; });
}

// The fused decode step: tile blockIdx.x (request t / Hkv, kv head t % Hkv)
// of the device-built plan, if its chunks span more than one warp segment.
// The fused kernel cut its flat chunk sequence into `warps` equal segments;
// split s is warp w0 + s (one warp per chunk when there are fewer chunks
// than warps), whose partial rows sit in its second 16-row slot for the
// tile its segment ends in, and in its first for the one it starts in.
template <int D>
__global__ void __launch_bounds__(kMergeThreads) merge_step_kernel(const AttnParams p, const StepParams sp,
                                                                 int64_t warps) {
  const int t = blockIdx.x;
  // (the caller's input, as the fused kernel read it before its barrier --
  // host memory when that kernel stages the inputs; the plan is the fused
  // kernel's, read after the wait)
  const int q0 = sp.in_query_start_loc[t / p.heads_kv];
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int64_t T = __ldcg(sp.prefix + sp.num_tiles);
  const int64_t f0 = __ldcg(sp.prefix + t), f1 = __ldcg(sp.prefix + t + 1);
  if (T <= 0 || f1 <= f0) return;
  // warp whose segment holds flat chunk f: floor(((f + 1) W - 1) / T)
  auto warp_of = [&](int64_t f) { return ((f + 1) * warps - 1) / T; };
  const bool dense = T >= warps;
  const int64_t w0 = warp_of(f0);
  const int64_t ns = dense ? warp_of(f1 - 1) - w0 + 1 : f1 - f0;
  if (ns <= 1) return;  // one piece: written by its warp
  const bool first_is_last = (w0 * T) / warps < f0;
  const int4 ti = __ldcg(sp.tiles + t);
  const MergeItem m{t / p.heads_kv, t % p.heads_kv, 0, ti.w, 0, (int32_t)ns, 0, 0};
  merge_tile<D, false>(p, m, q0, (int)ns, [&](int s) {
    const int64_t w = dense ? w0 + s : warp_of(f0 + s);
    return (int)((2 * w + (s == 0 && first_is_last ? 1 : 0)) * kTileMaxRows);
  });
}

}  // namespace kvq
