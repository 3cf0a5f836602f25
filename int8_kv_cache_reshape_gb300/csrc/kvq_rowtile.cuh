// kvq_rowtile.cuh -- split-KV attention over the quantised paged cache for
// small row tiles (decode: one query token x G heads of a kv head).
//
// What it computes: for each packed row (query token, q head) of the tile,
// o = softmax_j(z_j) v_j over the visible keys j, with
//   z_j = sm_scale * (q . k_j) [* k_scale or the row's k scale],
//   optional soft cap z <- cap * tanh(z / cap), causal / sliding-window
//   masks; k_j, v_j are dequantised codes.  vllm PR 39445 page, Breakdown
//   items 2-3 (tile GEMMs for Q K^T and P V with the fp8 dequantisation
//   fused into the B-operand load, load_b_pair_vec) and Risks (scale
//   folding); vllm PR 38378 page, Breakdown item 3 (_prepare_kv_tile:
//   per-token-head scales applied inside the attention tile); vllm PR 50194
//   page, Key source snippet (enable_kv_split: the KV axis split across
//   workers and merged).
//
// GB300 design:
//   * HBM bound: every K/V byte is read once per tile; no dequantised copy
//     is written anywhere.  Each warp streams its chunks (16 tokens) through
//     a lane-private cp.async ring in shared memory (each lane reads back
//     only the bytes it copied: no barriers, no bank conflicts), several
//     chunks in flight per warp.  Every copy instruction covers whole
//     32-byte sectors, and the physical block of each chunk is fetched
//     ahead, 32 chunks per warp-wide load, so no copy waits on the block
//     table.
//   * Tensor cores at the register level: S^T = K Q^T and O^T = V^T P^T as
//     m16n8k16 f16 MMAs with tokens as M (one chunk), packed rows as N.
//     Codes convert exactly to f16 (e4m3 / e5m2 / int8 all fit), Q enters
//     exactly (a power-of-two shift of its bf16 values), and every scale
//     stays in fp32: sm_scale, log2(e) and the per-tensor k_scale multiply
//     the scores, v_scale the output; per-token-head scales multiply score
//     rows and P columns.
//   * The dot-product index order is permuted so that each lane reads
//     contiguous bytes; Q and the output use the same permutation, which
//     leaves the sums unchanged.
//   * Online softmax in log2 units with warp shuffles; the 4 warps of a CTA
//     and the CTAs of a split tile are merged with the log-sum-exp rule.
#pragma once

#include <cuda_runtime.h>

#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {

template <int DT, int D>
struct RowtileGeom {
  static constexpr int kKsteps = D / 16;     // MMA k-steps over head_dim (QK)
  static constexpr int kMtiles = D / 16;     // MMA m-tiles over head_dim (PV)
  static constexpr int kK16 = D / 64;        // 16-byte K pieces per lane per row
  static constexpr int kVBytes = D / 8;      // V bytes per lane per row
  static constexpr int kVPieces = kVBytes >= 16 ? kVBytes / 16 : 1;
  static constexpr int kVSlots = D / 32;     // 16-byte V slots per lane
  static constexpr bool kPth = is_per_token_head(DT);
  static constexpr int kSlots = 2 * kK16 + kVSlots + (kPth ? 1 : 0);
  static constexpr int kStageBytes = kSlots * 32 * 16;
  static constexpr int kStages = rowtile_stages(DT, D);
  static constexpr int kRow = row_bytes(DT, D);
  static_assert(kStageBytes == rowtile_chunk_bytes(DT, D), "stage size must follow the geometry");
  static_assert((size_t)kStageBytes * kStages * kRowtileWarps == rowtile_pipeline_smem(DT, D),
                "pipeline size must follow the geometry");
};

// Head dim of element k (0: MMA row g, 1: row g + 8) of P.V m-tile mi for a
// lane of group g: each lane owns 16-byte runs of every V row (8 bytes for
// head_dim 64), the runs of the 8 groups side by side.
template <int D>
__device__ __forceinline__ int pv_dim(int mi, int g, int k) {
  constexpr int run = D / 8 >= 16 ? 16 : D / 8;
  return (mi / 8) * 128 + g * run + 2 * (mi % 8) + k;
}

// Merge of a tile's KV splits (vllm PR 50194 page, Key source snippet:
// enable_kv_split).  Each split s left o_s = (sum_j p_j v_j) / l_s and
// lse_s = m_s + log2(l_s) (log2 units); the merged row is
//   o = sum_s 2^(lse_s - M) o_s / sum_s 2^(lse_s - M),  M = max_s lse_s.
// Run by the last CTA of the split group to finish; warp w merges rows
// w, w + 4, ...; each lane owns D/32 consecutive dims.  Partials are read
// through L2 (other CTAs wrote them).
template <int D>
__device__ __forceinline__ void merge_splits(const AttnParams& p, const MergeItem& m, int warp,
                                             int lane) {
  constexpr int kPer = D / 32;
  const int G = p.group;
  const int q0 = p.query_start_loc[m.req];
  for (int n = warp; n < m.nrows; n += kRowtileWarps) {
    float M = -INFINITY;
    for (int s = lane; s < m.nsplits; s += 32)
      M = fmaxf(M, __ldcg(p.part_lse + m.part + s * m.nrows + n));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    float acc[kPer];
#pragma unroll
    for (int e = 0; e < kPer; ++e) acc[e] = 0.0f;
    float wsum = 0.0f;
    for (int s = 0; s < m.nsplits; ++s) {
      const int row = m.part + s * m.nrows + n;
      const float lse = __ldcg(p.part_lse + row);
      const float w = (lse == -INFINITY || M == -INFINITY) ? 0.0f : exp2f(lse - M);
      wsum += w;
      const float* src = p.part_o + (int64_t)row * D + lane * kPer;
#pragma unroll
      for (int e = 0; e < kPer; e += 2) {
        const float2 v = __ldcg(reinterpret_cast<const float2*>(src + e));
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

template <int DT, int D, int NT>
__global__ void __launch_bounds__(kRowtileThreads, rowtile_min_ctas(DT, D, NT))
rowtile_attention_kernel(const AttnParams p, int64_t item_offset) {
  using Geo = RowtileGeom<DT, D>;
  extern __shared__ __align__(128) uint8_t smem[];
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int g = lane >> 2;
  const int c = lane & 3;

  const RowtileItem it = p.items[item_offset + blockIdx.x];
  const int G = p.group;
  const int q0 = p.query_start_loc[it.req];
  const int Q = p.query_start_loc[it.req + 1] - q0;
  const int L = p.seq_lens[it.req];
  const int p_min = L - Q + it.row0 / G;
  const int p_max = L - Q + (it.row0 + it.nrows - 1) / G;
  const int W = p.window;
  // Keys any row of the tile can see, and keys every row sees.
  const int any_lo = W > 0 ? p_min - W + 1 : 0;
  const int any_hi = p.causal ? p_max + 1 : L;
  const int all_lo = W > 0 ? p_max - W + 1 : 0;
  const int all_hi = p.causal ? p_min + 1 : L;

  // ---- chunk pipeline: the first chunks are requested before Q is loaded --
  const int nchunks = it.chunk_hi - it.chunk_lo;
  const int nk = nchunks > warp ? (nchunks - warp + kRowtileWarps - 1) / kRowtileWarps : 0;
  const uint32_t ring =
      dev::smem_u32(smem) + (uint32_t)(warp * Geo::kStages * Geo::kStageBytes) + lane * 16;
  const int32_t* btab = p.block_table + (int64_t)it.req * p.block_table_stride;
  const uint8_t* kbase = p.key_cache;
  const uint8_t* vbase = p.value_cache;
  const int64_t row_stride = (int64_t)p.heads_kv * Geo::kRow;  // bytes between tokens
  const uint32_t rs = (uint32_t)row_stride;
  const uint32_t head_off = (uint32_t)it.kv_head * Geo::kRow;
  // Byte offsets, from a chunk's first row, of what this lane copies:
  // K rows g, g+8, bytes 64i + 16c (piece i); V rows 2c, 2c+1, 2c+8, 2c+9,
  // bytes 128i + 16g (8g for head_dim 64); the scale tail of K row g (c=0),
  // K row g+8 (c=1), V row g (c=2) or V row g+8 (c=3).
  const uint32_t koff0 = g * rs + head_off + 16 * c;
  const uint32_t koff1 = koff0 + 8 * rs;
  uint32_t voff[4];
#pragma unroll
  for (int vr = 0; vr < 4; ++vr)
    voff[vr] = (2 * c + (vr & 1) + 8 * (vr >> 1)) * rs + head_off +
               g * (Geo::kVBytes >= 16 ? 16 : Geo::kVBytes);
  const uint32_t toff = (g + 8 * (c & 1)) * rs + head_off + D;
  const int cpb = p.block_size / kChunkTokens;  // chunks per cache block
  int64_t slot_reg = -1;  // first slot of this lane's chunk in the batch (-1: no block)
  uint32_t ok_bits = 0;

  auto issue = [&](int k, int stage) {
    if ((k & 31) == 0) {
      // Block ids of the next 32 chunks of this warp, one per lane.
      const int kk = k + lane;
      int64_t s0 = -1;
      if (kk < nk) {
        const int chunk = it.chunk_lo + warp + kk * kRowtileWarps;
        const int lb = chunk / cpb;
        const int blk = btab[lb];
        if (blk >= 0 && (int64_t)blk < p.num_blocks)
          s0 = (int64_t)blk * p.block_size + (int64_t)(chunk - lb * cpb) * kChunkTokens;
      }
      slot_reg = s0;
    }
    const int src_lane = k & 31;
    const uint32_t lo = __shfl_sync(0xffffffffu, (uint32_t)(uint64_t)slot_reg, src_lane);
    const uint32_t hi = __shfl_sync(0xffffffffu, (uint32_t)((uint64_t)slot_reg >> 32), src_lane);
    const int64_t slot0 = (int64_t)(((uint64_t)hi << 32) | lo);
    const bool ok = slot0 >= 0;
    ok_bits = (ok_bits & ~(1u << stage)) | ((ok ? 1u : 0u) << stage);
    const int tok0 = (it.chunk_lo + warp + k * kRowtileWarps) * kChunkTokens;
    const bool all_live = ok && tok0 >= any_lo && tok0 + kChunkTokens <= any_hi;
    auto live = [&](int r) {
      return all_live || (ok && tok0 + r >= any_lo && tok0 + r < any_hi);
    };
    const uint8_t* kchunk = kbase + (ok ? slot0 * row_stride : 0);
    const uint8_t* vchunk = vbase + (ok ? slot0 * row_stride : 0);
    const uint32_t dst = ring + stage * Geo::kStageBytes;
    if (all_live) {  // warp-uniform: every row of the chunk is copied
#pragma unroll
      for (int i = 0; i < Geo::kK16; ++i) {
        dev::cp_async_16(dst + i * 512, kchunk + koff0 + 64 * i, 16);
        dev::cp_async_16(dst + (Geo::kK16 + i) * 512, kchunk + koff1 + 64 * i, 16);
      }
#pragma unroll
      for (int vr = 0; vr < 4; ++vr) {
        if constexpr (Geo::kVBytes == 8) {
          dev::cp_async_8(dst + (2 * Geo::kK16 + vr / 2) * 512 + (vr & 1) * 8, vchunk + voff[vr], 8);
        } else {
#pragma unroll
          for (int i = 0; i < Geo::kVPieces; ++i)
            dev::cp_async_16(dst + (2 * Geo::kK16 + vr * Geo::kVPieces + i) * 512,
                             vchunk + voff[vr] + 128 * i, 16);
        }
      }
      if constexpr (Geo::kPth)
        dev::cp_async_16(dst + (Geo::kSlots - 1) * 512, (c < 2 ? kchunk : vchunk) + toff, 16);
      return;
    }
    // K rows g and g + 8.
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      const bool lv = live(g + 8 * rr);
      const uint8_t* src = lv ? kchunk + (rr ? koff1 : koff0) : kbase;
#pragma unroll
      for (int i = 0; i < Geo::kK16; ++i)
        dev::cp_async_16(dst + (rr * Geo::kK16 + i) * 512, src + (lv ? 64 * i : 0), lv ? 16 : 0);
    }
    // V rows 2c, 2c+1, 2c+8, 2c+9.
#pragma unroll
    for (int vr = 0; vr < 4; ++vr) {
      const bool lv = live(2 * c + (vr & 1) + 8 * (vr >> 1));
      const uint8_t* src = lv ? vchunk + voff[vr] : vbase;
      if constexpr (Geo::kVBytes == 8) {
        dev::cp_async_8(dst + (2 * Geo::kK16 + vr / 2) * 512 + (vr & 1) * 8, src, lv ? 8 : 0);
      } else {
#pragma unroll
        for (int i = 0; i < Geo::kVPieces; ++i)
          dev::cp_async_16(dst + (2 * Geo::kK16 + vr * Geo::kVPieces + i) * 512,
                           src + (lv ? 128 * i : 0), lv ? 16 : 0);
      }
    }
    if constexpr (Geo::kPth) {
      const bool lv = live(g + 8 * (c & 1));
      const uint8_t* src = lv ? (c < 2 ? kchunk : vchunk) + toff : kbase;
      dev::cp_async_16(dst + (Geo::kSlots - 1) * 512, src, lv ? 16 : 0);
    }
  };

#pragma unroll
  for (int s = 0; s < Geo::kStages - 1; ++s) {
    if (s < nk) issue(s, s);
    dev::cp_async_commit();
  }

  // ---- Q fragments (B operand of S^T = K Q^T) -----------------------------
  // Q enters the MMA exactly: bf16 values scaled by a power of two only
  // (8 significant bits fit f16's 11); sm_scale and log2(e) are applied to
  // the fp32 scores, so no rounding of Q * sm_scale perturbs large scores.
  // Lane c holds dims 64i + 16c + [0, 16) of its rows (K piece i).
  const float log2e = 1.4426950408889634f;
  const float base_scale = p.sm_scale * (p.soft_cap > 0.0f ? 1.0f : log2e);
  float qv[NT][D / 4];
  float qmax = 0.0f;
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    const int n = 8 * t + g;
    const bool valid = n < it.nrows;
    const int R = it.row0 + (valid ? n : 0);
    const int tok = q0 + R / G;
    const int head = it.kv_head * G + R % G;
    const uint16_t* src = p.q + ((int64_t)tok * p.heads_q + head) * D + 16 * c;
#pragma unroll
    for (int i = 0; i < Geo::kK16; ++i) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint4 w = valid ? *reinterpret_cast<const uint4*>(src + 64 * i + 8 * h)
                              : make_uint4(0, 0, 0, 0);
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int e = 16 * i + 8 * h + 2 * k;
          qv[t][e] = dev::bf16_lo(ws[k]);
          qv[t][e + 1] = dev::bf16_hi(ws[k]);
          qmax = fmaxf(qmax, fmaxf(fabsf(qv[t][e]), fabsf(qv[t][e + 1])));
        }
      }
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) qmax = fmaxf(qmax, __shfl_xor_sync(0xffffffffu, qmax, off));
  // Power-of-two shift that puts the largest |q| just under 2^15.
  int shift = 0;
  if (qmax > 0.0f && qmax < 3.0e38f) {
    int e;
    frexpf(qmax, &e);
    shift = max(-126, min(126, 15 - e));
  }
  const float q_mul = __int_as_float((127 + shift) << 23);
  const float q_unmul = __int_as_float((127 - shift) << 23);
  uint32_t qf[NT][Geo::kKsteps][2];
#pragma unroll
  for (int t = 0; t < NT; ++t)
#pragma unroll
    for (int j = 0; j < Geo::kKsteps; ++j) {
      qf[t][j][0] = dev::pack_f16x2(qv[t][4 * j] * q_mul, qv[t][4 * j + 1] * q_mul);
      qf[t][j][1] = dev::pack_f16x2(qv[t][4 * j + 2] * q_mul, qv[t][4 * j + 3] * q_mul);
    }

  // Per-column (packed row) key limits for this lane's columns 2c, 2c+1.
  int col_lo[NT][2], col_hi[NT][2];
#pragma unroll
  for (int t = 0; t < NT; ++t)
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int n = min(8 * t + 2 * c + k, it.nrows - 1);
      const int pn = L - Q + (it.row0 + n) / G;
      col_hi[t][k] = p.causal ? pn + 1 : L;
      col_lo[t][k] = W > 0 ? pn - W + 1 : 0;
    }
  const float score_mul = q_unmul * base_scale * (Geo::kPth ? 1.0f : p.k_scale);
  const float cap = p.soft_cap;
  const float cap_l2 = cap * log2e;
  const float inv_cap = cap > 0.0f ? 1.0f / cap : 0.0f;

  // ---- running softmax state ------------------------------------------
  // P enters the P.V MMA as f16 scaled by 2^14 (l carries the same factor,
  // so it cancels in O / l): weights down to 2^-28 of the running maximum
  // stay normal f16 numbers.  Per-token-head V scales multiply P as
  // s_v * 2^-ev, ev the exponent of the largest s_v seen so far (a running
  // reference like the softmax maximum; O is rescaled when it grows), so
  // that small scales keep P inside the f16 range.
  float o[NT][Geo::kMtiles][4];
  float m_run[NT][2], l_run[NT][2];
  int ev = -1000;
#pragma unroll
  for (int t = 0; t < NT; ++t) {
#pragma unroll
    for (int i = 0; i < Geo::kMtiles; ++i) o[t][i][0] = o[t][i][1] = o[t][i][2] = o[t][i][3] = 0.0f;
    m_run[t][0] = m_run[t][1] = -INFINITY;
    l_run[t][0] = l_run[t][1] = 0.0f;
  }

  for (int k = 0; k < nk; ++k) {
    dev::cp_async_wait<Geo::kStages - 2>();
    {
      const int nxt = k + Geo::kStages - 1;
      if (nxt < nk) issue(nxt, nxt % Geo::kStages);
      dev::cp_async_commit();
    }
    const int stage = k % Geo::kStages;
    const uint32_t src = ring + stage * Geo::kStageBytes;
    const int tok0 = (it.chunk_lo + warp + k * kRowtileWarps) * kChunkTokens;
    const bool chunk_ok = (ok_bits >> stage) & 1u;

    // Per-token-head scales of tokens g and g + 8 (K and V).
    float sk0 = 1.0f, sk1 = 1.0f, sv0 = 1.0f, sv1 = 1.0f;
    float alpha_v = 1.0f;
    bool rescale_v = false;
    if constexpr (Geo::kPth) {
      const uint4 tail = dev::lds128(src + (Geo::kSlots - 1) * 512);
      const float mine = __uint_as_float(tail.x);
      sk0 = __shfl_sync(0xffffffffu, mine, 4 * g + 0);
      sk1 = __shfl_sync(0xffffffffu, mine, 4 * g + 1);
      sv0 = __shfl_sync(0xffffffffu, mine, 4 * g + 2);
      sv1 = __shfl_sync(0xffffffffu, mine, 4 * g + 3);
      float mx = fmaxf(sv0, sv1);
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      if (mx > 0.0f) {
        const int e = max(-100, min(100, (int)((__float_as_uint(mx) >> 23) & 0xFFu) - 127));
        if (e > ev) {
          alpha_v = ldexpf(1.0f, ev - e);
          rescale_v = true;
          ev = e;
        }
      }
      const float to_ref = ldexpf(1.0f, -ev);
      sv0 *= to_ref;
      sv1 *= to_ref;
    }

    // S^T = K Q^T : 16 tokens x 8 rows per n-tile; even and odd k-steps in
    // separate accumulators to halve the dependent MMA chain.
    float s[NT][4], s2[NT][4];
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
      for (int e = 0; e < 4; ++e) s[t][e] = s2[t][e] = 0.0f;
#pragma unroll
    for (int i = 0; i < Geo::kK16; ++i) {
      const uint4 kg = dev::lds128(src + i * 512);
      const uint4 kg8 = dev::lds128(src + (Geo::kK16 + i) * 512);
      const uint32_t wg[4] = {kg.x, kg.y, kg.z, kg.w};
      const uint32_t wg8[4] = {kg8.x, kg8.y, kg8.z, kg8.w};
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const int j = 4 * i + w;
        uint32_t a[4];
        dev::word_to_f16x2x2<DT>(wg[w], a[0], a[2]);
        dev::word_to_f16x2x2<DT>(wg8[w], a[1], a[3]);
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          if (w & 1) dev::mma_f16_16816(s2[t], a, qf[t][j][0], qf[t][j][1]);
          else dev::mma_f16_16816(s[t], a, qf[t][j][0], qf[t][j][1]);
        }
      }
    }

    // Scores in log2 units, masks, running max.
    const bool full = chunk_ok && tok0 >= all_lo && tok0 + kChunkTokens <= all_hi;
    uint32_t pb0[NT], pb1[NT];
    bool rescale = false;
    float alpha[NT][2];
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      float z[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float sk = (e < 2) ? sk0 : sk1;
        float v = (s[t][e] + s2[t][e]) * score_mul * sk;
        if (cap > 0.0f) v = cap_l2 * tanhf(v * inv_cap);
        if (!full) {
          const int tok = tok0 + g + 8 * (e >> 1);
          const int col = e & 1;
          const bool vis = chunk_ok && tok >= col_lo[t][col] && tok < col_hi[t][col];
          v = vis ? v : -INFINITY;
        }
        z[e] = v;
      }
      float cm0 = fmaxf(z[0], z[2]), cm1 = fmaxf(z[1], z[3]);
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        cm0 = fmaxf(cm0, __shfl_xor_sync(0xffffffffu, cm0, off));
        cm1 = fmaxf(cm1, __shfl_xor_sync(0xffffffffu, cm1, off));
      }
      const float mn0 = fmaxf(m_run[t][0], cm0), mn1 = fmaxf(m_run[t][1], cm1);
      const float ref0 = mn0 == -INFINITY ? 0.0f : mn0;
      const float ref1 = mn1 == -INFINITY ? 0.0f : mn1;
      alpha[t][0] = dev::fast_exp2(m_run[t][0] - ref0);
      alpha[t][1] = dev::fast_exp2(m_run[t][1] - ref1);
      rescale |= (alpha[t][0] != 1.0f) || (alpha[t][1] != 1.0f);
      m_run[t][0] = mn0;
      m_run[t][1] = mn1;
      // P * 2^14 (see above); l_run and O carry the same factor.
      const float e0 = ref0 - 14.0f, e1 = ref1 - 14.0f;
      const float p0 = dev::fast_exp2(z[0] - e0), p1 = dev::fast_exp2(z[1] - e1);
      const float p2 = dev::fast_exp2(z[2] - e0), p3 = dev::fast_exp2(z[3] - e1);
      l_run[t][0] = l_run[t][0] * alpha[t][0] + (p0 + p2);
      l_run[t][1] = l_run[t][1] * alpha[t][1] + (p1 + p3);
      // P^T (tokens x rows) -> B operand of O^T = V^T P^T via transposes.
      pb0[t] = dev::movmatrix_trans(dev::pack_f16x2(p0 * sv0, p1 * sv0));
      pb1[t] = dev::movmatrix_trans(dev::pack_f16x2(p2 * sv1, p3 * sv1));
    }
    if (__any_sync(0xffffffffu, rescale) || rescale_v) {
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        const float a0 = alpha[t][0] * alpha_v, a1 = alpha[t][1] * alpha_v;
#pragma unroll
        for (int i = 0; i < Geo::kMtiles; ++i) {
          o[t][i][0] *= a0;
          o[t][i][1] *= a1;
          o[t][i][2] *= a0;
          o[t][i][3] *= a1;
        }
      }
    }

    // O^T += V^T P^T : head_dim x 8 rows per n-tile.
    constexpr int kWords = Geo::kVBytes == 8 ? 2 : 4;  // words per row per piece
#pragma unroll
    for (int vs = 0; vs < Geo::kVPieces; ++vs) {
      uint32_t r0[4], r1[4], r2[4], r3[4];
      if constexpr (Geo::kVBytes == 8) {
        // head_dim 64: slot 0 holds rows 2c | 2c+1, slot 1 rows 2c+8 | 2c+9.
        const uint4 x01 = dev::lds128(src + (2 * Geo::kK16 + 0) * 512);
        const uint4 x23 = dev::lds128(src + (2 * Geo::kK16 + 1) * 512);
        r0[0] = x01.x; r0[1] = x01.y; r1[0] = x01.z; r1[1] = x01.w;
        r2[0] = x23.x; r2[1] = x23.y; r3[0] = x23.z; r3[1] = x23.w;
        r0[2] = r0[3] = r1[2] = r1[3] = r2[2] = r2[3] = r3[2] = r3[3] = 0u;
      } else {
        const uint4 a0 = dev::lds128(src + (2 * Geo::kK16 + 0 * Geo::kVPieces + vs) * 512);
        const uint4 a1 = dev::lds128(src + (2 * Geo::kK16 + 1 * Geo::kVPieces + vs) * 512);
        const uint4 a2 = dev::lds128(src + (2 * Geo::kK16 + 2 * Geo::kVPieces + vs) * 512);
        const uint4 a3 = dev::lds128(src + (2 * Geo::kK16 + 3 * Geo::kVPieces + vs) * 512);
        r0[0] = a0.x; r0[1] = a0.y; r0[2] = a0.z; r0[3] = a0.w;
        r1[0] = a1.x; r1[1] = a1.y; r1[2] = a1.z; r1[3] = a1.w;
        r2[0] = a2.x; r2[1] = a2.y; r2[2] = a2.z; r2[3] = a2.w;
        r3[0] = a3.x; r3[1] = a3.y; r3[2] = a3.z; r3[3] = a3.w;
      }
      // Word w of rows 2c / 2c+1 -> bytes (b0, b1) and (b2, b3) paired across
      // the two tokens: m-tiles 2(vs*kWords + w) and 2(vs*kWords + w) + 1.
#pragma unroll
      for (int w = 0; w < kWords; ++w) {
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const uint32_t sel = half ? 0x7362u : 0x5140u;
          const uint32_t x01 = dev::prmt(r0[w], r1[w], sel);
          const uint32_t x23 = dev::prmt(r2[w], r3[w], sel);
          uint32_t a[4];
          dev::word_to_f16x2x2<DT>(x01, a[0], a[1]);
          dev::word_to_f16x2x2<DT>(x23, a[2], a[3]);
          const int i = (vs * kWords + w) * 2 + half;  // m-tile
#pragma unroll
          for (int t = 0; t < NT; ++t) dev::mma_f16_16816(o[t][i], a, pb0[t], pb1[t]);
        }
      }
    }
  }
  dev::cp_async_wait<0>();

  // ---- combine the 4 warps ------------------------------------------------
#pragma unroll
  for (int t = 0; t < NT; ++t)
#pragma unroll
    for (int k = 0; k < 2; ++k)
#pragma unroll
      for (int off = 4; off < 32; off <<= 1)
        l_run[t][k] += __shfl_xor_sync(0xffffffffu, l_run[t][k], off);
  __syncthreads();  // every warp is done with its ring
  float* comb_o = reinterpret_cast<float*>(smem);                       // [W][16][D]
  float* comb_m = comb_o + kRowtileWarps * kRowtileMaxRows * D;        // [W][16]
  float* comb_l = comb_m + kRowtileWarps * kRowtileMaxRows;            // [W][16]
  const float unit = Geo::kPth && ev > -1000 ? ldexpf(1.0f, ev) : 1.0f;
#pragma unroll
  for (int t = 0; t < NT; ++t)
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int n = 8 * t + 2 * c + k;
      if (g == 0) {
        comb_m[warp * kRowtileMaxRows + n] = m_run[t][k];
        comb_l[warp * kRowtileMaxRows + n] = l_run[t][k];
      }
      float* dst = comb_o + (warp * kRowtileMaxRows + n) * D;
#pragma unroll
      for (int i = 0; i < Geo::kMtiles; ++i)
        *reinterpret_cast<float2*>(dst + pv_dim<D>(i, g, 0)) =
            make_float2(o[t][i][k] * unit, o[t][i][k + 2] * unit);
    }
  __syncthreads();

  const int per_row = D / 8;
  for (int idx = threadIdx.x; idx < it.nrows * per_row; idx += kRowtileThreads) {
    const int n = idx / per_row;
    const int d0 = (idx % per_row) * 8;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kRowtileWarps; ++w) M = fmaxf(M, comb_m[w * kRowtileMaxRows + n]);
    float f[kRowtileWarps];
    float lsum = 0.0f;
#pragma unroll
    for (int w = 0; w < kRowtileWarps; ++w) {
      const float mw = comb_m[w * kRowtileMaxRows + n];
      f[w] = mw == -INFINITY ? 0.0f : exp2f(mw - M);
      lsum += f[w] * comb_l[w * kRowtileMaxRows + n];
    }
    float acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.0f;
#pragma unroll
    for (int w = 0; w < kRowtileWarps; ++w) {
      const float* srcp = comb_o + (w * kRowtileMaxRows + n) * D + d0;
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] += f[w] * srcp[e];
    }
    const float inv_l = lsum > 0.0f ? 1.0f / lsum : 0.0f;
    const float vmul = Geo::kPth ? 1.0f : p.v_scale;
    const int R = it.row0 + n;
    const float sc = inv_l * vmul;
    if (it.part < 0) {
      const int tok = q0 + R / G;
      const int head = it.kv_head * G + R % G;
      uint16_t* dst = p.out + ((int64_t)tok * p.heads_q + head) * D + d0;
      *reinterpret_cast<uint4*>(dst) =
          make_uint4(dev::pack_bf16x2(acc[0] * sc, acc[1] * sc), dev::pack_bf16x2(acc[2] * sc, acc[3] * sc),
                     dev::pack_bf16x2(acc[4] * sc, acc[5] * sc), dev::pack_bf16x2(acc[6] * sc, acc[7] * sc));
    } else {
      float* dst = p.part_o + (int64_t)(it.part + n) * D + d0;
      *reinterpret_cast<float4*>(dst) = make_float4(acc[0] * sc, acc[1] * sc, acc[2] * sc, acc[3] * sc);
      *reinterpret_cast<float4*>(dst + 4) = make_float4(acc[4] * sc, acc[5] * sc, acc[6] * sc, acc[7] * sc);
      if (d0 == 0) p.part_lse[it.part + n] = lsum > 0.0f ? M + log2f(lsum) : -INFINITY;
    }
  }

  // ---- split tiles: the last CTA of the group to finish merges ----------
  // (threadfence-reduction pattern: publish the partials, count arrivals;
  // nothing waits, so no CTA can block on another.)
  if (it.part >= 0) {
    __shared__ int is_last;
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
      const MergeItem& m = p.merges[it.merge];
      const int prev = atomicAdd(p.merge_counters + it.merge, 1);
      is_last = prev == m.nsplits - 1;
    }
    __syncthreads();
    if (is_last) {
      __threadfence();
      const MergeItem m = p.merges[it.merge];
      merge_splits<D>(p, m, warp, lane);
      if (threadIdx.x == 0) atomicExch(p.merge_counters + it.merge, 0);  // ready for the next call
    }
  }
}

// Launch one instance (used by the per-head_dim translation units).
template <int DT, int D, int NT>
int launch_rowtile_instance(const AttnParams& p, int64_t item_offset, int64_t num_items,
                            cudaStream_t stream) {
  const size_t smem = rowtile_smem_bytes(DT, D);
  auto kern = rowtile_attention_kernel<DT, D, NT>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return KVQ_E_CUDA;
  kern<<<(unsigned)num_items, kRowtileThreads, smem, stream>>>(p, item_offset);
  return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_E_CUDA;
}

template <int D>
int launch_rowtile_d(const AttnParams& p, int dtype, int ntiles, int64_t item_offset,
                     int64_t num_items, cudaStream_t stream) {
#define KVQ_ROWTILE_CASE(DT)                                                          \
  case DT:                                                                            \
    return ntiles == 1 ? launch_rowtile_instance<DT, D, 1>(p, item_offset, num_items, stream) \
                       : launch_rowtile_instance<DT, D, 2>(p, item_offset, num_items, stream);
  switch (dtype) {
    KVQ_ROWTILE_CASE(KVQ_FP8_E4M3)
    KVQ_ROWTILE_CASE(KVQ_FP8_E5M2)
    KVQ_ROWTILE_CASE(KVQ_INT8_PER_TOKEN_HEAD)
    KVQ_ROWTILE_CASE(KVQ_FP8_PER_TOKEN_HEAD)
    default:
      return KVQ_E_UNSUPPORTED;
  }
#undef KVQ_ROWTILE_CASE
}

}  // namespace kvq
