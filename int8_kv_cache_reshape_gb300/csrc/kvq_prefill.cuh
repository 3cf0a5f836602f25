// kvq_prefill.cuh -- prefill attention over the quantised paged cache on the
// 5th-generation tensor cores (tcgen05, accumulators in tensor memory).
//
// What it computes is the attention of kvq_decode.cuh (same masks, soft cap,
// scales) for tiles of 128 packed (query token, head) rows of one kv head:
// vllm PR 39445 page, Breakdown items 2-3 (tile GEMMs for Q K^T and P V with
// the fp8 cache dequantised into a bf16 tile first, deq_tile_amx /
// prepare_b_tile) and Risks (scale folding); vllm PR 38378 page, Breakdown
// item 3 (_prepare_kv_tile); vllm PR 50194 page, Key source snippet (the
// large fp8 prefill with block_size 2176).
//
// GB300 design:
//   * One CTA of 4 warps per 128-row tile; thread t owns row t (tensor-memory
//     lane t) for the softmax and the epilogue.
//   * Per 64-key tile: the threads load the key and value codes of the paged
//     cache, convert them exactly (every e4m3 / e5m2 / int8 value is both a
//     bf16 and an f16 value) and store K (64 x D, bf16: Q is bf16) and V^T
//     (D x 64, f16) in shared memory in the 128-byte-swizzled K-major layout
//     the tensor core reads; one thread issues S = Q K^T (M 128, N 64, K D)
//     into tensor memory; each thread reads its row of S, applies scales /
//     soft cap / masks and the online softmax (lazy: the reference maximum
//     moves only when a score exceeds it by 2^8; P is lifted by 2^6, so
//     P <= 2^14), writes its row of P in f16 (11 significant bits) to
//     shared memory; one thread
//     issues O += P V (M 128, N D, K 64) into tensor memory.  O is read back
//     once at the end.
//   * Per-token-head value scales are folded into P relative to a running
//     power-of-two reference 2^ev (the largest scale exponent seen so far),
//     so P * sv * 2^-ev < 2^14 stays in f16 range; O is rescaled by a power
//     of two when ev grows and multiplied by 2^ev at the end.
//   * Scales stay in fp32: sm_scale, log2(e), k_scale (per tensor) or the
//     key's scale (per token-head) multiply the fp32 scores; v_scale the
//     output.
//   * Every mbarrier wait is bounded: on a timeout the kernel sets the
//     schedule's error word, frees its tensor memory and returns.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "kvq_device.cuh"
#include "kvq_internal.h"
#include "kvq_tcgen05.cuh"

namespace kvq {

template <int DT, int D>
struct PrefillGeom {
  static constexpr int kM = kPrefillRows;   // packed rows per tile
  static constexpr int kN = kPrefillKeys;   // keys per KV tile
  static constexpr int kThreads = 128;
  static constexpr bool kPth = is_per_token_head(DT);
  static constexpr int kRow = row_bytes(DT, D);
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kM * D * 2;
  static constexpr int kOffV = kOffK + kN * D * 2;
  static constexpr int kOffP = kOffV + D * kN * 2;
  static constexpr int kOffSk = kOffP + kM * kN * 2;  // kN fp32 key scales
  static constexpr int kOffSv = kOffSk + kN * 4;      // kN fp32 value scales
  static constexpr int kOffValid = kOffSv + kN * 4;   // kN bytes: key has a block
  static constexpr int kOffBar = kOffValid + kN;      // 2 mbarriers + tmem address
  static constexpr int kBytes = kOffBar + 32;
  static constexpr int kColO = 0;                     // O: D fp32 columns
  static constexpr int kColS = D;                     // S: kN fp32 columns
  static constexpr int kTmemCols = prefill_tmem_cols(D);
  static_assert(kOffK % 1024 == 0 && kOffV % 1024 == 0 && kOffP % 1024 == 0, "1024-byte tiles");
  static_assert((size_t)kBytes + 1024 == prefill_smem_bytes(D), "smem must follow the geometry");
};

// 16 codes -> 16 bf16 (two 16-byte chunks), exact.
template <int DT>
__device__ __forceinline__ void codes16_to_bf16(uint4 c, uint4& lo, uint4& hi) {
  const uint32_t w[4] = {c.x, c.y, c.z, c.w};
  uint32_t o[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if constexpr (DT == KVQ_INT8_PER_TOKEN_HEAD) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const float f0 = (float)(int)(int8_t)((w[i] >> (16 * h)) & 0xFF);
        const float f1 = (float)(int)(int8_t)((w[i] >> (16 * h + 8)) & 0xFF);
        o[2 * i + h] = dev::prmt(__float_as_uint(f0), __float_as_uint(f1), 0x7632u);
      }
    } else {
      uint32_t p0, p1;  // f16x2 pairs (bytes 0-1, 2-3)
      dev::word_to_f16x2x2<DT>(w[i], p0, p1);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const __half2 hv = *reinterpret_cast<const __half2*>(h ? &p1 : &p0);
        const float2 f = __half22float2(hv);
        o[2 * i + h] = dev::prmt(__float_as_uint(f.x), __float_as_uint(f.y), 0x7632u);
      }
    }
  }
  lo = make_uint4(o[0], o[1], o[2], o[3]);
  hi = make_uint4(o[4], o[5], o[6], o[7]);
}

__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" :: "r"(addr), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w) : "memory");
}

template <int DT, int D>
__global__ void __launch_bounds__(128, 1) prefill_attention_kernel(const AttnParams p) {
  using Geo = PrefillGeom<DT, D>;
  constexpr int kM = Geo::kM, kN = Geo::kN;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = dev::smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* sm = smem_raw + (base - raw);
  const int tid = threadIdx.x;
  const int warp = tid >> 5;

  const PrefillTile t = p.prefill_tiles[blockIdx.x];
  const int G = p.group;
  const int q0 = p.query_start_loc[t.req];
  const int Q = p.query_start_loc[t.req + 1] - q0;
  const int L = p.seq_lens[t.req];
  const int32_t* btab = p.block_table + (int64_t)t.req * p.block_table_stride;
  const int64_t row_stride = (int64_t)p.heads_kv * Geo::kRow;
  const uint8_t* kcache = p.key_cache + (int64_t)t.kv_head * Geo::kRow;
  const uint8_t* vcache = p.value_cache + (int64_t)t.kv_head * Geo::kRow;

  const uint32_t bar_s = base + Geo::kOffBar;
  const uint32_t bar_o = bar_s + 8;
  const uint32_t tmem_slot = bar_s + 16;
  float* sk = reinterpret_cast<float*>(sm + Geo::kOffSk);
  float* sv = reinterpret_cast<float*>(sm + Geo::kOffSv);
  uint8_t* kvalid = sm + Geo::kOffValid;

  if (tid == 0) {
    tc::mbar_init(bar_s, 1);
    tc::mbar_init(bar_o, 1);
    tc::mbar_fence_init();
  }
  if (warp == 0) {
    tc::tmem_alloc(tmem_slot, Geo::kTmemCols);
    tc::tmem_relinquish();
  }

  // ---- Q tile -> shared memory (bf16, 128-byte swizzle, K-major) ----------
  for (int idx = tid; idx < kM * (D / 8); idx += Geo::kThreads) {
    const int m = idx / (D / 8);
    const int cc = idx % (D / 8);
    uint4 v = make_uint4(0, 0, 0, 0);
    if (m < t.nrows) {
      const int R = t.row0 + m;
      const int tok = q0 + R / G;
      const int head = t.kv_head * G + R % G;
      v = *reinterpret_cast<const uint4*>(p.q + ((int64_t)tok * p.heads_q + head) * D + cc * 8);
    }
    sts128(base + Geo::kOffQ + tc::sw128_offset(kM, m, cc * 8), v);
  }
  tc::fence_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(sm + Geo::kOffBar + 16);
  const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
  const uint32_t tmem_o = tmem + Geo::kColO;
  const uint32_t tmem_s = tmem + Geo::kColS;

  // ---- this thread's row -------------------------------------------------
  const int m = tid;
  const bool row_valid = m < t.nrows;
  const int R = t.row0 + (row_valid ? m : 0);
  const int pos = L - Q + R / G;
  const int W = p.window;
  const int row_hi = row_valid ? (p.causal ? pos + 1 : L) : 0;  // invalid rows see nothing
  const int row_lo = W > 0 ? pos - W + 1 : 0;
  const float log2e = 1.4426950408889634f;
  const float cap = p.soft_cap;
  const float score_mul = p.sm_scale * (cap > 0.0f ? 1.0f : log2e) * (Geo::kPth ? 1.0f : p.k_scale);
  const float cap_l2 = cap * log2e;
  const float inv_cap = cap > 0.0f ? 1.0f / cap : 0.0f;
  float m_ref = -INFINITY, l_sum = 0.0f;
  int ev = -1000;  // exponent of the value-scale reference (per-token-head)

  bool failed = false;
  uint32_t pending_bar = bar_s, pending_parity = 0;  // the MMA group last waited for
  int it = 0;
  for (int kv0 = (t.kv_lo / kN) * kN; kv0 < t.kv_hi; kv0 += kN, ++it) {
    // ---- K and V codes -> bf16 tiles -------------------------------------
    for (int idx = tid; idx < kN * (D / 16); idx += Geo::kThreads) {
      const int n = idx / (D / 16);
      const int s = idx % (D / 16);
      const int j = kv0 + n;
      uint4 codes = make_uint4(0, 0, 0, 0);
      bool live = false;
      const uint8_t* row = nullptr;
      if (j >= t.kv_lo && j < t.kv_hi) {
        const int blk = btab[j / p.block_size];
        if (blk >= 0 && (int64_t)blk < p.num_blocks) {
          live = true;
          row = kcache + ((int64_t)blk * p.block_size + j % p.block_size) * row_stride;
          codes = *reinterpret_cast<const uint4*>(row + 16 * s);
        }
      }
      uint4 lo, hi;
      codes16_to_bf16<DT>(codes, lo, hi);
      sts128(base + Geo::kOffK + tc::sw128_offset(kN, n, 16 * s), lo);
      sts128(base + Geo::kOffK + tc::sw128_offset(kN, n, 16 * s + 8), hi);
      if (s == 0) {
        kvalid[n] = live ? 1 : 0;
        if constexpr (Geo::kPth) sk[n] = live ? *reinterpret_cast<const float*>(row + D) : 0.0f;
      }
    }
    for (int idx = tid; idx < (kN / 8) * (D / 8); idx += Geo::kThreads) {
      const int kg = idx / (D / 8);  // 8 keys
      const int dg = idx % (D / 8);  // 8 dims
      uint4 x[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int j = kv0 + 8 * kg + i;
        uint2 c8 = make_uint2(0, 0);
        float scale = 0.0f;
        if (j >= t.kv_lo && j < t.kv_hi) {
          const int blk = btab[j / p.block_size];
          if (blk >= 0 && (int64_t)blk < p.num_blocks) {
            const uint8_t* row = vcache + ((int64_t)blk * p.block_size + j % p.block_size) * row_stride;
            c8 = *reinterpret_cast<const uint2*>(row + 8 * dg);
            if constexpr (Geo::kPth) scale = *reinterpret_cast<const float*>(row + D);
          }
        }
        uint32_t h0, h1, h2, h3;  // dims 8dg .. 8dg+7 of key 8kg+i as 4 f16x2 words
        dev::word_to_f16x2x2<DT>(c8.x, h0, h1);
        dev::word_to_f16x2x2<DT>(c8.y, h2, h3);
        x[i] = make_uint4(h0, h1, h2, h3);
        if constexpr (Geo::kPth)
          if (dg == 0) sv[8 * kg + i] = scale;
      }
      // Transpose 8 keys x 8 dims: row d of V^T holds keys 8kg .. 8kg+7.
      const uint32_t xs[8][4] = {{x[0].x, x[0].y, x[0].z, x[0].w}, {x[1].x, x[1].y, x[1].z, x[1].w},
                                 {x[2].x, x[2].y, x[2].z, x[2].w}, {x[3].x, x[3].y, x[3].z, x[3].w},
                                 {x[4].x, x[4].y, x[4].z, x[4].w}, {x[5].x, x[5].y, x[5].z, x[5].w},
                                 {x[6].x, x[6].y, x[6].z, x[6].w}, {x[7].x, x[7].y, x[7].z, x[7].w}};
#pragma unroll
      for (int w = 0; w < 4; ++w)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint32_t sel = h ? 0x7632u : 0x5410u;
          const uint4 out = make_uint4(dev::prmt(xs[0][w], xs[1][w], sel), dev::prmt(xs[2][w], xs[3][w], sel),
                                       dev::prmt(xs[4][w], xs[5][w], sel), dev::prmt(xs[6][w], xs[7][w], sel));
          sts128(base + Geo::kOffV + tc::sw128_offset(D, 8 * dg + 2 * w + h, 8 * kg), out);
        }
    }
    tc::fence_async_smem();
    __syncthreads();

    // ---- S = Q K^T ---------------------------------------------------------
    if (tid == 0) {
      tc::fence_after_sync();
      constexpr uint32_t idesc = tc::idesc_bf16(kM, kN);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t aoff = (kk >> 2) * (kM * 128) + (kk & 3) * 32;
        const uint32_t boff = (kk >> 2) * (kN * 128) + (kk & 3) * 32;
        tc::mma_bf16(tmem_s, tc::desc_sw128(base + Geo::kOffQ + aoff),
                     tc::desc_sw128(base + Geo::kOffK + boff), idesc, kk > 0 ? 1u : 0u);
      }
      tc::mma_commit(bar_s);
    }
    pending_bar = bar_s;
    pending_parity = (uint32_t)(it & 1);
    const bool ok_s = tc::mbar_wait(bar_s, (uint32_t)(it & 1));
    if (__syncthreads_or(!ok_s)) {
      failed = true;
      break;
    }
    tc::fence_after_sync();

    // ---- softmax on this thread's row --------------------------------------
    float z[kN];
#pragma unroll
    for (int c0 = 0; c0 < kN; c0 += 32) {
      uint32_t v[32];
      tc::tmem_ld32(tmem_s + lane_base + c0, v);
      tc::tmem_wait_ld();
#pragma unroll
      for (int e = 0; e < 32; ++e) z[c0 + e] = __uint_as_float(v[e]);
    }
    float mx = -INFINITY;
#pragma unroll
    for (int n = 0; n < kN; ++n) {
      const int j = kv0 + n;
      float v = z[n] * score_mul * (Geo::kPth ? sk[n] : 1.0f);
      if (cap > 0.0f) v = cap_l2 * tanhf(v * inv_cap);
      const bool vis = kvalid[n] && j >= row_lo && j < row_hi;
      v = vis ? v : -INFINITY;
      z[n] = v;
      mx = fmaxf(mx, v);
    }
    float alpha = 1.0f;
    if (mx > m_ref + 8.0f) {
      alpha = m_ref == -INFINITY ? 0.0f : exp2f(m_ref - mx);
      m_ref = mx;
      l_sum *= alpha;
    }
    // P = 2^(z - ref + 6) <= 2^14: the 2^6 lifts small weights clear of the
    // f16 subnormal range; l carries the same factor.
    const float ref = (m_ref == -INFINITY ? 0.0f : m_ref) - 6.0f;
    float v_mul = 1.0f;  // 2^-ev
    if constexpr (Geo::kPth) {
      // Value-scale reference: the largest exponent of this tile's scales.
      float smax = 0.0f;
#pragma unroll
      for (int n = 0; n < kN; ++n) smax = fmaxf(smax, sv[n]);
      if (smax > 0.0f) {
        int e;
        (void)frexpf(smax, &e);  // smax < 2^e
        if (e > ev) {
          if (ev > -1000) alpha *= ldexpf(1.0f, ev - e);  // O accumulated against 2^ev
          ev = e;
        }
      }
      v_mul = ldexpf(1.0f, -ev);
    }
    float lsum_tile = 0.0f;
#pragma unroll
    for (int c0 = 0; c0 < kN; c0 += 8) {
      uint32_t w[4];
#pragma unroll
      for (int e = 0; e < 8; e += 2) {
        const float p0 = dev::fast_exp2(z[c0 + e] - ref);
        const float p1 = dev::fast_exp2(z[c0 + e + 1] - ref);
        lsum_tile += p0 + p1;
        const float v0 = Geo::kPth ? p0 * (sv[c0 + e] * v_mul) : p0;
        const float v1 = Geo::kPth ? p1 * (sv[c0 + e + 1] * v_mul) : p1;
        w[e / 2] = dev::pack_f16x2(v0, v1);
      }
      sts128(base + Geo::kOffP + tc::sw128_offset(kM, m, c0), make_uint4(w[0], w[1], w[2], w[3]));
    }
    l_sum += lsum_tile;
    // Rescale O in tensor memory when this warp's reference moved.
    if (it > 0 && __any_sync(0xffffffffu, alpha != 1.0f)) {
#pragma unroll 1
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t v[32];
        tc::tmem_ld32(tmem_o + lane_base + c0, v);
        tc::tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
        tc::tmem_st32(tmem_o + lane_base + c0, v);
      }
      tc::tmem_wait_st();
    }
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncthreads();

    // ---- O += P V ------------------------------------------------------------
    if (tid == 0) {
      tc::fence_after_sync();
      constexpr uint32_t idesc = tc::idesc_f16(kM, D);
#pragma unroll
      for (int kk = 0; kk < kN / 16; ++kk) {
        const uint32_t aoff = (kk >> 2) * (kM * 128) + (kk & 3) * 32;
        const uint32_t boff = (kk >> 2) * (D * 128) + (kk & 3) * 32;
        tc::mma_bf16(tmem_o, tc::desc_sw128(base + Geo::kOffP + aoff),
                     tc::desc_sw128(base + Geo::kOffV + boff), idesc,
                     (it > 0 || kk > 0) ? 1u : 0u);
      }
      tc::mma_commit(bar_o);
    }
    pending_bar = bar_o;
    pending_parity = (uint32_t)(it & 1);
    const bool ok_o = tc::mbar_wait(bar_o, (uint32_t)(it & 1));
    if (__syncthreads_or(!ok_o)) {
      failed = true;
      break;
    }
    tc::fence_after_sync();
  }

  // ---- epilogue: O / l -> bf16 ---------------------------------------------
  if (!failed && it > 0) {
    const float sc = (l_sum > 0.0f ? 1.0f / l_sum : 0.0f) *
                     (Geo::kPth ? (ev > -1000 ? ldexpf(1.0f, ev) : 0.0f) : p.v_scale);
    uint16_t* dst = nullptr;
    if (row_valid) {
      const int tok = q0 + R / G;
      const int head = t.kv_head * G + R % G;
      dst = p.out + ((int64_t)tok * p.heads_q + head) * D;
    }
#pragma unroll 1
    for (int c0 = 0; c0 < D; c0 += 32) {
      uint32_t v[32];
      tc::tmem_ld32(tmem_o + lane_base + c0, v);
      tc::tmem_wait_ld();
      if (row_valid) {
#pragma unroll
        for (int e = 0; e < 32; e += 8) {
          uint4 o;
          o.x = dev::pack_bf16x2(__uint_as_float(v[e]) * sc, __uint_as_float(v[e + 1]) * sc);
          o.y = dev::pack_bf16x2(__uint_as_float(v[e + 2]) * sc, __uint_as_float(v[e + 3]) * sc);
          o.z = dev::pack_bf16x2(__uint_as_float(v[e + 4]) * sc, __uint_as_float(v[e + 5]) * sc);
          o.w = dev::pack_bf16x2(__uint_as_float(v[e + 6]) * sc, __uint_as_float(v[e + 7]) * sc);
          *reinterpret_cast<uint4*>(dst + c0 + e) = o;
        }
      }
    }
  }
  if (!failed && it == 0 && row_valid) {
    // No key tile at all (an empty key range): the output row is zero.
    uint16_t* dst = p.out + ((int64_t)(q0 + R / G) * p.heads_q + t.kv_head * G + R % G) * D;
#pragma unroll 1
    for (int c = 0; c < D; c += 8) *reinterpret_cast<uint4*>(dst + c) = make_uint4(0, 0, 0, 0);
  }
  if (failed) {
    // An MMA did not complete in time: record it, give the outstanding MMA a
    // last bounded chance to finish, then release the tensor memory.
    if (tid == 0) atomicExch(p.error_flag, 1);
    (void)tc::mbar_wait(pending_bar, pending_parity, 200000000LL);
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, Geo::kTmemCols);
}

template <int DT, int D>
int launch_prefill_instance(const AttnParams& p, int64_t num_tiles, cudaStream_t stream) {
  const size_t smem = prefill_smem_bytes(D);
  auto kern = prefill_attention_kernel<DT, D>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return KVQ_E_CUDA;
  kern<<<(unsigned)num_tiles, 128, smem, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_E_CUDA;
}

template <int D>
int launch_prefill_d(const AttnParams& p, int dtype, int64_t num_tiles, cudaStream_t stream) {
  switch (dtype) {
    case KVQ_FP8_E4M3: return launch_prefill_instance<KVQ_FP8_E4M3, D>(p, num_tiles, stream);
    case KVQ_FP8_E5M2: return launch_prefill_instance<KVQ_FP8_E5M2, D>(p, num_tiles, stream);
    case KVQ_INT8_PER_TOKEN_HEAD:
      return launch_prefill_instance<KVQ_INT8_PER_TOKEN_HEAD, D>(p, num_tiles, stream);
    case KVQ_FP8_PER_TOKEN_HEAD:
      return launch_prefill_instance<KVQ_FP8_PER_TOKEN_HEAD, D>(p, num_tiles, stream);
    default:
      return KVQ_E_UNSUPPORTED;
  }
}

}  // namespace kvq
