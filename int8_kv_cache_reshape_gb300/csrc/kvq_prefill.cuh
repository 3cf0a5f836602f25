// kvq_prefill.cuh -- prefill attention over the quantised paged cache on the
// 5th-generation tensor cores (tcgen05, accumulators in tensor memory).
//
// What it computes is the attention of kvq_decode.cuh (same masks, soft cap,
// scales) for tiles of 128 packed (query token, head) rows of one kv head:
// vllm PR 39445 page, Breakdown items 2-3 (tile GEMMs for Q K^T and P V with
// the fp8 cache dequantised into a 16-bit tile first, deq_tile_amx /
// prepare_b_tile) and Risks (scale folding); vllm PR 38378 page, Breakdown
// item 3 (_prepare_kv_tile); vllm PR 50194 page, Key source snippet (the
// large fp8 prefill with block_size 2176).
//
// GB300 design: one CTA of 12 warps per 128-row tile, warp-specialised and
// pipelined through mbarriers.
//   * Converter warps (1-3, 8-11): stream the key and value codes of the
//     paged cache (16-byte loads, a whole 32-byte sector per key row and
//     load pair), convert them exactly to f16 (every e4m3 / e5m2 / int8
//     value is an f16 value) and store K (keys x D) and V^T (D x keys) in the
//     128-byte-swizzled K-major layout the tensor core reads, into a 2-stage
//     ring; per-token-head scales and key-valid flags go beside them.
//   * Warp 0, one thread: issues S(j+1) = Q K(j+1)^T into the free one of
//     two tensor-memory S buffers while the softmax works on S(j), then
//     O += P(j) V(j) once P(j) is in shared memory; commits free the ring.
//   * Softmax warps (4-7): thread t owns row t (tensor-memory lane t).  It
//     reads its row of S twice (maximum, then weights), applies scales,
//     soft cap and masks, keeps a lazy reference maximum (moved only when a
//     score exceeds it by 2^8; weights are lifted by 2^6, so P <= 2^14),
//     writes its row of P in f16 and, when the reference moved, rescales its
//     row of O in tensor memory.  At the end it reads O and writes bf16.
//   * Q enters as f16 exactly: each row is scaled by a power of two that puts
//     its largest |q| in [2^14, 2^15) (a bf16 significand fits in f16's);
//     the scale, sm_scale, log2(e) and k_scale (per tensor) or the key's
//     scale (per token-head) multiply the fp32 scores; v_scale the output.
//   * Per-token-head value scales are folded into P relative to a running
//     power-of-two reference 2^ev (the largest scale exponent seen so far),
//     so P * sv * 2^-ev < 2^14 stays in f16 range; O is rescaled by a power
//     of two when ev grows and multiplied by 2^ev at the end.
//   * Every mbarrier wait is bounded: on a timeout the kernel sets the
//     schedule's error word, the other roles stop at their next wait, the
//     MMA thread drains its tensor-core work and the tensor memory is freed.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <type_traits>

#include "kvq_device.cuh"
#include "kvq_internal.h"
#include "kvq_tcgen05.cuh"

namespace kvq {

template <int DT, int D>
struct PrefillGeom {
  static constexpr int kM = kPrefillRows;      // packed rows per tile
  static constexpr int kN = prefill_keys(D);   // keys per KV tile
  static constexpr int kThreads = kPrefillThreads;
  static constexpr int kConv = kPrefillConvThreads;
  static constexpr int kStages = kPrefillStages;
  static constexpr bool kPth = is_per_token_head(DT);
  static constexpr int kRow = row_bytes(DT, D);
  static constexpr int kOffQ = 0;                                   // kM x D f16
  static constexpr int kOffK = kOffQ + kM * D * 2;                  // stages x kN x D f16
  static constexpr int kOffV = kOffK + kStages * kN * D * 2;        // stages x D x kN f16
  static constexpr int kOffP = kOffV + kStages * D * kN * 2;        // kM x kN f16
  static constexpr int kOffSk = kOffP + kM * kN * 2;                // stages x kN f32
  static constexpr int kOffSv = kOffSk + kStages * kN * 4;          // stages x kN f32
  static constexpr int kOffValid = kOffSv + kStages * kN * 4;       // stages x kN bytes
  static constexpr int kOffQScale = kOffValid + kStages * kN;       // kM f32: 2^-sh of each Q row
  static constexpr int kOffBar = kOffQScale + kM * 4;               // mbarriers, tmem slot, flags
  static constexpr int kBytes = kOffBar + 128;
  static constexpr int kColO = 0;   // O: D fp32 columns
  static constexpr int kColS = D;   // S buffers: kN fp32 columns each
  static constexpr int kTmemCols = prefill_tmem_cols(D);
  static_assert(D + 2 * kN <= kTmemCols, "tensor memory: O + 2 S buffers");
  static_assert(kOffK % 1024 == 0 && kOffV % 1024 == 0 && kOffP % 1024 == 0, "1024-byte tiles");
  static_assert((kN * D * 2) % 1024 == 0, "stage tiles stay 1024-byte aligned");
  static_assert(kOffBar % 8 == 0, "mbarrier alignment");
  static_assert((size_t)kBytes + 1024 == prefill_smem_bytes(D), "smem must follow the geometry");
  // barrier slots (8 bytes each)
  static constexpr int kBarKFull = 0, kBarVFull = 2, kBarKvEmpty = 4, kBarSFull = 6, kBarPFull = 8,
                       kBarODone = 9, kBarDrain = 10, kNumBars = 11;
  static constexpr int kOffTmemSlot = kOffBar + 8 * kNumBars;   // u32
  static constexpr int kOffAbort = kOffTmemSlot + 4;            // u32
  static constexpr int kOffBadTile = kOffAbort + 4;             // stages x i32
  static_assert(kOffBadTile + 4 * kStages <= kBytes, "flag space");
};

__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" :: "r"(addr), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" :: "r"(bar) : "memory");
}

// Bounded wait that also gives up when another role has aborted.
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, volatile uint32_t* abort) {
  if (tc::mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (tc::mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (clock64() - t0 > 2000000000LL) {  // about a second
      *abort = 1u;
      return false;
    }
  }
}

// 8 codes (two words) -> 8 f16 (four f16x2 words), exact.
template <int DT>
__device__ __forceinline__ void codes8_to_f16(uint32_t w0, uint32_t w1, uint32_t (&h)[4]) {
  dev::word_to_f16x2x2<DT>(w0, h[0], h[1]);
  dev::word_to_f16x2x2<DT>(w1, h[2], h[3]);
}

template <int DT, int D>
__global__ void __launch_bounds__(kPrefillThreads, 1) prefill_attention_kernel(const AttnParams p) {
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
  const int kv_first = (t.kv_lo / kN) * kN;
  const int T = t.kv_hi > kv_first ? (t.kv_hi - kv_first + kN - 1) / kN : 0;  // KV tiles

  const uint32_t bars = base + Geo::kOffBar;
  auto bar = [&](int i) { return bars + 8u * (uint32_t)i; };
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(sm + Geo::kOffAbort);
  volatile int32_t* bad_tile = reinterpret_cast<volatile int32_t*>(sm + Geo::kOffBadTile);

  if (tid == 0) {
    for (int s = 0; s < Geo::kStages; ++s) {
      tc::mbar_init(bar(Geo::kBarKFull + s), Geo::kConv);
      tc::mbar_init(bar(Geo::kBarVFull + s), Geo::kConv);
      tc::mbar_init(bar(Geo::kBarKvEmpty + s), 1);
      tc::mbar_init(bar(Geo::kBarSFull + s), 1);
      bad_tile[s] = -1;
    }
    tc::mbar_init(bar(Geo::kBarPFull), 128);
    tc::mbar_init(bar(Geo::kBarODone), 1);
    tc::mbar_init(bar(Geo::kBarDrain), 1);
    *abort_flag = 0u;
    tc::mbar_fence_init();
  }
  if (warp == 0) {
    tc::tmem_alloc(base + Geo::kOffTmemSlot, Geo::kTmemCols);
    tc::tmem_relinquish();
  }

  // ---- Q tile -> shared memory, all warps: lanes_per_row lanes hold one
  // row (16 bytes each, coalesced); the row's largest exponent comes from a
  // shuffle reduction over those lanes, and the row is scaled by the power of
  // two that puts its largest |q| in [2^14, 2^15) (exact in f16: a bf16
  // significand fits in f16's).
  {
    constexpr int kLpr = D / 8;            // lanes per row
    constexpr int kRps = 32 / kLpr;        // rows per warp step
    constexpr int kWarps = Geo::kThreads / 32;
    constexpr int kSteps = (kM / kRps + kWarps - 1) / kWarps;
    const int lane = tid & 31;
    const int sub = lane / kLpr, c = lane % kLpr;
    float* qscale = reinterpret_cast<float*>(sm + Geo::kOffQScale);
    uint4 v[kSteps];
#pragma unroll
    for (int i = 0; i < kSteps; ++i) {  // all loads first
      const int m = (warp + i * kWarps) * kRps + sub;
      v[i] = make_uint4(0, 0, 0, 0);
      if (m < t.nrows) {
        const int R = t.row0 + m;
        v[i] = *reinterpret_cast<const uint4*>(
            p.q + ((int64_t)(q0 + R / G) * p.heads_q + t.kv_head * G + R % G) * D + 8 * c);
      }
    }
#pragma unroll
    for (int i = 0; i < kSteps; ++i) {
      const int m = (warp + i * kWarps) * kRps + sub;
      const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
      int emax = 0;
#pragma unroll
      for (int k = 0; k < 4; ++k) emax = max(emax, (int)max((w[k] >> 7) & 0xFFu, (w[k] >> 23) & 0xFFu));
#pragma unroll
      for (int o = kLpr / 2; o > 0; o >>= 1) emax = max(emax, __shfl_xor_sync(0xffffffffu, emax, o));
      // largest |q| < 2^(emax - 126)
      const int sh = emax > 0 ? min(140 - emax, 126) : 0;
      const float up = ldexpf(1.0f, sh);
      if (m < kM) {
        uint4 o;
        o.x = dev::pack_f16x2(dev::bf16_lo(w[0]) * up, dev::bf16_hi(w[0]) * up);
        o.y = dev::pack_f16x2(dev::bf16_lo(w[1]) * up, dev::bf16_hi(w[1]) * up);
        o.z = dev::pack_f16x2(dev::bf16_lo(w[2]) * up, dev::bf16_hi(w[2]) * up);
        o.w = dev::pack_f16x2(dev::bf16_lo(w[3]) * up, dev::bf16_hi(w[3]) * up);
        sts128(base + Geo::kOffQ + tc::sw128_offset(kM, m, 8 * c), o);
        if (c == 0) qscale[m] = ldexpf(1.0f, -sh);
      }
    }
    tc::fence_async_smem();
  }
  const bool is_softmax = warp >= 4 && warp < 8;
  const int m = tid - 128;  // row (softmax warps)
  const bool row_valid = is_softmax && m < t.nrows;
  const int R = t.row0 + (row_valid ? m : 0);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(sm + Geo::kOffTmemSlot);

  if (warp == 0) {
    // ======================= MMA issuer ========================================
    if (tid == 0 && T > 0) {
      constexpr uint32_t idesc_s = tc::idesc_f16(kM, kN);
      constexpr uint32_t idesc_o = tc::idesc_f16(kM, D);
      auto issue_s = [&](int j) {
        const int st = j & 1;
        const uint32_t tmem_s = tmem + Geo::kColS + (uint32_t)(st * kN);
        const uint32_t kbase = base + Geo::kOffK + (uint32_t)(st * kN * D * 2);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t aoff = (kk >> 2) * (kM * 128) + (kk & 3) * 32;
          const uint32_t boff = (kk >> 2) * (kN * 128) + (kk & 3) * 32;
          tc::mma_bf16(tmem_s, tc::desc_sw128(base + Geo::kOffQ + aoff), tc::desc_sw128(kbase + boff),
                       idesc_s, kk > 0 ? 1u : 0u);
        }
        tc::mma_commit(bar(Geo::kBarSFull + st));
      };
      bool ok = wait_or_abort(bar(Geo::kBarKFull + 0), 0u, abort_flag);
      if (ok) {
        tc::fence_after_sync();
        issue_s(0);
      }
      for (int j = 0; ok && j < T; ++j) {
        const int st = j & 1;
        if (j + 1 < T) {
          ok = wait_or_abort(bar(Geo::kBarKFull + ((j + 1) & 1)), (uint32_t)(((j + 1) >> 1) & 1),
                             abort_flag);
          if (!ok) break;
          tc::fence_after_sync();
          issue_s(j + 1);
        }
        ok = wait_or_abort(bar(Geo::kBarPFull), (uint32_t)(j & 1), abort_flag) &&
             wait_or_abort(bar(Geo::kBarVFull + st), (uint32_t)((j >> 1) & 1), abort_flag);
        if (!ok) break;
        tc::fence_after_sync();
        const uint32_t vbase = base + Geo::kOffV + (uint32_t)(st * D * kN * 2);
#pragma unroll
        for (int kk = 0; kk < kN / 16; ++kk) {
          const uint32_t aoff = (kk >> 2) * (kM * 128) + (kk & 3) * 32;
          const uint32_t boff = (kk >> 2) * (D * 128) + (kk & 3) * 32;
          tc::mma_bf16(tmem + Geo::kColO, tc::desc_sw128(base + Geo::kOffP + aoff),
                       tc::desc_sw128(vbase + boff), idesc_o, (j > 0 || kk > 0) ? 1u : 0u);
        }
        tc::mma_commit(bar(Geo::kBarODone));
        tc::mma_commit(bar(Geo::kBarKvEmpty + st));
      }
      if (!ok) {
        // Drain whatever was issued before the tensor memory is freed.
        tc::mma_commit(bar(Geo::kBarDrain));
        (void)tc::mbar_wait(bar(Geo::kBarDrain), 0u, 200000000LL);
      }
    }
    __syncwarp();
  } else if (!is_softmax) {
    // ======================= converters ========================================
    const int ctid = warp < 4 ? tid - 32 : tid - 256 + 96;
    const int32_t* btab = p.block_table + (int64_t)t.req * p.block_table_stride;
    const int64_t row_stride = (int64_t)p.heads_kv * Geo::kRow;
    const uint8_t* kcache = p.key_cache + (int64_t)t.kv_head * Geo::kRow;
    const uint8_t* vcache = p.value_cache + (int64_t)t.kv_head * Geo::kRow;
    float* sk = reinterpret_cast<float*>(sm + Geo::kOffSk);
    float* sv = reinterpret_cast<float*>(sm + Geo::kOffSv);
    uint8_t* kvalid = sm + Geo::kOffValid;
    // Logical key j -> (table entry, offset) without a divide: q0 = hi32(j *
    // floor((2^32 - 1) / B)) is q or q - 1 for every 32-bit j.
    const uint32_t bsz = (uint32_t)p.block_size;
    const uint32_t bdiv = 0xFFFFFFFFu / bsz;
    // Row of logical key j (j >= 0), or nullptr when its block is missing.
    // Keys j .. j + k within one 8-aligned group share a block (block sizes
    // are multiples of 16), so their rows are consecutive slots.
    auto key_row = [&](const uint8_t* cache, int j) -> const uint8_t* {
      uint32_t q = __umulhi((uint32_t)j, bdiv);
      uint32_t r = (uint32_t)j - q * bsz;
      if (r >= bsz) {
        ++q;
        r -= bsz;
      }
      const int blk = btab[q];
      if (blk < 0 || (int64_t)blk >= p.num_blocks) return nullptr;
      return cache + ((int64_t)blk * bsz + r) * row_stride;
    };
    constexpr int kKUnits = kN * (D / 32);        // key x 32-code pieces
    constexpr int kVUnits = (kN / 8) * (D / 16);  // 8 keys x 16 dims
    constexpr int kKSlots = (kKUnits + Geo::kConv - 1) / Geo::kConv;
    constexpr int kVSlots = (kVUnits + Geo::kConv - 1) / Geo::kConv;
    // Codes of the next tile, loaded while the current one is in use.
    uint4 kraw[kKSlots][2];
    uint4 vraw[kVSlots][8];
    float kscale[kKSlots];
    float vscale[kVSlots][8];
    uint32_t kdead = 0;  // bit i: K slot i's key has no row (in range, no block)
    uint32_t kmiss = 0;  // bit i: K slot i's key has no row at all
    auto load_tile = [&](int j) {
      const int kv0 = kv_first + j * kN;
      kdead = kmiss = 0;
#pragma unroll
      for (int i = 0; i < kKSlots; ++i) {
        const int u = ctid + i * Geo::kConv;
        kraw[i][0] = kraw[i][1] = make_uint4(0, 0, 0, 0);
        kscale[i] = 0.0f;
        if (u < kKUnits) {
          const int n = u % kN, pc = u / kN;
          const int jj = kv0 + n;
          const bool in_range = jj >= t.kv_lo && jj < t.kv_hi;
          const uint8_t* row = in_range ? key_row(kcache, jj) : nullptr;
          if (row) {
            kraw[i][0] = *reinterpret_cast<const uint4*>(row + 32 * pc);
            kraw[i][1] = *reinterpret_cast<const uint4*>(row + 32 * pc + 16);
            if constexpr (Geo::kPth)
              if (pc == 0) kscale[i] = *reinterpret_cast<const float*>(row + D);
          } else {
            kmiss |= 1u << i;
            if (in_range) kdead |= 1u << i;
          }
        }
      }
#pragma unroll
      for (int i = 0; i < kVSlots; ++i) {
        const int u = ctid + i * Geo::kConv;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          vraw[i][k] = make_uint4(0, 0, 0, 0);
          vscale[i][k] = 0.0f;
        }
        if (u < kVUnits) {
          const int kg = u % (kN / 8), d16 = u / (kN / 8);
          const int j8 = kv0 + 8 * kg;  // 8-aligned: one block for all 8 keys
          const uint8_t* row0 =
              (j8 + 8 > t.kv_lo && j8 < t.kv_hi) ? key_row(vcache, j8) : nullptr;
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            if (row0 && j8 + k >= t.kv_lo && j8 + k < t.kv_hi) {
              const uint8_t* row = row0 + (int64_t)k * row_stride;
              vraw[i][k] = *reinterpret_cast<const uint4*>(row + 16 * d16);
              if constexpr (Geo::kPth)
                if (d16 == 0) vscale[i][k] = *reinterpret_cast<const float*>(row + D);
            }
          }
        }
      }
    };
    if (T > 0) load_tile(0);
    for (int j = 0; j < T; ++j) {
      const int st = j & 1;
      if (j >= 2 && !__all_sync(0xffffffffu, wait_or_abort(bar(Geo::kBarKvEmpty + st),
                                                            (uint32_t)(((j >> 1) - 1) & 1), abort_flag)))
        break;
      // ---- K: thread -> (key n, 32 codes); 8 consecutive threads take 8
      // consecutive keys, so the swizzled 16-byte stores hit 8 bank groups.
      const uint32_t kbase = base + Geo::kOffK + (uint32_t)(st * kN * D * 2);
#pragma unroll
      for (int i = 0; i < kKSlots; ++i) {
        const int u = ctid + i * Geo::kConv;
        if (u < kKUnits) {
          const int n = u % kN, pc = u / kN;
          uint32_t h[4];
          codes8_to_f16<DT>(kraw[i][0].x, kraw[i][0].y, h);
          sts128(kbase + tc::sw128_offset(kN, n, 32 * pc), make_uint4(h[0], h[1], h[2], h[3]));
          codes8_to_f16<DT>(kraw[i][0].z, kraw[i][0].w, h);
          sts128(kbase + tc::sw128_offset(kN, n, 32 * pc + 8), make_uint4(h[0], h[1], h[2], h[3]));
          codes8_to_f16<DT>(kraw[i][1].x, kraw[i][1].y, h);
          sts128(kbase + tc::sw128_offset(kN, n, 32 * pc + 16), make_uint4(h[0], h[1], h[2], h[3]));
          codes8_to_f16<DT>(kraw[i][1].z, kraw[i][1].w, h);
          sts128(kbase + tc::sw128_offset(kN, n, 32 * pc + 24), make_uint4(h[0], h[1], h[2], h[3]));
          if (pc == 0) {
            kvalid[st * kN + n] = (kmiss >> i) & 1u ? 0 : 1;
            if constexpr (Geo::kPth) sk[st * kN + n] = kscale[i];
            if ((kdead >> i) & 1u) bad_tile[st] = j;
          }
        }
      }
      tc::fence_async_smem();
      mbar_arrive(bar(Geo::kBarKFull + st));
      // ---- V^T: thread -> (8 keys, 16 dims); threads with consecutive key
      // groups share dims, so the stores of one row hit distinct bank groups.
      const uint32_t vbase = base + Geo::kOffV + (uint32_t)(st * D * kN * 2);
#pragma unroll
      for (int i = 0; i < kVSlots; ++i) {
        const int u = ctid + i * Geo::kConv;
        if (u < kVUnits) {
          const int kg = u % (kN / 8), d16 = u / (kN / 8);
          uint32_t x[8][8];  // key k: 16 dims as 8 f16x2 words
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            uint32_t h[4];
            codes8_to_f16<DT>(vraw[i][k].x, vraw[i][k].y, h);
            x[k][0] = h[0]; x[k][1] = h[1]; x[k][2] = h[2]; x[k][3] = h[3];
            codes8_to_f16<DT>(vraw[i][k].z, vraw[i][k].w, h);
            x[k][4] = h[0]; x[k][5] = h[1]; x[k][6] = h[2]; x[k][7] = h[3];
            if constexpr (Geo::kPth)
              if (d16 == 0) sv[st * kN + 8 * kg + k] = vscale[i][k];
          }
          // Row d of V^T holds keys 8kg .. 8kg+7: the d-th half of each word.
#pragma unroll
          for (int w = 0; w < 8; ++w)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              const uint32_t sel = hh ? 0x7632u : 0x5410u;
              const uint4 out =
                  make_uint4(dev::prmt(x[0][w], x[1][w], sel), dev::prmt(x[2][w], x[3][w], sel),
                             dev::prmt(x[4][w], x[5][w], sel), dev::prmt(x[6][w], x[7][w], sel));
              sts128(vbase + tc::sw128_offset(D, 16 * d16 + 2 * w + hh, 8 * kg), out);
            }
        }
      }
      tc::fence_async_smem();
      mbar_arrive(bar(Geo::kBarVFull + st));
      if (j + 1 < T) load_tile(j + 1);
    }
    __syncwarp();
  } else {
    // ======================= softmax ===========================================
    const uint32_t lane_base = (uint32_t)((warp - 4) * 32) << 16;
    const float* sk = reinterpret_cast<const float*>(sm + Geo::kOffSk);
    const float* sv = reinterpret_cast<const float*>(sm + Geo::kOffSv);
    const uint8_t* kvalid = sm + Geo::kOffValid;
    const int pos = L - Q + R / G;
    const int W = p.window;
    const int row_hi = row_valid ? (p.causal ? pos + 1 : L) : 0;  // padding rows see nothing
    const int row_lo = W > 0 ? pos - W + 1 : 0;
    const float log2e = 1.4426950408889634f;
    const float cap = p.soft_cap;
    // scores in log2 units (natural units under a soft cap, which converts)
    const float q_unscale = reinterpret_cast<const float*>(sm + Geo::kOffQScale)[m];  // 2^-sh
    const float score_mul =
        p.sm_scale * q_unscale * (cap > 0.0f ? 1.0f : log2e) * (Geo::kPth ? 1.0f : p.k_scale);
    const float cap_l2 = cap * log2e;
    const float inv_cap = cap > 0.0f ? 1.0f / cap : 0.0f;
    float m_ref = -INFINITY, l_sum = 0.0f;
    int ev = -1000;  // exponent of the value-scale reference (per-token-head)
    bool ok = true;
    for (int j = 0; j < T; ++j) {
      const int st = j & 1;
      const int kv0 = kv_first + j * kN;
      // S(j) is in tensor memory; K(j) (and V(j)) side data is in smem.
      ok = wait_or_abort(bar(Geo::kBarSFull + st), (uint32_t)((j >> 1) & 1), abort_flag) &&
           wait_or_abort(bar(Geo::kBarKFull + st), (uint32_t)((j >> 1) & 1), abort_flag) &&
           (!Geo::kPth || wait_or_abort(bar(Geo::kBarVFull + st), (uint32_t)((j >> 1) & 1), abort_flag));
      ok = __all_sync(0xffffffffu, ok);  // warp-uniform: the warp's tensor-memory loads are collective
      if (!ok) break;
      tc::fence_after_sync();
      const uint32_t tmem_s = tmem + Geo::kColS + (uint32_t)(st * kN) + lane_base;
      // Masks are needed when some row of the warp does not see the whole
      // tile, or the tile has a key without a block.
      const bool full =
          __all_sync(0xffffffffu, kv0 >= row_lo && kv0 + kN <= row_hi) && bad_tile[st] != j;
      // Value-scale reference (per-token-head): the largest exponent so far.
      float alpha = 1.0f;  // factor for O (score reference and value reference)
      float v_mul = 1.0f;  // 2^-ev
      if constexpr (Geo::kPth) {
        float smax = 0.0f;
#pragma unroll
        for (int n = 0; n < kN; n += 4) {
          const float4 s4 = *reinterpret_cast<const float4*>(sv + st * kN + n);
          smax = fmaxf(fmaxf(smax, fmaxf(s4.x, s4.y)), fmaxf(s4.z, s4.w));
        }
        if (smax > 0.0f) {
          int e;
          (void)frexpf(smax, &e);  // smax < 2^e
          if (e > ev) {
            if (ev > -1000) alpha = ldexpf(1.0f, ev - e);  // O was accumulated against 2^ev
            ev = e;
          }
        }
        v_mul = ldexpf(1.0f, -ev);
      }
      // Weights against the current reference: P = 2^(z - m_ref + 6) <= 2^14
      // while no score exceeds m_ref + 8 (the 2^6 lifts small weights clear
      // of the f16 subnormal range; l carries the same factor).  Specialised
      // on a tile every row sees whole (no masks) and on the soft cap.
      uint32_t pw[kN / 2];
      float lsum_tile = 0.0f, mx = -INFINITY;
      auto weights = [&](auto full_c, auto cap_c) {
        constexpr bool kFull = decltype(full_c)::value, kCap = decltype(cap_c)::value;
        const float ref = m_ref == -INFINITY ? 0.0f : m_ref - 6.0f;
        float mr = -INFINITY;  // max of r (r * score_mul is the score without a cap)
        lsum_tile = 0.0f;
        constexpr int kBatch = kN >= 128 ? 32 : 64;  // columns per tensor-memory wait (registers)
#pragma unroll
        for (int c0 = 0; c0 < kN; c0 += kBatch) {
          uint32_t v[kBatch];
#pragma unroll
          for (int c = 0; c < kBatch; c += 32)
            tc::tmem_ld32(tmem_s + c0 + c, *reinterpret_cast<uint32_t(*)[32]>(v + c));
          tc::tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < kBatch; e += 2) {
            const int n = c0 + e;
            float r0 = __uint_as_float(v[e]), r1 = __uint_as_float(v[e + 1]);
            if constexpr (Geo::kPth) {
              const float2 k2 = *reinterpret_cast<const float2*>(sk + st * kN + n);
              r0 *= k2.x;
              r1 *= k2.y;
            }
            bool vis0 = true, vis1 = true;
            if constexpr (!kFull) {
              const int jj = kv0 + n;
              vis0 = kvalid[st * kN + n] && jj >= row_lo && jj < row_hi;
              vis1 = kvalid[st * kN + n + 1] && jj + 1 >= row_lo && jj + 1 < row_hi;
              if constexpr (!kCap) {
                r0 = vis0 ? r0 : -INFINITY;
                r1 = vis1 ? r1 : -INFINITY;
              }
            }
            float p0, p1;
            if constexpr (kCap) {
              // the cap first, then the mask (a capped -inf would be finite)
              float z0 = cap_l2 * tanhf(r0 * score_mul * inv_cap);
              float z1 = cap_l2 * tanhf(r1 * score_mul * inv_cap);
              z0 = vis0 ? z0 : -INFINITY;
              z1 = vis1 ? z1 : -INFINITY;
              mr = fmaxf(mr, fmaxf(z0, z1));
              p0 = dev::fast_exp2(z0 - ref);
              p1 = dev::fast_exp2(z1 - ref);
            } else {
              mr = fmaxf(mr, fmaxf(r0, r1));
              p0 = dev::fast_exp2(fmaf(r0, score_mul, -ref));
              p1 = dev::fast_exp2(fmaf(r1, score_mul, -ref));
            }
            lsum_tile += p0 + p1;
            if constexpr (Geo::kPth) {
              const float2 v2 = *reinterpret_cast<const float2*>(sv + st * kN + n);
              p0 *= v2.x * v_mul;
              p1 *= v2.y * v_mul;
            }
            pw[n / 2] = dev::pack_f16x2(p0, p1);
          }
        }
        mx = kCap ? mr : mr * score_mul;  // score_mul > 0
      };
      auto run_weights = [&]() {
        if (cap > 0.0f) {
          if (full) weights(std::true_type{}, std::true_type{});
          else weights(std::false_type{}, std::true_type{});
        } else {
          if (full) weights(std::true_type{}, std::false_type{});
          else weights(std::false_type{}, std::false_type{});
        }
      };
      run_weights();
      // A score above the reference by more than 2^8 moves it (lazily); the
      // warp then recomputes its weights against the new reference.
      if (__any_sync(0xffffffffu, mx > m_ref + 8.0f)) {
        if (mx > m_ref + 8.0f) {
          const float a = m_ref == -INFINITY ? 0.0f : exp2f(m_ref - mx);
          alpha *= a;
          l_sum *= a;
          m_ref = mx;
        }
        run_weights();
      }
      l_sum += lsum_tile;
      // PV(j-1) must be complete: it reads the P buffer and accumulates O.
      if (j > 0) {
        ok = __all_sync(0xffffffffu, wait_or_abort(bar(Geo::kBarODone), (uint32_t)((j - 1) & 1), abort_flag));
        if (!ok) break;
        tc::fence_after_sync();
        if (__any_sync(0xffffffffu, alpha != 1.0f)) {
#pragma unroll 1
          for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t v[32];
            tc::tmem_ld32(tmem + Geo::kColO + lane_base + c0, v);
            tc::tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
            tc::tmem_st32(tmem + Geo::kColO + lane_base + c0, v);
          }
          tc::tmem_wait_st();
        }
      }
#pragma unroll
      for (int c0 = 0; c0 < kN; c0 += 8)
        sts128(base + Geo::kOffP + tc::sw128_offset(kM, m, c0),
               make_uint4(pw[c0 / 2], pw[c0 / 2 + 1], pw[c0 / 2 + 2], pw[c0 / 2 + 3]));
      tc::fence_async_smem();
      tc::fence_before_sync();
      mbar_arrive(bar(Geo::kBarPFull));
    }
    // ---- epilogue: O / l -> bf16 -------------------------------------------
    if (ok && T > 0)
      ok = __all_sync(0xffffffffu, wait_or_abort(bar(Geo::kBarODone), (uint32_t)((T - 1) & 1), abort_flag));
    // ok is warp-uniform here: the whole warp reads O (tcgen05.ld is a
    // warp-collective instruction), only valid rows are stored.
    if (ok) {
      uint16_t* dst =
          row_valid ? p.out + ((int64_t)(q0 + R / G) * p.heads_q + t.kv_head * G + R % G) * D : nullptr;
      if (T > 0) {
        tc::fence_after_sync();
        const float sc = (l_sum > 0.0f ? 1.0f / l_sum : 0.0f) *
                         (Geo::kPth ? (ev > -1000 ? ldexpf(1.0f, ev) : 0.0f) : p.v_scale);
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t v[32];
          tc::tmem_ld32(tmem + Geo::kColO + lane_base + c0, v);
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
          __syncwarp();
        }
      } else if (row_valid) {
        // No key tile at all (an empty key range): the output row is zero.
#pragma unroll 1
        for (int c = 0; c < D; c += 8) *reinterpret_cast<uint4*>(dst + c) = make_uint4(0, 0, 0, 0);
      }
    }
    // Order this warp's tensor-memory accesses before the teardown barrier.
    tc::fence_before_sync();
    __syncwarp();
  }

  __syncthreads();
  if (tid == 0 && *abort_flag) atomicExch(p.error_flag, 1);
  if (warp == 0) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, Geo::kTmemCols);
  }
}

template <int DT, int D>
int launch_prefill_instance(const AttnParams& p, int64_t num_tiles, cudaStream_t stream) {
  const size_t smem = prefill_smem_bytes(D);
  auto kern = prefill_attention_kernel<DT, D>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return KVQ_E_CUDA;
  kern<<<(unsigned)num_tiles, kPrefillThreads, smem, stream>>>(p);
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
