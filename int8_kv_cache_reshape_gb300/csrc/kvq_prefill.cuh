// kvq_prefill.cuh -- prefill attention over the quantised paged cache on the
// 5th-generation tensor cores (tcgen05, operands and accumulators in tensor
// memory).
//
// What it computes is the attention of kvq_decode.cuh (same masks, soft cap,
// scales) for tiles of 128 packed (query token, head) rows of one kv head:
// vllm PR 39445 page, Breakdown items 2-3 (tile GEMMs for Q K^T and P V with
// the fp8 cache dequantised into a 16-bit tile first, deq_tile_amx /
// prepare_b_tile) and Risks (scale folding); vllm PR 38378 page, Breakdown
// item 3 (_prepare_kv_tile); vllm PR 50194 page, Key source snippet (the
// large fp8 prefill with block_size 2176).
//
// GB300 design: one CTA of 16 warps (12 at head_dim 256) per 128-row tile,
// warp-specialised and pipelined through mbarriers.
//   * Tensor memory (512 columns): O (D fp32 columns), two S buffers (keys
//     fp32 columns each; P(j) is written as f16 pairs over the first half of
//     S(j)'s buffer), and Q (D/2 columns of f16 pairs).  Both MMAs take A
//     from tensor memory: S = Q K^T and O += P V read only K and V from
//     shared memory.
//   * Copy warp (the last): bulk tensor copies (TMA) of each tile's K codes
//     (with both per-token-head scale tails) and V codes into a two-stage
//     code ring, in two groups with a barrier each; the K group of tile
//     j + 2 goes out once K(j) is converted, the V group once V(j) is.
//   * Converter warps (1-3, and 8 up to the copy warp): a thread takes (key,
//     16 codes) units, converts the codes exactly to f16 (every e4m3 / e5m2
//     / int8 value is an f16 value) and stores them as key-major rows in the
//     128-byte swizzle into a two-stage K ring and V ring.  K is read by the
//     tensor core K-major, V MN-major, so neither needs a transpose.  Step i
//     converts K(i) (its buffer is free once S(i-2) is complete) and then
//     V(i-1) (free once P(i-3) V(i-3) is): K runs a tile ahead of V.
//     Per-key scales, the tile's chunk mask and its largest value scale go
//     to one of four side-data slots for the softmax.
//   * MMA warp (0): one elected lane issues S(j) as soon as K(j) is in and
//     PV(j-2) was issued (P(j-2) shares the buffer; one thread's MMAs run in
//     order), and O += P(j) V(j) as soon as P(j) and V(j) are in; one
//     warp-wide non-blocking barrier test per pass decides for the warp.
//   * Softmax warps (4-7): thread t owns row t (tensor-memory lane t).  One
//     pass over its row of S, 64 scores per tensor-memory round trip: the
//     round's maximum, then the weights, written as f16 straight into
//     tensor memory.  The reference maximum is an integer (log2 units) and
//     lazy: it moves only when a score exceeds it by 2^8 (weights are lifted
//     by 2^6, so P <= 2^14), to the next integer at or above the maximum,
//     and the weights, O and l already accumulated are rescaled by the exact
//     power of two (O only after P(j-1) V(j-1) is complete).  At the end it
//     reads O and writes bf16.
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
//     MMA warp drains its tensor-core work, the copy warp waits for its
//     copies in flight, and the tensor memory is freed.
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
  // bf16 ("auto") rows need no conversion: the bulk copies write K and V
  // straight into the operand tiles, and the MMAs take bf16 operands.
  static constexpr bool kAuto = DT == KVQ_AUTO;
  static constexpr int kM = kPrefillRows;      // packed rows per tile
  static constexpr int kN = prefill_keys(D);   // keys per KV tile
  static constexpr int kThreads = prefill_threads(D);
  static constexpr int kConv = prefill_conv_threads(D);
  static constexpr int kStages = kPrefillStages;
  static constexpr bool kPth = is_per_token_head(DT);
  static constexpr int kTileBytes = kN * D * 2;                     // one K or V tile (f16)
  static constexpr int kOffK = 0;                                   // stages x K tile
  static constexpr int kOffV = kOffK + kStages * kTileBytes;        // stages x V tile
  static constexpr int kOffCodeK = kOffV + kStages * kTileBytes;   // stages x kN x D code bytes
  static constexpr int kOffCodeV = kOffCodeK + kStages * kN * D;    // stages x kN x D code bytes
  static constexpr int kOffTailK = kOffCodeV + kStages * kN * D;    // stages x kN x 16 (scale tails)
  static constexpr int kOffTailV = kOffTailK + kStages * kN * 16;   // stages x kN x 16
  // Side data of tile j, for the softmax, in slot j % kSide: per-key scales,
  // the 16-key chunk mask and, per converter warp, the largest value scale
  // of its keys (bits of a float >= 0).
  static constexpr int kSide = kPrefillSideSlots;
  static constexpr int kOffSk = kOffTailV + kStages * kN * 16;      // kSide x kN f32
  static constexpr int kOffSv = kOffSk + kSide * kN * 4;            // kSide x kN f32
  static constexpr int kOffSMask = kOffSv + kSide * kN * 4;         // kSide x u32
  static constexpr int kOffVMax = kOffSMask + 4 * kSide;            // kSide x 8 u32
  static constexpr int kOffQScale = kOffVMax + 32 * kSide;          // kM f32: 2^-sh of each Q row
  static constexpr int kOffBar = kOffQScale + kM * 4;               // mbarriers, tmem slot, flags
  static constexpr int kBytes = kOffBar + 256;
  // Q (kM x D, swizzled) is staged over the K ring -- or, for bf16 rows,
  // whose first K tiles land in the K ring while Q is staged, over the
  // (unused) code rings.
  static constexpr int kOffQStage = kAuto ? kOffCodeK : kOffK;
  static constexpr int kOffOStage = kOffK;  // O (kM x D bf16) staged over the K ring at the end
  static constexpr int kColO = 0;                 // O: D fp32 columns
  static constexpr int kColS = D;                 // S buffers: kN fp32 columns each
  static constexpr int kColQ = D + 2 * kN;        // Q: D/2 columns of f16 pairs
  static constexpr int kTmemCols = prefill_tmem_cols(D);
  static_assert(kColQ + D / 2 <= kTmemCols, "tensor memory: O + 2 S buffers + Q");
  static_assert(kM * D * 2 <= kStages * kTileBytes, "Q / O staging fits the K ring");
  static_assert(!kAuto || kM * D * 2 <= 2 * kStages * kN * D, "Q staging fits the code rings");
  static_assert(kTileBytes % 1024 == 0 && kOffV % 1024 == 0 && kOffCodeK % 1024 == 0 &&
                    kOffCodeV % 128 == 0 && kOffTailK % 128 == 0 && kOffTailV % 128 == 0,
                "1024-byte operand tiles, 128-byte copy destinations");
  static_assert(kOffBar % 8 == 0, "mbarrier alignment");
  static_assert((kN + 31) / 32 <= 8 && kSide == 4, "side data space");
  static_assert((size_t)kBytes + 1024 == prefill_smem_bytes(D), "smem must follow the geometry");
  // barrier slots (8 bytes each).  K and V travel separately: the K codes
  // of tile j + 2 are copied once K(j) is converted, K(j + 2) is converted
  // once S(j) is complete, V(j + 2) once P(j) V(j) is.  One P barrier per
  // S buffer: P(j+1) may be ready before PV(j) is issued.  A parity wait is
  // unambiguous only while the waiter is at most one phase behind, so the
  // epilogue (which may be several PVs ahead of the last phase it saw)
  // waits on a one-shot barrier for the last PV, and the side data (which
  // the converters may write two tiles ahead) has four slots.
  static constexpr int kBarCodesK = 0, kBarCodesV = 2, kBarCodesKFree = 4, kBarCodesVFree = 6,
                       kBarKFull = 8, kBarVFull = 10, kBarVEmpty = 12, kBarSFull = 14, kBarPFull = 16,
                       kBarSide = 18, kBarODone = 22, kBarOFinal = 23, kBarDrain = 24, kNumBars = 25;
  static constexpr int kOffTmemSlot = kOffBar + 8 * kNumBars;   // u32
  static constexpr int kOffAbort = kOffTmemSlot + 4;            // u32
  static constexpr int kOffChunkValid = kOffAbort + 4;          // stages x u32: 16-key chunks copied
  static_assert(kOffChunkValid + 4 * kStages <= kBytes, "flag space");
  static_assert(kN / 16 <= 32, "chunk mask");
};

__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" :: "r"(addr), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w) : "memory");
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

// One lane of the (converged) warp, the same one on every lane's view.
__device__ __forceinline__ bool elect_one() {
  uint32_t pred;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "elect.sync _|p, 0xffffffff;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(pred));
  return pred != 0;
}

// Bulk tensor copy of a {x, y, z} box of a rank-3 tensor map into shared
// memory, completing on an mbarrier's transaction count.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y, int z,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];"
      :: "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" :: "r"(bar), "r"(bytes)
               : "memory");
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
__device__ __forceinline__ uint4 codes8_to_f16(uint32_t w0, uint32_t w1) {
  uint4 h;
  dev::word_to_f16x2x2<DT>(w0, h.x, h.y);
  dev::word_to_f16x2x2<DT>(w1, h.z, h.w);
  return h;
}

template <int DT, int D, bool AL>
__global__ void __launch_bounds__(prefill_threads(D), 1)
    prefill_attention_kernel(const AttnParams p, const __grid_constant__ PrefillMaps maps) {
  using Geo = PrefillGeom<DT, D>;
  constexpr int kM = Geo::kM, kN = Geo::kN;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = dev::smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* sm = smem_raw + (base - raw);
  const int tid = threadIdx.x;
  const int warp = tid >> 5;

  // The tile record carries the request's first query token and the
  // position of its query 0, so the Q loads depend on one load only.
  const PrefillTile t = p.prefill_tiles[blockIdx.x];
  const int G = p.group;
  const int q0 = t.q0;
  const int kv_first = (t.kv_lo / kN) * kN;
  const int T = t.kv_hi > kv_first ? (t.kv_hi - kv_first + kN - 1) / kN : 0;  // KV tiles

  const uint32_t bars = base + Geo::kOffBar;
  auto bar = [&](int i) { return bars + 8u * (uint32_t)i; };
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(sm + Geo::kOffAbort);

  if (tid == 0) {
    for (int s = 0; s < Geo::kStages; ++s) {
      tc::mbar_init(bar(Geo::kBarCodesK + s), 1);
      tc::mbar_init(bar(Geo::kBarCodesV + s), 1);
      tc::mbar_init(bar(Geo::kBarCodesKFree + s), Geo::kConv);
      tc::mbar_init(bar(Geo::kBarCodesVFree + s), Geo::kConv);
      tc::mbar_init(bar(Geo::kBarKFull + s), Geo::kConv);
      tc::mbar_init(bar(Geo::kBarVFull + s), Geo::kConv);
      tc::mbar_init(bar(Geo::kBarVEmpty + s), 1);
      tc::mbar_init(bar(Geo::kBarSFull + s), 1);
      tc::mbar_init(bar(Geo::kBarPFull + s), 128);
    }
    for (int s = 0; s < Geo::kSide; ++s)
      tc::mbar_init(bar(Geo::kBarSide + s), Geo::kAuto ? 1 : Geo::kConv);
    tc::mbar_init(bar(Geo::kBarODone), 1);
    tc::mbar_init(bar(Geo::kBarOFinal), 1);
    tc::mbar_init(bar(Geo::kBarDrain), 1);
    *abort_flag = 0u;
    tc::mbar_fence_init();
  }
  if (warp == 0) {
    tc::tmem_alloc(base + Geo::kOffTmemSlot, Geo::kTmemCols);
    tc::tmem_relinquish();
  }

  // ---- roles: warp 0 issues the MMAs, warps 4-7 run the softmax, the last
  // warp issues the bulk tensor copies, the others convert codes to f16.
  constexpr int kCopyWarp = Geo::kThreads / 32 - 1;  // issues the bulk tensor copies
  const bool is_conv = (warp >= 1 && warp < 4) || (warp >= 8 && warp < kCopyWarp);
  const int ctid = warp < 4 ? tid - 32 : tid - 256 + 96;
  const int32_t* btab = p.block_table + (int64_t)t.req * p.block_table_stride;
  float* sk = reinterpret_cast<float*>(sm + Geo::kOffSk);
  float* sv = reinterpret_cast<float*>(sm + Geo::kOffSv);
  uint32_t* smask = reinterpret_cast<uint32_t*>(sm + Geo::kOffSMask);
  volatile uint32_t* smask_w = smask;  // written by the copy warp for bf16 rows
  uint32_t* vmaxw = reinterpret_cast<uint32_t*>(sm + Geo::kOffVMax);
  volatile uint32_t* chunk_valid = reinterpret_cast<volatile uint32_t*>(sm + Geo::kOffChunkValid);
  // Logical key j -> (table entry, offset) without a divide: q0 = hi32(j *
  // floor((2^32 - 1) / B)) is q or q - 1 for every 32-bit j.
  const uint32_t bsz = (uint32_t)p.block_size;
  const uint32_t bdiv = 0xFFFFFFFFu / bsz;
  // Tile j's 16-key chunks: their table entries are loaded one tile ahead
  // (fetch_chunks, whose loads nobody waits for until the copies are issued),
  // then resolved to first slots and a mask of the chunks with a key in the
  // tile's range and a block (resolve_chunks).
  constexpr int kChunks = kN / 16;
  auto fetch_chunks = [&](int j, int (&blk)[kChunks], uint32_t (&off)[kChunks]) {
    const int kv0 = kv_first + j * kN;
#pragma unroll
    for (int c = 0; c < kChunks; ++c) {
      const int j0 = kv0 + 16 * c;
      blk[c] = -1;
      off[c] = 0;
      if (j0 + 16 > t.kv_lo && j0 < t.kv_hi) {
        uint32_t q = __umulhi((uint32_t)j0, bdiv);
        uint32_t r = (uint32_t)j0 - q * bsz;
        if (r >= bsz) {
          ++q;
          r -= bsz;
        }
        blk[c] = btab[q];
        off[c] = r;
      }
    }
  };
  auto resolve_chunks = [&](const int (&blk)[kChunks], const uint32_t (&off)[kChunks],
                            int (&slot0)[kChunks], uint32_t& valid) {
    valid = 0;
#pragma unroll
    for (int c = 0; c < kChunks; ++c) {
      slot0[c] = 0;
      if (blk[c] >= 0 && (int64_t)blk[c] < p.num_blocks) {
        valid |= 1u << c;
        slot0[c] = blk[c] * (int)bsz + (int)off[c];  // < num_blocks * block_size < 2^31
      }
    }
  };
  // Copies of those chunks into code stage j & 1, in two groups with a
  // barrier each: the K codes (and, per token-head, both scale tails), and
  // the V codes.  The chunk list of each stage stays in registers (static
  // indices, selected by the uniform stage) for the V group.
  int kept_slot[2][kChunks];
  uint32_t kept_valid[2] = {0u, 0u};
  // bf16 rows ("auto"): a chunk's rows go straight into the operand tile,
  // one {64 values, 1, 16 slots} box per 64-dim column block, which the
  // copy writes in the 128-byte swizzle the MMAs read.  Chunks that are not
  // copied are zeroed by the copy warp (the tile must hold no stale NaN).
  auto zero_chunk = [&](uint32_t tile, int c) {
    const int lane = tid & 31;
#pragma unroll 1
    for (int cb = 0; cb < D / 64; ++cb)
      for (int u = lane; u < 16 * 8; u += 32)
        sts128(tile + (uint32_t)(cb * kN * 128 + (16 * c) * 128 + u * 16), make_uint4(0, 0, 0, 0));
  };
  auto issue_auto = [&](uint32_t tile, const CUtensorMap* map, const int (&slot0)[kChunks],
                        uint32_t valid, uint32_t cb_bar, bool leader) {
    if ((valid & ((1u << kChunks) - 1u)) != ((1u << kChunks) - 1u)) {
#pragma unroll 1
      for (int c = 0; c < kChunks; ++c)
        if (!((valid >> c) & 1u)) zero_chunk(tile, c);
      tc::fence_async_smem();
    }
    __syncwarp();
    if (leader) {
      mbar_arrive_expect_tx(cb_bar, (uint32_t)__popc(valid) * 16u * D * 2u);
#pragma unroll
      for (int c = 0; c < kChunks; ++c)
        if ((valid >> c) & 1u)
#pragma unroll
          for (int cb = 0; cb < D / 64; ++cb)
            tma_load_3d(tile + (uint32_t)(cb * kN * 128 + (16 * c) * 128), map, 64 * cb, t.kv_head,
                        slot0[c], cb_bar);
    }
  };
  auto issue_k = [&](int j, const int (&slot0)[kChunks], uint32_t valid, bool leader) {
    const int st = j & 1;
    constexpr uint32_t kChunkBytes = 16u * D + (Geo::kPth ? 2u * 16u * 16u : 0u);
    const uint32_t cb = bar(Geo::kBarCodesK + st);
#pragma unroll
    for (int s2 = 0; s2 < 2; ++s2) {
      if (s2 == st) {
#pragma unroll
        for (int c = 0; c < kChunks; ++c) kept_slot[s2][c] = slot0[c];
        kept_valid[s2] = valid;
      }
    }
    if constexpr (Geo::kAuto) {
      issue_auto(base + Geo::kOffK + (uint32_t)(st * Geo::kTileBytes), &maps.k, slot0, valid, cb, leader);
      // The tile's chunk mask for the softmax (side slot j % 4).
      if (leader) smask_w[j & (Geo::kSide - 1)] = valid;
      __syncwarp();
      if (leader) mbar_arrive(bar(Geo::kBarSide + (j & (Geo::kSide - 1))));
    } else if (leader) {
      chunk_valid[st] = valid;
      mbar_arrive_expect_tx(cb, (uint32_t)__popc(valid) * kChunkBytes);
#pragma unroll
      for (int c = 0; c < kChunks; ++c) {
        if ((valid >> c) & 1u) {
          const uint32_t off = (uint32_t)(st * kN + 16 * c);
          tma_load_3d(base + Geo::kOffCodeK + off * D, &maps.k, 0, t.kv_head, slot0[c], cb);
          if constexpr (Geo::kPth) {
            tma_load_3d(base + Geo::kOffTailK + off * 16, &maps.ks, D, t.kv_head, slot0[c], cb);
            tma_load_3d(base + Geo::kOffTailV + off * 16, &maps.vs, D, t.kv_head, slot0[c], cb);
          }
        }
      }
    }
  };
  auto issue_v = [&](int j, bool leader) {
    const int st = j & 1;
    const uint32_t cb = bar(Geo::kBarCodesV + st);
    int slot0[kChunks];
    uint32_t valid = 0;
#pragma unroll
    for (int s2 = 0; s2 < 2; ++s2) {
      if (s2 == st) {
#pragma unroll
        for (int c = 0; c < kChunks; ++c) slot0[c] = kept_slot[s2][c];
        valid = kept_valid[s2];
      }
    }
    if constexpr (Geo::kAuto) {
      issue_auto(base + Geo::kOffV + (uint32_t)(st * Geo::kTileBytes), &maps.v, slot0, valid, cb, leader);
    } else if (leader) {
      mbar_arrive_expect_tx(cb, (uint32_t)__popc(valid) * 16u * D);
#pragma unroll
      for (int c = 0; c < kChunks; ++c) {
        if ((valid >> c) & 1u) {
          const uint32_t off = (uint32_t)(st * kN + 16 * c);
          tma_load_3d(base + Geo::kOffCodeV + off * D, &maps.v, 0, t.kv_head, slot0[c], cb);
        }
      }
    }
  };
  // The copy warp issues the copies: tiles 0 and 1 before Q is staged; then
  // the K group of tile j + 2 once every converter has released the K codes
  // of stage j & 1 (the V group of tile j is out by then: the chunk list is
  // per stage), the V group once the V codes are released.  The table
  // entries of the next tile to copy are read ahead.
  int nk = 0, nv = 0;  // tiles whose K / V copies are issued
  int nx_blk[kChunks];
  uint32_t nx_off[kChunks];
  // Run by the whole copy warp (uniform state); the leader issues.
  auto issue_next_k = [&](bool leader) {  // K copies of tile nk (entries fetched), fetch tile nk + 1
    int slot0[kChunks];
    uint32_t valid;
    resolve_chunks(nx_blk, nx_off, slot0, valid);
    issue_k(nk, slot0, valid, leader);
    ++nk;
    if (nk < T) fetch_chunks(nk, nx_blk, nx_off);
  };
  // ---- Q tile -> staging (swizzled rows), all warps: lanes_per_row lanes
  // hold one row (16 bytes each, coalesced); the row's largest exponent
  // comes from a shuffle reduction over those lanes, and the row is scaled
  // by the power of two that puts its largest |q| in [2^14, 2^15).  The
  // loads are issued first: their latency overlaps the table reads and the
  // first copies.
  constexpr int kLpr = D / 8;            // lanes per row
  constexpr int kRps = 32 / kLpr;        // rows per warp step
  constexpr int kQWarps = Geo::kThreads / 32;
  constexpr int kQSteps = (kM / kRps + kQWarps - 1) / kQWarps;
  const int q_sub = (tid & 31) / kLpr, q_c = (tid & 31) % kLpr;
  uint4 qv[kQSteps];
#pragma unroll
  for (int i = 0; i < kQSteps; ++i) {
    const int m = (warp + i * kQWarps) * kRps + q_sub;
    qv[i] = make_uint4(0, 0, 0, 0);
    if (m < t.nrows) {
      const int R = t.row0 + m;
      qv[i] = *reinterpret_cast<const uint4*>(
          p.q + ((int64_t)(q0 + R / G) * p.heads_q + t.kv_head * G + R % G) * D + 8 * q_c);
    }
  }
  int blk1[kChunks];
  uint32_t off1[kChunks];
  if (warp == kCopyWarp && (tid & 31) == 0) {
    // the tensor maps' descriptors, ahead of the first copies
    asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(&maps.k)) : "memory");
    asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(&maps.v)) : "memory");
    if constexpr (Geo::kPth) {
      asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(&maps.ks)) : "memory");
      asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(&maps.vs)) : "memory");
    }
  }
  if (warp == kCopyWarp && T > 0) {
    fetch_chunks(0, nx_blk, nx_off);
    if (T > 1) fetch_chunks(1, blk1, off1);
  }
  __syncthreads();  // barriers initialised
  if (warp == kCopyWarp && T > 0) {
    const bool leader = elect_one();
    int slot0[kChunks];
    uint32_t valid;
    resolve_chunks(nx_blk, nx_off, slot0, valid);
    issue_k(0, slot0, valid, leader);
    issue_v(0, leader);
    nk = nv = 1;
    if (T > 1) {
      resolve_chunks(blk1, off1, slot0, valid);
      issue_k(1, slot0, valid, leader);
      issue_v(1, leader);
      nk = nv = 2;
      if (nk < T) fetch_chunks(nk, nx_blk, nx_off);
    }
    __syncwarp();
  }
  {
    float* qscale = reinterpret_cast<float*>(sm + Geo::kOffQScale);
#pragma unroll
    for (int i = 0; i < kQSteps; ++i) {
      const int m = (warp + i * kQWarps) * kRps + q_sub;
      const uint32_t w[4] = {qv[i].x, qv[i].y, qv[i].z, qv[i].w};
      int emax = 0;
#pragma unroll
      for (int k = 0; k < 4; ++k) emax = max(emax, (int)max((w[k] >> 7) & 0xFFu, (w[k] >> 23) & 0xFFu));
#pragma unroll
      for (int o = kLpr / 2; o > 0; o >>= 1) emax = max(emax, __shfl_xor_sync(0xffffffffu, emax, o));
      // largest |q| < 2^(emax - 126)
      const int sh = emax > 0 && !Geo::kAuto ? min(140 - emax, 126) : 0;
      const float up = ldexpf(1.0f, sh);
      if (m < kM) {
        uint4 o = qv[i];  // bf16 rows: Q enters the bf16 MMA as it is
        if constexpr (!Geo::kAuto) {
          o.x = dev::pack_f16x2(dev::bf16_lo(w[0]) * up, dev::bf16_hi(w[0]) * up);
          o.y = dev::pack_f16x2(dev::bf16_lo(w[1]) * up, dev::bf16_hi(w[1]) * up);
          o.z = dev::pack_f16x2(dev::bf16_lo(w[2]) * up, dev::bf16_hi(w[2]) * up);
          o.w = dev::pack_f16x2(dev::bf16_lo(w[3]) * up, dev::bf16_hi(w[3]) * up);
        }
        sts128(base + Geo::kOffQStage + tc::sw128_offset(kM, m, 8 * q_c), o);
        if (q_c == 0) qscale[m] = ldexpf(1.0f, -sh);
      }
    }
  }
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(sm + Geo::kOffTmemSlot);
  const bool is_softmax = warp >= 4 && warp < 8;
  const int m = tid - 128;  // row (softmax warps)
  const bool row_valid = is_softmax && m < t.nrows;
  const int R = t.row0 + (row_valid ? m : 0);
  const uint32_t lane_base = (uint32_t)(((warp - 4) & 3) * 32) << 16;
  if (is_softmax) {
    // The softmax warps move Q rows (their own lanes) into tensor memory.
#pragma unroll
    for (int c0 = 0; c0 < D / 2; c0 += 16) {
      uint32_t w[16];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 x = lds128(base + Geo::kOffQStage + tc::sw128_offset(kM, m, 2 * c0 + 8 * q));
        w[4 * q] = x.x; w[4 * q + 1] = x.y; w[4 * q + 2] = x.z; w[4 * q + 3] = x.w;
      }
      tc::tmem_st16(tmem + Geo::kColQ + lane_base + c0, w);
    }
    tc::tmem_wait_st();
  }
  tc::fence_before_sync();
  __syncthreads();  // Q is in tensor memory; the staging area is free
  tc::fence_after_sync();

  if (warp == 0) {
    // ======================= MMA issuer ========================================
    // The whole warp runs the loop with warp-uniform state (descriptors and
    // counters stay in the uniform datapath); one elected lane issues every
    // MMA (the tensor core runs one thread's MMAs in order).
    if (T > 0) {
      const int lane = tid & 31;
      const bool leader = elect_one();
      constexpr uint32_t idesc_s = Geo::kAuto ? tc::idesc_bf16(kM, kN) : tc::idesc_f16(kM, kN);
      constexpr uint32_t idesc_o =
          (Geo::kAuto ? tc::idesc_bf16(kM, D) : tc::idesc_f16(kM, D)) | tc::kBMajorMN;
      auto issue_s = [&](int j) {
        const int st = j & 1;
        // (descriptor start addresses are in 16-byte units in the low bits)
        const uint64_t d0 = tc::desc_sw128(base + Geo::kOffK + (uint32_t)(st * Geo::kTileBytes));
        if (leader) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t boff = (kk >> 2) * (kN * 128) + (kk & 3) * 32;
            tc::mma_ts(tmem + Geo::kColS + (uint32_t)(st * kN), tmem + Geo::kColQ + (uint32_t)(kk * 8),
                       d0 + (uint64_t)(boff >> 4), idesc_s, kk > 0 ? 1u : 0u);
          }
          tc::mma_commit(bar(Geo::kBarSFull + st));
        }
        __syncwarp();
      };
      auto issue_pv = [&](int j) {
        const int st = j & 1;
        const uint64_t d0 =
            tc::desc_sw128_mn(base + Geo::kOffV + (uint32_t)(st * Geo::kTileBytes), kN * 128, 1024);
        if (leader) {
#pragma unroll
          for (int kk = 0; kk < kN / 16; ++kk) {
            if constexpr (Geo::kAuto) {
              // P = hi + lo, both bf16: round c0 of the softmax wrote the hi
              // halves of keys c0 .. c0 + 63 to columns c0 .. c0 + 31 and the
              // lo halves to c0 + 32 .. c0 + 63.
              const uint32_t pc = (uint32_t)(st * kN + 64 * (kk / 4) + 8 * (kk % 4));
              tc::mma_ts(tmem + Geo::kColO, tmem + Geo::kColS + pc, d0 + (uint64_t)(kk * (2048 >> 4)),
                         idesc_o, (j > 0 || kk > 0) ? 1u : 0u);
              tc::mma_ts(tmem + Geo::kColO, tmem + Geo::kColS + pc + 32u,
                         d0 + (uint64_t)(kk * (2048 >> 4)), idesc_o, 1u);
            } else {
              tc::mma_ts(tmem + Geo::kColO, tmem + Geo::kColS + (uint32_t)(st * kN + kk * 8),
                         d0 + (uint64_t)(kk * (2048 >> 4)), idesc_o, (j > 0 || kk > 0) ? 1u : 0u);
            }
          }
          tc::mma_commit(bar(Geo::kBarODone));
          tc::mma_commit(bar(Geo::kBarVEmpty + st));
          if (j == T - 1) tc::mma_commit(bar(Geo::kBarOFinal));
        }
        __syncwarp();
      };
      // S(j) needs K(j) and PV(j-2) issued (P(j-2) shares its buffer; the
      // tensor core runs one thread's MMAs in order).  PV(j) needs P(j) and
      // V(j).  One warp-wide non-blocking test per pass (lane 0: K(ns) in,
      // lane 1: P(npv), lane 2: V(npv)) and one ballot decide for the warp;
      // everything ready is issued, PV first.
      int ns = 0, npv = 0;
      bool ok = true;
      long long t_idle = clock64();
      // (bf16 rows: the copies themselves fill K and V)
      constexpr int kBarK = Geo::kAuto ? Geo::kBarCodesK : Geo::kBarKFull;
      constexpr int kBarV = Geo::kAuto ? Geo::kBarCodesV : Geo::kBarVFull;
      while (npv < T) {
        uint32_t tb = bar(kBarK + (ns & 1)), tp = (uint32_t)((ns >> 1) & 1);
        bool cond = ns < T && ns <= npv + 1;
        if (lane == 1 || lane == 2) {
          tb = bar((lane == 1 ? Geo::kBarPFull : kBarV) + (npv & 1));
          tp = (uint32_t)((npv >> 1) & 1);
          cond = npv < ns;
        }
        const bool r = tc::mbar_test_wait(tb, tp) && cond;
        const uint32_t rb = __ballot_sync(0xffffffffu, r);
        __syncwarp();  // orders the testing lanes' acquires before the leader's issues
        if ((rb & 6u) == 6u) {
          tc::fence_after_sync();
          issue_pv(npv);
          ++npv;
        }
        if (rb & 1u) {
          tc::fence_after_sync();
          issue_s(ns);
          ++ns;
        }
        if ((rb & 1u) || (rb & 6u) == 6u) {
          t_idle = clock64();
        } else if (clock64() - t_idle > 20000) {  // idle a while: look for an abort
          const bool give_up = __shfl_sync(0xffffffffu, (*abort_flag != 0u) ? 1 : 0, 0) != 0;
          const bool timeout = __shfl_sync(0xffffffffu, (clock64() - t_idle > 2000000000LL) ? 1 : 0, 0) != 0;
          if (give_up || timeout) {
            if (timeout && leader) *abort_flag = 1u;
            ok = false;
            break;
          }
        }
      }
      if (!ok && leader) {
        // Drain whatever was issued before the tensor memory is freed.
        tc::mma_commit(bar(Geo::kBarDrain));
        (void)tc::mbar_wait(bar(Geo::kBarDrain), 0u, 200000000LL);
      }
    }
    __syncwarp();
  } else if (warp == kCopyWarp) {
    // ======================= copy producer =====================================
    // One CTA fits on an SM, so the tile that will start when this one ends
    // is about a grid's worth of SMs later in launch order: pull its record
    // and its Q rows into L2 now (its prologue then reads them from L2).
    {
      uint32_t nsm;
      asm("mov.u32 %0, %%nsmid;" : "=r"(nsm));
      const int nb = (int)(blockIdx.x + nsm);
      if (nb < p.num_prefill_tiles) {
        const PrefillTile tn = p.prefill_tiles[nb];
        const int lane = tid & 31;
        // rows R of the tile: token q0 + R / G, heads kv_head * G .. + G - 1
        // contiguous (G * D * 2 bytes per token)
        const int tok0 = tn.row0 / G, tok1 = (tn.row0 + tn.nrows - 1) / G;
        const int64_t run = (int64_t)G * D * 2;
        for (int tk = tok0; tk <= tok1; ++tk) {
          const char* base_q = reinterpret_cast<const char*>(
              p.q + ((int64_t)(tn.q0 + tk) * p.heads_q + (int64_t)tn.kv_head * G) * D);
          for (int64_t off = (int64_t)lane * 128; off < run; off += 32 * 128)
            asm volatile("prefetch.global.L2 [%0];" :: "l"(base_q + off));
        }
      }
    }
    // Tiles 0 and 1 went out before Q was staged.  Step i copies the K codes
    // of tile i + 1 (once K(i - 1) is converted) and then the V codes of
    // tile i (once V(i - 2) is), the order in which the converters release
    // them.
    if (T > 2) {
      const bool leader = elect_one();
      bool ok = true;
      for (int i = 1; i < T; ++i) {
        // (bf16 rows: K(j) waits for S(j - 2) to complete, V(i) for
        // P(i - 2) V(i - 2); code rows wait for the converters.)
        constexpr int kBarKFree = Geo::kAuto ? Geo::kBarSFull : Geo::kBarCodesKFree;
        constexpr int kBarVFree = Geo::kAuto ? Geo::kBarVEmpty : Geo::kBarCodesVFree;
        if (i + 1 < T) {
          const int j = i + 1;
          ok = __all_sync(0xffffffffu, wait_or_abort(bar(kBarKFree + (j & 1)),
                                                      (uint32_t)(((j >> 1) - 1) & 1), abort_flag));
          if (!ok) break;
          issue_next_k(leader);
        }
        if (i >= 2) {
          ok = __all_sync(0xffffffffu, wait_or_abort(bar(kBarVFree + (i & 1)),
                                                      (uint32_t)(((i >> 1) - 1) & 1), abort_flag));
          if (!ok) break;
          issue_v(i, leader);
          ++nv;
        }
      }
      if (!ok && leader) {
        // Let the last copies (at most two tiles of each group in flight)
        // land before the shared memory is released.
        for (int j = nk >= 2 ? nk - 2 : 0; j < nk; ++j)
          (void)tc::mbar_wait(bar(Geo::kBarCodesK + (j & 1)), (uint32_t)((j >> 1) & 1), 200000000LL);
        for (int j = nv >= 2 ? nv - 2 : 0; j < nv; ++j)
          (void)tc::mbar_wait(bar(Geo::kBarCodesV + (j & 1)), (uint32_t)((j >> 1) & 1), 200000000LL);
      }
    }
    __syncwarp();
  } else if (is_conv) {
    if constexpr (!Geo::kAuto) {
    // ======================= converters ========================================
    // A unit is (key n, 16 codes pc): consecutive threads take consecutive
    // 16-byte pieces of a code row (conflict-free reads).  The two 16-byte f16
    // chunks go out in the order that keeps the 8 lanes of a quarter-warp on
    // 8 bank groups (lanes in odd 64-dim blocks store their odd chunk first).
    // A unit's offsets do not change from tile to tile.
    constexpr int kPieces = D / 16;
    constexpr int kUnits = kN * kPieces;
    constexpr int kSlots = (kUnits + Geo::kConv - 1) / Geo::kConv;
    uint32_t code_off[kSlots], st_first[kSlots], st_second[kSlots];
    int unit_key[kSlots];
    uint32_t odd_mask = 0;
#pragma unroll
    for (int i = 0; i < kSlots; ++i) {
      const int u = min(ctid + i * Geo::kConv, kUnits - 1);
      const int n = u / kPieces, pc = u % kPieces;
      const bool odd = (pc >> 2) & 1;
      const uint32_t a_lo = tc::sw128_offset(kN, n, 16 * pc), a_hi = tc::sw128_offset(kN, n, 16 * pc + 8);
      code_off[i] = (uint32_t)(n * D + 16 * pc);
      st_first[i] = odd ? a_hi : a_lo;
      st_second[i] = odd ? a_lo : a_hi;
      unit_key[i] = n;
      odd_mask |= (odd ? 1u : 0u) << i;
    }
    auto convert = [&](int j, uint32_t tile, uint32_t codes, uint32_t valid, bool whole) {
      const int kv0 = kv_first + j * kN;
#pragma unroll
      for (int i = 0; i < kSlots; ++i) {
        if (ctid + i * Geo::kConv < kUnits) {
          uint4 c = make_uint4(0, 0, 0, 0);
          const int n = unit_key[i];
          if (whole || (((valid >> (n >> 4)) & 1u) && kv0 + n >= t.kv_lo && kv0 + n < t.kv_hi))
            c = lds128(codes + code_off[i]);
          const bool odd = (odd_mask >> i) & 1u;
          sts128(tile + st_first[i], codes8_to_f16<DT>(odd ? c.z : c.x, odd ? c.w : c.y));
          sts128(tile + st_second[i], codes8_to_f16<DT>(odd ? c.x : c.z, odd ? c.y : c.w));
        }
      }
    };
    // Step i converts K(i), then V(i - 1): K(i) needs S(i - 2) complete
    // (its buffer), V(i - 1) needs P(i - 3) V(i - 3) complete, which the
    // tensor core finishes later.  The chunk mask of a tile is read with its
    // K codes and kept for its V codes (the issuer rewrites it for tile
    // i + 2 once K(i) is converted).
    uint32_t valid_k = 0, valid_v = 0;
    bool whole_k = false, whole_v = false;
    for (int i = 0; i <= T; ++i) {
      if (i < T) {
        const int st = i & 1, sd = i & (Geo::kSide - 1);
        const int kv0 = kv_first + i * kN;
        if (!__all_sync(0xffffffffu, wait_or_abort(bar(Geo::kBarCodesK + st), (uint32_t)((i >> 1) & 1),
                                                   abort_flag)))
          break;
        if (i >= 2 && !__all_sync(0xffffffffu, wait_or_abort(bar(Geo::kBarSFull + st),
                                                              (uint32_t)(((i >> 1) - 1) & 1), abort_flag)))
          break;
        valid_k = chunk_valid[st];
        // every key of the tile in range and copied: no per-unit checks
        whole_k = valid_k == (1u << kChunks) - 1u && kv0 >= t.kv_lo && kv0 + kN <= t.kv_hi;
        // Side data for the softmax in slot i % 4 (its reader, the softmax
        // of tile i - 4, is done: S(i - 2) was issued after P(i - 4) V(i - 4)).
        if (ctid == 0) smask[sd] = valid_k;
        if constexpr (Geo::kPth) {
          // Per-key scales, one thread per key (0 for a key without a copied
          // row); each converter warp publishes the largest value scale it saw.
          float vmax = 0.0f;
          for (int n = ctid; n < kN; n += Geo::kConv) {
            const int jj = kv0 + n;
            const bool live = jj >= t.kv_lo && jj < t.kv_hi && ((valid_k >> (n >> 4)) & 1u);
            const uint32_t off = (uint32_t)((st * kN + n) * 16);
            const float ks = live ? *reinterpret_cast<const float*>(sm + Geo::kOffTailK + off) : 0.0f;
            const float vs = live ? *reinterpret_cast<const float*>(sm + Geo::kOffTailV + off) : 0.0f;
            sk[sd * kN + n] = ks;
            sv[sd * kN + n] = vs;
            vmax = fmaxf(vmax, vs);  // stays >= 0 (a NaN or negative scale is ignored)
          }
          const uint32_t wmax = __reduce_max_sync(0xffffffffu, __float_as_uint(vmax));
          // (only the first (kN + 31) / 32 converter warps hold keys)
          if ((ctid & 31) == 0 && (ctid >> 5) < (kN + 31) / 32) vmaxw[sd * 8 + (ctid >> 5)] = wmax;
        }
        mbar_arrive(bar(Geo::kBarSide + sd));
        convert(i, base + Geo::kOffK + (uint32_t)(st * Geo::kTileBytes),
                base + Geo::kOffCodeK + (uint32_t)(st * kN * D), valid_k, whole_k);
        tc::fence_async_smem();
        mbar_arrive(bar(Geo::kBarKFull + st));
        // done with the K codes and tails of stage st
        mbar_arrive(bar(Geo::kBarCodesKFree + st));
      }
      if (i >= 1) {
        const int jv = i - 1, st = jv & 1;
        if (!__all_sync(0xffffffffu, wait_or_abort(bar(Geo::kBarCodesV + st), (uint32_t)((jv >> 1) & 1),
                                                   abort_flag)))
          break;
        if (jv >= 2 && !__all_sync(0xffffffffu, wait_or_abort(bar(Geo::kBarVEmpty + st),
                                                               (uint32_t)(((jv >> 1) - 1) & 1), abort_flag)))
          break;
        convert(jv, base + Geo::kOffV + (uint32_t)(st * Geo::kTileBytes),
                base + Geo::kOffCodeV + (uint32_t)(st * kN * D), valid_v, whole_v);
        tc::fence_async_smem();
        mbar_arrive(bar(Geo::kBarVFull + st));
        mbar_arrive(bar(Geo::kBarCodesVFree + st));
      }
      valid_v = valid_k;
      whole_v = whole_k;
    }
    }
    __syncwarp();
  } else {
    // ======================= softmax ===========================================
    const float* sk = reinterpret_cast<const float*>(sm + Geo::kOffSk);
    const float* sv = reinterpret_cast<const float*>(sm + Geo::kOffSv);
    const uint32_t* smask = reinterpret_cast<const uint32_t*>(sm + Geo::kOffSMask);
    const uint32_t* vmaxw = reinterpret_cast<const uint32_t*>(sm + Geo::kOffVMax);
    constexpr uint32_t kAllChunks = (kChunks >= 32) ? 0xFFFFFFFFu : ((1u << kChunks) - 1u);
    constexpr int kVMaxSlots = (kN + 31) / 32;  // converter warps that hold keys
    const int pos = t.pos0 + R / G;
    const int W = p.window;
    // (without causality every row sees the request's L keys: the tile's kv_hi)
    const int row_hi = row_valid ? (p.causal ? pos + 1 : t.kv_hi) : 0;  // padding rows see nothing
    const int row_lo = W > 0 ? pos - W + 1 : 0;
    const float log2e = 1.4426950408889634f;
    const float cap = p.soft_cap;
    // scores in log2 units (natural units under a soft cap, which converts)
    const float q_unscale = reinterpret_cast<const float*>(sm + Geo::kOffQScale)[m];  // 2^-sh
    const float score_mul = p.sm_scale * q_unscale * (cap > 0.0f ? 1.0f : log2e) *
                            (Geo::kPth || Geo::kAuto ? 1.0f : p.k_scale);
    // ALiBi: this row's slope in log2 units (the bias uses the exact integer
    // distance key - position, added after the soft cap).
    const float al_slope = AL ? p.alibi_slopes[t.kv_head * G + R % G] * log2e : 0.0f;
    const float cap_l2 = cap * log2e;
    const float inv_cap = cap > 0.0f ? 1.0f / cap : 0.0f;
    // m_ref: the reference maximum, an integer (log2 units) once set, so
    // that moving it scales weights, O and l by exact powers of two.
    float m_ref = -INFINITY, l_sum = 0.0f;
    int ev = -1000;  // exponent of the value-scale reference (per-token-head)
    bool ok = true;
    for (int j = 0; j < T; ++j) {
      const int st = j & 1;
      const int kv0 = kv_first + j * kN;
      const int sd = j & (Geo::kSide - 1);
      // S(j) is in tensor memory; tile j's side data is in slot sd.
      ok = wait_or_abort(bar(Geo::kBarSFull + st), (uint32_t)((j >> 1) & 1), abort_flag) &&
           wait_or_abort(bar(Geo::kBarSide + sd), (uint32_t)((j >> 2) & 1), abort_flag);
      ok = __all_sync(0xffffffffu, ok);  // warp-uniform: the warp's tensor-memory accesses are collective
      if (!ok) break;
      tc::fence_after_sync();
      const uint32_t tmem_s = tmem + Geo::kColS + (uint32_t)(st * kN) + lane_base;
      // Visible keys n of this row: lo_n <= n < hi_n, in a 16-key chunk
      // that was copied.  Masks are needed unless every row of the warp
      // sees the whole tile and every chunk is in.
      const uint32_t cmask = smask[sd];
      const int lo_n = row_lo - kv0, hi_n = row_hi - kv0;
      const bool full = __all_sync(0xffffffffu, lo_n <= 0 && hi_n >= kN) && cmask == kAllChunks;
      float alpha = 1.0f;  // factor for O (score reference and value reference)
      // Value-scale reference (per-token-head): the largest exponent so far.
      float v_mul = 1.0f;  // 2^-ev
      if constexpr (Geo::kPth) {
        uint32_t mb = 0;
#pragma unroll
        for (int w = 0; w < kVMaxSlots; ++w) mb = max(mb, vmaxw[sd * 8 + w]);
        const float smax = __uint_as_float(mb);
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
      // The score in log2 units from r (the raw score, times the key's scale
      // per token-head; -inf when masked).  Under a cap, masked r stays
      // masked (a capped -inf would be finite).
      auto score = [&](auto cap_c, float r) -> float {
        if constexpr (decltype(cap_c)::value)
          return r == -INFINITY ? -INFINITY : cap_l2 * dev::tanh_exp(r * score_mul * inv_cap);
        else
          return r * score_mul;
      };
      // 64 scores from column c0: r in place, the row's maximum of r.  With
      // ALiBi the bias differs per key, so the final scores (log2 units) are
      // stored and maximised instead.
      auto raw64 = [&](auto full_c, uint32_t* v, int c0) -> float {
        const float* skp = sk + sd * kN + c0;
        const int lo = lo_n - c0, hi = hi_n - c0;
        const uint32_t cm = cmask >> (c0 >> 4);
        const int dist0 = kv0 + c0 - pos;  // key - position of column c0
        float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int e = 0; e < 64; e += 2) {
          float r0 = __uint_as_float(v[e]), r1 = __uint_as_float(v[e + 1]);
          if constexpr (Geo::kPth) {
            const float2 k2 = *reinterpret_cast<const float2*>(skp + e);
            r0 *= k2.x;
            r1 *= k2.y;
          }
          if constexpr (AL) {
            if (cap > 0.0f) {
              r0 = cap_l2 * dev::tanh_exp(r0 * score_mul * inv_cap);
              r1 = cap_l2 * dev::tanh_exp(r1 * score_mul * inv_cap);
            } else {
              r0 *= score_mul;
              r1 *= score_mul;
            }
            r0 = fmaf(al_slope, (float)(dist0 + e), r0);
            r1 = fmaf(al_slope, (float)(dist0 + e + 1), r1);
          }
          if constexpr (!decltype(full_c)::value) {
            const bool in = (cm >> (e >> 4)) & 1u;
            r0 = in && e >= lo && e < hi ? r0 : -INFINITY;
            r1 = in && e + 1 >= lo && e + 1 < hi ? r1 : -INFINITY;
          }
          v[e] = __float_as_uint(r0);
          v[e + 1] = __float_as_uint(r1);
          mx4[(e >> 1) & 3] = fmaxf(mx4[(e >> 1) & 3], fmaxf(r0, r1));
        }
        return fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
      };
      // P = 2^(z - m_ref + 6) <= 2^14 in f16 pairs: the 2^6 lifts small
      // weights clear of the f16 subnormal range; l carries the same factor.
      float lsum_tile = 0.0f;
      auto weights64 = [&](auto cap_c, const uint32_t* v, int c0, float ref, uint32_t* pw) {
        const float* svp = sv + sd * kN + c0;
        float ls0 = 0.0f, ls1 = 0.0f;
#pragma unroll
        for (int e = 0; e < 64; e += 2) {
          const float r0 = __uint_as_float(v[e]), r1 = __uint_as_float(v[e + 1]);
          float p0, p1;
          if constexpr (AL) {  // v holds the final scores
            p0 = dev::fast_exp2(r0 - ref);
            p1 = dev::fast_exp2(r1 - ref);
          } else if constexpr (decltype(cap_c)::value) {
            p0 = dev::fast_exp2(score(cap_c, r0) - ref);
            p1 = dev::fast_exp2(score(cap_c, r1) - ref);
          } else {
            p0 = dev::fast_exp2(fmaf(r0, score_mul, -ref));
            p1 = dev::fast_exp2(fmaf(r1, score_mul, -ref));
          }
          ls0 += p0;
          ls1 += p1;
          if constexpr (Geo::kPth) {
            const float2 v2 = *reinterpret_cast<const float2*>(svp + e);
            p0 *= v2.x * v_mul;
            p1 *= v2.y * v_mul;
          }
          if constexpr (Geo::kAuto) {
            // bf16 MMA: P = hi + lo, both bf16 (16 significant bits); hi in
            // pw[0 .. 31], lo in pw[32 .. 63].
            const uint32_t h = dev::pack_bf16x2(p0, p1);
            pw[e / 2] = h;
            pw[32 + e / 2] = dev::pack_bf16x2(p0 - dev::bf16_lo(h), p1 - dev::bf16_hi(h));
          } else {
            pw[e / 2] = dev::pack_f16x2(p0, p1);
          }
        }
        lsum_tile += ls0 + ls1;
      };
      // One pass over the row, 64 scores per tensor-memory round trip: the
      // round's maximum, then its weights against the reference, written
      // as f16 pairs over columns of S(j) already read.  A round maximum
      // more than 2^8 above the reference moves it (lazily) to the next
      // integer at or above; weights already written in this tile are then
      // scaled by the same power of two.
#pragma unroll 1
      for (int c0 = 0; c0 < kN; c0 += 64) {
        uint32_t v[64];
        tc::tmem_ld32(tmem_s + c0, *reinterpret_cast<uint32_t(*)[32]>(v));
        tc::tmem_ld32(tmem_s + c0 + 32, *reinterpret_cast<uint32_t(*)[32]>(v + 32));
        tc::tmem_wait_ld();
        const float mr = full ? raw64(std::true_type{}, v, c0) : raw64(std::false_type{}, v, c0);
        // the score is monotonic in r (score_mul > 0, tanh increasing); with
        // ALiBi mr is the largest final score already
        const float mx = AL ? mr : cap > 0.0f ? score(std::true_type{}, mr) : score(std::false_type{}, mr);
        float a = 1.0f;
        if (mx > m_ref + 8.0f) {
          const float nref = ceilf(mx);
          if (m_ref != -INFINITY) a = ldexpf(1.0f, (int)fmaxf(m_ref - nref, -200.0f));
          m_ref = nref;
          alpha *= a;
          l_sum *= a;
          lsum_tile *= a;
        }
        const float ref = m_ref == -INFINITY ? 0.0f : m_ref - 6.0f;
        constexpr int kPw = Geo::kAuto ? 64 : 32;  // P words of the round (bf16: hi and lo)
        uint32_t pw[kPw];
        if (cap > 0.0f)
          weights64(std::true_type{}, v, c0, ref, pw);
        else
          weights64(std::false_type{}, v, c0, ref, pw);
        // f16 P of the round goes to columns c0 / 2 .. c0 / 2 + 31; bf16 hi
        // and lo halves to c0 .. c0 + 63 (the columns this round read).
        const int pcol = Geo::kAuto ? c0 : c0 / 2;
#pragma unroll
        for (int h = 0; h < kPw; h += 16)
          tc::tmem_st16(tmem_s + pcol + h, *reinterpret_cast<uint32_t(*)[16]>(pw + h));
        if (c0 > 0 && __any_sync(0xffffffffu, a != 1.0f)) {
          // Weights of the earlier rounds against the new reference: a
          // power-of-two scaling, exact unless subnormal.
          tc::tmem_wait_st();
#pragma unroll 1
          for (int c = 0; c < pcol; c += 32) {
            uint32_t w[32];
            tc::tmem_ld32(tmem_s + c, w);
            tc::tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              if constexpr (Geo::kAuto) {
                w[e] = dev::pack_bf16x2(dev::bf16_lo(w[e]) * a, dev::bf16_hi(w[e]) * a);
              } else {
                const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[e]));
                w[e] = dev::pack_f16x2(f.x * a, f.y * a);
              }
            }
            tc::tmem_st32(tmem_s + c, w);
          }
        }
      }
      l_sum += lsum_tile;
      // A moved reference rescales O: PV(j-1) must be complete first.  (S(j)
      // being complete implies PV(j-2) is, and PV(j) waits for this tile's
      // P, so the barrier is at completion j-1 or j: the wait is exact.)
      if (j > 0 && __any_sync(0xffffffffu, alpha != 1.0f)) {
        ok = __all_sync(0xffffffffu,
                        wait_or_abort(bar(Geo::kBarODone), (uint32_t)((j - 1) & 1), abort_flag));
        if (!ok) break;
        tc::fence_after_sync();
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t v[32];
          tc::tmem_ld32(tmem + Geo::kColO + lane_base + c0, v);
          tc::tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
          tc::tmem_st32(tmem + Geo::kColO + lane_base + c0, v);
        }
      }
      tc::tmem_wait_st();
      tc::fence_before_sync();
      mbar_arrive(bar(Geo::kBarPFull + st));
    }
    // ---- epilogue: O / l -> bf16 -------------------------------------------
    if (ok && T > 0)
      ok = __all_sync(0xffffffffu, wait_or_abort(bar(Geo::kBarOFinal), 0u, abort_flag));
    // ok is warp-uniform here: the whole warp reads O (tcgen05.ld is a
    // warp-collective instruction).  Each thread writes its row in bf16 to
    // the (now idle) K ring, row-major with the 16-byte chunks of row m
    // rotated by m mod 8; all warps then copy the tile out coalesced.
    if (ok) {
      const uint32_t orow = base + Geo::kOffOStage + (uint32_t)(m * D * 2);
      if (T > 0) {
        tc::fence_after_sync();
        // An attention sink joins the normaliser (the weights carry
        // 2^-(m_ref - 6)).
        if (p.sinks && row_valid && m_ref != -INFINITY) {
          const float sk = p.sinks[t.kv_head * G + R % G] * log2e;
          if (sk != -INFINITY) l_sum += exp2f(fminf(sk - m_ref + 6.0f, 126.0f));
        }
        const float sc = (l_sum > 0.0f ? 1.0f / l_sum : 0.0f) *
                         (Geo::kPth ? (ev > -1000 ? ldexpf(1.0f, ev) : 0.0f)
                                    : Geo::kAuto ? 1.0f : p.v_scale);
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t v[32];
          tc::tmem_ld32(tmem + Geo::kColO + lane_base + c0, v);
          tc::tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; e += 8) {
            uint4 o;
            o.x = dev::pack_bf16x2(__uint_as_float(v[e]) * sc, __uint_as_float(v[e + 1]) * sc);
            o.y = dev::pack_bf16x2(__uint_as_float(v[e + 2]) * sc, __uint_as_float(v[e + 3]) * sc);
            o.z = dev::pack_bf16x2(__uint_as_float(v[e + 4]) * sc, __uint_as_float(v[e + 5]) * sc);
            o.w = dev::pack_bf16x2(__uint_as_float(v[e + 6]) * sc, __uint_as_float(v[e + 7]) * sc);
            const int c = (c0 + e) / 8;
            sts128(orow + (uint32_t)(((c ^ (m & 7)) << 4)), o);
          }
        }
      } else {
        // No key tile at all (an empty key range): the output row is zero.
#pragma unroll 1
        for (int c = 0; c < D / 8; ++c) sts128(orow + (uint32_t)(c << 4), make_uint4(0, 0, 0, 0));
      }
    }
    // Order this warp's tensor-memory accesses before the teardown barrier.
    tc::fence_before_sync();
    __syncwarp();
  }

  __syncthreads();
  const bool aborted = *abort_flag != 0u;
  if (tid == 0 && aborted) atomicExch(p.error_flag, 1);
  if (warp == 0) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, Geo::kTmemCols);
  }
  // ---- O tile -> global, coalesced: lanes_per_row lanes write one row.  A
  // tile that gave up a bounded wait writes NaN rows instead, so its failure
  // shows in the output even where nobody reads the error word.
  {
    constexpr int kLpr = D / 8;
    constexpr int kRps = 32 / kLpr;
    const int lane = tid & 31;
    const int sub = lane / kLpr, c = lane % kLpr;
    const uint4 nan4 = make_uint4(0x7FC07FC0u, 0x7FC07FC0u, 0x7FC07FC0u, 0x7FC07FC0u);
    for (int r = warp * kRps + sub; r < t.nrows; r += (Geo::kThreads / 32) * kRps) {
      const uint4 o = aborted ? nan4
                              : lds128(base + Geo::kOffOStage + (uint32_t)(r * D * 2 + ((c ^ (r & 7)) << 4)));
      const int Rr = t.row0 + r;
      *reinterpret_cast<uint4*>(p.out + ((int64_t)(q0 + Rr / G) * p.heads_q + t.kv_head * G + Rr % G) * D +
                                8 * c) = o;
    }
  }
}

template <int DT, int D, bool AL>
int launch_prefill_instance(const AttnParams& p, const PrefillMaps& maps, int64_t num_tiles,
                            cudaStream_t stream) {
  const size_t smem = prefill_smem_bytes(D);
  auto kern = prefill_attention_kernel<DT, D, AL>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return KVQ_E_CUDA;
  kern<<<(unsigned)num_tiles, prefill_threads(D), smem, stream>>>(p, maps);
  return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_E_CUDA;
}

// The instances of one head_dim and one ALiBi setting (one translation unit
// each keeps the build parallel).
template <int D, bool AL>
int launch_prefill_d(const AttnParams& p, const PrefillMaps& maps, int dtype, int64_t num_tiles,
                     cudaStream_t stream) {
  switch (dtype) {
    case KVQ_AUTO: return launch_prefill_instance<KVQ_AUTO, D, AL>(p, maps, num_tiles, stream);
    case KVQ_FP8_E4M3: return launch_prefill_instance<KVQ_FP8_E4M3, D, AL>(p, maps, num_tiles, stream);
    case KVQ_FP8_E5M2: return launch_prefill_instance<KVQ_FP8_E5M2, D, AL>(p, maps, num_tiles, stream);
    case KVQ_INT8_PER_TOKEN_HEAD:
      return launch_prefill_instance<KVQ_INT8_PER_TOKEN_HEAD, D, AL>(p, maps, num_tiles, stream);
    case KVQ_FP8_PER_TOKEN_HEAD:
      return launch_prefill_instance<KVQ_FP8_PER_TOKEN_HEAD, D, AL>(p, maps, num_tiles, stream);
    case KVQ_FP8_E5M2_PER_TOKEN_HEAD:
      return launch_prefill_instance<KVQ_FP8_E5M2_PER_TOKEN_HEAD, D, AL>(p, maps, num_tiles, stream);
    default:
      return KVQ_E_UNSUPPORTED;
  }
}

}  // namespace kvq
