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
// GB300 design: persistent CTAs (one per SM) walking a dealt list of tiles,
// 16 warps (12 at head_dim 256), warp-specialised and pipelined through
// mbarriers.
//   * Tensor memory (512 columns): O (D fp32 columns), two S buffers (keys
//     fp32 columns each; P(j) is written as f16 pairs over the first half of
//     S(j)'s buffer), and Q (D/2 columns of f16 pairs).  Both MMAs take A
//     from tensor memory: S = Q K^T and O += P V read only K and V from
//     shared memory.
//   * Copy warp (the last): resolves each KV tile's 16-key chunks through
//     the block table into first slots (a slot table per KV tile, up to four
//     ahead).  bf16 ("auto") rows: bulk tensor copies (TMA) of the chunks
//     straight into the K and V operand tiles.
//   * Converter warps (1-3, and 8 up to the copy warp): a thread takes (key,
//     16 codes) units, loads the codes from global memory one KV tile ahead,
//     converts them exactly to f16 (every e4m3 / e5m2 / int8 value is an f16
//     value) and stores them as key-major rows in the 128-byte swizzle into a
//     two-stage K ring and V ring.  K is read by the tensor core K-major, V
//     MN-major, so neither needs a transpose.  Step i converts K(i) (its
//     buffer is free once S(i-2) is complete) and then V(i-1) (free once
//     P(i-3) V(i-3) is).  Per-key scales, the tile's chunk mask and its
//     largest value scale go to one of four side-data slots for the softmax.
//   * MMA warp (0): one elected lane issues, in a fixed order, S(j+1) and
//     then O += P(j) V(j), each once its operands are in (blocking waits).
//   * Softmax warps (4-7): thread t owns row t (tensor-memory lane t).  One
//     pass over its row of S, 64 scores per tensor-memory round trip: the
//     round's maximum, then the weights, written as f16 straight into
//     tensor memory.  The reference maximum is an integer (log2 units) and
//     lazy: it moves only when a score exceeds it by 2^8 (weights are lifted
//     by 2^6, so P <= 2^14), to the next integer at or above the maximum,
//     and the weights, O and l already accumulated are rescaled by the exact
//     power of two (O only after P(j-1) V(j-1) is complete; 32 columns a
//     round, the next round's tensor-memory load in flight).  At the end it
//     reads O and stages bf16 rows for one bulk store per row.
//   * Q rows of the next tile are bulk-copied into shared memory (the output
//     staging area, free between epilogues) when a tile starts, and moved
//     into tensor memory once the tile's last S is complete, so that the
//     next tile's first S runs beside the last softmax.
//   * Q enters as f16 exactly: each row is scaled by a power of two that puts
//     its largest |q| in [2^13, 2^14) (a bf16 significand fits in f16's);
//     the scale, sm_scale, log2(e) and k_scale (per tensor) or the key's
//     scale (per token-head) multiply the fp32 scores; v_scale the output.
//     Elements more than about 2^27 below the row's largest fall into f16's
//     subnormals and lose low bits (further down, flush to zero).
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

#include <algorithm>
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
  // CTA pair (kCG = 2): this CTA holds keys [r * kN / 2, (r + 1) * kN / 2) of
  // each K tile (all D dims) and dims [r * D / 2, (r + 1) * D / 2) of each V
  // tile (all kN keys), r its rank in the cluster.
  static constexpr int kCG = prefill_cta_group(DT, D);
  static constexpr int kKeysK = kN / kCG;                           // keys of a K tile held here
  static constexpr int kDimsV = D / kCG;                            // dims of a V tile held here
  static constexpr int kTileBytes = kN * D * 2 / kCG;               // this CTA's K or V tile (f16)
  static constexpr int kOffK = 0;                                   // stages x K tile
  static constexpr int kOffV = kOffK + kStages * kTileBytes;        // stages x V tile
  // Side data of KV tile g, for the softmax, in slot g % kSide: per-key
  // scales, the 16-key chunk mask and, per converter warp, the largest
  // value scale of its keys (bits of a float >= 0).
  static constexpr int kSide = kPrefillSideSlots;
  static constexpr int kOffSk = kOffV + kStages * kTileBytes;       // kSide x kN f32
  static constexpr int kOffSv = kOffSk + kSide * kN * 4;            // kSide x kN f32
  static constexpr int kOffSMask = kOffSv + kSide * kN * 4;         // kSide x u32
  static constexpr int kOffVMax = kOffSMask + 4 * kSide;            // kSide x 8 u32
  // Slot tables of KV tiles g, in entry g % kSlotRing: the first slot of
  // each 16-key chunk (entries 0 .. kN / 16 - 1) and the chunk mask (15).
  static constexpr int kSlotRing = kPrefillSlotRing;
  static constexpr int kOffSlots = kOffVMax + 32 * kSide;           // kSlotRing x 16 i32
  // O of a finished tile, bf16 rows for the bulk stores: kM rows of D * 2
  // bytes, 16 bytes of padding after each (a warp's 16-byte stores of one
  // column chunk then cover all 32 banks).
  static constexpr int kOutPitch = D * 2 + 16;
  static constexpr int kOffOut = kOffSlots + kSlotRing * 64;         // kM x kOutPitch
  static constexpr int kOffBar = kOffOut + kM * kOutPitch;          // mbarriers, tmem slot, flags
  static constexpr int kBytes = kOffBar + 512;
  static constexpr int kColO = 0;                 // O: D fp32 columns
  static constexpr int kColS = D;                 // S buffers: kN fp32 columns each
  static constexpr int kColQ = D + 2 * kN;        // Q: D/2 columns of f16 pairs
  static constexpr int kTmemCols = prefill_tmem_cols(D);
  static_assert(kColQ + D / 2 <= kTmemCols, "tensor memory: O + 2 S buffers + Q");
  static_assert(kTileBytes % 1024 == 0 && kOffV % 1024 == 0, "1024-byte operand tiles");
  static_assert(kOffBar % 8 == 0, "mbarrier alignment");
  static_assert((kN + 31) / 32 <= 8 && kSide == 4, "side data space");
  static_assert(kN / 16 <= 15 && (kSlotRing & (kSlotRing - 1)) == 0, "slot table layout");
  static_assert(kConv >= kN && kConv % 32 == 0, "a converter thread per key, whole warps");
  static_assert((size_t)kBytes + 1024 == prefill_smem_bytes(D, kCG), "smem must follow the geometry");
  static_assert(kCG == 1 || (!kAuto && kDimsV % 64 == 0 && kKeysK % 8 == 0), "pair halves in the swizzle");
  // barrier slots (8 bytes each).  Quantised rows: the copy warp publishes
  // KV tile g's slot table (Slots, ring entry g % 4) once the converters
  // released entry g - 4 (SlotsFree); K(g) is converted once S(g - 2) is
  // complete, V(g) once P(g - 2) V(g - 2) is (KFull / VFull).  bf16 rows:
  // bulk copies fill the K and V tiles (CodesK / CodesV).  One P barrier
  // per S buffer: P(g+1) may be ready before PV(g) is issued.  A parity
  // wait is unambiguous only while the waiter is at most one phase behind,
  // so the epilogue (which may be several PVs ahead of the last phase it
  // saw) waits on a barrier of its own for a tile's last PV (one phase per
  // tile), and the side data (which the converters may write two tiles
  // ahead) has four slots.  Across tiles: Q full (the softmax warps wrote
  // the tile's Q; the tile's first S waits) and O free (the epilogue read
  // O; the next tile's first PV waits) and Q staged (the softmax threads'
  // bulk copies of a tile's Q rows landed), one phase per tile each.  A CTA
  // pair: the barriers the MMA warp waits on (KFull, VFull, PFull, QFull,
  // OFree) are the even CTA's, counting the warps of both CTAs; each commit
  // arrives on both CTAs' barriers.
  static constexpr int kBarCodesK = 0, kBarCodesV = 2, kBarKFull = 4, kBarVFull = 6, kBarVEmpty = 8,
                       kBarSFull = 10, kBarPFull = 12, kBarSide = 14, kBarODone = 18, kBarOFinal = 19,
                       kBarDrain = 20, kBarQFull = 21, kBarOFree = 22, kBarQStage = 23, kBarSlots = 24,
                       kBarSlotsFree = kBarSlots + kSlotRing, kNumBars = kBarSlotsFree + kSlotRing;
  static constexpr int kOffTmemSlot = kOffBar + 8 * kNumBars;   // u32
  static constexpr int kOffAbort = kOffTmemSlot + 4;            // u32
  static_assert(kOffAbort + 4 <= kBytes, "flag space");
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

// One arrival for the (converged) warp, after every lane's prior writes:
// the barriers count warps.  Per-thread arrivals would put hundreds of
// shared-memory atomics per KV tile in front of the MMA warp's polls.
__device__ __forceinline__ void warp_arrive(uint32_t bar) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}

// One arrival of the (converged) warp on a barrier of the CTA that issues
// the MMAs: this CTA's, or for the odd CTA of a pair the even CTA's (a
// release at cluster scope).
template <int CG>
__device__ __forceinline__ void warp_arrive_mma(uint32_t bar, uint32_t rank) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) {
    if (CG == 2 && rank != 0)
      tc::mbar_arrive_remote(bar, 0u);
    else
      mbar_arrive(bar);
  }
}

// Bounded wait that also gives up when another role has aborted (CG = 2:
// acquire at cluster scope, for the MMA warp of a pair, whose barriers see
// arrivals from both CTAs).
template <int CG = 1>
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, volatile uint32_t* abort) {
  auto test = [&]() {
    if constexpr (CG == 2)
      return tc::mbar_try_wait_cluster(bar, parity);
    else
      return tc::mbar_try_wait(bar, parity);
  };
  if (test()) return true;
  const long long t0 = clock64();
  while (true) {
    if (test()) return true;
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

// This CTA's k-th tile: the longest-first tile list dealt out over the grid
// in serpentine order (CTA b takes tile b of the first round, tile 2G-1-b of
// the second, ...), so every CTA gets a similar amount of work.  CTA pairs
// (CG = 2) deal pair tiles (list entries 2i, 2i + 1: two consecutive row
// tiles of one kv head) to the clusters; the CTA of rank r takes entry 2i + r.
template <int CG>
__device__ __forceinline__ int dealt_tile(int k) {
  const int G = (int)gridDim.x / CG, b = (int)blockIdx.x / CG;
  const int i = k * G + ((k & 1) ? G - 1 - b : b);
  return CG == 1 ? i : 2 * i + (int)(blockIdx.x & 1u);
}

// A tile and its run of KV tiles: kN-key tiles from kv_first (the key range's
// start rounded down to a tile) up to its end.  For a CTA pair the key range
// is the union of both halves' (both CTAs walk the same KV tiles; each row
// masks the keys it does not see).
template <int kN>
struct TileRun {
  PrefillTile t;
  int lo, hi, kv_first, T;
  __device__ __forceinline__ void set(const PrefillTile& x, const PrefillTile& y) {
    t = x;
    lo = min(x.kv_lo, y.kv_lo);
    hi = max(x.kv_hi, y.kv_hi);
    kv_first = (lo / kN) * kN;
    T = hi > kv_first ? (hi - kv_first + kN - 1) / kN : 0;
  }
};

// The record of list entry idx and, for a pair, its partner's.
template <int CG>
__device__ __forceinline__ void load_tiles(const AttnParams& p, int idx, PrefillTile& x, PrefillTile& y) {
  x = p.prefill_tiles[idx];
  if constexpr (CG == 2)
    y = p.prefill_tiles[idx ^ 1];
  else
    y = x;
}

// Walks this CTA's KV tiles in order: KV tile j of its tile ordinal k
// (tiles without keys skipped), n = the tiles with keys before this one.
// The next tile's record is loaded a tile ahead, so that a move to it does
// not wait for memory.
template <int kN, int CG>
struct KvCursor {
  TileRun<kN> cur;
  PrefillTile nxt, nxt_y;
  int k, j, n;
  bool valid, nxt_valid;
  __device__ __forceinline__ void start(const AttnParams& p) {
    k = -1;
    n = -1;
    nxt_valid = dealt_tile<CG>(0) < p.num_prefill_tiles;
    if (nxt_valid) load_tiles<CG>(p, dealt_tile<CG>(0), nxt, nxt_y);
    next_tile(p);
  }
  __device__ __forceinline__ void next_tile(const AttnParams& p) {
    valid = false;
    while (nxt_valid) {
      cur.set(nxt, nxt_y);
      ++k;
      const int idx = dealt_tile<CG>(k + 1);
      nxt_valid = idx < p.num_prefill_tiles;
      if (nxt_valid) load_tiles<CG>(p, idx, nxt, nxt_y);
      if (cur.T > 0) {
        valid = true;
        ++n;
        j = 0;
        return;
      }
    }
  }
  __device__ __forceinline__ void advance(const AttnParams& p) {
    if (++j >= cur.T) next_tile(p);
  }
};

template <int DT, int D, bool AL>
__global__ void __launch_bounds__(prefill_threads(D), 1)
    prefill_attention_kernel(const AttnParams p, const __grid_constant__ PrefillMaps maps) {
  using Geo = PrefillGeom<DT, D>;
  constexpr int kM = Geo::kM, kN = Geo::kN, CG = Geo::kCG;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = dev::smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* sm = smem_raw + (base - raw);
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int G = p.group;
  // rank in the CTA pair (0: issues the MMAs of both)
  const uint32_t rank = CG == 2 ? tc::cluster_ctarank() : 0u;

  const uint32_t bars = base + Geo::kOffBar;
  auto bar = [&](int i) { return bars + 8u * (uint32_t)i; };
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(sm + Geo::kOffAbort);
  constexpr int kCopyWarp = Geo::kThreads / 32 - 1;  // issues the bulk tensor copies

  if (tid == 0) {
    for (int s = 0; s < Geo::kSlotRing; ++s) {
      tc::mbar_init(bar(Geo::kBarSlots + s), 1);
      tc::mbar_init(bar(Geo::kBarSlotsFree + s), Geo::kConv / 32);
    }
    for (int s = 0; s < Geo::kStages; ++s) {
      tc::mbar_init(bar(Geo::kBarCodesK + s), 1);
      tc::mbar_init(bar(Geo::kBarCodesV + s), 1);
      tc::mbar_init(bar(Geo::kBarKFull + s), CG * Geo::kConv / 32);
      tc::mbar_init(bar(Geo::kBarVFull + s), CG * Geo::kConv / 32);
      tc::mbar_init(bar(Geo::kBarVEmpty + s), 1);
      tc::mbar_init(bar(Geo::kBarSFull + s), 1);
      tc::mbar_init(bar(Geo::kBarPFull + s), 4 * CG);
    }
    for (int s = 0; s < Geo::kSide; ++s)
      tc::mbar_init(bar(Geo::kBarSide + s), Geo::kAuto ? 1 : Geo::kConv / 32);
    tc::mbar_init(bar(Geo::kBarODone), 1);
    tc::mbar_init(bar(Geo::kBarOFinal), 1);
    tc::mbar_init(bar(Geo::kBarDrain), 1);
    tc::mbar_init(bar(Geo::kBarQFull), 4 * CG);
    tc::mbar_init(bar(Geo::kBarQStage), 128);
    tc::mbar_init(bar(Geo::kBarOFree), 4 * CG);
    *abort_flag = 0u;
    tc::mbar_fence_init();
  }
  if (warp == 0) {
    // (a pair: warp 0 of both CTAs, the same columns in both)
    tc::tmem_alloc<CG>(base + Geo::kOffTmemSlot, Geo::kTmemCols);
    tc::tmem_relinquish<CG>();
  }
  if (Geo::kAuto && warp == kCopyWarp && (tid & 31) == 0) {
    // the tensor maps' descriptors, ahead of the first copies
    asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(&maps.k)) : "memory");
    asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(&maps.v)) : "memory");
  }
  tc::fence_before_sync();
  // barriers initialised, tensor memory allocated (a pair: in both CTAs,
  // before either arrives on the other's barriers)
  if constexpr (CG == 2)
    tc::cluster_sync();
  else
    __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(sm + Geo::kOffTmemSlot);

  // ---- roles: warp 0 issues the MMAs, warps 4-7 run the softmax, the last
  // warp issues the bulk tensor copies, the others convert codes to f16.
  // Every role walks the same sequence of KV tiles g = 0, 1, ... (over all
  // of this CTA's tiles), so the rings' stages and phases follow g.
  const bool is_conv = (warp >= 1 && warp < 4) || (warp >= 8 && warp < kCopyWarp);
  const int ctid = warp < 4 ? tid - 32 : tid - 256 + 96;
  float* sk = reinterpret_cast<float*>(sm + Geo::kOffSk);
  float* sv = reinterpret_cast<float*>(sm + Geo::kOffSv);
  uint32_t* smask = reinterpret_cast<uint32_t*>(sm + Geo::kOffSMask);
  uint32_t* vmaxw = reinterpret_cast<uint32_t*>(sm + Geo::kOffVMax);
  constexpr int kChunks = kN / 16;

  if (warp == 0) {
    if (rank == 0) {
    // ======================= MMA issuer ========================================
    // The whole warp runs the loop with warp-uniform state (descriptors and
    // counters stay in the uniform datapath); one elected lane issues every
    // MMA (the tensor core runs one thread's MMAs in order).  A CTA pair's
    // MMAs (M = 256) are issued by the even CTA: rows 128-255 are the odd
    // CTA's tile, and the B operands' halves are read from both CTAs' shared
    // memory at the same offsets.
    const bool leader = elect_one();
    KvCursor<kN, CG> cs;
    cs.start(p);
    constexpr uint32_t idesc_s = Geo::kAuto ? tc::idesc_bf16(kM, kN) : tc::idesc_f16(kM * CG, kN);
    constexpr uint32_t idesc_o =
        (Geo::kAuto ? tc::idesc_bf16(kM, D) : tc::idesc_f16(kM * CG, D)) | tc::kBMajorMN;
    auto issue_s = [&](int g) {
      const int st = g & 1;
      // (descriptor start addresses are in 16-byte units in the low bits)
      const uint64_t d0 = tc::desc_sw128(base + Geo::kOffK + (uint32_t)(st * Geo::kTileBytes));
      if (leader) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t boff = (kk >> 2) * (Geo::kKeysK * 128) + (kk & 3) * 32;
          tc::mma_ts<CG>(tmem + Geo::kColS + (uint32_t)(st * kN), tmem + Geo::kColQ + (uint32_t)(kk * 8),
                         d0 + (uint64_t)(boff >> 4), idesc_s, kk > 0 ? 1u : 0u);
        }
        tc::mma_commit<CG>(bar(Geo::kBarSFull + st));
      }
      __syncwarp();
    };
    auto issue_pv = [&](int g, bool first, bool last) {
      const int st = g & 1;
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
                       idesc_o, (!first || kk > 0) ? 1u : 0u);
            tc::mma_ts(tmem + Geo::kColO, tmem + Geo::kColS + pc + 32u,
                       d0 + (uint64_t)(kk * (2048 >> 4)), idesc_o, 1u);
          } else {
            tc::mma_ts<CG>(tmem + Geo::kColO, tmem + Geo::kColS + (uint32_t)(st * kN + kk * 8),
                           d0 + (uint64_t)(kk * (2048 >> 4)), idesc_o, (!first || kk > 0) ? 1u : 0u);
          }
        }
        tc::mma_commit<CG>(bar(Geo::kBarODone));
        tc::mma_commit<CG>(bar(Geo::kBarVEmpty + st));
        if (last) tc::mma_commit<CG>(bar(Geo::kBarOFinal));
      }
      __syncwarp();
    };
    // S(g) needs K(g), PV(g-2) issued (P(g-2) shares its buffer; the tensor
    // core runs one thread's MMAs in order) and, for a tile's first KV
    // tile, the tile's Q in tensor memory.  PV(g) needs P(g), V(g) and, for
    // a tile's first KV tile after the CTA's first tile, O read out by the
    // previous tile's epilogue.  So the issue order is fixed -- S(0), then
    // per g: S(g+1), PV(g) -- and the warp waits for each barrier in turn
    // (a blocking wait wakes as soon as the phase completes; polling several
    // barriers costs a shared-memory round trip per pass).  At a tile
    // boundary S(g+1) needs the next tile's Q, which the softmax writes as
    // soon as S(g) is complete, before P(g).  Flags of S(g) for its PV, 4 bits in
    // slot g % 4: first KV tile of its tile, last, the tile's ordinal (with
    // keys) odd, ordinal 0.
    int ns = 0;
    uint32_t flags = 0;
    bool ok = true;
    // (bf16 rows: the copies themselves fill K and V)
    constexpr int kBarK = Geo::kAuto ? Geo::kBarCodesK : Geo::kBarKFull;
    constexpr int kBarV = Geo::kAuto ? Geo::kBarCodesV : Geo::kBarVFull;
    auto wait = [&](int b, uint32_t parity) {
      return __all_sync(0xffffffffu, wait_or_abort<CG>(bar(b), parity, abort_flag));
    };
    auto next_s = [&]() -> bool {  // S(ns) at the cursor
      if (cs.j == 0 && !wait(Geo::kBarQFull, (uint32_t)(cs.n & 1))) return false;
      if (!wait(kBarK + (ns & 1), (uint32_t)((ns >> 1) & 1))) return false;
      tc::fence_after_sync();
      issue_s(ns);
      const uint32_t nf = (cs.j == 0 ? 1u : 0u) | (cs.j == cs.cur.T - 1 ? 2u : 0u) |
                          ((uint32_t)(cs.n & 1) << 2) | (cs.n == 0 ? 8u : 0u);
      flags = (flags & ~(0xFu << (4 * (ns & 3)))) | (nf << (4 * (ns & 3)));
      ++ns;
      cs.advance(p);
      return true;
    };
    if (cs.valid) ok = next_s();
    for (int g = 0; ok && g < ns; ++g) {
      if (cs.valid && !(ok = next_s())) break;
      const uint32_t f = (flags >> (4 * (g & 3))) & 0xFu;
      // O of the previous tile read out: its OFree completion (ordinal - 1)
      if ((f & 1u) && !(f & 8u) && !(ok = wait(Geo::kBarOFree, ((f >> 2) & 1u) ^ 1u))) break;
      if (!(ok = wait(Geo::kBarPFull + (g & 1), (uint32_t)((g >> 1) & 1)) &&
                 wait(kBarV + (g & 1), (uint32_t)((g >> 1) & 1))))
        break;
      tc::fence_after_sync();
      issue_pv(g, (f & 1u) != 0, (f & 2u) != 0);
    }
    if (!ok && leader) {
      // Drain whatever was issued before the tensor memory is freed.
      tc::mma_commit<CG>(bar(Geo::kBarDrain), 1);
      (void)tc::mbar_wait(bar(Geo::kBarDrain), 0u, 200000000LL);
    }
    }
    __syncwarp();
  } else if (warp == kCopyWarp) {
    // ======================= copy producer =====================================
    // Logical key j of a tile's request -> (table entry, offset) without a
    // divide: q0 = hi32(j * floor((2^32 - 1) / B)) is q or q - 1 for every
    // 32-bit j.  KV tile g's 16-key chunks: their table entries are loaded
    // one KV tile ahead (fetch_chunks, whose loads nobody waits for until
    // they are used), then resolved to first slots and a mask of the chunks
    // with a key in the tile's range and a block (resolve_chunks).  (A
    // chunk's 16 slots are consecutive: the block size is a multiple of 16.)
    const uint32_t bsz = (uint32_t)p.block_size;
    const uint32_t bdiv = 0xFFFFFFFFu / bsz;
    auto fetch_chunks = [&](const TileRun<kN>& r, int j, int (&blk)[kChunks], uint32_t (&off)[kChunks]) {
      const int32_t* btab = p.block_table + (int64_t)r.t.req * p.block_table_stride;
      const int kv0 = r.kv_first + j * kN;
#pragma unroll
      for (int c = 0; c < kChunks; ++c) {
        const int j0 = kv0 + 16 * c;
        blk[c] = -1;
        off[c] = 0;
        if (j0 + 16 > r.lo && j0 < r.hi) {
          uint32_t q = __umulhi((uint32_t)j0, bdiv);
          uint32_t rr = (uint32_t)j0 - q * bsz;
          if (rr >= bsz) {
            ++q;
            rr -= bsz;
          }
          blk[c] = btab[q];
          off[c] = rr;
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
    const bool leader = elect_one();
    KvCursor<kN, CG> ck;
    ck.start(p);
    int nx_blk[kChunks];
    uint32_t nx_off[kChunks];
    if (ck.valid) fetch_chunks(ck.cur, 0, nx_blk, nx_off);
    if constexpr (!Geo::kAuto) {
      // Quantised rows: the converters load the codes themselves.  KV tile
      // g's slot table (first slot of each chunk, then the chunk mask in
      // entry 15) goes to ring entry g % 4 once the converters are done
      // with KV tile g - 4's.
      int32_t* table = reinterpret_cast<int32_t*>(sm + Geo::kOffSlots);
      for (int g = 0; ck.valid; ++g) {
        const int e = g & (Geo::kSlotRing - 1);
        if (g >= Geo::kSlotRing &&
            !__all_sync(0xffffffffu, wait_or_abort(bar(Geo::kBarSlotsFree + e),
                                                    (uint32_t)(((g / Geo::kSlotRing) - 1) & 1), abort_flag)))
          break;
        int slot0[kChunks];
        uint32_t valid;
        resolve_chunks(nx_blk, nx_off, slot0, valid);
        if (leader) {
#pragma unroll
          for (int c = 0; c < kChunks; ++c) table[e * 16 + c] = slot0[c];
          table[e * 16 + 15] = (int32_t)valid;
          mbar_arrive(bar(Geo::kBarSlots + e));
        }
        __syncwarp();
        ck.advance(p);
        if (ck.valid) fetch_chunks(ck.cur, ck.j, nx_blk, nx_off);
      }
    } else {
      // bf16 rows ("auto"): a chunk's rows go straight into the operand
      // tile, one {64 values, 1, 16 slots} box per 64-dim column block, which
      // the copy writes in the 128-byte swizzle the MMAs read.  Chunks that
      // are not copied are zeroed by the copy warp (the tile must hold no
      // stale NaN).  The chunk list and kv head of each stage stay in
      // registers (static indices, selected by the uniform stage) for the V
      // copies.
      volatile uint32_t* smask_w = smask;
      int kept_slot[2][kChunks];
      uint32_t kept_valid[2] = {0u, 0u};
      int kept_head[2] = {0, 0};
      auto zero_chunk = [&](uint32_t tile, int c) {
        const int lane = tid & 31;
#pragma unroll 1
        for (int cb = 0; cb < D / 64; ++cb)
          for (int u = lane; u < 16 * 8; u += 32)
            sts128(tile + (uint32_t)(cb * kN * 128 + (16 * c) * 128 + u * 16), make_uint4(0, 0, 0, 0));
      };
      auto issue_auto = [&](uint32_t tile, const CUtensorMap* map, int head, const int (&slot0)[kChunks],
                            uint32_t valid, uint32_t cb_bar) {
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
                tma_load_3d(tile + (uint32_t)(cb * kN * 128 + (16 * c) * 128), map, 64 * cb, head, slot0[c],
                            cb_bar);
        }
      };
      auto issue_k = [&](int g, int head, const int (&slot0)[kChunks], uint32_t valid) {
        const int st = g & 1;
#pragma unroll
        for (int s2 = 0; s2 < 2; ++s2) {
          if (s2 == st) {
#pragma unroll
            for (int c = 0; c < kChunks; ++c) kept_slot[s2][c] = slot0[c];
            kept_valid[s2] = valid;
            kept_head[s2] = head;
          }
        }
        issue_auto(base + Geo::kOffK + (uint32_t)(st * Geo::kTileBytes), &maps.k, head, slot0, valid,
                   bar(Geo::kBarCodesK + st));
        // The tile's chunk mask for the softmax (side slot g % 4).
        if (leader) smask_w[g & (Geo::kSide - 1)] = valid;
        __syncwarp();
        if (leader) mbar_arrive(bar(Geo::kBarSide + (g & (Geo::kSide - 1))));
      };
      auto issue_v = [&](int g) {
        const int st = g & 1;
        int slot0[kChunks];
        uint32_t valid = 0;
        int head = 0;
#pragma unroll
        for (int s2 = 0; s2 < 2; ++s2) {
          if (s2 == st) {
#pragma unroll
            for (int c = 0; c < kChunks; ++c) slot0[c] = kept_slot[s2][c];
            valid = kept_valid[s2];
            head = kept_head[s2];
          }
        }
        issue_auto(base + Geo::kOffV + (uint32_t)(st * Geo::kTileBytes), &maps.v, head, slot0, valid,
                   bar(Geo::kBarCodesV + st));
      };
      // Step g copies K(g) (once S(g - 2) is complete: its buffer) and then
      // V(g - 1) (once P(g - 3) V(g - 3) is).
      int nk = 0, nv = 0;  // KV tiles whose K / V copies are issued
      bool ok = true;
      for (int g = 0;; ++g) {
        const bool have_k = ck.valid;
        if (have_k) {
          if (g >= 2) {
            ok = __all_sync(0xffffffffu, wait_or_abort(bar(Geo::kBarSFull + (g & 1)),
                                                        (uint32_t)(((g >> 1) - 1) & 1), abort_flag));
            if (!ok) break;
          }
          int slot0[kChunks];
          uint32_t valid;
          resolve_chunks(nx_blk, nx_off, slot0, valid);
          issue_k(g, ck.cur.t.kv_head, slot0, valid);
          ++nk;
          ck.advance(p);
          if (ck.valid) fetch_chunks(ck.cur, ck.j, nx_blk, nx_off);
        }
        if (g >= 1) {
          const int gv = g - 1;
          if (gv >= 2) {
            ok = __all_sync(0xffffffffu, wait_or_abort(bar(Geo::kBarVEmpty + (gv & 1)),
                                                        (uint32_t)(((gv >> 1) - 1) & 1), abort_flag));
            if (!ok) break;
          }
          issue_v(gv);
          ++nv;
        }
        if (!have_k) break;
      }
      if (!ok && leader) {
        // Let the last copies (at most two KV tiles of each group in flight)
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
    // 16-byte pieces of a key's row (coalesced loads).  The codes come from
    // global memory into registers one KV tile ahead of their conversion (K
    // of tile g + 1 and V of tile g while tile g is converted), so their
    // latency hides behind a step; dead keys (outside the key range or in a
    // chunk without a block) load as zero.  The two 16-byte f16 chunks go
    // out in the order that keeps the 8 lanes of a quarter-warp on 8 bank
    // groups (lanes in odd 64-dim blocks store their odd chunk first).  A
    // unit's offsets do not change from tile to tile.  A CTA of a pair
    // converts its half of each tile: of K, keys [r * kN / 2, (r + 1) * kN / 2)
    // (rows of its K tile); of V, dims [r * D / 2, (r + 1) * D / 2) of every
    // key (columns of its V tile).
    constexpr int kUnits = kN * D / 16 / CG;
    constexpr int kSlots = (kUnits + Geo::kConv - 1) / Geo::kConv;
    constexpr int64_t kRow = row_bytes(DT, D);
    struct Units {
      uint32_t code_off[kSlots];  // key in the tile * D + dim in the row
      uint32_t st_first[kSlots], st_second[kSlots], odd_mask;
    };
    // units of a tile held as `rows` rows of `pieces` 16-code pieces, its
    // row n being key key0 + n, dims from dim0
    auto make_units = [&](int rows, int pieces, int key0, int dim0) {
      Units t;
      t.odd_mask = 0;
#pragma unroll
      for (int i = 0; i < kSlots; ++i) {
        const int u = min(ctid + i * Geo::kConv, kUnits - 1);
        const int n = u / pieces, pc = u % pieces;
        const bool odd = (pc >> 2) & 1;
        const uint32_t a_lo = tc::sw128_offset(rows, n, 16 * pc), a_hi = tc::sw128_offset(rows, n, 16 * pc + 8);
        t.code_off[i] = (uint32_t)((key0 + n) * D + dim0 + 16 * pc);
        t.st_first[i] = odd ? a_hi : a_lo;
        t.st_second[i] = odd ? a_lo : a_hi;
        t.odd_mask |= (odd ? 1u : 0u) << i;
      }
      return t;
    };
    const Units uk = make_units(Geo::kKeysK, D / 16, (int)rank * Geo::kKeysK, 0);
    const Units uv = CG == 1 ? uk : make_units(kN, Geo::kDimsV / 16, 0, (int)rank * Geo::kDimsV);
    const int32_t* table = reinterpret_cast<const int32_t*>(sm + Geo::kOffSlots);
    // Codes of KV tile g (slot table entry e, kv head `head`, live keys
    // [win & 0xFFFF, win >> 16) of the tile) into registers; returns the
    // tile's chunk mask.
    auto load_codes = [&](const Units& un, const uint8_t* cache, int e, int head, uint32_t win,
                          uint4 (&dst)[kSlots]) {
      const uint32_t valid = (uint32_t)table[e * 16 + 15];
#pragma unroll
      for (int i = 0; i < kSlots; ++i) {
        dst[i] = make_uint4(0, 0, 0, 0);
        const int n = (int)(un.code_off[i] / D);
        if (ctid + i * Geo::kConv < kUnits && ((valid >> (n >> 4)) & 1u) && n >= (int)(win & 0xFFFFu) &&
            n < (int)(win >> 16)) {
          const int64_t slot = table[e * 16 + (n >> 4)] + (n & 15);
          dst[i] = dev::ldg_stream(cache + (slot * p.heads_kv + head) * kRow + (un.code_off[i] & (D - 1)));
        }
      }
      return valid;
    };
    // Per token-head: key ctid's two scales (the fp32 after the codes; 0 for
    // a dead key), loaded with the tile's K codes.
    auto load_scales = [&](int e, int head, uint32_t win, uint32_t valid, float& ks, float& vs) {
      ks = vs = 0.0f;
      if constexpr (Geo::kPth) {
        const int n = ctid;
        if (n < kN && ((valid >> (n >> 4)) & 1u) && n >= (int)(win & 0xFFFFu) && n < (int)(win >> 16)) {
          const int64_t off = ((int64_t)(table[e * 16 + (n >> 4)] + (n & 15)) * p.heads_kv + head) * kRow + D;
          ks = __ldg(reinterpret_cast<const float*>(p.key_cache + off));
          vs = __ldg(reinterpret_cast<const float*>(p.value_cache + off));
        }
      }
    };
    auto convert = [&](const Units& un, uint32_t tile, const uint4 (&c)[kSlots]) {
#pragma unroll
      for (int i = 0; i < kSlots; ++i) {
        if (ctid + i * Geo::kConv < kUnits) {
          const bool odd = (un.odd_mask >> i) & 1u;
          sts128(tile + un.st_first[i], codes8_to_f16<DT>(odd ? c[i].z : c[i].x, odd ? c[i].w : c[i].y));
          sts128(tile + un.st_second[i], codes8_to_f16<DT>(odd ? c[i].x : c[i].z, odd ? c[i].y : c[i].w));
        }
      }
    };
    // The converted tile is visible to the tensor core (for a pair, the MMAs
    // the even CTA issues read it after that CTA's barrier wait).
    auto fence_operands = [&]() { tc::fence_async_smem(); };
    // A KV tile's live keys relative to its first key, packed lo | hi << 16.
    auto window_of = [&](const KvCursor<kN, CG>& c) {
      const int kv0 = c.cur.kv_first + c.j * kN;
      const int klo = min(max(c.cur.lo - kv0, 0), kN), khi = min(max(c.cur.hi - kv0, 0), kN);
      return (uint32_t)klo | ((uint32_t)khi << 16);
    };
    // Step g: convert K(g) (its buffer is free once S(g - 2) is complete)
    // and publish its side data; load K(g + 1); convert V(g - 1) (its buffer
    // is free once P(g - 3) V(g - 3) is complete); load V(g), after which
    // slot table g is released.
    KvCursor<kN, CG> ck;
    ck.start(p);
    uint4 ka[kSlots], vb[kSlots];
    float ks_a = 0.0f, vs_a = 0.0f;
    uint32_t valid_a = 0, win_a = 0;
    bool ok = true;
    if (ck.valid) {
      ok = __all_sync(0xffffffffu, wait_or_abort(bar(Geo::kBarSlots), 0u, abort_flag));
      if (ok) {
        win_a = window_of(ck);
        valid_a = load_codes(uk, p.key_cache, 0, ck.cur.t.kv_head, win_a, ka);
        load_scales(0, ck.cur.t.kv_head, win_a, valid_a, ks_a, vs_a);
      }
    }
    for (int g = 0; ok; ++g) {
      const bool have_k = ck.valid;
      const int head_g = ck.cur.t.kv_head;
      const uint32_t win_g = win_a;
      if (have_k) {
        const int st = g & 1, sd = g & (Geo::kSide - 1);
        if (g >= 2 && !(ok = __all_sync(0xffffffffu, wait_or_abort(bar(Geo::kBarSFull + st),
                                                                    (uint32_t)(((g >> 1) - 1) & 1), abort_flag))))
          break;
        // Side data for the softmax in slot g % 4 (its reader, the softmax
        // of KV tile g - 4, is done: S(g - 2) was issued after P(g - 4) V(g - 4)).
        if (ctid == 0) smask[sd] = valid_a;
        if constexpr (Geo::kPth) {
          // per-key scales (0 for a dead key); each converter warp publishes
          // the largest value scale of its keys
          if (ctid < kN) {
            sk[sd * kN + ctid] = ks_a;
            sv[sd * kN + ctid] = vs_a;
          }
          const float vmax = ctid < kN ? fmaxf(vs_a, 0.0f) : 0.0f;  // (a NaN or negative scale is ignored)
          const uint32_t wmax = __reduce_max_sync(0xffffffffu, __float_as_uint(vmax));
          // (only the first (kN + 31) / 32 converter warps hold keys)
          if ((ctid & 31) == 0 && (ctid >> 5) < (kN + 31) / 32) vmaxw[sd * 8 + (ctid >> 5)] = wmax;
        }
        warp_arrive(bar(Geo::kBarSide + sd));
        convert(uk, base + Geo::kOffK + (uint32_t)(st * Geo::kTileBytes), ka);
        fence_operands();
        warp_arrive_mma<CG>(bar(Geo::kBarKFull + st), rank);
        ck.advance(p);
      }
      // K(g + 1) into registers.  The odd CTA of a pair issues it after
      // V(g - 1)'s arrival: an arrival on the other CTA's barrier releases at
      // cluster scope, which waits for this thread's loads in flight.
      auto load_next_k = [&]() -> bool {
        if (have_k && ck.valid) {
          const int e1 = (g + 1) & (Geo::kSlotRing - 1);
          if (!__all_sync(0xffffffffu, wait_or_abort(bar(Geo::kBarSlots + e1),
                                                     (uint32_t)(((g + 1) / Geo::kSlotRing) & 1), abort_flag)))
            return false;
          win_a = window_of(ck);
          valid_a = load_codes(uk, p.key_cache, e1, ck.cur.t.kv_head, win_a, ka);
          load_scales(e1, ck.cur.t.kv_head, win_a, valid_a, ks_a, vs_a);
        }
        return true;
      };
      const bool defer_k = CG == 2 && rank != 0;
      if (!defer_k && !(ok = load_next_k())) break;
      if (g >= 1) {
        const int gv = g - 1, st = gv & 1;
        if (gv >= 2 && !(ok = __all_sync(0xffffffffu, wait_or_abort(bar(Geo::kBarVEmpty + st),
                                                                     (uint32_t)(((gv >> 1) - 1) & 1), abort_flag))))
          break;
        convert(uv, base + Geo::kOffV + (uint32_t)(st * Geo::kTileBytes), vb);
        fence_operands();
        warp_arrive_mma<CG>(bar(Geo::kBarVFull + st), rank);
      }
      if (defer_k && !(ok = load_next_k())) break;
      if (!have_k) break;
      const int e = g & (Geo::kSlotRing - 1);
      (void)load_codes(uv, p.value_cache, e, head_g, win_g, vb);
      warp_arrive(bar(Geo::kBarSlotsFree + e));
    }
    }
    __syncwarp();
  } else {
    // ======================= softmax ===========================================
    constexpr uint32_t kAllChunks = (kChunks >= 32) ? 0xFFFFFFFFu : ((1u << kChunks) - 1u);
    constexpr int kVMaxSlots = (kN + 31) / 32;  // converter warps that hold keys
    const int m = tid - 128;  // row (tensor-memory lane m)
    const uint32_t lane_base = (uint32_t)(((warp - 4) & 3) * 32) << 16;
    const float log2e = 1.4426950408889634f;
    const float cap = p.soft_cap;
    const float cap_l2 = cap * log2e;
    const float inv_cap = cap > 0.0f ? 1.0f / cap : 0.0f;
    const int W = p.window;
    // Output row m of a tile, bf16: D values from `dst` (null: not a row).
    auto out_row = [&](const PrefillTile& t) -> uint16_t* {
      if (m >= t.nrows) return nullptr;
      const int Rr = t.row0 + m;
      return p.out + ((int64_t)(t.q0 + Rr / G) * p.heads_q + t.kv_head * G + Rr % G) * D;
    };
    // Tiles without keys (an empty key range) get zero rows as they are passed.
    auto zero_rows = [&](const PrefillTile& t) {
      uint16_t* dst = out_row(t);
      if (dst)
        for (int c = 0; c < D / 8; ++c) reinterpret_cast<uint4*>(dst)[c] = make_uint4(0, 0, 0, 0);
    };
    // Next tile with keys after ordinal k (k moves to it); false: none.
    auto next_run = [&](int& k, TileRun<kN>& r) -> bool {
      while (true) {
        const int idx = dealt_tile<CG>(++k);
        if (idx >= p.num_prefill_tiles) return false;
        PrefillTile x, y;
        load_tiles<CG>(p, idx, x, y);
        r.set(x, y);
        if (r.T > 0) return true;
        zero_rows(r.t);
      }
    };
    // Q rows of a tile are staged in shared memory a tile ahead: each thread
    // copies its row of the next tile (one bulk copy, completing on the
    // QStage barrier) into its row of the output staging area, which is free
    // from the previous tile's bulk store until this tile's epilogue.  Rows
    // past the tile's end copy nothing.
    const uint32_t srow = base + Geo::kOffOut + (uint32_t)(m * Geo::kOutPitch);
    auto stage_q = [&](const PrefillTile& t) {
      const bool valid = m < t.nrows;
      // (this thread's previous bulk store has read its staging row)
      asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
      mbar_arrive_expect_tx(bar(Geo::kBarQStage), valid ? (uint32_t)(D * 2) : 0u);
      if (valid) {
        const int Rq = t.row0 + m;
        const uint16_t* src = p.q + ((int64_t)(t.q0 + Rq / G) * p.heads_q + t.kv_head * G + Rq % G) * D;
        asm volatile(
            "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
            :: "r"(srow), "l"(reinterpret_cast<uint64_t>(src)), "n"(D * 2), "r"(bar(Geo::kBarQStage))
            : "memory");
      }
    };
    // Staged Q row m of the tile with ordinal (with keys) n_tile -> tensor
    // memory (columns kColQ.., f16 pairs), and the arrival that lets the
    // tile's first S go.  Q enters as f16 exactly: the row is scaled by the
    // power of two that puts its largest |q| in [2^13, 2^14) (a bf16
    // significand fits in f16's).  Elements more than about 2^27 below the
    // row's largest land in f16's subnormal range (bits lost) or flush to
    // zero: a Q row with that dynamic range loses them.  bf16 rows ("auto")
    // enter the bf16 MMA as they are.  Returns the row's 2^-shift.
    auto load_q = [&](int nrows, int n_tile) -> float {
      const bool valid = m < nrows;
      (void)__all_sync(0xffffffffu, wait_or_abort(bar(Geo::kBarQStage), (uint32_t)(n_tile & 1), abort_flag));
      int emax = 0;
      if (valid && !Geo::kAuto) {
#pragma unroll 8
        for (int c = 0; c < D / 8; ++c) {
          const uint4 x4 = lds128(srow + (uint32_t)(16 * c));
          const uint32_t x[4] = {x4.x, x4.y, x4.z, x4.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) emax = max(emax, (int)max((x[e] >> 7) & 0xFFu, (x[e] >> 23) & 0xFFu));
        }
      }
      // largest |q| < 2^(emax - 126): scaled into [2^13, 2^14)
      const int sh = emax == 0 || Geo::kAuto ? 0 : min(140 - emax, 126);
      const float up = ldexpf(1.0f, sh);
#pragma unroll 1
      for (int h = 0; h < D / 2; h += 16) {
        uint32_t w[16];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint4 x4 = valid ? lds128(srow + (uint32_t)(4 * h + 16 * c)) : make_uint4(0, 0, 0, 0);
          const uint32_t x[4] = {x4.x, x4.y, x4.z, x4.w};
#pragma unroll
          for (int e = 0; e < 4; ++e)
            w[4 * c + e] = Geo::kAuto ? x[e] : dev::pack_f16x2(dev::bf16_lo(x[e]) * up, dev::bf16_hi(x[e]) * up);
        }
        tc::tmem_st16(tmem + Geo::kColQ + lane_base + (uint32_t)h, w);
      }
      tc::tmem_wait_st();
      tc::fence_before_sync();
      warp_arrive_mma<CG>(bar(Geo::kBarQFull), rank);
      return ldexpf(1.0f, -sh);
    };

    TileRun<kN> cur;
    int k = -1;
    bool have = next_run(k, cur);
    if (have) stage_q(cur.t);
    float q_unscale = have ? load_q(cur.t.nrows, 0) : 1.0f;
    bool ok = true;
    int g = 0;
    int staged = 0;  // tiles whose Q was staged
    if (have) staged = 1;
    for (int n = 0; have; ++n) {
      // The next tile with keys (its record is read again when its Q is
      // staged and after this tile's loop, from L1: only its ordinal stays
      // in registers).
      int k2 = k;
      {
        TileRun<kN> nxt;
        if (!next_run(k2, nxt)) k2 = -1;
      }
      // the next tile's Q rows into the staging area (free from this
      // thread's previous bulk store until this tile's epilogue)
      if (k2 >= 0) {
        stage_q(p.prefill_tiles[dealt_tile<CG>(k2)]);
        ++staged;
      }
      float q_next = 1.0f;
      const PrefillTile& t = cur.t;
      const int kv_first = cur.kv_first, T = cur.T;
      const bool row_valid = m < t.nrows;
      const int R = t.row0 + (row_valid ? m : 0);
      const int pos = t.pos0 + R / G;

      // (without causality every row sees the request's L keys: the tile's kv_hi)
      const int row_hi = row_valid ? (p.causal ? pos + 1 : t.kv_hi) : 0;  // padding rows see nothing
      const int row_lo = W > 0 ? pos - W + 1 : 0;
      // scores in log2 units (natural units under a soft cap, which converts)
      const float score_mul = p.sm_scale * q_unscale * (cap > 0.0f ? 1.0f : log2e) *
                              (Geo::kPth || Geo::kAuto ? 1.0f : p.k_scale);
      // ALiBi: this row's slope in log2 units (the bias uses the exact integer
      // distance key - position, added after the soft cap).
      const float al_slope = AL ? p.alibi_slopes[t.kv_head * G + R % G] * log2e : 0.0f;
      // m_ref: the reference maximum, an integer (log2 units) once set, so
      // that moving it scales weights, O and l by exact powers of two.
      float m_ref = -INFINITY, l_sum = 0.0f;
      int ev = -1000;  // exponent of the value-scale reference (per-token-head)
      for (int j = 0; j < T; ++j, ++g) {
        const int st = g & 1;
        const int kv0 = kv_first + j * kN;
        const int sd = g & (Geo::kSide - 1);
        // S(g) is in tensor memory; KV tile g's side data is in slot sd.
        ok = wait_or_abort(bar(Geo::kBarSFull + st), (uint32_t)((g >> 1) & 1), abort_flag) &&
             wait_or_abort(bar(Geo::kBarSide + sd), (uint32_t)((g >> 2) & 1), abort_flag);
        ok = __all_sync(0xffffffffu, ok);  // warp-uniform: the warp's tensor-memory accesses are collective
        if (!ok) break;
        tc::fence_after_sync();
        // S(g), this tile's last, is complete: Q's tensor memory takes the
        // next tile's Q now, so that its first S runs beside this softmax.
        if (j == T - 1 && k2 >= 0) q_next = load_q(p.prefill_tiles[dealt_tile<CG>(k2)].nrows, n + 1);
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
        // A moved reference rescales O: PV(g-1) must be complete first.  (S(g)
        // being complete implies PV(g-2) is, and PV(g) waits for this KV
        // tile's P, so the barrier is at completion g-1 or g: the wait is
        // exact.  The tile's first KV tile starts O afresh.)
        if (j > 0 && __any_sync(0xffffffffu, alpha != 1.0f)) {
          ok = __all_sync(0xffffffffu,
                          wait_or_abort(bar(Geo::kBarODone), (uint32_t)((g - 1) & 1), abort_flag));
          if (!ok) break;
          tc::fence_after_sync();
          // 32 columns per round, the next round's load in flight while
          // this one is scaled and stored
          const uint32_t orow_t = tmem + Geo::kColO + lane_base;
          auto scale32 = [&](uint32_t (&v)[32]) {
#pragma unroll
            for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
          };
          uint32_t va[32], vb[32];
          tc::tmem_ld32(orow_t, va);
          tc::tmem_wait_ld_for(va);
#pragma unroll 1
          for (int c0 = 0; c0 < D; c0 += 64) {
            tc::tmem_ld32(orow_t + (uint32_t)(c0 + 32), vb);
            scale32(va);
            tc::tmem_st32(orow_t + (uint32_t)c0, va);
            tc::tmem_wait_ld_for(vb);
            if (c0 + 64 < D) tc::tmem_ld32(orow_t + (uint32_t)(c0 + 64), va);
            scale32(vb);
            tc::tmem_st32(orow_t + (uint32_t)(c0 + 32), vb);
            if (c0 + 64 < D) tc::tmem_wait_ld_for(va);
          }
        }
        tc::tmem_wait_st();
        tc::fence_before_sync();
        warp_arrive_mma<CG>(bar(Geo::kBarPFull + st), rank);
      }
      if (!ok) break;
      // (the next tile's Q is in tensor memory: loaded at this tile's last
      // KV tile)
      TileRun<kN> nxt;
      if (k2 >= 0) {
        PrefillTile x, y;
        load_tiles<CG>(p, dealt_tile<CG>(k2), x, y);
        nxt.set(x, y);
      }
      // ---- epilogue: O / l -> bf16 rows in shared memory; then O is free
      // for the next tile's first P V, and each row goes to global memory by
      // one bulk copy of its thread (coalesced, asynchronous).
      ok = __all_sync(0xffffffffu, wait_or_abort(bar(Geo::kBarOFinal), (uint32_t)(n & 1), abort_flag));
      if (!ok) break;
      tc::fence_after_sync();
      // An attention sink joins the normaliser (the weights carry
      // 2^-(m_ref - 6)).
      // (this tile's record again, from L1: not kept in registers over the loop)
      const PrefillTile te = p.prefill_tiles[dealt_tile<CG>(k)];
      if (p.sinks && m < te.nrows && m_ref != -INFINITY) {
        const float skl = p.sinks[te.kv_head * G + (te.row0 + m) % G] * log2e;
        if (skl != -INFINITY) l_sum += exp2f(fminf(skl - m_ref + 6.0f, 126.0f));
      }
      uint16_t* const dst = out_row(te);
      const float sc = (l_sum > 0.0f ? 1.0f / l_sum : 0.0f) *
                       (Geo::kPth ? (ev > -1000 ? ldexpf(1.0f, ev) : 0.0f) : Geo::kAuto ? 1.0f : p.v_scale);
      // (the previous tile's bulk copy of this row has read its staging row)
      asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
      const uint32_t orow = base + Geo::kOffOut + (uint32_t)(m * Geo::kOutPitch);
      // 32 columns per round, the next round's load in flight while this one
      // is packed and staged
      const uint32_t orow_t = tmem + Geo::kColO + lane_base;
      auto stage32 = [&](const uint32_t (&v)[32], int c0) {
#pragma unroll
        for (int e = 0; e < 32; e += 8) {
          uint4 o;
          o.x = dev::pack_bf16x2(__uint_as_float(v[e]) * sc, __uint_as_float(v[e + 1]) * sc);
          o.y = dev::pack_bf16x2(__uint_as_float(v[e + 2]) * sc, __uint_as_float(v[e + 3]) * sc);
          o.z = dev::pack_bf16x2(__uint_as_float(v[e + 4]) * sc, __uint_as_float(v[e + 5]) * sc);
          o.w = dev::pack_bf16x2(__uint_as_float(v[e + 6]) * sc, __uint_as_float(v[e + 7]) * sc);
          sts128(orow + (uint32_t)((c0 + e) * 2), o);
        }
      };
      {
        uint32_t va[32], vb[32];
        tc::tmem_ld32(orow_t, va);
        tc::tmem_wait_ld_for(va);
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 64) {
          tc::tmem_ld32(orow_t + (uint32_t)(c0 + 32), vb);
          stage32(va, c0);
          tc::tmem_wait_ld_for(vb);
          if (c0 + 64 < D) tc::tmem_ld32(orow_t + (uint32_t)(c0 + 64), va);
          stage32(vb, c0 + 32);
          if (c0 + 64 < D) tc::tmem_wait_ld_for(va);
        }
      }
      tc::fence_before_sync();
      warp_arrive_mma<CG>(bar(Geo::kBarOFree), rank);
      if (dst) {
        tc::fence_async_smem();
        asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;\n\t"
                     "cp.async.bulk.commit_group;"
                     :: "l"(reinterpret_cast<uint64_t>(dst)), "r"(orow), "n"(D * 2) : "memory");
      }
      cur = nxt;
      k = k2;
      have = k2 >= 0;
      q_unscale = q_next;
    }
    // The rows' bulk copies are complete before the shared memory goes (and
    // a staged Q that was not used, after an abort, has landed).
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    if (staged > 0) (void)tc::mbar_wait(bar(Geo::kBarQStage), (uint32_t)((staged - 1) & 1), 200000000LL);
    // Order this warp's tensor-memory accesses before the teardown barrier.
    tc::fence_before_sync();
    __syncwarp();
  }

  // (a pair: neither CTA leaves while the other's MMAs may read its shared
  // or tensor memory, or its warps may arrive on its barriers)
  if constexpr (CG == 2)
    tc::cluster_sync();
  else
    __syncthreads();
  const bool aborted = *abort_flag != 0u;
  if (warp == 0) {
    tc::fence_after_sync();
    tc::tmem_dealloc<CG>(tmem, Geo::kTmemCols);
  }
  // A CTA that gave up a bounded wait writes NaN over every row of its
  // tiles, so its failure shows in the output even where nobody reads the
  // error word.
  if (aborted) {
    if (tid == 0) atomicExch(p.error_flag, 1);
    constexpr int kLpr = D / 8;
    constexpr int kRps = 32 / kLpr;
    const int lane = tid & 31;
    const int sub = lane / kLpr, c = lane % kLpr;
    const uint4 nan4 = make_uint4(0x7FC07FC0u, 0x7FC07FC0u, 0x7FC07FC0u, 0x7FC07FC0u);
    for (int k = 0; dealt_tile<CG>(k) < p.num_prefill_tiles; ++k) {
      const PrefillTile t = p.prefill_tiles[dealt_tile<CG>(k)];
      for (int r = warp * kRps + sub; r < t.nrows; r += (Geo::kThreads / 32) * kRps) {
        const int Rr = t.row0 + r;
        *reinterpret_cast<uint4*>(p.out + ((int64_t)(t.q0 + Rr / G) * p.heads_q + t.kv_head * G + Rr % G) * D +
                                  8 * c) = nan4;
      }
    }
  }
}

// `ctas`: CTAs wanted (one per SM, or fewer).  CTA pairs launch as clusters
// of two: max(1, ctas / 2) of them, at most as many as fit on the device at
// once (the kernel is persistent: a second wave would run its pairs' whole
// tile lists after the first).
template <int DT, int D, bool AL>
int launch_prefill_instance(const AttnParams& p, const PrefillMaps& maps, int64_t ctas,
                            cudaStream_t stream) {
  constexpr int CG = prefill_cta_group(DT, D);
  const size_t smem = prefill_smem_bytes(D, CG);
  auto kern = prefill_attention_kernel<DT, D, AL>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return KVQ_E_CUDA;
  if constexpr (CG == 1) {
    kern<<<(unsigned)ctas, prefill_threads(D), smem, stream>>>(p, maps);
  } else {
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(prefill_threads(D));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    static const int max_pairs = [&]() {
      cudaLaunchConfig_t q = cfg;
      q.gridDim = dim3(2);
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, kern, &q) != cudaSuccess) {
        cudaGetLastError();
        n = 0;
      }
      return n;
    }();
    int64_t pairs = std::max<int64_t>(1, ctas / 2);
    if (max_pairs > 0) pairs = std::min<int64_t>(pairs, max_pairs);
    cfg.gridDim = dim3((unsigned)(2 * pairs));
    if (cudaLaunchKernelEx(&cfg, kern, p, maps) != cudaSuccess) {
      cudaGetLastError();
      return KVQ_E_CUDA;
    }
  }
  return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_E_CUDA;
}

// The instances of one head_dim and one ALiBi setting (one translation unit
// each keeps the build parallel).
template <int D, bool AL>
int launch_prefill_d(const AttnParams& p, const PrefillMaps& maps, int dtype, int64_t ctas,
                     cudaStream_t stream) {
  switch (dtype) {
    case KVQ_AUTO: return launch_prefill_instance<KVQ_AUTO, D, AL>(p, maps, ctas, stream);
    case KVQ_FP8_E4M3: return launch_prefill_instance<KVQ_FP8_E4M3, D, AL>(p, maps, ctas, stream);
    case KVQ_FP8_E5M2: return launch_prefill_instance<KVQ_FP8_E5M2, D, AL>(p, maps, ctas, stream);
    case KVQ_INT8_PER_TOKEN_HEAD:
      return launch_prefill_instance<KVQ_INT8_PER_TOKEN_HEAD, D, AL>(p, maps, ctas, stream);
    case KVQ_FP8_PER_TOKEN_HEAD:
      return launch_prefill_instance<KVQ_FP8_PER_TOKEN_HEAD, D, AL>(p, maps, ctas, stream);
    case KVQ_FP8_E5M2_PER_TOKEN_HEAD:
      return launch_prefill_instance<KVQ_FP8_E5M2_PER_TOKEN_HEAD, D, AL>(p, maps, ctas, stream);
    default:
      return KVQ_E_UNSUPPORTED;
  }
}

}  // namespace kvq
