// kvq_internal.h -- definitions shared by the host scheduler and the kernels.
//
// The tile geometry lives here, in one set of constexpr functions of the KV
// cache dtype and head_dim.  The scheduler sizes shared memory and scratch
// from these functions and the kernels are instantiated from the same ones,
// so the two cannot disagree about the KV element size -- the failure of
// the vllm PR 50194 page (Motivation: tiles chosen from one element size,
// scratch sized for another, out-of-bounds writes during a large prefill).
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda.h>  // CUtensorMap

#include "../../include/kvq.h"

#ifdef __CUDACC__
#define KVQ_HD __host__ __device__
#else
#define KVQ_HD
#endif

// Bounds-checked build (-DKVQ_CHECKED=1, libkvq_checked.so): the kernels
// also check the indices they derive from device arrays the host did not
// plan from (query_start_loc's row offsets, block-table positions); an index
// outside its array sets the error word to 2 and the access is skipped.
// Never a trap: the word is read by kvq_sched_check_device.
#ifndef KVQ_CHECKED
#define KVQ_CHECKED 0
#endif

namespace kvq {

// ---- cache rows --------------------------------------------------------
KVQ_HD constexpr bool is_per_token_head(int dtype) {
  return dtype == KVQ_INT8_PER_TOKEN_HEAD || dtype == KVQ_FP8_PER_TOKEN_HEAD ||
         dtype == KVQ_FP8_E5M2_PER_TOKEN_HEAD;
}
KVQ_HD constexpr bool is_valid_dtype(int dtype) { return dtype >= 0 && dtype <= 5; }
// The code format of a quantised dtype: KVQ_FP8_E4M3, KVQ_FP8_E5M2 or
// KVQ_INT8_PER_TOKEN_HEAD (int8 codes).
KVQ_HD constexpr int code_format(int dtype) {
  return dtype == KVQ_FP8_E5M2 || dtype == KVQ_FP8_E5M2_PER_TOKEN_HEAD ? KVQ_FP8_E5M2
         : dtype == KVQ_INT8_PER_TOKEN_HEAD                          ? KVQ_INT8_PER_TOKEN_HEAD
                                                                      : KVQ_FP8_E4M3;
}
// Largest code magnitude a per-token-head scale maps the row's absmax to.
KVQ_HD constexpr float per_token_head_qmax(int dtype) {
  return dtype == KVQ_INT8_PER_TOKEN_HEAD ? 127.0f
         : dtype == KVQ_FP8_E5M2_PER_TOKEN_HEAD ? 57344.0f : 448.0f;
}
// Bytes of one cached K or V element (the KV element size).
KVQ_HD constexpr int kv_elem_bytes(int dtype) { return dtype == KVQ_AUTO ? 2 : 1; }
// Bytes of one (token, kv_head) row: codes plus, per-token-head, a 16-byte
// tail holding the fp32 scale and 12 zero bytes.
KVQ_HD constexpr int row_bytes(int dtype, int head_dim) {
  return head_dim * kv_elem_bytes(dtype) + (is_per_token_head(dtype) ? 16 : 0);
}
KVQ_HD constexpr bool head_dim_supported(int d) { return d == 64 || d == 128 || d == 256; }
// Dtypes with built attention kernels: all of them (the bf16 "auto" cache
// reads its rows as they are).
KVQ_HD constexpr bool attention_dtype_supported(int dtype) { return is_valid_dtype(dtype); }

// ---- split-KV decode kernel (stream decomposition) -------------------------
// A row tile is up to 16 packed (query token, head) rows of one kv head with
// the range of 16-token KV chunks its rows can see.  The tiles' chunks are
// laid end to end and the sequence is cut into equal contiguous segments,
// one per warp; a tile cut by a segment boundary becomes several pieces whose
// partial results are merged.  The 4 warps of a CTA are independent.
constexpr int kChunkTokens = 16;
constexpr int kDecodeWarps = 4;
constexpr int kDecodeThreads = 32 * kDecodeWarps;
constexpr int kTileMaxRows = 16;
constexpr int kRecordRing = 32;       // per-warp ring of chunk records (16 B each)
constexpr int kMinChunksPerWarp = 8;  // smallest segment worth a warp

// Bytes of one 16-token chunk of K and V codes (plus the per-token-head
// scale tails) -- what a warp loads per step, straight into registers.
KVQ_HD constexpr int decode_chunk_bytes(int dtype, int head_dim) {
  return 2 * kChunkTokens * head_dim * kv_elem_bytes(dtype) +
         (is_per_token_head(dtype) ? 32 * 16 : 0);
}
// Resident CTAs per SM the kernel is compiled for (register budget): a
// bf16 ("auto") chunk is twice the bytes of a code chunk, so its register
// lead is too.
KVQ_HD constexpr int decode_min_ctas(int dtype, int head_dim, int ntiles) {
  return dtype == KVQ_AUTO ? (head_dim >= 256 ? 1 : head_dim >= 128 ? 3 : 4)
                           : (head_dim >= 256 ? 2 : (ntiles == 1 ? 4 : 3));
}
// Shared memory: only each warp's ring of chunk records.
KVQ_HD constexpr size_t decode_warp_smem(int dtype, int head_dim) {
  return (size_t)kRecordRing * 16;
}
KVQ_HD constexpr size_t decode_smem_bytes(int dtype, int head_dim) {
  return (size_t)kDecodeWarps * decode_warp_smem(dtype, head_dim);
}

// ---- tensor-core prefill kernel -----------------------------------------
// A prefill tile is 128 packed (query token, head) rows of one kv head; its
// keys stream through in tiles of 64.  Requests whose rows per kv head
// exceed kTileMaxRows go to this kernel.
constexpr int kPrefillRows = 128;
constexpr int kPrefillStages = 2;        // K / V^T tiles in flight
// Threads of a prefill CTA: 1 MMA warp, 4 softmax warps, 1 copy warp and
// the converter warps.  16 warps of at most 128 registers (the SM's 65,536)
// at head_dim 64 and 128; at head_dim 256 the softmax and converters need
// more registers than that without spilling, so 12 warps.
KVQ_HD constexpr int prefill_threads(int head_dim) { return head_dim >= 256 ? 384 : 512; }
KVQ_HD constexpr int prefill_conv_threads(int head_dim) { return prefill_threads(head_dim) - 6 * 32; }
// Keys per KV tile: 128, or 64 at head_dim 256 (shared memory).
KVQ_HD constexpr int prefill_keys(int head_dim) { return head_dim >= 256 ? 64 : 128; }
// Tensor-memory columns: O (head_dim fp32), two S buffers (keys fp32 each,
// P in f16 pairs over the first half), Q (head_dim / 2 columns of f16
// pairs); always 512.
KVQ_HD constexpr int prefill_tmem_cols(int /*head_dim*/) { return 512; }
// Side-data slots of the prefill (per-key scales, chunk mask, largest value
// scale): KV tile g uses slot g % 4, so the converters may run two tiles
// ahead of the softmax.
constexpr int kPrefillSideSlots = 4;
// Slot tables of the prefill's KV tiles (first slot of each 16-key chunk and
// the chunk mask), published by the copy warp up to 4 tiles ahead.
constexpr int kPrefillSlotRing = 4;
// CTA pairs for the prefill (-DKVQ_PREFILL_PAIR=1; measured slower than
// single CTAs on the prefill workloads, so off by default).
#ifndef KVQ_PREFILL_PAIR
#define KVQ_PREFILL_PAIR 0
#endif
// CTAs per tile MMA: quantised caches at head_dim 128 and 256 run on CTA
// pairs (cta_group::2, M = 256: two 128-row tiles of one kv head share each
// converted KV tile, each CTA converting half of it); bf16 caches and
// head_dim 64 (a V half of 32 dims is narrower than the 128-byte swizzle)
// on single CTAs.
KVQ_HD constexpr int prefill_cta_group(int dtype, int head_dim) {
  return KVQ_PREFILL_PAIR && dtype != KVQ_AUTO && head_dim >= 128 ? 2 : 1;
}
// Shared memory: 2 x K and 2 x V (keys x D f16 each, halves for a pair); 4 x
// the tile's key / value scales; 4 x the tile's chunk mask and per-warp
// largest value scales (144 bytes); 4 x 64-byte slot tables; the finished
// tile's O rows (128 x (D * 2 + 16) bytes); barriers and flags (512 bytes);
// +1 KB for 1024-byte alignment.  (The codes go from global memory to the
// converters' registers, Q from global memory to tensor memory.)
KVQ_HD constexpr size_t prefill_smem_bytes(int head_dim, int cta_group = 1) {
  return 2 * (size_t)kPrefillStages * prefill_keys(head_dim) * head_dim * 2 / cta_group +
         (size_t)kPrefillSideSlots * prefill_keys(head_dim) * 8 + 144 + kPrefillSlotRing * 64 +
         (size_t)kPrefillRows * (head_dim * 2 + 16) + 512 + 1024;
}

// Tensor maps of bf16 ("auto") caches for the prefill's bulk tensor copies:
// a cache is a rank-3 bf16 tensor {head_dim, kv heads, slots} copied in
// boxes of {64, 1, 16 slots} in the 128-byte swizzle.
struct PrefillMaps {
  CUtensorMap k, v;
};

struct PrefillTile {
  int32_t req, kv_head, row0, nrows;
  int32_t kv_lo, kv_hi;  // keys some row of the tile can see
  int32_t q0;            // the request's first query token (query_start_loc[req])
  int32_t pos0;          // position of its query 0: L - Q
};
static_assert(sizeof(PrefillTile) == 32, "PrefillTile layout");

// One piece of a row tile (32 bytes).
struct DecodePiece {
  int32_t req;       // request index
  int32_t kv_head;   // kv head
  int32_t row0;      // first packed row: row = q_index * G + (head % G)
  int32_t nrows;     // rows in the tile, 1..16
  int32_t part;      // -1: write `out`; else first partial row in workspace
  int32_t merge;     // merge item of a split tile (-1: not split)
  int32_t any_lo;    // keys some row of the tile can see: [any_lo, any_hi)
  int32_t any_hi;
  int32_t flat0;     // position of the piece's first chunk in its launch's flat sequence
  int32_t chunk0;    // that chunk's 16-token index in the request
  int32_t pad0, pad1;
};
static_assert(sizeof(DecodePiece) == 48, "DecodePiece layout");

// One decode warp's work: the segment [seg0, seg0 + n) of its launch's flat
// chunk sequence and the piece holding chunk seg0.
struct WarpSeg {
  int32_t piece, seg0, n, pad;
};
static_assert(sizeof(WarpSeg) == 16, "WarpSeg layout");

// One merge item: the partial rows of a tile that was split along KV.
struct MergeItem {
  int32_t req, kv_head, row0, nrows;
  int32_t part;      // partial row of (split 0, row 0); split s row n at
                     // part + s * nrows + n
  int32_t nsplits;
  int32_t pad0, pad1;
};
static_assert(sizeof(MergeItem) == 32, "MergeItem layout");

// Workspace layout: partial outputs [P][head_dim] fp32, then partial
// log2-sum-exp [P] fp32, each 256-byte aligned.
KVQ_HD constexpr size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }
KVQ_HD constexpr size_t workspace_o_bytes(int64_t partial_rows, int head_dim) {
  return align256((size_t)partial_rows * head_dim * 4);
}
KVQ_HD constexpr size_t workspace_bytes(int64_t partial_rows, int head_dim) {
  return partial_rows == 0 ? 0
                           : workspace_o_bytes(partial_rows, head_dim) +
                                 align256((size_t)partial_rows * 4);
}

// Kernel arguments of the attention kernels (passed by value).
struct AttnParams {
  const uint16_t* q;           // bf16 [sum Q, Hq, D]
  const uint8_t* key_cache;    // [NB, B, Hkv, row]
  const uint8_t* value_cache;
  const int32_t* query_start_loc;
  const int32_t* seq_lens;
  const int32_t* block_table;
  uint16_t* out;               // bf16 [sum Q, Hq, D]
  float* part_o;               // [P, D]
  float* part_lse;             // [P]
  const DecodePiece* pieces;   // this launch's pieces, in flat order
  int32_t num_pieces;
  const struct WarpSeg* warp_seg;  // per warp: its segment and the piece of its first chunk
  int64_t num_chunks;          // length of the launch's flat chunk sequence
  int num_warps;               // warps it is cut among (grid * kDecodeWarps)
  const MergeItem* merges;
  const PrefillTile* prefill_tiles;
  int32_t num_prefill_tiles;
  int32_t total_q_tokens;      // rows of q and out (the host plan's sum Q)
  int32_t* error_flag;         // 1: a bounded wait timed out; 2: an index outside its array
  int64_t num_blocks;
  int block_table_stride;
  int block_size;
  int heads_q, heads_kv, group;  // group = Hq / Hkv
  int causal, window;
  float sm_scale, soft_cap, k_scale, v_scale;
  const float* alibi_slopes;   // [Hq] or null: score += slope * (key - query position)
  const float* sinks;          // [Hq] or null: one extra logit in the softmax normaliser
};

// ---- fused decode step (cache write + device-built plan + decode) --------
// Extra kernel arguments of the fused step: the new tokens' rows for the
// cache write and the plan the kernel builds in its workspace.  Each
// (request, kv head) is one row tile of the request's Q * G <= 16 rows.
struct StepParams {
  const uint16_t* key;          // bf16 [num_tokens, Hkv, D] (token stride given)
  const uint16_t* value;
  int64_t num_tokens, key_stride, value_stride;
  const int64_t* slot_mapping;  // [num_tokens]
  uint8_t* key_cache;           // the caches the attention reads, writable
  uint8_t* value_cache;
  int64_t num_slots;            // num_blocks * block_size
  int32_t* prefix;              // [num_tiles + 1]: flat index of each tile's first chunk
  int4* tiles;                  // [num_tiles]: {first chunk, key_lo, key_hi, rows}
  int32_t* warp_tile;           // [warps]: the tile holding each warp's first chunk
  uint32_t* barrier;            // [2]: arrivals, generation (grid barrier)
  int num_req, num_tiles;       // num_tiles = num_req * Hkv
  int max_rows;                 // 8 or 16: rows per tile the launch is built for
  // The lengths as read before the grid barrier (the plan; the merge reads
  // query_start_loc before it waits): AttnParams' own pointers, or their
  // host mappings when the kernel stages the inputs itself.
  const int32_t* in_query_start_loc;
  const int32_t* in_seq_lens;
  // Staged inputs: stage_bytes copied from a mapped host buffer to the device
  // buffer the attention reads after the barrier (by every CTA but the
  // planner); 0 when the inputs are already on the device.
  const uint8_t* stage_src;
  uint8_t* stage_dst;
  int64_t stage_bytes;
};

// Workspace of the fused step for `warps` decode warps: an error word and
// the grid barrier's two words (256 bytes), the prefix, the tile table, each
// warp's first tile, then partial log-sum-exps and outputs: each warp owns
// two 16-row slots (the tile its segment starts in and the one it ends in).
struct StepWorkspace {
  size_t prefix, tiles, warp_tile, lse, o, total;
};
KVQ_HD constexpr StepWorkspace step_workspace(int num_tiles, int head_dim, int64_t warps) {
  StepWorkspace w{};
  w.prefix = 256;
  w.tiles = w.prefix + align256((size_t)(num_tiles + 1) * 4);
  w.warp_tile = w.tiles + align256((size_t)num_tiles * 16);
  w.lse = w.warp_tile + align256((size_t)warps * 4);
  w.o = w.lse + align256((size_t)warps * 2 * kTileMaxRows * 4);
  w.total = w.o + (size_t)warps * 2 * kTileMaxRows * head_dim * 4;
  return w;
}
// Largest num_req * heads_kv of one fused step.
constexpr int kMaxStepTiles = 1 << 16;
// Devices whose launch configuration the host code keeps (others query it
// on every call).
constexpr int kMaxCachedDevices = 64;

}  // namespace kvq

// Launchers (defined in the .cu files; return KVQ_OK or KVQ_E_CUDA).
namespace kvq {
int launch_reshape_and_cache(const void* key, const void* value,
                             int64_t num_tokens, int64_t key_stride,
                             int64_t value_stride, int num_heads_kv,
                             int head_dim, void* key_cache, void* value_cache,
                             int64_t num_blocks, int block_size,
                             const int64_t* slot_mapping, int dtype,
                             float k_scale, float v_scale, void* stream);
int launch_decode(const AttnParams& p, int dtype, int head_dim, int ntiles, void* stream);
// The fused step's kernel (cooperative launch of `warps` / 4 CTAs); `warps`
// from step_warps().
int launch_decode_step(const AttnParams& p, const StepParams& sp, int dtype, int head_dim,
                       int64_t warps, void* stream);
// Decode warps of the fused step's grid on the current device (every CTA
// resident at once) in *warps; KVQ_OK or a KVQ_E_* status.
int step_warps(int dtype, int head_dim, bool alibi, int max_rows, int64_t* warps);
// The merge of the decode's cut tiles (p.merges, one CTA each), after the
// decode kernels of a host-planned call.
int launch_merge(const AttnParams& p, int head_dim, int64_t num_merges, void* stream);
// The fused step's merge of its cut tiles: one CTA per tile of the device
// plan (tiles left whole return at once), a programmatic dependent of the
// fused kernel, whose `warps` warps cut the chunk sequence.
int launch_merge_step(const AttnParams& p, const StepParams& sp, int head_dim, int64_t warps,
                      void* stream);
// The persistent prefill over p.num_prefill_tiles tiles on `ctas` CTAs
// (at most one per SM is resident).
int launch_prefill(const AttnParams& p, const PrefillMaps& maps, int dtype, int head_dim,
                   int64_t ctas, void* stream);
// Whether a launch needs the ALiBi instances of the kernels.
inline bool uses_alibi(const AttnParams& p) { return p.alibi_slopes != nullptr; }
}  // namespace kvq
