// kvq_decode.cuh -- split-KV attention over the quantised paged cache for
// small row tiles (decode: the query token(s) x G heads of one kv head).
//
// What it computes: for each packed row (query token, q head) of a tile,
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
//   * Work: the tiles' 16-token chunks are laid end to end and cut into equal
//     contiguous segments, one per warp (a stream-K split of the KV axis).
//     Every warp is independent: it streams its segment, writes each tile's
//     output (or partial, for a tile cut by a segment boundary) straight from
//     registers, and the last piece of a cut tile to finish merges it.  No
//     barriers, no shared-memory combine, no per-CTA start-up per tile.
//   * HBM bound: every K/V byte is read once; no dequantised copy is
//     written.  Each lane loads its own bytes of the next chunk straight into
//     registers with 16-byte streaming loads (every load instruction covers
//     whole 32-byte sectors), one chunk ahead of the MMAs.  On GB300 this
//     path streams the paged rows faster than cp.async or bulk copies into
//     shared memory (measured: about 4.8-4.9 vs 3.9-4.0 TB/s for the
//     decode batch's access pattern with no compute).  Block lookups and
//     visibility masks are prepared 16-32 chunks ahead in a small per-warp
//     record ring in shared memory, so no load waits on the block table.
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
//   * Online softmax in log2 units with warp shuffles; pieces of a tile are
//     merged with the log-sum-exp rule.
#pragma once

#include <cuda_runtime.h>

#include <atomic>

#include "kvq_cache_row.cuh"
#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {

template <int DT, int D>
struct DecodeGeom {
  static constexpr bool kAuto = DT == KVQ_AUTO;  // bf16 rows, bf16 MMAs
  static constexpr int kEB = kv_elem_bytes(DT);
  static constexpr int kKsteps = D / 16;     // MMA k-steps over head_dim (QK)
  static constexpr int kMtiles = D / 16;     // MMA m-tiles over head_dim (PV)
  static constexpr int kK16 = D * kEB / 64;  // 16-byte K pieces per lane per row
  static constexpr int kVBytes = D * kEB / 8;  // V bytes per lane per row
  static constexpr int kVPieces = kVBytes >= 16 ? kVBytes / 16 : 1;
  static constexpr int kVSlots = D / 32;     // 16-byte V slots per lane
  static constexpr bool kPth = is_per_token_head(DT);
  static constexpr int kRow = row_bytes(DT, D);
  static constexpr int kWarpSmem = kRecordRing * 16;
  static_assert((size_t)kWarpSmem == decode_warp_smem(DT, D), "warp smem must follow the geometry");
};

// Head dim of element k (0: MMA row g, 1: row g + 8) of P.V m-tile mi for a
// lane of group g: each lane owns 16-byte runs of every V row (8 bytes for
// head_dim 64), the runs of the 8 groups side by side.  A 16-byte run is 16
// codes (two per m-tile) or, for bf16 rows, 8 values (two per m-tile).
template <int DT, int D>
__device__ __forceinline__ int pv_dim(int mi, int g, int k) {
  if constexpr (DT == KVQ_AUTO) {
    return (mi / 4) * 64 + g * 8 + 2 * (mi % 4) + k;
  } else {
    constexpr int run = D / 8 >= 16 ? 16 : D / 8;
    return (mi / 8) * 128 + g * run + 2 * (mi % 8) + k;
  }
}

// ---- fused decode step: the plan built on the device ----------------------
// One row tile per (request, kv head): its first 16-token chunk, the keys
// some of its rows see and its rows; the tiles' chunk counts are
// prefix-summed by the kernel's first CTA (kDecodeThreads threads).  A
// request with more rows than the launch was built for (or more queries
// than keys) is left out and flags the error word.  (The lengths are read
// where the step's inputs are before the barrier: host memory when the
// kernel stages them.  Issuing a batch of tiles' loads together measured
// slower, also from host memory.)
__device__ __forceinline__ void plan_step(const AttnParams& p, const StepParams& sp) {
  __shared__ int32_t warp_sums[kDecodeWarps];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nt = sp.num_tiles;
  const int per = (nt + kDecodeThreads - 1) / kDecodeThreads;
  const int t0 = min(nt, tid * per), t1 = min(nt, t0 + per);
  // A thread's tiles are consecutive, mostly the kv heads of one request:
  // the last request's lengths stay in registers.
  int last_r = -1, last_q = 0, last_l = 0;
  auto chunks_of = [&](int t, bool store) {
    const int r = t / p.heads_kv;
    if (r != last_r) {
      last_r = r;
      last_q = sp.in_query_start_loc[r + 1] - sp.in_query_start_loc[r];
      last_l = sp.in_seq_lens[r];
    }
    const int Q = last_q;
    const int L = last_l;
    const int rows = Q * p.group;
    if (Q <= 0 || L < Q || rows > sp.max_rows) {
      if (store) {
        if (Q != 0) atomicExch(p.error_flag, 2);  // (1 is the barrier's timeout)
        sp.tiles[t] = make_int4(0, 0, 0, 0);
      }
      return 0;
    }
    const int lo = p.window > 0 ? max(0, L - Q - p.window + 1) : 0;
    if (store) sp.tiles[t] = make_int4(lo / kChunkTokens, lo, L, rows);
    return (L + kChunkTokens - 1) / kChunkTokens - lo / kChunkTokens;
  };
  int local = 0;
  for (int t = t0; t < t1; ++t) local += chunks_of(t, true);
  // exclusive scan of the threads' sums
  int incl = local;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += v;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  int run = incl - local;
  for (int w = 0; w < warp; ++w) run += warp_sums[w];
  for (int t = t0; t < t1; ++t) {
    sp.prefix[t] = run;
    run += chunks_of(t, false);
  }
  __shared__ int32_t total;
  if (tid == kDecodeThreads - 1) {
    sp.prefix[nt] = run;
    total = run;
  }
  __syncthreads();
  // Each warp's first tile: warp w's segment starts at floor(w T / W), which
  // lies in tile t for w in [ceil(f0 W / T), ceil(f1 W / T)).
  const int64_t T = total, W = (int64_t)gridDim.x * kDecodeWarps;
  if (T > 0) {
    int64_t f0 = t0 < t1 ? sp.prefix[t0] : 0;  // (this thread's own stores)
    for (int t = t0; t < t1; ++t) {
      const int64_t f1 = t + 1 < t1 ? sp.prefix[t + 1] : (t + 1 == nt ? T : f0 + chunks_of(t, false));
      for (int64_t w = (f0 * W + T - 1) / T; w < (f1 * W + T - 1) / T && w < W; ++w)
        sp.warp_tile[w] = t;
      f0 = f1;
    }
  }
}

// Staged inputs: every CTA but the planner (CTA 0, unless it is alone)
// copies 16 bytes a thread from the mapped host buffer to the device one.
// The loads are issued before the cache write and stored after it, so the
// two host round trips overlap.
constexpr int kStageRegs = 2;
struct StageLane {
  bool on;
  int64_t i0, step, n16;
  uint4 v[kStageRegs];
};
__device__ __forceinline__ void stage_issue(const StepParams& sp, StageLane& st) {
  st.on = sp.stage_bytes > 0 && !(gridDim.x > 1 && blockIdx.x == 0);
  if (!st.on) return;
  const int64_t ctas = gridDim.x > 1 ? gridDim.x - 1 : 1;
  const int64_t cta = gridDim.x > 1 ? blockIdx.x - 1 : 0;
  st.i0 = cta * kDecodeThreads + threadIdx.x;
  st.step = ctas * kDecodeThreads;
  st.n16 = sp.stage_bytes >> 4;
  const uint4* src = reinterpret_cast<const uint4*>(sp.stage_src);
#pragma unroll
  for (int k = 0; k < kStageRegs; ++k) {
    const int64_t i = st.i0 + k * st.step;
    if (i < st.n16) st.v[k] = src[i];
  }
}
__device__ __forceinline__ void stage_finish(const StepParams& sp, const StageLane& st) {
  if (!st.on) return;
  const uint4* src = reinterpret_cast<const uint4*>(sp.stage_src);
  uint4* dst = reinterpret_cast<uint4*>(sp.stage_dst);
#pragma unroll
  for (int k = 0; k < kStageRegs; ++k) {
    const int64_t i = st.i0 + k * st.step;
    if (i < st.n16) dst[i] = st.v[k];
  }
  for (int64_t i = st.i0 + kStageRegs * st.step; i < st.n16; i += st.step) dst[i] = src[i];
  // the tail of a size that is not a multiple of 16
  for (int64_t b = (st.n16 << 4) + st.i0; b < sp.stage_bytes; b += st.step)
    sp.stage_dst[b] = sp.stage_src[b];
}

// Grid-wide barrier of a cooperative launch (every CTA resident): arrival
// count and generation in global memory; the last CTA to arrive resets the
// count and advances the generation.  Bounded: a CTA that waits about a
// second flags the error word and the call gives up.
__device__ __forceinline__ bool grid_barrier(uint32_t* bar, int32_t* error_flag) {
  __syncthreads();
  int ok = 1;
  if (threadIdx.x == 0) {
    volatile uint32_t* gen = bar + 1;
    const uint32_t g0 = *gen;
    __threadfence();
    const uint32_t prev = atomicAdd(bar, 1u);
    if (prev == gridDim.x - 1) {
      atomicExch(bar, 0u);
      __threadfence();
      atomicAdd(bar + 1, 1u);
    } else {
      const long long t0 = clock64();
      while (*gen == g0) {
        if (clock64() - t0 > 2000000000LL) {  // about a second
          ok = 0;
          atomicExch(error_flag, 1);
          break;
        }
      }
    }
    __threadfence();
  }
  return __syncthreads_and(ok) != 0;
}

// DEV: the fused decode step -- the new tokens are written to the caches,
// the plan is built from the device's lengths (and, when the inputs come
// from a mapped host buffer, that buffer is copied to the device), and a
// grid barrier separates all of it from the attention (which then reads the
// caches with coherent loads).
template <int DT, int D, int NT, bool AL, bool DEV>
__global__ void __launch_bounds__(kDecodeThreads, decode_min_ctas(DT, D, NT))
splitkv_decode_kernel(const AttnParams p, const StepParams sp) {
  using Geo = DecodeGeom<DT, D>;
  extern __shared__ __align__(128) uint8_t smem[];
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int g = lane >> 2;
  const int c = lane & 3;

  // The merge of the cut tiles (its own kernel, after this one) may be
  // scheduled now: it waits for this grid to complete before it reads a
  // partial row.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // ---- the fused step's prologue -------------------------------------------
  int64_t total_chunks = p.num_chunks;
  int64_t total_warps = p.num_warps;
  if constexpr (DEV) {
    StageLane st;
    stage_issue(sp, st);
    row::write_rows<DT, D>(sp.key, sp.value, sp.num_tokens, sp.key_stride, sp.value_stride,
                           p.heads_kv, sp.key_cache, sp.value_cache, sp.num_slots,
                           sp.slot_mapping, p.k_scale, p.v_scale, kDecodeThreads, threadIdx.x,
                           blockIdx.x, gridDim.x);
    stage_finish(sp, st);
    if (blockIdx.x == 0) plan_step(p, sp);
    if (!grid_barrier(sp.barrier, p.error_flag)) return;
    total_chunks = __ldcg(sp.prefix + sp.num_tiles);
    total_warps = (int64_t)gridDim.x * kDecodeWarps;
  }
  auto load16 = [&](const void* a) {
    if constexpr (DEV) return dev::ldg_stream_coherent(a);
    else return dev::ldg_stream(a);
  };

  // ---- this warp's segment of the flat chunk sequence -------------------
  // (host plan: from the schedule's warp table; fused step: equal cuts)
  const int gw = blockIdx.x * kDecodeWarps + warp;
  int64_t seg0;
  int n;
  int first_piece = 0;
  if constexpr (DEV) {
    seg0 = (int64_t)gw * total_chunks / total_warps;
    n = (int)((int64_t)(gw + 1) * total_chunks / total_warps - seg0);
  } else {
    const WarpSeg ws = p.warp_seg[gw];
    seg0 = ws.seg0;
    n = ws.n;
    first_piece = ws.piece;
  }
  // The piece of each position: the warp's first piece comes from the
  // schedule; a lane's cursor only moves forward as its positions grow.
  // (Fused step: the pieces are the tiles themselves -- the part of a tile
  // inside this warp's segment -- found in the device-built prefix.)
  uint4* records = reinterpret_cast<uint4*>(smem + warp * Geo::kWarpSmem);

  const uint8_t* kbase = p.key_cache;
  const uint8_t* vbase = p.value_cache;
  const int64_t row_stride = (int64_t)p.heads_kv * Geo::kRow;  // bytes between tokens
  const uint32_t rs = (uint32_t)row_stride;
  const int cpb = p.block_size / kChunkTokens;                 // chunks per cache block
  // Byte offsets, from a chunk's first row of the head, of what this lane
  // copies: K rows g, g+8 at bytes 64i + 16c (piece i); V rows 2c, 2c+1,
  // 2c+8, 2c+9 at bytes 128i + 16g (8g for head_dim 64); the scale tail of
  // K row g (c=0), K row g+8 (c=1), V row g (c=2) or V row g+8 (c=3).
  const uint32_t koff0 = g * rs + 16 * c;
  const uint32_t koff1 = koff0 + 8 * rs;
  uint32_t voff[4];
#pragma unroll
  for (int vr = 0; vr < 4; ++vr)
    voff[vr] = (2 * c + (vr & 1) + 8 * (vr >> 1)) * rs + g * (Geo::kVBytes >= 16 ? 16 : Geo::kVBytes);
  const uint32_t toff = (g + 8 * (c & 1)) * rs + D;

  // ---- chunk records: {slot of the chunk's first row (-1: no block),
  // first token, piece, visible-row mask | kv_head << 16}, built by lanes
  // 0-15 for 16 positions at a time in three steps a few chunks apart so
  // that the dependent loads (chunk ref -> piece -> block table) overlap
  // with the streaming; the first 32 positions before streaming starts.
  int f_piece = -1, f_chunk = 0;
  int cur_piece = 0;
  if constexpr (DEV) {
    if (n > 0) cur_piece = __ldcg(sp.warp_tile + gw);  // the tile holding position seg0
  } else {
    cur_piece = n > 0 ? first_piece : 0;
  }
  int4 f_pc = make_int4(0, 0, 0, 0);  // req, kv_head, any_lo, any_hi
  int f_blk = -1;
  auto fill_load_ref = [&](int pos, int lanes) {
    f_piece = -1;
    if (lane < lanes && pos + lane < n) {
      const int64_t flat = seg0 + pos + lane;
      if constexpr (DEV) {
        while (cur_piece + 1 < sp.num_tiles && (int64_t)__ldcg(sp.prefix + cur_piece + 1) <= flat)
          ++cur_piece;
        f_piece = cur_piece;
        f_chunk = __ldcg(&sp.tiles[cur_piece].x) + (int)(flat - __ldcg(sp.prefix + cur_piece));
      } else {
        while (cur_piece + 1 < p.num_pieces &&
               (int64_t)__ldg(&p.pieces[cur_piece + 1].flat0) <= flat)
          ++cur_piece;
        f_piece = cur_piece;
        f_chunk = __ldg(&p.pieces[cur_piece].chunk0) + (int)(flat - __ldg(&p.pieces[cur_piece].flat0));
      }
    }
  };
  auto fill_load_piece = [&]() {
    if (f_piece >= 0) {
      if constexpr (DEV) {
        const int4 ti = __ldcg(sp.tiles + f_piece);
        f_pc = make_int4(f_piece / p.heads_kv, f_piece % p.heads_kv, ti.y, ti.z);
      } else {
        const DecodePiece* pc = p.pieces + f_piece;
        f_pc = make_int4(pc->req, pc->kv_head, pc->any_lo, pc->any_hi);
      }
    }
  };
  auto fill_load_block = [&]() {
    f_blk = -1;
    // (the fused step's table width is not known on the host: check it here;
    // the bounds-checked build checks the host plan's positions too)
    if (f_piece >= 0) {
      const bool in_table = f_chunk / cpb < p.block_table_stride;
      if constexpr (KVQ_CHECKED && !DEV)
        if (!in_table) atomicExch(p.error_flag, 2);
      if (!(DEV || KVQ_CHECKED) || in_table)
        f_blk = p.block_table[(int64_t)f_pc.x * p.block_table_stride + f_chunk / cpb];
    }
  };
  auto fill_store = [&](int pos, int lanes) {
    if (lane < lanes && pos + lane < n) {
      const int chunk = f_chunk;
      const int tok0 = chunk * kChunkTokens;
      const bool ok = f_blk >= 0 && (int64_t)f_blk < p.num_blocks;
      const int slot0 = ok ? f_blk * p.block_size + (chunk % cpb) * kChunkTokens : -1;
      const int lo = min(max(f_pc.z - tok0, 0), kChunkTokens);
      const int hi = min(max(f_pc.w - tok0, 0), kChunkTokens);
      const uint32_t live = ok ? (((1u << hi) - 1u) & ~((1u << lo) - 1u)) : 0u;
      records[(pos + lane) % kRecordRing] =
          make_uint4((uint32_t)slot0, (uint32_t)tok0, (uint32_t)f_piece,
                     live | ((uint32_t)f_pc.y << 16));
    }
  };
  // Positions [0, 32) are prepared before streaming starts: one per lane
  // (the fused step walks its device prefix per lane: 16 at a time there).
  if constexpr (DEV) {
#pragma unroll
    for (int b = 0; b < 2; ++b) {
      fill_load_ref(16 * b, 16);
      fill_load_piece();
      fill_load_block();
      fill_store(16 * b, 16);
    }
  } else {
    fill_load_ref(0, 32);
    fill_load_piece();
    fill_load_block();
    fill_store(0, 32);
  }
  __syncwarp();

  // K and V codes of the next chunk are loaded straight into registers
  // (16-byte streaming loads), K right after the current chunk's Q K^T has
  // consumed its K registers and V right after P V: one chunk of lead, no
  // shared-memory staging.  Rows outside the visible range (or a missing
  // block) read as zeros.
  uint4 kreg[2][Geo::kK16];
  uint4 vreg[4][Geo::kVPieces];
  uint4 treg = make_uint4(0, 0, 0, 0);  // per-token-head scale tail (see toff)
  int nx_tok = 0, nx_piece = -1;         // record of the chunk whose K is loaded
  bool nx_ok = false;
  uint32_t nx_live = 0;
  int64_t nx_base = 0;
  auto load_k = [&](int q) {
    const uint4 rec = records[q % kRecordRing];
    nx_ok = (int)rec.x >= 0;
    nx_tok = (int)rec.y;
    nx_piece = (int)rec.z;
    nx_live = rec.w & 0xFFFFu;
    nx_base = nx_ok ? (int64_t)(int)rec.x * row_stride + (rec.w >> 16) * Geo::kRow : 0;
    const uint8_t* kchunk = kbase + nx_base;
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      const bool lv = (nx_live >> (g + 8 * rr)) & 1u;
#pragma unroll
      for (int i = 0; i < Geo::kK16; ++i)
        kreg[rr][i] = lv ? load16(kchunk + (rr ? koff1 : koff0) + 64 * i) : make_uint4(0, 0, 0, 0);
    }
    if constexpr (Geo::kPth) {
      const bool lv = (nx_live >> (g + 8 * (c & 1))) & 1u;
      treg = lv ? load16((c < 2 ? kbase : vbase) + nx_base + toff) : make_uint4(0, 0, 0, 0);
    }
  };
  auto load_v = [&]() {  // V codes of the chunk whose K was loaded last
    const uint8_t* vchunk = vbase + nx_base;
#pragma unroll
    for (int vr = 0; vr < 4; ++vr) {
      const bool lv = (nx_live >> (2 * c + (vr & 1) + 8 * (vr >> 1))) & 1u;
      if constexpr (Geo::kVBytes == 8) {
        uint2 w = make_uint2(0, 0);
        if (lv) w = *reinterpret_cast<const uint2*>(vchunk + voff[vr]);
        vreg[vr][0] = make_uint4(w.x, w.y, 0, 0);
      } else {
#pragma unroll
        for (int i = 0; i < Geo::kVPieces; ++i)
          vreg[vr][i] = lv ? load16(vchunk + voff[vr] + 128 * i) : make_uint4(0, 0, 0, 0);
      }
    }
  };

  if (n > 0) {
    load_k(0);
    load_v();
  }

  // ---- per-piece state ---------------------------------------------------
  const float log2e = 1.4426950408889634f;
  const float base_scale = p.sm_scale * (p.soft_cap > 0.0f ? 1.0f : log2e);
  const float cap = p.soft_cap;
  const float cap_l2 = cap * log2e;
  const float inv_cap = cap > 0.0f ? 1.0f / cap : 0.0f;
  const int G = p.group;
  const int W = p.window;
  int cur = -1;                 // current piece
  DecodePiece pc;               // its descriptor
  bool piece_bad = false;       // (bounds-checked build) its rows lie outside q / out
  int q0 = 0, all_lo = 0, all_hi = 0;
  int col_lo[NT][2], col_hi[NT][2];
  float score_mul = 0.0f;
  uint32_t qf[NT][Geo::kKsteps][2];
  float o[NT][Geo::kMtiles][4];
  float m_run[NT][2], l_run[NT][2];
  int ev = -1000;
  // ALiBi: per column, the slope in log2 units and the query position.
  float al_slope[NT][2];
  int al_pos[NT][2];

  // Start a piece: Q fragments (B operand of S^T = K Q^T) and masks.  Q
  // enters the MMA exactly: bf16 values scaled by a power of two only (8
  // significant bits fit f16's 11); sm_scale and log2(e) are applied to the
  // fp32 scores.  Lane c holds dims 64i + 16c + [0, 16) of its rows.
  auto start_piece = [&](int piece) {
    if constexpr (DEV) {
      // The tile's part inside this warp's segment; a cut tile's partial
      // rows go to one of the warp's two 16-row slots: 2 gw for the tile the
      // segment starts in, 2 gw + 1 for the one it ends in.
      const int4 ti = __ldcg(sp.tiles + piece);
      const int64_t f0 = __ldcg(sp.prefix + piece), f1 = __ldcg(sp.prefix + piece + 1);
      const bool cut = f0 < seg0 || f1 > seg0 + n;
      pc.req = piece / p.heads_kv;
      pc.kv_head = piece % p.heads_kv;
      pc.row0 = 0;
      pc.nrows = ti.w;
      pc.part = cut ? (2 * gw + (f0 <= seg0 ? 0 : 1)) * kTileMaxRows : -1;
      pc.merge = piece;
      pc.any_lo = ti.y;
      pc.any_hi = ti.z;
      pc.flat0 = (int32_t)f0;
      pc.chunk0 = ti.x;
    } else {
      pc = p.pieces[piece];
    }
    q0 = p.query_start_loc[pc.req];
    if constexpr (KVQ_CHECKED && !DEV) {
      // the piece's rows must lie in q and out (the device offsets are the
      // caller's copy of the planned ones)
      piece_bad = q0 < 0 || q0 + (pc.row0 + pc.nrows - 1) / G >= p.total_q_tokens;
      if (piece_bad && lane == 0) atomicExch(p.error_flag, 2);
    }
    const int Q = p.query_start_loc[pc.req + 1] - q0;
    const int L = p.seq_lens[pc.req];
    const int p_min = L - Q + pc.row0 / G;
    const int p_max = L - Q + (pc.row0 + pc.nrows - 1) / G;
    all_lo = W > 0 ? p_max - W + 1 : 0;
    all_hi = p.causal ? p_min + 1 : L;
    float q_unmul = 1.0f;
    if constexpr (Geo::kAuto) {
      // bf16 rows: Q enters the bf16 MMA as it is.  Lane c holds dims
      // 32i + 8c + [0, 8) of its rows (k-steps 2i and 2i + 1).
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        const int nr = 8 * t + g;
        const bool valid = nr < pc.nrows && !piece_bad;
        const int R = pc.row0 + (valid ? nr : 0);
        const int tok = q0 + R / G;
        const int head = pc.kv_head * G + R % G;
        const uint16_t* src = p.q + ((int64_t)tok * p.heads_q + head) * D + 8 * c;
#pragma unroll
        for (int i = 0; i < D / 32; ++i) {
          const uint4 w = valid ? *reinterpret_cast<const uint4*>(src + 32 * i) : make_uint4(0, 0, 0, 0);
          qf[t][2 * i][0] = w.x;
          qf[t][2 * i][1] = w.y;
          qf[t][2 * i + 1][0] = w.z;
          qf[t][2 * i + 1][1] = w.w;
        }
      }
    } else {
    float qv[NT][D / 4];
    float qmax = 0.0f;
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const int nr = 8 * t + g;
      const bool valid = nr < pc.nrows && !piece_bad;
      const int R = pc.row0 + (valid ? nr : 0);
      const int tok = q0 + R / G;
      const int head = pc.kv_head * G + R % G;
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
    q_unmul = __int_as_float((127 - shift) << 23);
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
      for (int j = 0; j < Geo::kKsteps; ++j) {
        qf[t][j][0] = dev::pack_f16x2(qv[t][4 * j] * q_mul, qv[t][4 * j + 1] * q_mul);
        qf[t][j][1] = dev::pack_f16x2(qv[t][4 * j + 2] * q_mul, qv[t][4 * j + 3] * q_mul);
      }
    }
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int nr = min(8 * t + 2 * c + k, pc.nrows - 1);
        const int pn = L - Q + (pc.row0 + nr) / G;
        col_hi[t][k] = p.causal ? pn + 1 : L;
        col_lo[t][k] = W > 0 ? pn - W + 1 : 0;
        if constexpr (AL) {
          al_slope[t][k] = p.alibi_slopes[pc.kv_head * G + (pc.row0 + nr) % G] * log2e;
          al_pos[t][k] = pn;
        }
      }
    score_mul = q_unmul * base_scale * (Geo::kPth || Geo::kAuto ? 1.0f : p.k_scale);
#pragma unroll
    for (int t = 0; t < NT; ++t) {
#pragma unroll
      for (int i = 0; i < Geo::kMtiles; ++i) o[t][i][0] = o[t][i][1] = o[t][i][2] = o[t][i][3] = 0.0f;
      m_run[t][0] = m_run[t][1] = -INFINITY;
      l_run[t][0] = l_run[t][1] = 0.0f;
    }
    ev = -1000;
  };

  // Finish a piece: its rows' outputs (or partials) straight from the MMA
  // fragments; the last piece of a cut tile merges the tile.
  auto finish_piece = [&]() {
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
      for (int k = 0; k < 2; ++k)
#pragma unroll
        for (int off = 4; off < 32; off <<= 1)
          l_run[t][k] += __shfl_xor_sync(0xffffffffu, l_run[t][k], off);
    const float unit = Geo::kPth && ev > -1000 ? ldexpf(1.0f, ev) : 1.0f;
    const float vmul = Geo::kPth || Geo::kAuto ? 1.0f : p.v_scale;
    // An attention sink joins the normaliser of a whole (uncut) tile here;
    // a cut tile's merge adds it once.  The weights carry 2^-(m_run - 6).
    if (p.sinks && pc.part < 0) {
#pragma unroll
      for (int t = 0; t < NT; ++t)
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const int nr = min(8 * t + 2 * c + k, pc.nrows - 1);
          const float sk = p.sinks[pc.kv_head * G + (pc.row0 + nr) % G] * log2e;
          if (m_run[t][k] != -INFINITY && sk != -INFINITY)
            l_run[t][k] += exp2f(fminf(sk - m_run[t][k] + 6.0f, 126.0f));
        }
    }
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int nr = 8 * t + 2 * c + k;
        if (nr >= pc.nrows) continue;
        const float l = l_run[t][k];
        const float sc = (l > 0.0f ? 1.0f / l : 0.0f) * unit * vmul;
        const int R = pc.row0 + nr;
        if (pc.part < 0) {
          if (piece_bad) continue;
          const int tok = q0 + R / G;
          const int head = pc.kv_head * G + R % G;
          uint16_t* dst = p.out + ((int64_t)tok * p.heads_q + head) * D;
          // m-tiles 8r .. 8r+7 cover 16 consecutive dims (8 for head_dim 64).
#pragma unroll
          for (int r0 = 0; r0 < Geo::kMtiles; r0 += 4) {
            uint2 w;
            w.x = dev::pack_bf16x2(o[t][r0][k] * sc, o[t][r0][k + 2] * sc);
            w.y = dev::pack_bf16x2(o[t][r0 + 1][k] * sc, o[t][r0 + 1][k + 2] * sc);
            uint2 w2;
            w2.x = dev::pack_bf16x2(o[t][r0 + 2][k] * sc, o[t][r0 + 2][k + 2] * sc);
            w2.y = dev::pack_bf16x2(o[t][r0 + 3][k] * sc, o[t][r0 + 3][k + 2] * sc);
            *reinterpret_cast<uint4*>(dst + pv_dim<DT, D>(r0, g, 0)) = make_uint4(w.x, w.y, w2.x, w2.y);
          }
        } else {
          float* dst = p.part_o + (int64_t)(pc.part + nr) * D;
#pragma unroll
          for (int r0 = 0; r0 < Geo::kMtiles; r0 += 2)
            *reinterpret_cast<float4*>(dst + pv_dim<DT, D>(r0, g, 0)) =
                make_float4(o[t][r0][k] * sc, o[t][r0][k + 2] * sc, o[t][r0 + 1][k] * sc,
                            o[t][r0 + 1][k + 2] * sc);
          if (g == 0) p.part_lse[pc.part + nr] = l > 0.0f ? m_run[t][k] + log2f(l) : -INFINITY;
        }
      }
  };

  // ---- stream the segment -------------------------------------------------
  for (int q = 0; q < n; ++q) {
    const int tok0 = nx_tok;
    const int rec_piece = nx_piece;
    const bool chunk_ok = nx_ok;
    if (rec_piece != cur) {
      if (cur >= 0) finish_piece();
      cur = rec_piece;
      start_piece(cur);
    }

    // Per-token-head scales of tokens g and g + 8 (K and V).
    float sk0 = 1.0f, sk1 = 1.0f, sv0 = 1.0f, sv1 = 1.0f;
    float alpha_v = 1.0f;
    bool rescale_v = false;
    if constexpr (Geo::kPth) {
      const float mine = __uint_as_float(treg.x);
      sk0 = __shfl_sync(0xffffffffu, mine, 4 * g + 0);
      sk1 = __shfl_sync(0xffffffffu, mine, 4 * g + 1);
      sv0 = __shfl_sync(0xffffffffu, mine, 4 * g + 2);
      sv1 = __shfl_sync(0xffffffffu, mine, 4 * g + 3);
      // V scales multiply P as s_v * 2^-ev, ev the exponent of the largest
      // s_v seen so far in the piece (O is rescaled when it grows), so that
      // small scales keep P inside the f16 range.
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
      const uint4 kg = kreg[0][i];
      const uint4 kg8 = kreg[1][i];
      const uint32_t wg[4] = {kg.x, kg.y, kg.z, kg.w};
      const uint32_t wg8[4] = {kg8.x, kg8.y, kg8.z, kg8.w};
      if constexpr (Geo::kAuto) {
        // 8 bf16 per piece: k-steps 2i (words 0, 1) and 2i + 1 (words 2, 3).
#pragma unroll
        for (int w2 = 0; w2 < 2; ++w2) {
          const int j = 2 * i + w2;
          const uint32_t a[4] = {wg[2 * w2], wg8[2 * w2], wg[2 * w2 + 1], wg8[2 * w2 + 1]};
#pragma unroll
          for (int t = 0; t < NT; ++t) {
            if (w2 & 1) dev::mma_bf16_16816(s2[t], a, qf[t][j][0], qf[t][j][1]);
            else dev::mma_bf16_16816(s[t], a, qf[t][j][0], qf[t][j][1]);
          }
        }
      } else {
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
    }

    if (q + 1 < n) load_k(q + 1);   // K registers are free now

    // Scores in log2 units, masks, softmax reference.  The reference m_run
    // of a row only moves when some score exceeds it by more than 2^8
    // (a warp vote; the cross-lane maximum is reduced only then), so
    // P = 2^(z - m_run + 6) <= 2^14 fits f16 and the common chunk needs no
    // shuffles.  l carries the same 2^6 factor, which cancels in O / l.
    const bool full = chunk_ok && tok0 >= all_lo && tok0 + kChunkTokens <= all_hi;
    uint32_t pb0[NT], pb1[NT];
    uint32_t pl0[NT], pl1[NT];  // bf16 rows: the low halves of P (P = hi + lo)
    float z[NT][4];
    bool grow = false;
#pragma unroll
    for (int t = 0; t < NT; ++t) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float sk = (e < 2) ? sk0 : sk1;
        float v = (s[t][e] + s2[t][e]) * score_mul * sk;
        if (cap > 0.0f) v = cap_l2 * dev::tanh_exp(v * inv_cap);
        if constexpr (AL)  // bias from the exact integer distance, after the cap
          v = fmaf(al_slope[t][e & 1], (float)(tok0 + g + 8 * (e >> 1) - al_pos[t][e & 1]), v);
        if (!full) {
          const int tok = tok0 + g + 8 * (e >> 1);
          const int col = e & 1;
          const bool vis = chunk_ok && tok >= col_lo[t][col] && tok < col_hi[t][col];
          v = vis ? v : -INFINITY;
        }
        z[t][e] = v;
      }
      grow |= fmaxf(z[t][0], z[t][2]) > m_run[t][0] + 8.0f;
      grow |= fmaxf(z[t][1], z[t][3]) > m_run[t][1] + 8.0f;
    }
    float alpha[NT][2];
    const bool rescale = __any_sync(0xffffffffu, grow);
    if (rescale) {
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        float cm0 = fmaxf(z[t][0], z[t][2]), cm1 = fmaxf(z[t][1], z[t][3]);
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
          cm0 = fmaxf(cm0, __shfl_xor_sync(0xffffffffu, cm0, off));
          cm1 = fmaxf(cm1, __shfl_xor_sync(0xffffffffu, cm1, off));
        }
        const float mn0 = fmaxf(m_run[t][0], cm0), mn1 = fmaxf(m_run[t][1], cm1);
        alpha[t][0] = m_run[t][0] == -INFINITY ? 0.0f : dev::fast_exp2(m_run[t][0] - mn0);
        alpha[t][1] = m_run[t][1] == -INFINITY ? 0.0f : dev::fast_exp2(m_run[t][1] - mn1);
        m_run[t][0] = mn0;
        m_run[t][1] = mn1;
        l_run[t][0] *= alpha[t][0];
        l_run[t][1] *= alpha[t][1];
      }
    }
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const float e0 = m_run[t][0] == -INFINITY ? 0.0f : m_run[t][0] - 6.0f;
      const float e1 = m_run[t][1] == -INFINITY ? 0.0f : m_run[t][1] - 6.0f;
      const float p0 = dev::fast_exp2(z[t][0] - e0), p1 = dev::fast_exp2(z[t][1] - e1);
      const float p2 = dev::fast_exp2(z[t][2] - e0), p3 = dev::fast_exp2(z[t][3] - e1);
      l_run[t][0] += p0 + p2;
      l_run[t][1] += p1 + p3;
      // P^T (tokens x rows) -> B operand of O^T = V^T P^T via transposes.
      if constexpr (Geo::kAuto) {
        // bf16 MMA: P as the sum of two bf16 numbers (16 significant bits).
        const uint32_t h01 = dev::pack_bf16x2(p0, p1), h23 = dev::pack_bf16x2(p2, p3);
        pb0[t] = dev::movmatrix_trans(h01);
        pb1[t] = dev::movmatrix_trans(h23);
        pl0[t] = dev::movmatrix_trans(dev::pack_bf16x2(p0 - dev::bf16_lo(h01), p1 - dev::bf16_hi(h01)));
        pl1[t] = dev::movmatrix_trans(dev::pack_bf16x2(p2 - dev::bf16_lo(h23), p3 - dev::bf16_hi(h23)));
      } else {
        pb0[t] = dev::movmatrix_trans(dev::pack_f16x2(p0 * sv0, p1 * sv0));
        pb1[t] = dev::movmatrix_trans(dev::pack_f16x2(p2 * sv1, p3 * sv1));
      }
    }
    if (rescale || rescale_v) {
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        const float a0 = (rescale ? alpha[t][0] : 1.0f) * alpha_v;
        const float a1 = (rescale ? alpha[t][1] : 1.0f) * alpha_v;
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
      {
        const uint4 a0 = vreg[0][vs];
        const uint4 a1 = vreg[1][vs];
        const uint4 a2 = vreg[2][vs];
        const uint4 a3 = vreg[3][vs];
        r0[0] = a0.x; r0[1] = a0.y; r0[2] = a0.z; r0[3] = a0.w;
        r1[0] = a1.x; r1[1] = a1.y; r1[2] = a1.z; r1[3] = a1.w;
        r2[0] = a2.x; r2[1] = a2.y; r2[2] = a2.z; r2[3] = a2.w;
        r3[0] = a3.x; r3[1] = a3.y; r3[2] = a3.z; r3[3] = a3.w;
      }
      if constexpr (Geo::kAuto) {
        // Word w of rows 2c / 2c+1 holds dims (2w, 2w + 1) of the run: the
        // two tokens' values of one dim pair up per half (m-tile 4 vs + w).
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const uint32_t a[4] = {dev::prmt(r0[w], r1[w], 0x5410u), dev::prmt(r0[w], r1[w], 0x7632u),
                                 dev::prmt(r2[w], r3[w], 0x5410u), dev::prmt(r2[w], r3[w], 0x7632u)};
          const int i = vs * 4 + w;  // m-tile
#pragma unroll
          for (int t = 0; t < NT; ++t) {
            dev::mma_bf16_16816(o[t][i], a, pb0[t], pb1[t]);
            dev::mma_bf16_16816(o[t][i], a, pl0[t], pl1[t]);
          }
        }
      } else {
        // Word w of rows 2c / 2c+1 -> bytes (b0, b1) and (b2, b3) paired
        // across the two tokens: m-tiles 2(vs*kWords + w) and 2(vs*kWords + w) + 1.
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

    if (q + 1 < n) load_v();        // V registers are free now

    // Records for positions q + 17 .. q + 32, in three steps (see above).
    {
      const int phase = q % 16;
      if (phase == 0) fill_load_ref(q + 32, 16);
      else if (phase == 5) fill_load_piece();
      else if (phase == 10) fill_load_block();
      else if (phase == 15) {
        fill_store(q + 17, 16);
        __syncwarp();
      }
    }
  }
  if (cur >= 0) finish_piece();
}

// Launch one instance (used by the per-head_dim translation units).
template <int DT, int D, int NT, bool AL>
int launch_decode_instance(const AttnParams& p, cudaStream_t stream) {
  const size_t smem = decode_smem_bytes(DT, D);
  auto kern = splitkv_decode_kernel<DT, D, NT, AL, false>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return KVQ_E_CUDA;
  StepParams none{};
  kern<<<(unsigned)(p.num_warps / kDecodeWarps), kDecodeThreads, smem, stream>>>(p, none);
  return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_E_CUDA;
}

// The fused step: every CTA resident at once (a cooperative launch), as many
// as fit on the device.  `warps` == 0 asks for that number instead.
template <int DT, int D, int NT, bool AL>
int launch_step_instance(const AttnParams& p, const StepParams& sp, int64_t* warps,
                         cudaStream_t stream) {
  const size_t smem = decode_smem_bytes(DT, D);
  auto kern = splitkv_decode_kernel<DT, D, NT, AL, true>;
  // The grid of each device, found once (the attribute and occupancy queries
  // cost microseconds of host time, and a step calls this twice).
  static std::atomic<int64_t> grid_of[kMaxCachedDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return KVQ_E_CUDA;
  }
  int64_t grid = dev < kMaxCachedDevices ? grid_of[dev].load(std::memory_order_acquire) : 0;
  if (grid <= 0) {
    int sms = 0, per_sm = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
            cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kDecodeThreads, smem) !=
            cudaSuccess || per_sm <= 0) {
      cudaGetLastError();
      return KVQ_E_CUDA;
    }
    grid = (int64_t)sms * per_sm;
    if (dev < kMaxCachedDevices) grid_of[dev].store(grid, std::memory_order_release);
  }
  if (*warps == 0) {
    *warps = grid * kDecodeWarps;
    return KVQ_OK;
  }
  if (*warps != grid * kDecodeWarps) return KVQ_E_INVALID_ARG;
  AttnParams pp = p;
  StepParams ss = sp;
  void* args[] = {&pp, &ss};
  if (cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(kern), dim3((unsigned)grid),
                                  dim3(kDecodeThreads), args, smem, stream) != cudaSuccess) {
    cudaGetLastError();
    return KVQ_E_CUDA;
  }
  return KVQ_OK;
}

// The instances of one head_dim and one ALiBi setting (one translation unit
// each keeps the build parallel).
// (tiles of up to 8 rows: one MMA n-tile; up to 16: two)
template <int D, bool AL>
int launch_step_d(const AttnParams& p, const StepParams& sp, int dtype, int64_t* warps,
                  cudaStream_t stream) {
#define KVQ_STEP_CASE(DT)                                                          \
  case DT:                                                                         \
    return sp.max_rows <= 8 ? launch_step_instance<DT, D, 1, AL>(p, sp, warps, stream) \
                            : launch_step_instance<DT, D, 2, AL>(p, sp, warps, stream);
  switch (dtype) {
    KVQ_STEP_CASE(KVQ_AUTO)
    KVQ_STEP_CASE(KVQ_FP8_E4M3)
    KVQ_STEP_CASE(KVQ_FP8_E5M2)
    KVQ_STEP_CASE(KVQ_INT8_PER_TOKEN_HEAD)
    KVQ_STEP_CASE(KVQ_FP8_PER_TOKEN_HEAD)
    KVQ_STEP_CASE(KVQ_FP8_E5M2_PER_TOKEN_HEAD)
    default:
      return KVQ_E_UNSUPPORTED;
  }
#undef KVQ_STEP_CASE
}

template <int D, bool AL>
int launch_decode_d(const AttnParams& p, int dtype, int ntiles, cudaStream_t stream) {
#define KVQ_DECODE_CASE(DT)                                                  \
  case DT:                                                                   \
    return ntiles == 1 ? launch_decode_instance<DT, D, 1, AL>(p, stream)     \
                       : launch_decode_instance<DT, D, 2, AL>(p, stream);
  switch (dtype) {
    KVQ_DECODE_CASE(KVQ_AUTO)
    KVQ_DECODE_CASE(KVQ_FP8_E4M3)
    KVQ_DECODE_CASE(KVQ_FP8_E5M2)
    KVQ_DECODE_CASE(KVQ_INT8_PER_TOKEN_HEAD)
    KVQ_DECODE_CASE(KVQ_FP8_PER_TOKEN_HEAD)
    KVQ_DECODE_CASE(KVQ_FP8_E5M2_PER_TOKEN_HEAD)
    default:
      return KVQ_E_UNSUPPORTED;
  }
#undef KVQ_DECODE_CASE
}

}  // namespace kvq
