// kvq_host.cpp -- the C ABI: argument checks, dtype parsing, the scheduler
// (get_scheduler_metadata) and the attention dispatch.
//
// vllm PR 50194 page, Breakdown item 1 and Key source snippet: the
// scheduler is given kv_cache_dtype (parsed to the enum 0 = auto,
// 1 = fp8_e4m3, 2 = fp8_e5m2) so that tile and scratch sizes follow the KV
// cache element size.  Here every size comes from kvq_internal.h's constexpr
// geometry, and the attention call refuses a schedule built for another
// dtype, head count or head size.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <atomic>
#include <mutex>
#include <new>
#include <utility>
#include <numeric>
#include <vector>

#include "kvq_internal.h"

using kvq::DecodePiece;
using kvq::MergeItem;
using kvq::PrefillTile;
using kvq::WarpSeg;

// One launch of the split-KV decode kernel: the tiles with one 8-row n-tile
// (class 0) or two (class 1).
struct DecodeLaunch {
  int64_t piece_off = 0;   // the launch's first piece
  int64_t num_pieces = 0;
  int64_t warp_off = 0;    // its first entry of the warp table
  int64_t num_chunks = 0;  // length of its flat chunk sequence
  int num_warps = 0;       // warps the sequence is cut among
  bool lockstep = false;   // every kv head of a request cut at the same chunks
};

struct kvq_sched {
  int num_req, heads_q, heads_kv, head_dim, dtype, causal, window, group;
  int device;
  int64_t total_q;
  // The plan lives in its host image (below): the pieces of both launches,
  // then per launch and warp its segment and first piece, the merge items.
  const DecodePiece* h_pieces;
  const WarpSeg* h_warps;
  const MergeItem* h_merges;
  int64_t num_pieces, num_merges;
  std::vector<PrefillTile> prefill;
  DecodeLaunch launch[2];
  int64_t num_tiles, max_splits, partial_rows;
  int32_t max_chunk;  // highest 16-token chunk index any tile reads
  size_t workspace_bytes;
  void* d_buf;  // device copy: pieces, warp table, merge items, prefill tiles, error word
  size_t d_buf_bytes;
  size_t d_pieces_off, d_warps_off, d_merges_off, d_prefill_off, d_error_off;
  size_t image_bytes;       // bytes of the plan image (host and device copies)
  void* h_image;            // host image (pinned with a device), uploaded by the first attention call
  size_t h_image_bytes;
  bool h_image_pinned;
  std::atomic<bool> uploaded;
};

namespace {

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Device buffers of destroyed schedules, kept for the next schedules (a
// serving loop plans every step; cudaMalloc / cudaFree there would cost more
// than the planning).  Bounded; sizes are powers of two from 64 KiB.
struct PooledBuf {
  int device;
  size_t bytes;
  void* ptr;
};
std::mutex g_pool_mutex;
std::vector<PooledBuf> g_pool;
constexpr size_t kPoolMax = 16;

size_t pool_size_class(size_t bytes) {
  size_t c = 64 * 1024;
  while (c < bytes) c <<= 1;
  return c;
}

void* pool_get(int device, size_t bytes, size_t* got) {
  const size_t want = pool_size_class(bytes);
  {
    std::lock_guard<std::mutex> lock(g_pool_mutex);
    for (size_t i = 0; i < g_pool.size(); ++i) {
      if (g_pool[i].device == device && g_pool[i].bytes >= want) {
        void* p = g_pool[i].ptr;
        *got = g_pool[i].bytes;
        g_pool.erase(g_pool.begin() + (std::ptrdiff_t)i);
        return p;
      }
    }
  }
  void* p = nullptr;
  if (cudaMalloc(&p, want) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  *got = want;
  return p;
}

// Pinned host images of destroyed schedules, kept for the next schedules
// (the same power-of-two classes; bounded).  A schedule's image is uploaded
// by its first attention call with an asynchronous copy on that call's
// stream, so it must stay untouched until the schedule is destroyed.
std::mutex g_pinned_mutex;
std::vector<std::pair<size_t, void*>> g_pinned;

void* pinned_get(size_t bytes, size_t* got, bool* pinned) {
  const size_t want = pool_size_class(bytes);
  {
    std::lock_guard<std::mutex> lock(g_pinned_mutex);
    for (size_t i = 0; i < g_pinned.size(); ++i) {
      if (g_pinned[i].first >= want) {
        void* p = g_pinned[i].second;
        *got = g_pinned[i].first;
        g_pinned.erase(g_pinned.begin() + (std::ptrdiff_t)i);
        *pinned = true;
        return p;
      }
    }
  }
  void* p = nullptr;
  if (cudaHostAlloc(&p, want, cudaHostAllocDefault) == cudaSuccess) {
    *got = want;
    *pinned = true;
    return p;
  }
  cudaGetLastError();
  // Without pinned memory the image is pageable; the upload then completes
  // before cudaMemcpyAsync returns.
  p = std::malloc(want);
  *got = p ? want : 0;
  *pinned = false;
  return p;
}

void pinned_put(void* p, size_t bytes, bool pinned) {
  if (!p) return;
  if (!pinned) {
    std::free(p);
    return;
  }
  {
    std::lock_guard<std::mutex> lock(g_pinned_mutex);
    if (g_pinned.size() < kPoolMax) {
      g_pinned.emplace_back(bytes, p);
      return;
    }
  }
  cudaFreeHost(p);
}

void pool_put(int device, void* ptr, size_t bytes) {
  {
    std::lock_guard<std::mutex> lock(g_pool_mutex);
    if (g_pool.size() < kPoolMax) {
      g_pool.push_back(PooledBuf{device, bytes, ptr});
      return;
    }
  }
  cudaFree(ptr);
}

// The driver's tensor-map encoder, fetched once through the runtime (no
// link against the driver library).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }();
  return fn;
}

// Map of a bf16 ("auto") cache for the prefill's bulk tensor copies:
// {head_dim values, kv heads, slots} with boxes {64, 1, 16} written in the
// 128-byte swizzle, i.e. straight into the tensor core's operand layout.
bool encode_auto_map(CUtensorMap* map, const void* cache, int head_dim, int heads_kv,
                     int64_t slots) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t row = 2 * (cuuint64_t)head_dim;
  const cuuint64_t dims[3] = {(cuuint64_t)head_dim, (cuuint64_t)heads_kv, (cuuint64_t)slots};
  const cuuint64_t strides[2] = {row, row * (cuuint64_t)heads_kv};
  const cuuint32_t box[3] = {64u, 1u, 16u};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(cache), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return sms;
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Prefill tiles in order of key range, longest first, equal ranges in their
// given order: a stable LSD radix sort of (longest range - range), 11 bits a
// pass (a mixed batch has thousands of tiles).
void sort_longest_first(std::vector<PrefillTile>& v) {
  const size_t n = v.size();
  if (n < 2) return;
  uint32_t longest = 0;
  for (const PrefillTile& t : v) longest = std::max(longest, (uint32_t)std::max(0, t.kv_hi - t.kv_lo));
  std::vector<uint32_t> key(n), idx(n), key2(n), idx2(n);
  for (size_t i = 0; i < n; ++i) {
    key[i] = longest - (uint32_t)std::max(0, v[i].kv_hi - v[i].kv_lo);
    idx[i] = (uint32_t)i;
  }
  constexpr int kBits = 11;
  constexpr uint32_t kMask = (1u << kBits) - 1;
  uint32_t count[1u << kBits];
  for (int shift = 0; shift < 32 && (longest >> shift) != 0; shift += kBits) {
    std::memset(count, 0, sizeof(count));
    for (size_t i = 0; i < n; ++i) ++count[(key[i] >> shift) & kMask];
    uint32_t run = 0;
    for (uint32_t d = 0; d <= kMask; ++d) {
      const uint32_t c = count[d];
      count[d] = run;
      run += c;
    }
    for (size_t i = 0; i < n; ++i) {
      const uint32_t pos = count[(key[i] >> shift) & kMask]++;
      key2[pos] = key[i];
      idx2[pos] = idx[i];
    }
    key.swap(key2);
    idx.swap(idx2);
  }
  std::vector<PrefillTile> sorted(n);
  for (size_t i = 0; i < n; ++i) sorted[i] = v[idx[i]];
  v.swap(sorted);
}

// SM count assumed when planning without a device (GB300: 152 SMs).
constexpr int kDefaultSmCount = 152;

// A row tile: packed rows [row0, row0 + nrows) of one (request, kv head)
// and the 16-token chunks [c_lo, c_hi) those rows can see.
struct Tile {
  int req, kv_head, row0, nrows;
  int64_t c_lo, c_hi, any_lo, any_hi;
};

}  // namespace

extern "C" {

const char* kvq_status_string(int status) {
  switch (status) {
    case KVQ_OK: return "ok";
    case KVQ_E_INVALID_ARG: return "invalid argument";
    case KVQ_E_UNSUPPORTED: return "unsupported dtype, head_dim or shape";
    case KVQ_E_SCHED_MISMATCH: return "schedule built for another dtype, head count, head_dim, causal or window";
    case KVQ_E_WORKSPACE_TOO_SMALL: return "workspace smaller than the schedule requires";
    case KVQ_E_CUDA: return "CUDA runtime error";
    case KVQ_E_NO_MEMORY: return "allocation failed";
    case KVQ_E_TIMEOUT: return "a kernel's bounded wait for the tensor core timed out";
    default: return "unknown status";
  }
}

int kvq_parse_kv_cache_dtype(const char* s, kvq_dtype_t* out) {
  if (!out) return KVQ_E_INVALID_ARG;
  if (!s || !*s || !std::strcmp(s, "auto")) { *out = KVQ_AUTO; return KVQ_OK; }
  if (!std::strcmp(s, "fp8") || !std::strcmp(s, "fp8_e4m3")) { *out = KVQ_FP8_E4M3; return KVQ_OK; }
  if (!std::strcmp(s, "fp8_e5m2")) { *out = KVQ_FP8_E5M2; return KVQ_OK; }
  if (!std::strcmp(s, "int8_per_token_head")) { *out = KVQ_INT8_PER_TOKEN_HEAD; return KVQ_OK; }
  if (!std::strcmp(s, "fp8_per_token_head")) { *out = KVQ_FP8_PER_TOKEN_HEAD; return KVQ_OK; }
  if (!std::strcmp(s, "fp8_e5m2_per_token_head")) {
    *out = KVQ_FP8_E5M2_PER_TOKEN_HEAD;
    return KVQ_OK;
  }
  return KVQ_E_INVALID_ARG;
}

int kvq_cache_row_bytes(kvq_dtype_t dtype, int head_dim, size_t* out) {
  if (!out || !kvq::is_valid_dtype(dtype) || head_dim <= 0 || head_dim % 16)
    return KVQ_E_INVALID_ARG;
  *out = (size_t)kvq::row_bytes(dtype, head_dim);
  return KVQ_OK;
}

int kvq_reshape_and_cache(const void* key, const void* value, int64_t num_tokens,
                          int64_t key_stride_tok, int64_t value_stride_tok, int num_heads_kv,
                          int head_dim, void* key_cache, void* value_cache, int64_t num_blocks,
                          int block_size, const int64_t* slot_mapping, kvq_dtype_t dtype,
                          float k_scale, float v_scale, void* stream) {
  if (!kvq::is_valid_dtype(dtype)) return KVQ_E_INVALID_ARG;
  if (!kvq::head_dim_supported(head_dim)) return KVQ_E_UNSUPPORTED;
  if (num_tokens < 0 || num_heads_kv <= 0 || num_blocks < 0 || block_size <= 0)
    return KVQ_E_INVALID_ARG;
  if (num_tokens == 0) return KVQ_OK;
  if (!key || !value || !key_cache || !value_cache || !slot_mapping) return KVQ_E_INVALID_ARG;
  const int64_t min_stride = (int64_t)num_heads_kv * head_dim;
  if (key_stride_tok < min_stride || value_stride_tok < min_stride || key_stride_tok % 8 ||
      value_stride_tok % 8)
    return KVQ_E_INVALID_ARG;
  if (!aligned(key, 16) || !aligned(value, 16) || !aligned(key_cache, 16) ||
      !aligned(value_cache, 16) || !aligned(slot_mapping, 8))
    return KVQ_E_INVALID_ARG;
  if (dtype == KVQ_FP8_E4M3 || dtype == KVQ_FP8_E5M2) {
    if (!(std::isfinite(k_scale) && k_scale > 0.0f && std::isfinite(v_scale) && v_scale > 0.0f))
      return KVQ_E_INVALID_ARG;
  }
  return kvq::launch_reshape_and_cache(key, value, num_tokens, key_stride_tok, value_stride_tok,
                                       num_heads_kv, head_dim, key_cache, value_cache, num_blocks,
                                       block_size, slot_mapping, dtype, k_scale, v_scale, stream);
}


void kvq_sched_destroy(kvq_sched_t* s) {
  if (!s) return;
  if (s->d_buf) pool_put(s->device, s->d_buf, s->d_buf_bytes);
  pinned_put(s->h_image, s->h_image_bytes, s->h_image_pinned);
  delete s;
}

int kvq_get_scheduler_metadata(int num_req, int heads_q, int heads_kv, int head_dim,
                               const int32_t* seq_lens_host, const int32_t* query_start_loc_host,
                               int causal, int window, kvq_dtype_t dtype, kvq_sched_t** out,
                               size_t* workspace_bytes) {
  if (!out || !workspace_bytes) return KVQ_E_INVALID_ARG;
  *out = nullptr;
  *workspace_bytes = 0;
  if (num_req < 0 || heads_kv <= 0 || heads_q <= 0) return KVQ_E_INVALID_ARG;
  if (num_req > 0 && (!seq_lens_host || !query_start_loc_host)) return KVQ_E_INVALID_ARG;
  if (!kvq::is_valid_dtype(dtype)) return KVQ_E_INVALID_ARG;
  if (heads_q % heads_kv) return KVQ_E_UNSUPPORTED;
  if (!kvq::head_dim_supported(head_dim) || !kvq::attention_dtype_supported(dtype))
    return KVQ_E_UNSUPPORTED;
  if (window > 0 && !causal) return KVQ_E_INVALID_ARG;
  if (num_req > 0 && query_start_loc_host[0] != 0) return KVQ_E_INVALID_ARG;
  for (int r = 0; r < num_req; ++r) {
    const int64_t Q = (int64_t)query_start_loc_host[r + 1] - query_start_loc_host[r];
    if (Q < 0 || seq_lens_host[r] < 0 || Q > seq_lens_host[r]) return KVQ_E_INVALID_ARG;
  }

  kvq_sched* s = new (std::nothrow) kvq_sched();
  if (!s) return KVQ_E_NO_MEMORY;
  s->num_req = num_req;
  s->heads_q = heads_q;
  s->heads_kv = heads_kv;
  s->head_dim = head_dim;
  s->dtype = dtype;
  s->causal = causal ? 1 : 0;
  s->window = window > 0 ? window : 0;
  s->group = heads_q / heads_kv;
  s->total_q = num_req > 0 ? query_start_loc_host[num_req] : 0;
  s->d_buf = nullptr;
  s->h_image = nullptr;
  s->h_image_bytes = 0;
  s->h_image_pinned = false;
  s->h_pieces = nullptr;
  s->h_warps = nullptr;
  s->h_merges = nullptr;
  s->num_pieces = 0;
  s->num_merges = 0;
  s->uploaded.store(false);
  // Without a usable CUDA device the plan is still built (host-only: its
  // attention calls return KVQ_E_CUDA), so that planning can be inspected
  // on machines without a GPU.
  const bool have_device = cudaGetDevice(&s->device) == cudaSuccess;
  if (!have_device) {
    cudaGetLastError();
    s->device = -1;
  }
  const int G = s->group;

  // 1) Row tiles: the packed rows (q_index * G + g) of each (request,
  //    kv_head) in tiles of up to 16, each with the chunks its rows can see,
  //    in (request, kv head) order so neighbouring warps read neighbouring
  //    rows of the same cache blocks.  Tiles of up to 8 rows use one MMA
  //    n-tile (class 0), larger ones two (class 1).
  std::vector<Tile> tiles[2];
  s->max_chunk = 0;
  {
    // capacities first (a prefill of many requests has thousands of tiles)
    size_t n_prefill = 0, n_tiles[2] = {0, 0};
    for (int r = 0; r < num_req; ++r) {
      const int64_t rows = ((int64_t)query_start_loc_host[r + 1] - query_start_loc_host[r]) * G;
      if (rows == 0) continue;
      if (rows > kvq::kTileMaxRows) {
        n_prefill += (size_t)heads_kv * (size_t)ceil_div(rows, kvq::kPrefillRows);
      } else {
        n_tiles[rows > 8 ? 1 : 0] += (size_t)heads_kv;
      }
    }
    s->prefill.reserve(n_prefill);
    tiles[0].reserve(n_tiles[0]);
    tiles[1].reserve(n_tiles[1]);
  }
  // A request's row tiles: their key ranges do not depend on the kv head, so
  // each is worked out once and copied for every head (heads outermost).
  std::vector<PrefillTile> row_prefill;
  std::vector<Tile> row_tiles;
  for (int r = 0; r < num_req; ++r) {
    const int64_t L = seq_lens_host[r];
    const int64_t Q = (int64_t)query_start_loc_host[r + 1] - query_start_loc_host[r];
    if (Q == 0) continue;
    const int64_t rows = Q * G;
    if (rows > kvq::kTileMaxRows) {
      // Prefill: 128-row tiles on the tensor cores.
      row_prefill.clear();
      for (int64_t row0 = 0; row0 < rows; row0 += kvq::kPrefillRows) {
        const int64_t nrows = std::min<int64_t>(kvq::kPrefillRows, rows - row0);
        const int64_t p_min = L - Q + row0 / G;
        const int64_t p_max = L - Q + (row0 + nrows - 1) / G;
        PrefillTile pt;
        pt.req = r;
        pt.kv_head = 0;
        pt.row0 = (int32_t)row0;
        pt.nrows = (int32_t)nrows;
        pt.kv_hi = (int32_t)(s->causal ? p_max + 1 : L);
        pt.kv_lo = (int32_t)(s->window > 0 ? std::max<int64_t>(0, p_min - s->window + 1) : 0);
        pt.q0 = query_start_loc_host[r];
        pt.pos0 = (int32_t)(L - Q);
        s->max_chunk = std::max<int32_t>(s->max_chunk, (int32_t)((pt.kv_hi - 1) / kvq::kChunkTokens));
        row_prefill.push_back(pt);
      }
      for (int h = 0; h < heads_kv; ++h)
        for (const PrefillTile& pt : row_prefill) {
          s->prefill.push_back(pt);
          s->prefill.back().kv_head = h;
        }
      continue;
    }
    row_tiles.clear();
    for (int64_t row0 = 0; row0 < rows; row0 += kvq::kTileMaxRows) {
      const int64_t nrows = std::min<int64_t>(kvq::kTileMaxRows, rows - row0);
      const int64_t p_min = L - Q + row0 / G;
      const int64_t p_max = L - Q + (row0 + nrows - 1) / G;
      Tile t;
      t.req = r;
      t.kv_head = 0;
      t.row0 = (int)row0;
      t.nrows = (int)nrows;
      t.any_hi = s->causal ? p_max + 1 : L;
      t.any_lo = s->window > 0 ? std::max<int64_t>(0, p_min - s->window + 1) : 0;
      t.c_lo = t.any_lo / kvq::kChunkTokens;
      t.c_hi = ceil_div(t.any_hi, kvq::kChunkTokens);
      s->max_chunk = std::max<int32_t>(s->max_chunk, (int32_t)(t.c_hi - 1));
      row_tiles.push_back(t);
    }
    for (int h = 0; h < heads_kv; ++h)
      for (const Tile& t : row_tiles) {
        std::vector<Tile>& v = tiles[t.nrows > 8 ? 1 : 0];
        v.push_back(t);
        v.back().kv_head = h;
      }
  }
  s->num_tiles = (int64_t)(tiles[0].size() + tiles[1].size());
  // Longest prefill tiles first, so the tail of the grid is short tiles.
  // CTA pairs take pair tiles: consecutive row tiles of one (request, kv
  // head) at list entries 2i and 2i + 1 (a last odd tile with an empty
  // partner: nrows 0, its key range), longest key-range union first.
  if (kvq::prefill_cta_group(s->dtype, s->head_dim) == 2 && !s->prefill.empty()) {
    std::vector<std::pair<PrefillTile, PrefillTile>> pairs;
    for (size_t i = 0; i < s->prefill.size();) {
      const PrefillTile& a = s->prefill[i];
      if (i + 1 < s->prefill.size() && s->prefill[i + 1].req == a.req &&
          s->prefill[i + 1].kv_head == a.kv_head) {
        pairs.emplace_back(a, s->prefill[i + 1]);
        i += 2;
      } else {
        PrefillTile e = a;
        e.row0 = a.row0 + a.nrows;
        e.nrows = 0;
        pairs.emplace_back(a, e);
        i += 1;
      }
    }
    auto span = [](const std::pair<PrefillTile, PrefillTile>& q) {
      return std::max(q.first.kv_hi, q.second.kv_hi) - std::min(q.first.kv_lo, q.second.kv_lo);
    };
    std::stable_sort(pairs.begin(), pairs.end(),
                     [&](const std::pair<PrefillTile, PrefillTile>& a,
                         const std::pair<PrefillTile, PrefillTile>& b) { return span(a) > span(b); });
    s->prefill.clear();
    for (const auto& q : pairs) {
      s->prefill.push_back(q.first);
      s->prefill.push_back(q.second);
    }
  } else {
    sort_longest_first(s->prefill);
  }

  // 2) Per class of row tiles: the chunk count, the tile order and the warp
  //    count.  Tile order:
  //    - request-major ((request, kv head) order) when a cache row is a whole
  //      number of 128-byte lines;
  //    - head lockstep otherwise (per-token-head rows of D + 16 bytes, 64-byte
  //      rows), where the rows of one token's neighbouring kv heads share a
  //      128-byte line: head-major order (every request's tile of kv head 0,
  //      then of kv head 1, ...) with a warp count that is a multiple of the
  //      kv heads, so every head's run of the sequence is cut at the same
  //      chunks, and the v-th segments of all heads go to neighbouring warps.
  //      Those warps stream the same tokens' rows side by side, and the
  //      second read of a shared line hits L2.
  //    KVQ_DECODE_WARPS (tests, benchmarks) forces the warp count;
  //    KVQ_DECODE_LOCKSTEP = 0 / 1 forces the order.
  const int sms = have_device ? std::max(1, sm_count()) : kDefaultSmCount;
  int64_t forced = 0;
  if (const char* env = std::getenv("KVQ_DECODE_WARPS")) forced = std::atoll(env);
  bool lockstep = kvq::row_bytes(dtype, head_dim) % 128 != 0;
  if (const char* env = std::getenv("KVQ_DECODE_LOCKSTEP")) lockstep = std::atoi(env) != 0;
  lockstep = lockstep && heads_kv > 1;
  s->partial_rows = 0;
  s->max_splits = 0;
  int64_t max_pieces = 0, max_merges = 0, num_warps = 0;
  for (int cls = 0; cls < 2; ++cls) {
    DecodeLaunch& dl = s->launch[cls];
    int64_t T = 0;
    for (const Tile& t : tiles[cls]) T += t.c_hi - t.c_lo;
    dl.num_chunks = T;
    if (T == 0) continue;
    // Head-major order when every request has one tile per kv head in this
    // class (row tiles of up to 16 rows: always, for decodes).
    bool ls = lockstep && tiles[cls].size() % (size_t)heads_kv == 0;
    for (size_t k = 0; ls && k < tiles[cls].size(); ++k)
      if (tiles[cls][k].kv_head != (int)(k % (size_t)heads_kv) ||
          tiles[cls][k].req != tiles[cls][k - k % (size_t)heads_kv].req)
        ls = false;
    if (ls)
      std::stable_sort(tiles[cls].begin(), tiles[cls].end(),
                       [](const Tile& a, const Tile& b) { return a.kv_head < b.kv_head; });
    dl.lockstep = ls;
    const int64_t max_ctas = (int64_t)sms * kvq::decode_min_ctas(dtype, head_dim, cls + 1);
    int64_t ctas = std::min<int64_t>(max_ctas, std::max<int64_t>(1, ceil_div(T, kvq::kDecodeWarps * kvq::kMinChunksPerWarp)));
    if (forced > 0) ctas = std::max<int64_t>(1, std::min<int64_t>(ceil_div(forced, kvq::kDecodeWarps), ceil_div(T, kvq::kDecodeWarps)));
    int64_t W = ctas * kvq::kDecodeWarps;
    if (ls && W >= heads_kv) {
      // a multiple of the kv head count (and of the CTA's warps)
      const int64_t unit = (int64_t)heads_kv * kvq::kDecodeWarps / std::gcd<int64_t>(heads_kv, kvq::kDecodeWarps);
      if (W >= unit) W = W / unit * unit;
    }
    dl.num_warps = (int)W;
    // a tile is cut at most at every segment boundary inside it
    max_pieces += (int64_t)tiles[cls].size() + W - 1;
    max_merges += (int64_t)tiles[cls].size();
    num_warps += W;
  }

  // 3) The plan image, laid out for the largest plan these tiles can give:
  //    pieces, per-launch warp table, merge items, prefill tiles, the error
  //    word.  With a device it is pinned host memory, and a pooled device
  //    buffer is reserved for it; the first attention call uploads it on its
  //    own stream (no synchronisation here).  The decomposition below writes
  //    the image directly.
  s->d_pieces_off = 0;
  s->d_warps_off = kvq::align256((size_t)max_pieces * sizeof(DecodePiece));
  s->d_merges_off = s->d_warps_off + kvq::align256((size_t)num_warps * sizeof(WarpSeg));
  s->d_prefill_off = s->d_merges_off + kvq::align256((size_t)max_merges * sizeof(MergeItem));
  s->d_error_off = s->d_prefill_off + kvq::align256(s->prefill.size() * sizeof(PrefillTile));
  const size_t total = s->d_error_off + sizeof(int32_t);
  s->image_bytes = total;
  if (have_device) {
    s->d_buf = pool_get(s->device, total, &s->d_buf_bytes);
    if (!s->d_buf) {
      delete s;
      return KVQ_E_NO_MEMORY;
    }
    s->h_image = pinned_get(total, &s->h_image_bytes, &s->h_image_pinned);
  } else {
    s->h_image = std::malloc(total);
    s->h_image_bytes = total;
    s->h_image_pinned = false;
  }
  if (!s->h_image) {
    kvq_sched_destroy(s);
    return KVQ_E_NO_MEMORY;
  }
  char* image = static_cast<char*>(s->h_image);
  DecodePiece* const P = reinterpret_cast<DecodePiece*>(image + s->d_pieces_off);
  WarpSeg* const WS = reinterpret_cast<WarpSeg*>(image + s->d_warps_off);
  MergeItem* const M = reinterpret_cast<MergeItem*>(image + s->d_merges_off);
  s->h_pieces = P;
  s->h_warps = WS;
  s->h_merges = M;
  if (!s->prefill.empty())
    std::memcpy(image + s->d_prefill_off, s->prefill.data(), s->prefill.size() * sizeof(PrefillTile));
  std::memset(image + s->d_error_off, 0, sizeof(int32_t));  // the error word starts at zero

  // 4) Work decomposition (stream-K): per class, lay the tiles' chunks end
  //    to end and cut the sequence into equal contiguous segments, one per
  //    warp.  A tile cut by a segment boundary becomes several pieces whose
  //    partial rows are merged.  (Counters in locals and stores through plain
  //    pointers into the image: this runs once per planned step.)
  int64_t npieces = 0, nmerges = 0, nwarps = 0, partial_rows = 0, max_splits = 0;
  std::vector<int64_t> seg;
  for (int cls = 0; cls < 2; ++cls) {
    DecodeLaunch& dl = s->launch[cls];
    dl.piece_off = npieces;
    dl.warp_off = nwarps;
    const int64_t T = dl.num_chunks;
    if (T == 0) continue;
    const int64_t W = dl.num_warps;
    // Stream-K: segment w is [floor(w T / W), floor((w + 1) T / W)),
    // incrementally (no divides in the loop).
    seg.resize((size_t)W + 1);
    int64_t* const sg = seg.data();
    {
      const int64_t qt = T / W, rt = T % W;
      int64_t q = 0, r = 0;
      for (int64_t w = 0; w <= W; ++w) {
        sg[w] = q;
        q += qt;
        r += rt;
        if (r >= W) {
          r -= W;
          ++q;
        }
      }
    }
    // Segment w goes to warp phys(w).  Head lockstep with W = Hkv * Wh: the
    // v-th segments of all kv heads go to neighbouring warps.
    const bool interleave = dl.lockstep && W % heads_kv == 0;
    const int64_t Wh = W / heads_kv;
    auto phys = [&](int64_t w) { return interleave ? (w % Wh) * heads_kv + w / Wh : w; };
    WarpSeg* const ws = WS + nwarps;
    for (int64_t w = 0; w < W; ++w) {
      WarpSeg& e = ws[phys(w)];
      e.piece = 0;
      e.seg0 = (int32_t)sg[w];
      e.n = (int32_t)(sg[w + 1] - sg[w]);
      e.pad = 0;
    }
    // Tiles and warps in one pass: w is the warp whose segment holds F; the
    // warps [w, we) hold the tile's chunks [F, Fe).
    int64_t F = 0;
    int64_t w = 0;
    for (const Tile& t : tiles[cls]) {
      const int64_t Fe = F + (t.c_hi - t.c_lo);
      while (w + 1 < W && sg[w + 1] <= F) ++w;
      int64_t np = 0, we = w;
      for (; we < W && sg[we] < Fe; ++we) np += std::min(Fe, sg[we + 1]) > std::max(F, sg[we]);
      // a tile cut into np > 1 pieces: a merge item, and partial rows after
      // the ones handed out so far
      int32_t merge = -1;
      int64_t part = -1;
      if (np > 1) {
        MergeItem& m = M[nmerges];
        m.req = t.req;
        m.kv_head = t.kv_head;
        m.row0 = t.row0;
        m.nrows = t.nrows;
        m.part = (int32_t)partial_rows;
        m.nsplits = (int32_t)np;
        m.pad0 = m.pad1 = 0;
        merge = (int32_t)nmerges++;
        part = partial_rows;
        partial_rows += np * t.nrows;
      }
      for (int64_t ww = w; ww < we; ++ww) {
        const int64_t lo = std::max(F, sg[ww]), hi = std::min(Fe, sg[ww + 1]);
        if (hi <= lo) continue;
        // a warp whose segment starts inside this tile starts with this piece
        if (sg[ww] >= F) ws[phys(ww)].piece = (int32_t)(npieces - dl.piece_off);
        DecodePiece& pc = P[npieces++];
        pc.req = t.req;
        pc.kv_head = t.kv_head;
        pc.row0 = t.row0;
        pc.nrows = t.nrows;
        pc.part = (int32_t)part;
        pc.merge = merge;
        pc.any_lo = (int32_t)t.any_lo;
        pc.any_hi = (int32_t)t.any_hi;
        pc.flat0 = (int32_t)lo;
        pc.chunk0 = (int32_t)(t.c_lo + (lo - F));
        pc.pad0 = pc.pad1 = 0;
        if (part >= 0) part += t.nrows;
      }
      max_splits = std::max(max_splits, np);
      F = Fe;
    }
    dl.num_pieces = npieces - dl.piece_off;
    nwarps += W;
  }
  s->num_pieces = npieces;
  s->num_merges = nmerges;
  s->partial_rows = partial_rows;
  s->max_splits = max_splits;
  s->workspace_bytes = kvq::workspace_bytes(s->partial_rows, head_dim);
  *workspace_bytes = s->workspace_bytes;
  *out = s;
  return KVQ_OK;
}

int kvq_sched_get_plan_sizes(const kvq_sched_t* s, kvq_plan_sizes_t* out) {
  if (!s || !out) return KVQ_E_INVALID_ARG;
  std::memset(out, 0, sizeof(*out));
  out->num_pieces = s->num_pieces;
  out->num_merges = s->num_merges;
  out->num_prefill_tiles = (int64_t)s->prefill.size();
  for (int c = 0; c < 2; ++c) {
    out->num_chunks[c] = s->launch[c].num_chunks;
    out->num_warps[c] = s->launch[c].num_warps;
    out->lockstep[c] = s->launch[c].lockstep ? 1 : 0;
  }
  return KVQ_OK;
}

int kvq_sched_export_plan(const kvq_sched_t* s, kvq_plan_piece_t* pieces, int64_t pieces_cap,
                          int32_t* warp_first_piece, int64_t warps_cap, kvq_plan_merge_t* merges,
                          int64_t merges_cap, kvq_plan_prefill_tile_t* tiles, int64_t tiles_cap) {
  if (!s) return KVQ_E_INVALID_ARG;
  const int64_t nw = (int64_t)s->launch[0].num_warps + s->launch[1].num_warps;
  if ((pieces && pieces_cap < s->num_pieces) || (warp_first_piece && warps_cap < nw) ||
      (merges && merges_cap < s->num_merges) ||
      (tiles && tiles_cap < (int64_t)s->prefill.size()))
    return KVQ_E_INVALID_ARG;
  for (int c = 0; c < 2; ++c) {
    const DecodeLaunch& dl = s->launch[c];
    if (pieces) {
      for (int64_t i = 0; i < dl.num_pieces; ++i) {
        const DecodePiece& pc = s->h_pieces[dl.piece_off + i];
        const int64_t end = i + 1 < dl.num_pieces ? s->h_pieces[dl.piece_off + i + 1].flat0
                                                  : dl.num_chunks;
        kvq_plan_piece_t& o = pieces[dl.piece_off + i];
        o.launch = c;
        o.req = pc.req;
        o.kv_head = pc.kv_head;
        o.row0 = pc.row0;
        o.nrows = pc.nrows;
        o.part = pc.part;
        o.merge = pc.merge;
        o.key_lo = pc.any_lo;
        o.key_hi = pc.any_hi;
        o.flat0 = pc.flat0;
        o.chunk0 = pc.chunk0;
        o.nchunks = (int32_t)(end - pc.flat0);
      }
    }
    if (warp_first_piece) {
      const int64_t base = c == 0 ? 0 : s->launch[0].num_warps;
      for (int w = 0; w < dl.num_warps; ++w) {
        const WarpSeg& ws = s->h_warps[dl.warp_off + w];
        warp_first_piece[base + w] = ws.n > 0 ? (int32_t)(dl.piece_off + ws.piece) : -1;
      }
    }
  }
  if (merges) {
    for (int64_t i = 0; i < s->num_merges; ++i) {
      const MergeItem& m = s->h_merges[i];
      merges[i] = kvq_plan_merge_t{m.req, m.kv_head, m.row0, m.nrows, m.part, m.nsplits};
    }
  }
  if (tiles) {
    for (size_t i = 0; i < s->prefill.size(); ++i) {
      const PrefillTile& t = s->prefill[i];
      tiles[i] = kvq_plan_prefill_tile_t{t.req, t.kv_head, t.row0, t.nrows, t.kv_lo, t.kv_hi};
    }
  }
  return KVQ_OK;
}

int kvq_sched_get_info(const kvq_sched_t* s, kvq_sched_info_t* out) {
  if (!s || !out) return KVQ_E_INVALID_ARG;
  std::memset(out, 0, sizeof(*out));
  out->num_req = s->num_req;
  out->heads_q = s->heads_q;
  out->heads_kv = s->heads_kv;
  out->head_dim = s->head_dim;
  out->dtype = s->dtype;
  out->kv_elem_bytes = kvq::kv_elem_bytes(s->dtype);
  out->row_bytes = kvq::row_bytes(s->dtype, s->head_dim);
  out->causal = s->causal;
  out->window = s->window;
  out->num_tiles = s->num_tiles;
  out->num_pieces = s->num_pieces;
  out->num_merge_items = s->num_merges;
  out->num_chunks = s->launch[0].num_chunks + s->launch[1].num_chunks;
  out->num_decode_warps = (int64_t)s->launch[0].num_warps + s->launch[1].num_warps;
  out->max_splits = s->max_splits;
  out->total_query_tokens = s->total_q;
  out->workspace_bytes = s->workspace_bytes;
  out->decode_smem_bytes = kvq::decode_smem_bytes(s->dtype, s->head_dim);
  out->decode_chunk_bytes = (size_t)kvq::decode_chunk_bytes(s->dtype, s->head_dim);
  out->num_prefill_tiles = (int64_t)s->prefill.size();
  out->prefill_smem_bytes =
      kvq::prefill_smem_bytes(s->head_dim, kvq::prefill_cta_group(s->dtype, s->head_dim));
  out->num_kernel_launches = (s->launch[0].num_chunks > 0) + (s->launch[1].num_chunks > 0) +
                             (s->num_merges > 0) + (!s->prefill.empty());
  out->prefill_cta_group = kvq::prefill_cta_group(s->dtype, s->head_dim);
  return KVQ_OK;
}

int kvq_sched_check_device(const kvq_sched_t* s) {
  if (!s) return KVQ_E_INVALID_ARG;
  if (!s->d_buf || !s->uploaded.load()) return KVQ_OK;
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess) return KVQ_E_CUDA;
  if (cur != s->device && cudaSetDevice(s->device) != cudaSuccess) return KVQ_E_CUDA;
  int32_t flag = 0;
  char* err = static_cast<char*>(s->d_buf) + s->d_error_off;
  int rc = KVQ_OK;
  if (cudaMemcpy(&flag, err, sizeof(flag), cudaMemcpyDeviceToHost) != cudaSuccess) rc = KVQ_E_CUDA;
  else if (flag != 0) {
    rc = flag == 1 ? KVQ_E_TIMEOUT : KVQ_E_INVALID_ARG;
    cudaMemset(err, 0, sizeof(flag));
  }
  if (cur != s->device) cudaSetDevice(cur);
  return rc;
}

int kvq_attention_with_kv_cache(const kvq_sched_t* s, int heads_q, int heads_kv, int head_dim,
                                kvq_dtype_t dtype, const void* q, const void* key_cache,
                                const void* value_cache, const int32_t* query_start_loc,
                                const int32_t* seq_lens, const int32_t* block_table,
                                int block_table_stride, int block_size, int64_t num_blocks,
                                float sm_scale, int causal, int window, float soft_cap,
                                const float* alibi_slopes, const float* sinks, float k_scale,
                                float v_scale, void* out, void* workspace, size_t workspace_bytes,
                                void* stream) {
  if (!s) return KVQ_E_INVALID_ARG;
  if (heads_q != s->heads_q || heads_kv != s->heads_kv || head_dim != s->head_dim ||
      (int)dtype != s->dtype || (causal ? 1 : 0) != s->causal ||
      (window > 0 ? window : 0) != s->window)
    return KVQ_E_SCHED_MISMATCH;
  if (s->launch[0].num_chunks + s->launch[1].num_chunks == 0 && s->prefill.empty()) return KVQ_OK;
  if (!s->d_buf) return KVQ_E_CUDA;  // planned without a device
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess) return KVQ_E_CUDA;
  if (cur != s->device) return KVQ_E_INVALID_ARG;
  if (!q || !key_cache || !value_cache || !query_start_loc || !seq_lens || !block_table || !out)
    return KVQ_E_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(key_cache, 16) || !aligned(value_cache, 16) ||
      !aligned(out, 16) || !aligned(block_table, 4) || !aligned(alibi_slopes, 4) ||
      !aligned(sinks, 4))
    return KVQ_E_INVALID_ARG;
  if (block_size <= 0 || block_size % kvq::kChunkTokens) return KVQ_E_UNSUPPORTED;
  if (num_blocks <= 0 || block_table_stride <= 0) return KVQ_E_INVALID_ARG;
  // Cache slots are addressed with 32-bit indices.
  if (num_blocks * (int64_t)block_size >= ((int64_t)1 << 31)) return KVQ_E_UNSUPPORTED;
  // The table must hold every logical block the schedule reads.
  const int64_t last_block = ((int64_t)s->max_chunk * kvq::kChunkTokens) / block_size;
  if (last_block >= block_table_stride) return KVQ_E_INVALID_ARG;
  if (!std::isfinite(sm_scale) || !std::isfinite(soft_cap)) return KVQ_E_INVALID_ARG;
  if (dtype == KVQ_FP8_E4M3 || dtype == KVQ_FP8_E5M2) {
    if (!(std::isfinite(k_scale) && std::isfinite(v_scale))) return KVQ_E_INVALID_ARG;
  }
  if (workspace_bytes < s->workspace_bytes) return KVQ_E_WORKSPACE_TOO_SMALL;
  if (s->workspace_bytes > 0 && (!workspace || !aligned(workspace, 256)))
    return KVQ_E_INVALID_ARG;

  kvq::AttnParams p;
  std::memset(&p, 0, sizeof(p));
  p.q = static_cast<const uint16_t*>(q);
  p.key_cache = static_cast<const uint8_t*>(key_cache);
  p.value_cache = static_cast<const uint8_t*>(value_cache);
  p.query_start_loc = query_start_loc;
  p.seq_lens = seq_lens;
  p.block_table = block_table;
  p.out = static_cast<uint16_t*>(out);
  p.part_o = static_cast<float*>(workspace);
  p.part_lse = s->workspace_bytes
                   ? reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                              kvq::workspace_o_bytes(s->partial_rows, head_dim))
                   : nullptr;
  char* b = static_cast<char*>(s->d_buf);
  p.pieces = reinterpret_cast<const DecodePiece*>(b + s->d_pieces_off);
  p.merges = reinterpret_cast<const MergeItem*>(b + s->d_merges_off);
  p.prefill_tiles = reinterpret_cast<const PrefillTile*>(b + s->d_prefill_off);
  p.num_prefill_tiles = (int32_t)s->prefill.size();
  p.total_q_tokens = (int32_t)s->total_q;
  p.error_flag = reinterpret_cast<int32_t*>(b + s->d_error_off);
  p.num_blocks = num_blocks;
  p.block_table_stride = block_table_stride;
  p.block_size = block_size;
  p.heads_q = heads_q;
  p.heads_kv = heads_kv;
  p.group = s->group;
  p.causal = s->causal;
  p.window = s->window;
  p.sm_scale = sm_scale;
  p.soft_cap = soft_cap > 0.0f ? soft_cap : 0.0f;
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  p.alibi_slopes = alibi_slopes;
  p.sinks = sinks;

  // bf16 rows: tensor maps for the prefill's bulk copies straight into the
  // operand tiles (quantised rows are loaded by the converter warps).
  kvq::PrefillMaps maps;
  std::memset(&maps, 0, sizeof(maps));
  if (!s->prefill.empty() && s->dtype == KVQ_AUTO) {
    const int64_t slots = num_blocks * (int64_t)block_size;
    if (!encode_auto_map(&maps.k, key_cache, head_dim, heads_kv, slots) ||
        !encode_auto_map(&maps.v, value_cache, head_dim, heads_kv, slots))
      return KVQ_E_CUDA;
  }
  // The first call with this schedule uploads its plan on the call's
  // stream, ahead of the kernels that read it.
  kvq_sched* ms = const_cast<kvq_sched*>(s);
  if (!ms->uploaded.exchange(true)) {
    if (cudaMemcpyAsync(s->d_buf, s->h_image, s->image_bytes, cudaMemcpyHostToDevice,
                        static_cast<cudaStream_t>(stream)) != cudaSuccess) {
      cudaGetLastError();
      ms->uploaded.store(false);
      return KVQ_E_CUDA;
    }
  }
  if (!s->prefill.empty()) {
    // One persistent CTA per SM (KVQ_PREFILL_CTAS, for tests, forces fewer),
    // never more than tiles (CTA pairs: list entries, two per pair tile).
    int64_t ctas = std::max(1, sm_count());
    if (const char* env = std::getenv("KVQ_PREFILL_CTAS"))
      if (std::atoll(env) > 0) ctas = std::atoll(env);
    ctas = std::min<int64_t>(ctas, (int64_t)s->prefill.size());
    const int rc = kvq::launch_prefill(p, maps, s->dtype, head_dim, ctas, stream);
    if (rc != KVQ_OK) return rc;
  }
  for (int cls = 0; cls < 2; ++cls) {
    const DecodeLaunch& dl = s->launch[cls];
    if (dl.num_chunks == 0) continue;
    p.pieces = reinterpret_cast<const DecodePiece*>(b + s->d_pieces_off) + dl.piece_off;
    p.num_pieces = (int32_t)dl.num_pieces;
    p.warp_seg = reinterpret_cast<const WarpSeg*>(b + s->d_warps_off) + dl.warp_off;
    p.num_chunks = dl.num_chunks;
    p.num_warps = dl.num_warps;
    const int rc = kvq::launch_decode(p, s->dtype, head_dim, cls + 1, stream);
    if (rc != KVQ_OK) return rc;
  }
  return kvq::launch_merge(p, head_dim, s->num_merges, stream);
}

// ---- the fused decode step ------------------------------------------------

namespace {
int step_rows(int max_query_len, int group) { return max_query_len * group <= 8 ? 8 : 16; }
}  // namespace

int kvq_decode_step_workspace_size(int num_req, int heads_q, int heads_kv, int head_dim,
                                   kvq_dtype_t dtype, int max_query_len, int use_alibi,
                                   size_t* workspace_bytes) {
  if (!workspace_bytes) return KVQ_E_INVALID_ARG;
  *workspace_bytes = 0;
  if (num_req < 0 || heads_q <= 0 || heads_kv <= 0 || max_query_len <= 0) return KVQ_E_INVALID_ARG;
  if (!kvq::is_valid_dtype(dtype)) return KVQ_E_INVALID_ARG;
  if (heads_q % heads_kv || !kvq::head_dim_supported(head_dim)) return KVQ_E_UNSUPPORTED;
  const int G = heads_q / heads_kv;
  if ((int64_t)max_query_len * G > kvq::kTileMaxRows) return KVQ_E_UNSUPPORTED;
  if ((int64_t)num_req * heads_kv > kvq::kMaxStepTiles) return KVQ_E_UNSUPPORTED;
  int64_t warps = 0;
  const int rc = kvq::step_warps(dtype, head_dim, use_alibi != 0, step_rows(max_query_len, G), &warps);
  if (rc != KVQ_OK) return rc;
  *workspace_bytes = kvq::step_workspace(num_req * heads_kv, head_dim, warps).total;
  return KVQ_OK;
}

namespace {
// Inputs the fused kernel stages itself: `bytes` at `dev` are a copy of the
// mapped host buffer `host`.  Before its grid barrier the kernel reads the
// inputs that lie in that range from `host` and copies the range to `dev`;
// after the barrier it reads `dev`.
struct StageRange {
  const char* host;
  char* dev;
  size_t bytes;
};

int decode_step_impl(int num_req, int heads_q, int heads_kv, int head_dim, kvq_dtype_t dtype,
                     const void* key, const void* value, int64_t num_new_tokens,
                     int64_t key_stride_tok, int64_t value_stride_tok,
                     const int64_t* slot_mapping, void* key_cache, void* value_cache,
                     int64_t num_blocks, int block_size, const void* q,
                     const int32_t* query_start_loc, const int32_t* seq_lens,
                     const int32_t* block_table, int block_table_stride, int max_query_len,
                     float sm_scale, int window, float soft_cap, const float* alibi_slopes,
                     const float* sinks, float k_scale, float v_scale, void* out,
                     void* workspace, size_t workspace_bytes, void* stream,
                     const StageRange* stage) {
  size_t need = 0;
  int rc = kvq_decode_step_workspace_size(num_req, heads_q, heads_kv, head_dim, dtype,
                                          max_query_len, alibi_slopes != nullptr, &need);
  if (rc != KVQ_OK) return rc;
  if (num_new_tokens < 0 || num_blocks <= 0 || block_table_stride <= 0) return KVQ_E_INVALID_ARG;
  if (block_size <= 0 || block_size % kvq::kChunkTokens) return KVQ_E_UNSUPPORTED;
  if (num_blocks * (int64_t)block_size >= ((int64_t)1 << 31)) return KVQ_E_UNSUPPORTED;
  if (!key_cache || !value_cache || !q || !out || !query_start_loc || !seq_lens || !block_table ||
      !workspace)
    return KVQ_E_INVALID_ARG;
  if (num_new_tokens > 0) {
    const int64_t min_stride = (int64_t)heads_kv * head_dim;
    if (!key || !value || !slot_mapping || key_stride_tok < min_stride ||
        value_stride_tok < min_stride || key_stride_tok % 8 || value_stride_tok % 8 ||
        !aligned(key, 16) || !aligned(value, 16) || !aligned(slot_mapping, 8))
      return KVQ_E_INVALID_ARG;
  }
  if (!aligned(q, 16) || !aligned(key_cache, 16) || !aligned(value_cache, 16) ||
      !aligned(out, 16) || !aligned(block_table, 4) || !aligned(alibi_slopes, 4) ||
      !aligned(sinks, 4) || !aligned(workspace, 256))
    return KVQ_E_INVALID_ARG;
  if (window < 0 || !std::isfinite(sm_scale) || !std::isfinite(soft_cap)) return KVQ_E_INVALID_ARG;
  if (dtype == KVQ_FP8_E4M3 || dtype == KVQ_FP8_E5M2) {
    if (!(std::isfinite(k_scale) && k_scale > 0.0f && std::isfinite(v_scale) && v_scale > 0.0f))
      return KVQ_E_INVALID_ARG;
  }
  if (workspace_bytes < need) return KVQ_E_WORKSPACE_TOO_SMALL;
  const int G = heads_q / heads_kv;
  const int max_rows = step_rows(max_query_len, G);
  int64_t warps = 0;
  rc = kvq::step_warps(dtype, head_dim, alibi_slopes != nullptr, max_rows, &warps);
  if (rc != KVQ_OK) return rc;
  const int num_tiles = num_req * heads_kv;
  const kvq::StepWorkspace lay = kvq::step_workspace(num_tiles, head_dim, warps);
  char* ws = static_cast<char*>(workspace);

  kvq::AttnParams p;
  std::memset(&p, 0, sizeof(p));
  p.q = static_cast<const uint16_t*>(q);
  p.key_cache = static_cast<const uint8_t*>(key_cache);
  p.value_cache = static_cast<const uint8_t*>(value_cache);
  p.query_start_loc = query_start_loc;
  p.seq_lens = seq_lens;
  p.block_table = block_table;
  p.out = static_cast<uint16_t*>(out);
  p.part_o = reinterpret_cast<float*>(ws + lay.o);
  p.part_lse = reinterpret_cast<float*>(ws + lay.lse);
  p.error_flag = reinterpret_cast<int32_t*>(ws);
  p.num_blocks = num_blocks;
  p.block_table_stride = block_table_stride;
  p.block_size = block_size;
  p.heads_q = heads_q;
  p.heads_kv = heads_kv;
  p.group = G;
  p.causal = 1;
  p.window = window;
  p.sm_scale = sm_scale;
  p.soft_cap = soft_cap > 0.0f ? soft_cap : 0.0f;
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  p.alibi_slopes = alibi_slopes;
  p.sinks = sinks;

  kvq::StepParams sp;
  std::memset(&sp, 0, sizeof(sp));
  sp.key = static_cast<const uint16_t*>(key);
  sp.value = static_cast<const uint16_t*>(value);
  sp.num_tokens = num_new_tokens;
  sp.key_stride = key_stride_tok;
  sp.value_stride = value_stride_tok;
  sp.slot_mapping = slot_mapping;
  sp.key_cache = static_cast<uint8_t*>(key_cache);
  sp.value_cache = static_cast<uint8_t*>(value_cache);
  sp.num_slots = num_blocks * (int64_t)block_size;
  sp.prefix = reinterpret_cast<int32_t*>(ws + lay.prefix);
  sp.tiles = reinterpret_cast<int4*>(ws + lay.tiles);
  sp.warp_tile = reinterpret_cast<int32_t*>(ws + lay.warp_tile);
  sp.barrier = reinterpret_cast<uint32_t*>(ws + 128);
  sp.num_req = num_req;
  sp.num_tiles = num_tiles;
  sp.max_rows = max_rows;
  sp.in_query_start_loc = query_start_loc;
  sp.in_seq_lens = seq_lens;
  if (stage && stage->bytes > 0) {
    // what the cache write and the plan read comes from the host buffer
    auto host_side = [&](const void* ptr) -> const void* {
      const char* a = static_cast<const char*>(ptr);
      if (a && a >= stage->dev && a < stage->dev + stage->bytes) return stage->host + (a - stage->dev);
      return ptr;
    };
    sp.key = static_cast<const uint16_t*>(host_side(key));
    sp.value = static_cast<const uint16_t*>(host_side(value));
    sp.slot_mapping = static_cast<const int64_t*>(host_side(slot_mapping));
    sp.in_query_start_loc = static_cast<const int32_t*>(host_side(query_start_loc));
    sp.in_seq_lens = static_cast<const int32_t*>(host_side(seq_lens));
    sp.stage_src = reinterpret_cast<const uint8_t*>(stage->host);
    sp.stage_dst = reinterpret_cast<uint8_t*>(stage->dev);
    sp.stage_bytes = (int64_t)stage->bytes;
  }
  // the fused kernel, then the merge of its cut tiles as a programmatic
  // dependent launch
  rc = kvq::launch_decode_step(p, sp, dtype, head_dim, warps, stream);
  if (rc != KVQ_OK) return rc;
  return kvq::launch_merge_step(p, sp, head_dim, warps, stream);
}
}  // namespace

int kvq_decode_step(int num_req, int heads_q, int heads_kv, int head_dim, kvq_dtype_t dtype,
                    const void* key, const void* value, int64_t num_new_tokens,
                    int64_t key_stride_tok, int64_t value_stride_tok, const int64_t* slot_mapping,
                    void* key_cache, void* value_cache, int64_t num_blocks, int block_size,
                    const void* q, const int32_t* query_start_loc, const int32_t* seq_lens,
                    const int32_t* block_table, int block_table_stride, int max_query_len,
                    float sm_scale, int window, float soft_cap, const float* alibi_slopes,
                    const float* sinks, float k_scale, float v_scale, void* out, void* workspace,
                    size_t workspace_bytes, void* stream) {
  return decode_step_impl(num_req, heads_q, heads_kv, head_dim, dtype, key, value, num_new_tokens,
                          key_stride_tok, value_stride_tok, slot_mapping, key_cache, value_cache,
                          num_blocks, block_size, q, query_start_loc, seq_lens, block_table,
                          block_table_stride, max_query_len, sm_scale, window, soft_cap,
                          alibi_slopes, sinks, k_scale, v_scale, out, workspace, workspace_bytes,
                          stream, nullptr);
}

#define KVQ_STEP_PARAMS                                                                      \
  int num_req, int heads_q, int heads_kv, int head_dim, kvq_dtype_t dtype, const void* key,  \
      const void* value, int64_t num_new_tokens, int64_t key_stride_tok,                      \
      int64_t value_stride_tok, const int64_t* slot_mapping, void* key_cache,                 \
      void* value_cache, int64_t num_blocks, int block_size, const void* q,                   \
      const int32_t* query_start_loc, const int32_t* seq_lens, const int32_t* block_table,    \
      int block_table_stride, int max_query_len, float sm_scale, int window, float soft_cap,  \
      const float* alibi_slopes, const float* sinks, float k_scale, float v_scale, void* out, \
      void* workspace, size_t workspace_bytes
#define KVQ_STEP_ARGS                                                                          \
  num_req, heads_q, heads_kv, head_dim, dtype, key, value, num_new_tokens, key_stride_tok,    \
      value_stride_tok, slot_mapping, key_cache, value_cache, num_blocks, block_size, q,      \
      query_start_loc, seq_lens, block_table, block_table_stride, max_query_len, sm_scale,    \
      window, soft_cap, alibi_slopes, sinks, k_scale, v_scale, out, workspace, workspace_bytes

namespace {
// Where a host-buffer step's bytes go: host_in mapped into the device's
// address space (pinned memory) is staged by the fused kernel itself
// (stage), otherwise copied first (copy_in); out NULL stores the output rows
// into host_out through its mapping (out_dev), otherwise out_bytes are
// copied back.  for_graph: a step to be captured, where a copy from memory
// the device cannot address is refused (KVQ_E_UNSUPPORTED).
struct HostIo {
  StageRange stage;
  bool copy_in;
  void* out_dev;
  size_t out_bytes;
};
int host_io_resolve(const void* host_in, void* dev_in, size_t in_bytes, void* host_out,
                    size_t out_bytes, void* out, bool for_graph, HostIo* io) {
  if ((in_bytes > 0 && (!host_in || !dev_in)) || (out_bytes > 0 && out && !host_out))
    return KVQ_E_INVALID_ARG;
  io->stage = StageRange{nullptr, static_cast<char*>(dev_in), 0};
  io->copy_in = false;
  io->out_dev = out;
  io->out_bytes = out_bytes;
  if (!out) {
    if (!host_out || cudaHostGetDevicePointer(&io->out_dev, host_out, 0) != cudaSuccess ||
        !io->out_dev) {
      cudaGetLastError();
      return KVQ_E_INVALID_ARG;
    }
    io->out_bytes = 0;
  }
  if (in_bytes > 0) {
    void* in_map = nullptr;
    if (cudaHostGetDevicePointer(&in_map, const_cast<void*>(host_in), 0) == cudaSuccess && in_map &&
        aligned(in_map, 16) && aligned(dev_in, 16)) {
      io->stage.host = static_cast<const char*>(in_map);
      io->stage.bytes = in_bytes;
    } else {
      cudaGetLastError();
      if (for_graph) return KVQ_E_UNSUPPORTED;
      io->copy_in = true;
    }
  }
  return KVQ_OK;
}

// The host-buffer step's work on stream s, without the final wait.
int host_io_enqueue(const HostIo& io, const void* host_in, void* dev_in, size_t in_bytes,
                    void* host_out, KVQ_STEP_PARAMS, cudaStream_t s) {
  if (io.copy_in &&
      cudaMemcpyAsync(dev_in, host_in, in_bytes, cudaMemcpyHostToDevice, s) != cudaSuccess) {
    cudaGetLastError();
    return KVQ_E_CUDA;
  }
  {
    // the step writes io.out_dev: `out` itself, or host_out's device mapping
    // (the local name is the one KVQ_STEP_ARGS passes on)
    void* out = io.out_dev;
    const int rc = decode_step_impl(KVQ_STEP_ARGS, s, &io.stage);
    if (rc != KVQ_OK) return rc;
  }
  // (a copy back only when `out` was given, so io.out_dev is `out`)
  if (io.out_bytes > 0 &&
      cudaMemcpyAsync(host_out, io.out_dev, io.out_bytes, cudaMemcpyDeviceToHost, s) != cudaSuccess) {
    cudaGetLastError();
    return KVQ_E_CUDA;
  }
  return KVQ_OK;
}
}  // namespace

int kvq_decode_step_host_io(const void* host_in, void* dev_in, size_t in_bytes, void* host_out,
                            size_t out_bytes, KVQ_STEP_PARAMS, void* stream) {
  HostIo io;
  int rc = host_io_resolve(host_in, dev_in, in_bytes, host_out, out_bytes, out, false, &io);
  if (rc != KVQ_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  rc = host_io_enqueue(io, host_in, dev_in, in_bytes, host_out, KVQ_STEP_ARGS, s);
  if (rc != KVQ_OK) return rc;
  if (cudaStreamSynchronize(s) != cudaSuccess) {
    cudaGetLastError();
    return KVQ_E_CUDA;
  }
  return KVQ_OK;
}

struct kvq_step_graph {
  cudaStream_t capture = nullptr;  // the private stream the step was captured on
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
};

void kvq_decode_step_graph_destroy(kvq_step_graph_t* g) {
  if (!g) return;
  if (g->exec) cudaGraphExecDestroy(g->exec);
  if (g->graph) cudaGraphDestroy(g->graph);
  if (g->capture) cudaStreamDestroy(g->capture);
  cudaGetLastError();
  delete g;
}

int kvq_decode_step_graph_create(const void* host_in, void* dev_in, size_t in_bytes,
                                 void* host_out, size_t out_bytes, KVQ_STEP_PARAMS,
                                 kvq_step_graph_t** graph) {
  if (!graph) return KVQ_E_INVALID_ARG;
  *graph = nullptr;
  HostIo io;
  int rc = host_io_resolve(host_in, dev_in, in_bytes, host_out, out_bytes, out, true, &io);
  if (rc != KVQ_OK) return rc;
  // the launch configuration is looked up (and kept) before the capture, so
  // the capture holds stream work only
  size_t need = 0;
  rc = kvq_decode_step_workspace_size(num_req, heads_q, heads_kv, head_dim, dtype, max_query_len,
                                      alibi_slopes != nullptr, &need);
  if (rc != KVQ_OK) return rc;
  kvq_step_graph_t* g = new (std::nothrow) kvq_step_graph_t();
  if (!g) return KVQ_E_NO_MEMORY;
  if (cudaStreamCreateWithFlags(&g->capture, cudaStreamNonBlocking) != cudaSuccess ||
      cudaStreamBeginCapture(g->capture, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
    cudaGetLastError();
    kvq_decode_step_graph_destroy(g);
    return KVQ_E_CUDA;
  }
  rc = host_io_enqueue(io, host_in, dev_in, in_bytes, host_out, KVQ_STEP_ARGS, g->capture);
  // the capture always ends (a failed step leaves an unusable graph)
  const cudaError_t end = cudaStreamEndCapture(g->capture, &g->graph);
  if (rc != KVQ_OK || end != cudaSuccess || !g->graph ||
      cudaGraphInstantiate(&g->exec, g->graph, 0) != cudaSuccess) {
    cudaGetLastError();
    kvq_decode_step_graph_destroy(g);
    return rc != KVQ_OK ? rc : KVQ_E_CUDA;
  }
  *graph = g;
  return KVQ_OK;
}

int kvq_decode_step_graph_launch(kvq_step_graph_t* g, void* stream) {
  if (!g || !g->exec) return KVQ_E_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaGraphLaunch(g->exec, s) != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess) {
    cudaGetLastError();
    return KVQ_E_CUDA;
  }
  return KVQ_OK;
}

#undef KVQ_STEP_PARAMS
#undef KVQ_STEP_ARGS

int kvq_decode_step_check(const void* workspace) {
  if (!workspace) return KVQ_E_INVALID_ARG;
  int32_t flag = 0;
  if (cudaMemcpy(&flag, workspace, sizeof(flag), cudaMemcpyDeviceToHost) != cudaSuccess) {
    cudaGetLastError();
    return KVQ_E_CUDA;
  }
  if (flag == 0) return KVQ_OK;
  if (cudaMemset(const_cast<void*>(workspace), 0, sizeof(flag)) != cudaSuccess) {
    cudaGetLastError();
    return KVQ_E_CUDA;
  }
  return flag == 1 ? KVQ_E_TIMEOUT : KVQ_E_INVALID_ARG;
}

}  // extern "C"
