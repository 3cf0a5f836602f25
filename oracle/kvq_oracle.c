/*
 * kvq_oracle.c -- plain, slow CPU oracle for quantized paged-KV attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test-suite, the smoke check and the
 * benchmark's CPU-baseline leg load this library.  The product (the CUDA
 * library in int8_kv_cache_reshape_gb300/) never calls it, and the two share
 * no code, header, table or constant generator.
 *
 * Every function restates one step of the method described on three pages
 * about vLLM's quantized KV cache (prhub.com.cn summaries of vLLM pull
 * requests 39445, 50194 and 38378):
 *
 *   [P1] "CPU 后端新增 FP8 KV 缓存量化支持" (vllm PR 39445)
 *        Breakdown item 1 / Key files (cpu_attn_fp8.hpp): scalar fp8 e4m3
 *        quantise and dequantise used to write and read the KV cache;
 *        Review: c10::Float8_e4m3fn / Float8_e5m2 are the two fp8 flavours;
 *        Risks: scale folding of the dequantisation into the attention.
 *   [P2] "修复 CPU FP8 注意力调度器临时缓冲区大小计算错误" (vllm PR 50194)
 *        Key source snippet: kv_cache_dtype "auto"/"fp8_e4m3"/"fp8_e5m2"
 *        = 0/1/2; window_size, soft_cap, causal options of the attention
 *        over a paged cache (block_size, num_blocks).
 *   [P3] "为 Triton 注意力后端引入 KV 缓存按令牌头 INT8/FP8 量化" (vllm PR 38378)
 *        Breakdown item 3 / Risks: per-(token, head) dynamic scale from the
 *        absolute maximum, stored inline in a padded head row; the test's
 *        reference quantiser reproduces the kernel's clamping.
 *
 * Readings where the pages are silent:
 *   - fp8 e4m3 is OCP E4M3FN (bias 7, no infinities, max 448); fp8 e5m2 is
 *     OCP E5M2 (bias 15, IEEE-like, max 57344).  Encoding rounds to nearest,
 *     ties to even, and saturates to the largest finite magnitude (the
 *     "clamping" of [P3] Review read as saturation, not truncation).
 *   - The quotient x / scale is a correctly rounded binary32 division.
 *   - int8 encoding: round half to even, clamp to [-128, 127].
 *   - Per-token-head: s = amax / qmax in binary32, qmax = 127 (int8), 448
 *     (fp8 = e4m3) or 57344 (fp8 e5m2, the "other scale granularities" of
 *     [P3] Risks applied to the e5m2 format); s == 0 gives all-zero codes.
 *     Row layout:
 *     [D codes][s as little-endian binary32][12 zero bytes].
 *   - Paged layout: cache[block][slot_in_block][kv_head][row bytes].
 *   - Query row i of a request with Q queries and L keys sits at position
 *     L - Q + i; key j is visible iff (!causal || j <= p) and
 *     (window <= 0 || p - j < window); soft cap is cap * tanh(z / cap),
 *     applied after the sm_scale and before the softmax.
 *
 * Arithmetic: binary32 exactly where the method fixes it (the quantiser),
 * binary64 everywhere else (dequantised values, scores, softmax, output).
 * No blocking, no fusion, no online softmax: one key at a time, in order.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* dtype numbering: 0..2 follow the kv_cache_dtype indices printed in [P2]'s
 * source snippet; 3 and 4 are the per-token-head modes of [P3]; 5 is the
 * per-token-head mode with e5m2 codes. */
enum { KVO_AUTO = 0, KVO_FP8_E4M3 = 1, KVO_FP8_E5M2 = 2,
       KVO_INT8_PER_TOKEN_HEAD = 3, KVO_FP8_PER_TOKEN_HEAD = 4,
       KVO_FP8_E5M2_PER_TOKEN_HEAD = 5 };
/* fp8 format selector for the scalar codec. */
enum { KVO_E4M3 = 0, KVO_E5M2 = 1 };

/* ------------------------------------------------------------------ */
/* Scalar codecs                                                       */
/* ------------------------------------------------------------------ */

/* bf16 -> binary32: a bf16 value is the top half of a binary32. */
double kvo_bf16_to_double(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

static float bf16_to_float(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* fp8 decode from the OCP 8-bit floating point definition.
 * E4M3FN: sign | 4-bit exponent (bias 7) | 3-bit mantissa; exponent 15 with
 *         mantissa 7 is NaN; there is no infinity; exponent 0 is subnormal,
 *         value m * 2^-9.
 * E5M2:   sign | 5-bit exponent (bias 15) | 2-bit mantissa; exponent 31 is
 *         inf (m = 0) or NaN; exponent 0 is subnormal, value m * 2^-16.
 * [P1] Key files: fp8e4m3_to_float_scalar. */
double kvo_fp8_decode(int fmt, uint8_t code) {
  int sign = code >> 7;
  int e, m;
  double v;
  if (fmt == KVO_E4M3) {
    e = (code >> 3) & 0xF;
    m = code & 0x7;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m, -9);
    else v = ldexp(1.0 + m / 8.0, e - 7);
  } else {
    e = (code >> 2) & 0x1F;
    m = code & 0x3;
    if (e == 31) return m == 0 ? (sign ? -INFINITY : INFINITY) : NAN;
    if (e == 0) v = ldexp((double)m, -16);
    else v = ldexp(1.0 + m / 4.0, e - 15);
  }
  return sign ? -v : v;
}

/* fp8 encode of a binary32: the nearest finite code, ties to the even code
 * (round half to even).  The non-negative finite codes 0 .. max_code have
 * strictly increasing values in both formats, so the nearest one is one of
 * the two codes that bracket |y|: a bisection over the code range finds the
 * largest code whose value is <= |y|, and the nearer of it and the next code
 * wins.  Magnitudes at or beyond the largest finite value saturate to it
 * (satfinite), infinities included.  The sign bit is copied, so a negative
 * value that rounds to zero gives the negative-zero code 0x80.
 *
 * Both distances are exact in binary64: |y| is a binary32 and the two
 * bracketing code values are short multiples of a power of two within a
 * binade of it, so the tie test is exact.
 * [P1] Key files: float_to_fp8e4m3_scalar; [P3] Review (clamping). */
uint8_t kvo_fp8_encode(int fmt, float y) {
  uint8_t max_code = fmt == KVO_E4M3 ? 0x7E : 0x7B;
  uint8_t sign = signbit(y) ? 0x80 : 0x00;
  int lo = 0, hi = max_code; /* invariant: dec(lo) <= a < dec(hi) */
  double a, d_lo, d_hi;
  if (isnan(y)) return 0x7F;
  a = fabs((double)y);
  if (a >= kvo_fp8_decode(fmt, max_code)) return (uint8_t)(sign | max_code);
  while (hi - lo > 1) {
    int mid = (lo + hi) / 2;
    if (kvo_fp8_decode(fmt, (uint8_t)mid) <= a) lo = mid;
    else hi = mid;
  }
  d_lo = a - kvo_fp8_decode(fmt, (uint8_t)lo);
  d_hi = kvo_fp8_decode(fmt, (uint8_t)hi) - a;
  if (d_lo < d_hi || (d_lo == d_hi && (lo & 1) == 0)) return (uint8_t)(sign | lo);
  return (uint8_t)(sign | hi);
}

/* int8 encode: round half to even (rint under the default rounding mode),
 * then clamp to the int8 range.  [P3] Breakdown item 3, Review. */
int8_t kvo_int8_encode(float y) {
  double r = rint((double)y);
  if (r > 127.0) r = 127.0;
  if (r < -128.0) r = -128.0;
  return (int8_t)r;
}

/* ------------------------------------------------------------------ */
/* Cache layout helpers                                                */
/* ------------------------------------------------------------------ */

/* Bytes of one (token, kv_head) row of the cache. */
int64_t kvo_row_bytes(int dtype, int head_dim) {
  switch (dtype) {
    case KVO_AUTO: return 2 * (int64_t)head_dim;
    case KVO_FP8_E4M3:
    case KVO_FP8_E5M2: return head_dim;
    case KVO_INT8_PER_TOKEN_HEAD:
    case KVO_FP8_PER_TOKEN_HEAD:
    case KVO_FP8_E5M2_PER_TOKEN_HEAD: return (int64_t)head_dim + 16;
    default: return -1;
  }
}

static void store_f32_le(uint8_t* p, float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  p[0] = (uint8_t)(u & 0xFF);
  p[1] = (uint8_t)((u >> 8) & 0xFF);
  p[2] = (uint8_t)((u >> 16) & 0xFF);
  p[3] = (uint8_t)((u >> 24) & 0xFF);
}

static float load_f32_le(const uint8_t* p) {
  uint32_t u = (uint32_t)p[0] | ((uint32_t)p[1] << 8) |
               ((uint32_t)p[2] << 16) | ((uint32_t)p[3] << 24);
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* Quantise one (token, head) row of D bf16 values into `row`. */
static void write_row(int dtype, const uint16_t* x, int D, float tensor_scale,
                      uint8_t* row) {
  if (dtype == KVO_AUTO) {
    /* bf16 cache: the row holds the input bytes unchanged (little endian). */
    for (int d = 0; d < D; ++d) {
      row[2 * d] = (uint8_t)(x[d] & 0xFF);
      row[2 * d + 1] = (uint8_t)(x[d] >> 8);
    }
    return;
  }
  if (dtype == KVO_FP8_E4M3 || dtype == KVO_FP8_E5M2) {
    /* per-tensor: code = enc(x / s) with a correctly rounded division. */
    int fmt = dtype == KVO_FP8_E4M3 ? KVO_E4M3 : KVO_E5M2;
    for (int d = 0; d < D; ++d) {
      float y = bf16_to_float(x[d]) / tensor_scale;
      row[d] = kvo_fp8_encode(fmt, y);
    }
    return;
  }
  /* per-token-head: dynamic scale from the row's absolute maximum. */
  {
    float amax = 0.0f, s;
    float qmax = dtype == KVO_INT8_PER_TOKEN_HEAD ? 127.0f
                 : dtype == KVO_FP8_E5M2_PER_TOKEN_HEAD ? 57344.0f : 448.0f;
    for (int d = 0; d < D; ++d) {
      float a = fabsf(bf16_to_float(x[d]));
      if (a > amax) amax = a;
    }
    s = amax / qmax;
    for (int d = 0; d < D; ++d) {
      float y;
      if (s == 0.0f) {
        row[d] = 0;
        continue;
      }
      y = bf16_to_float(x[d]) / s;
      if (dtype == KVO_INT8_PER_TOKEN_HEAD) {
        int8_t c = kvo_int8_encode(y);
        memcpy(&row[d], &c, 1);
      } else {
        row[d] = kvo_fp8_encode(dtype == KVO_FP8_E5M2_PER_TOKEN_HEAD ? KVO_E5M2 : KVO_E4M3, y);
      }
    }
    store_f32_le(row + D, s);
    memset(row + D + 4, 0, 12);
  }
}

/* reshape_and_cache: quantise each new token's K and V rows and place them
 * at slot_mapping[t] of the paged caches.  Negative slots, and slots beyond
 * num_blocks * block_size, are skipped; untouched rows keep their bytes.
 * key/value are bf16 [T, Hkv, D] with a token stride in elements.
 * [P1] Breakdown item 1 (reshape kernel); [P3] Breakdown item 3. */
int kvo_reshape_and_cache(const uint16_t* key, const uint16_t* value,
                          int64_t num_tokens, int64_t key_stride,
                          int64_t value_stride, int num_heads_kv,
                          int head_dim, uint8_t* key_cache,
                          uint8_t* value_cache, int64_t num_blocks,
                          int block_size, const int64_t* slot_mapping,
                          int dtype, float k_scale, float v_scale) {
  int64_t row = kvo_row_bytes(dtype, head_dim);
  if (row < 0) return -1;
  /* Tokens are independent (each slot is written by one token; a slot
   * named twice has no defined winner, here or in any parallel writer). */
#pragma omp parallel for schedule(dynamic, 64)
  for (int64_t t = 0; t < num_tokens; ++t) {
    int64_t slot = slot_mapping[t];
    int64_t blk, off;
    if (slot < 0 || slot >= num_blocks * (int64_t)block_size) continue;
    blk = slot / block_size;
    off = slot % block_size;
    for (int h = 0; h < num_heads_kv; ++h) {
      int64_t base = ((blk * block_size + off) * num_heads_kv + h) * row;
      write_row(dtype, key + t * key_stride + (int64_t)h * head_dim, head_dim,
                k_scale, key_cache + base);
      write_row(dtype, value + t * value_stride + (int64_t)h * head_dim,
                head_dim, v_scale, value_cache + base);
    }
  }
  return 0;
}

/* Dequantised values of one cache row (binary64): out[d] = dec(code_d) *
 * scale, with the per-tensor scale (fp8_e4m3 / fp8_e5m2) or the row's
 * inline scale (per-token-head); a bf16 row ("auto") is read as is.  `dec`
 * is the fp8 decode of the row's format, tabulated once per call from
 * kvo_fp8_decode (the same values). */
static void dequant_row(int dtype, const double* dec, const uint8_t* row, int D,
                        float tensor_scale, double* out) {
  switch (dtype) {
    case KVO_AUTO:
      for (int d = 0; d < D; ++d) {
        uint16_t b = (uint16_t)(row[2 * d] | (row[2 * d + 1] << 8));
        out[d] = kvo_bf16_to_double(b);
      }
      return;
    case KVO_FP8_E4M3:
    case KVO_FP8_E5M2:
      for (int d = 0; d < D; ++d) out[d] = dec[row[d]] * (double)tensor_scale;
      return;
    case KVO_INT8_PER_TOKEN_HEAD: {
      double s = (double)load_f32_le(row + D);
      for (int d = 0; d < D; ++d) {
        int8_t c;
        memcpy(&c, &row[d], 1);
        out[d] = (double)c * s;
      }
      return;
    }
    case KVO_FP8_PER_TOKEN_HEAD:
    case KVO_FP8_E5M2_PER_TOKEN_HEAD: {
      double s = (double)load_f32_le(row + D);
      for (int d = 0; d < D; ++d) out[d] = dec[row[d]] * s;
      return;
    }
    default:
      for (int d = 0; d < D; ++d) out[d] = NAN;
  }
}

/* ------------------------------------------------------------------ */
/* Attention over the paged cache                                      */
/* ------------------------------------------------------------------ */

typedef struct {
  int num_req, heads_q, heads_kv, head_dim;
  const uint16_t* q;
  const uint8_t *key_cache, *value_cache;
  int block_size;
  int dtype;
  int64_t row_bytes;
  const int32_t *query_start_loc, *seq_lens, *block_table;
  int block_table_stride;
  double sm_scale;
  int causal, window;
  double soft_cap;
  float k_scale, v_scale;
  const float* alibi_slopes; /* [heads_q] or NULL */
  const float* sinks;        /* [heads_q] or NULL */
  double dec[256];           /* fp8 decode of the cache's code format */
} attn_args;

/* Address of the cache row of logical key j of request r, kv head h. */
static const uint8_t* cache_row(const attn_args* a, const uint8_t* cache,
                                int r, int64_t j, int h) {
  int64_t phys = a->block_table[(int64_t)r * a->block_table_stride +
                                j / a->block_size];
  int64_t slot = phys * a->block_size + j % a->block_size;
  return cache + (slot * a->heads_kv + h) * a->row_bytes;
}

static int request_of(const attn_args* a, int64_t tok) {
  for (int r = 0; r < a->num_req; ++r)
    if (tok >= a->query_start_loc[r] && tok < a->query_start_loc[r + 1])
      return r;
  return -1;
}

/* Per-thread work buffers: D doubles each. */
typedef struct {
  double *q, *k, *v, *o, *e, *wv, *va;
} row_bufs;

/* Scores of query token `tok`, q head `hq` against every key of its request;
 * probs[j] is the softmax weight (0 for masked keys).  *sink_w receives the
 * weight of the attention sink (0 without one).  Returns L, or -1.
 *   z_j = sm_scale * (q . k_j);  z_j <- cap * tanh(z_j / cap) with a soft
 *   cap;  z_j <- z_j + slope * (j - p) with ALiBi;  P = softmax over the
 *   visible keys and, with a sink, the sink's logit s (no value). */
static int64_t row_probs(const attn_args* a, int64_t tok, int hq, double* probs,
                         double* sink_w, int64_t cap, const row_bufs* b) {
  int r = request_of(a, tok);
  int64_t L, Q, p;
  int G, hk, D = a->head_dim;
  const uint16_t* qrow;
  double m = -INFINITY, sum = 0.0, sink = -INFINITY;
  *sink_w = 0.0;
  if (r < 0) return -1;
  L = a->seq_lens[r];
  Q = a->query_start_loc[r + 1] - a->query_start_loc[r];
  p = L - Q + (tok - a->query_start_loc[r]);
  if (L > cap) return -1;
  G = a->heads_q / a->heads_kv;
  hk = hq / G;
  qrow = a->q + (tok * a->heads_q + hq) * (int64_t)D;
  for (int d = 0; d < D; ++d) b->q[d] = kvo_bf16_to_double(qrow[d]);
  for (int64_t j = 0; j < L; ++j) {
    int visible = (!a->causal || j <= p) && (a->window <= 0 || p - j < a->window);
    double z = 0.0;
    if (!visible) {
      probs[j] = -INFINITY;
      continue;
    }
    dequant_row(a->dtype, a->dec, cache_row(a, a->key_cache, r, j, hk), D, a->k_scale, b->k);
    for (int d = 0; d < D; ++d) z += b->q[d] * b->k[d];
    z *= a->sm_scale;
    if (a->soft_cap > 0.0) z = a->soft_cap * tanh(z / a->soft_cap);
    if (a->alibi_slopes) z += (double)a->alibi_slopes[hq] * (double)(j - p);
    probs[j] = z;
    if (z > m) m = z;
  }
  if (a->sinks) {
    sink = (double)a->sinks[hq];
    if (sink > m) m = sink;
  }
  for (int64_t j = 0; j < L; ++j) {
    if (probs[j] == -INFINITY) {
      probs[j] = 0.0;
      continue;
    }
    probs[j] = exp(probs[j] - m);
    sum += probs[j];
  }
  if (a->sinks) {
    *sink_w = exp(sink - m);
    sum += *sink_w;
  }
  if (sum > 0.0) {
    for (int64_t j = 0; j < L; ++j) probs[j] /= sum;
    *sink_w /= sum;
  }
  return L;
}

/* o = sum_j P_j * v_j for one (token, q head), accumulated key by key in
 * order for every d; returns 0 or -1. */
static int row_output(const attn_args* a, int64_t tok, int hq, float* out,
                      double* probs, int64_t cap, const row_bufs* b) {
  double sink_w;
  int64_t L = row_probs(a, tok, hq, probs, &sink_w, cap, b);
  int r = request_of(a, tok);
  int D = a->head_dim, G = a->heads_q / a->heads_kv, hk = hq / G;
  if (L < 0) return -1;
  for (int d = 0; d < D; ++d) b->o[d] = 0.0;
  for (int64_t j = 0; j < L; ++j) {
    if (probs[j] == 0.0) continue;
    dequant_row(a->dtype, a->dec, cache_row(a, a->value_cache, r, j, hk), D, a->v_scale, b->v);
    for (int d = 0; d < D; ++d) b->o[d] += probs[j] * b->v[d];
  }
  for (int d = 0; d < D; ++d) out[d] = (float)b->o[d];
  return 0;
}

static int code_format_of(int dtype) {
  return dtype == KVO_FP8_E5M2 || dtype == KVO_FP8_E5M2_PER_TOKEN_HEAD ? KVO_E5M2 : KVO_E4M3;
}

static attn_args make_args(int num_req, int heads_q, int heads_kv,
                           int head_dim, const uint16_t* q,
                           const uint8_t* key_cache, const uint8_t* value_cache,
                           int block_size, int dtype,
                           const int32_t* query_start_loc,
                           const int32_t* seq_lens, const int32_t* block_table,
                           int block_table_stride, double sm_scale, int causal,
                           int window, double soft_cap, float k_scale,
                           float v_scale, const float* alibi_slopes,
                           const float* sinks) {
  attn_args a;
  a.num_req = num_req;
  a.heads_q = heads_q;
  a.heads_kv = heads_kv;
  a.head_dim = head_dim;
  a.q = q;
  a.key_cache = key_cache;
  a.value_cache = value_cache;
  a.block_size = block_size;
  a.dtype = dtype;
  a.row_bytes = kvo_row_bytes(dtype, head_dim);
  a.query_start_loc = query_start_loc;
  a.seq_lens = seq_lens;
  a.block_table = block_table;
  a.block_table_stride = block_table_stride;
  a.sm_scale = sm_scale;
  a.causal = causal;
  a.window = window;
  a.soft_cap = soft_cap;
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  a.alibi_slopes = alibi_slopes;
  a.sinks = sinks;
  for (int c = 0; c < 256; ++c) a.dec[c] = kvo_fp8_decode(code_format_of(dtype), (uint8_t)c);
  return a;
}

static int64_t max_seq_len(const attn_args* a) {
  int64_t m = 1;
  for (int r = 0; r < a->num_req; ++r)
    if (a->seq_lens[r] > m) m = a->seq_lens[r];
  return m;
}

static double* alloc_bufs(row_bufs* b, int D) {
  double* mem = (double*)malloc(sizeof(double) * 7 * (size_t)D);
  if (mem) {
    b->q = mem;
    b->k = mem + D;
    b->v = mem + 2 * D;
    b->o = mem + 3 * D;
    b->e = mem + 4 * D;
    b->wv = mem + 5 * D;
    b->va = mem + 6 * D;
  }
  return mem;
}

/* Attention output (binary32) for the listed query tokens, all q heads:
 * out[i][hq][d] for tokens[i].  tokens == NULL means every token
 * 0 .. query_start_loc[num_req]-1 (then n_tokens is ignored).
 * alibi_slopes / sinks: per q head, or NULL for none.
 * [P1] Breakdown items 2-3 (attention over the fp8 cache, scale folding);
 * [P2] Key source snippet (causal, window_size, soft_cap, paged blocks,
 * use_alibi, use_sink). */
int kvo_attention(int num_req, int heads_q, int heads_kv, int head_dim,
                  const uint16_t* q, const uint8_t* key_cache,
                  const uint8_t* value_cache, int block_size, int dtype,
                  const int32_t* query_start_loc, const int32_t* seq_lens,
                  const int32_t* block_table, int block_table_stride,
                  double sm_scale, int causal, int window, double soft_cap,
                  float k_scale, float v_scale, const float* alibi_slopes,
                  const float* sinks, const int64_t* tokens, int64_t n_tokens,
                  float* out) {
  attn_args a;
  int64_t cap, n, work;
  int failed = 0;
  if (heads_kv <= 0 || heads_q % heads_kv != 0 || kvo_row_bytes(dtype, head_dim) < 0)
    return -1;
  a = make_args(num_req, heads_q, heads_kv, head_dim, q, key_cache, value_cache, block_size,
                dtype, query_start_loc, seq_lens, block_table, block_table_stride, sm_scale,
                causal, window, soft_cap, k_scale, v_scale, alibi_slopes, sinks);
  cap = max_seq_len(&a);
  n = tokens ? n_tokens : query_start_loc[num_req];
  work = n * heads_q;
#pragma omp parallel
  {
    double* probs = (double*)malloc(sizeof(double) * (size_t)cap);
    row_bufs b;
    double* mem = alloc_bufs(&b, head_dim);
#pragma omp for schedule(dynamic, 1)
    for (int64_t w = 0; w < work; ++w) {
      int64_t i = w / heads_q;
      int hq = (int)(w % heads_q);
      int64_t tok = tokens ? tokens[i] : i;
      if (!probs || !mem ||
          row_output(&a, tok, hq, out + (i * heads_q + hq) * (int64_t)head_dim, probs, cap,
                     &b) != 0) {
#pragma omp atomic write
        failed = 1;
      }
    }
    free(probs);
    free(mem);
  }
  return failed ? -1 : 0;
}

/* Softmax weights of one (token, q head) over its request's L keys
 * (masked keys get 0), and in *sink_w the sink's weight.  probs must hold
 * max seq_len doubles.  Returns L. */
int64_t kvo_attention_probs(int num_req, int heads_q, int heads_kv,
                            int head_dim, const uint16_t* q,
                            const uint8_t* key_cache, int block_size, int dtype,
                            const int32_t* query_start_loc,
                            const int32_t* seq_lens, const int32_t* block_table,
                            int block_table_stride, double sm_scale, int causal,
                            int window, double soft_cap, float k_scale,
                            const float* alibi_slopes, const float* sinks,
                            int64_t token, int head_q, double* probs, double* sink_w) {
  attn_args a;
  row_bufs b;
  double* mem;
  int64_t L;
  if (heads_kv <= 0 || heads_q % heads_kv != 0 || kvo_row_bytes(dtype, head_dim) < 0)
    return -1;
  a = make_args(num_req, heads_q, heads_kv, head_dim, q, key_cache, NULL, block_size, dtype,
                query_start_loc, seq_lens, block_table, block_table_stride, sm_scale, causal,
                window, soft_cap, k_scale, 1.0f, alibi_slopes, sinks);
  mem = alloc_bufs(&b, head_dim);
  if (!mem) return -1;
  L = row_probs(&a, token, head_q, probs, sink_w, max_seq_len(&a), &b);
  free(mem);
  return L;
}

/* ------------------------------------------------------------------ */
/* Forward error bound of a binary32 evaluation (test tolerance)       */
/* ------------------------------------------------------------------ */

/* First-order bound on |o_fp32 - o| for one output element when the
 * attention above is evaluated the way a GPU kernel does it: scores
 * s_j = sm_scale * (q . k_j) accumulated in binary32 (any order, up to
 * 2^-23 relative error per operation, so truncating accumulators are
 * covered), softmax weights rounded to a format with an 11-bit significand
 * (binary16: relative error <= 2^-11), and the weighted sums of values and
 * weights accumulated in binary32.
 *
 *   s_j -> s_j + e_j,  |e_j| <= gamma_{D+4} * A_j  (+ 2^-20 * cap with a soft
 *   cap: tanh evaluated to a few ulp; the cap's derivative is <= 1; + 2^-21
 *   * |slope (j - p)| with ALiBi: the bias formed and added in binary32),
 *   where A_j = sm_scale * sum_d |q_d| |k_jd| and gamma_n = n 2^-23 /
 *   (1 - n 2^-23); a score perturbation moves the output by
 *   sum_j w_j (v_j - o) e_j to first order (softmax derivative), and the
 *   weight / sum rounding by at most (2^-11 + gamma_{2n+8}) sum_j w_j |v_j|
 *   over the n visible keys (n + 1 with a sink), plus
 *   2^-25 sum_j |v_j| / sum_j p_j for weights that fall below the binary16
 *   normal range (absolute error 2^-25 with the largest unnormalised
 *   weight p at 1).
 *
 * The bound is the sum of those terms; it is zero only where nothing is
 * visible.  Used by the tests to widen the stated tolerance by what
 * binary32 arithmetic itself cannot avoid on inputs with outliers. */
static double gamma_n(double n) {
  const double u = 1.0 / 8388608.0; /* 2^-23 */
  return n * u / (1.0 - n * u);
}

static int row_bound(const attn_args* a, int64_t tok, int hq, float* out,
                     double* probs, double* err, int64_t cap, const row_bufs* b) {
  double sink_w;
  int64_t L = row_probs(a, tok, hq, probs, &sink_w, cap, b);
  int r = request_of(a, tok);
  int D = a->head_dim, G = a->heads_q / a->heads_kv, hk = hq / G;
  int64_t n = 0, p;
  if (L < 0) return -1;
  p = L - (a->query_start_loc[r + 1] - a->query_start_loc[r]) + (tok - a->query_start_loc[r]);
  for (int64_t j = 0; j < L; ++j) {
    double A = 0.0;
    err[j] = 0.0;
    if (probs[j] == 0.0) continue;
    ++n;
    dequant_row(a->dtype, a->dec, cache_row(a, a->key_cache, r, j, hk), D, a->k_scale, b->k);
    for (int d = 0; d < D; ++d) A += fabs(b->q[d] * b->k[d]);
    err[j] = gamma_n(D + 4) * A * fabs(a->sm_scale);
    if (a->soft_cap > 0.0) err[j] += a->soft_cap / 1048576.0; /* 2^-20 cap */
    if (a->alibi_slopes)
      err[j] += fabs((double)a->alibi_slopes[hq] * (double)(j - p)) / 2097152.0; /* 2^-21 */
  }
  if (a->sinks) ++n;
  /* sum_j p_j with the largest p at 1: the softmax normaliser of the
   * unnormalised weights a kernel rounds */
  double lsum = 0.0, pmax = sink_w;
  for (int64_t j = 0; j < L; ++j)
    if (probs[j] > pmax) pmax = probs[j];
  for (int64_t j = 0; j < L; ++j) lsum += probs[j] / (pmax > 0.0 ? pmax : 1.0);
  lsum += sink_w / (pmax > 0.0 ? pmax : 1.0);
  for (int d = 0; d < D; ++d) {
    b->o[d] = 0.0;
    b->e[d] = 0.0;
    b->wv[d] = 0.0;
    b->va[d] = 0.0;
  }
  for (int64_t j = 0; j < L; ++j) {
    if (probs[j] == 0.0) continue;
    dequant_row(a->dtype, a->dec, cache_row(a, a->value_cache, r, j, hk), D, a->v_scale, b->v);
    for (int d = 0; d < D; ++d) b->o[d] += probs[j] * b->v[d];
  }
  for (int64_t j = 0; j < L; ++j) {
    if (probs[j] == 0.0) continue;
    dequant_row(a->dtype, a->dec, cache_row(a, a->value_cache, r, j, hk), D, a->v_scale, b->v);
    for (int d = 0; d < D; ++d) {
      b->e[d] += probs[j] * fabs(b->v[d] - b->o[d]) * err[j];
      b->wv[d] += probs[j] * fabs(b->v[d]);
      b->va[d] += fabs(b->v[d]);
    }
  }
  for (int d = 0; d < D; ++d)
    out[d] = (float)(b->e[d] + (1.0 / 2048.0 + gamma_n(2.0 * (double)n + 8.0)) * b->wv[d] +
                     b->va[d] / 33554432.0 / (lsum > 0.0 ? lsum : 1.0));
  return 0;
}

/* The bound above for the listed query tokens, all q heads (layout and
 * arguments as kvo_attention). */
int kvo_attention_fp32_bound(int num_req, int heads_q, int heads_kv, int head_dim,
                             const uint16_t* q, const uint8_t* key_cache,
                             const uint8_t* value_cache, int block_size, int dtype,
                             const int32_t* query_start_loc, const int32_t* seq_lens,
                             const int32_t* block_table, int block_table_stride,
                             double sm_scale, int causal, int window, double soft_cap,
                             float k_scale, float v_scale, const float* alibi_slopes,
                             const float* sinks, const int64_t* tokens, int64_t n_tokens,
                             float* out) {
  attn_args a;
  int64_t cap, n, work;
  int failed = 0;
  if (heads_kv <= 0 || heads_q % heads_kv != 0 || kvo_row_bytes(dtype, head_dim) < 0)
    return -1;
  a = make_args(num_req, heads_q, heads_kv, head_dim, q, key_cache, value_cache, block_size,
                dtype, query_start_loc, seq_lens, block_table, block_table_stride, sm_scale,
                causal, window, soft_cap, k_scale, v_scale, alibi_slopes, sinks);
  cap = max_seq_len(&a);
  n = tokens ? n_tokens : query_start_loc[num_req];
  work = n * heads_q;
#pragma omp parallel
  {
    double* probs = (double*)malloc(sizeof(double) * (size_t)cap);
    double* err = (double*)malloc(sizeof(double) * (size_t)cap);
    row_bufs b;
    double* mem = alloc_bufs(&b, head_dim);
#pragma omp for schedule(dynamic, 1)
    for (int64_t w = 0; w < work; ++w) {
      int64_t i = w / heads_q;
      int hq = (int)(w % heads_q);
      int64_t tok = tokens ? tokens[i] : i;
      if (!probs || !err || !mem ||
          row_bound(&a, tok, hq, out + (i * heads_q + hq) * (int64_t)head_dim, probs, err, cap,
                    &b) != 0) {
#pragma omp atomic write
        failed = 1;
      }
    }
    free(probs);
    free(err);
    free(mem);
  }
  return failed ? -1 : 0;
}

/* Threads the OpenMP loops use (reported with CPU timings). */
int kvo_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
