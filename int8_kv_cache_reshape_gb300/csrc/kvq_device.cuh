// kvq_device.cuh -- small device helpers written as inline PTX for sm_103a:
// fp8 / int8 codecs, warp-level f16 MMA, register transposes, async copies.
#pragma once

#include <cstdint>

#include <cuda_runtime.h>

#include "../../include/kvq.h"
#include "kvq_internal.h"

namespace kvq {
namespace dev {

// ---- bf16 ------------------------------------------------------------------
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  // cvt packs its first operand into the upper half.
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// ---- fp8 / int8 encode (cache writer) --------------------------------------
// Two fp32 -> two fp8 codes, round to nearest even, saturating to the
// largest finite magnitude.  Result: lo code in bits 0-7, hi in 8-15.
__device__ __forceinline__ uint32_t enc_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ uint32_t enc_e5m2x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}
// int8: round half to even, then clamp to [-128, 127].
__device__ __forceinline__ uint32_t enc_int8(float y) {
  int v = __float2int_rn(y);
  v = max(-128, min(127, v));
  return (uint32_t)v & 0xFFu;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

// ---- code pairs -> f16x2 (exact) ---------------------------------------------
// `pair` holds two codes: bits 0-7 -> low half, bits 8-15 -> high half.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t pair) {
  uint32_t r;
  uint16_t p16 = (uint16_t)pair;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(p16));
  return r;
}
// An E5M2 code is the upper byte of the f16 with the same value.
__device__ __forceinline__ uint32_t e5m2x2_to_f16x2(uint32_t pair) {
  return ((pair & 0xFFu) << 8) | ((pair & 0xFF00u) << 16);
}
// int8 x2 -> f16x2: bias to unsigned, place under the f16 exponent of 1024
// (0x64 high byte: 1024 + u exactly), subtract 1024 + 128.
__device__ __forceinline__ uint32_t int8x2_to_f16x2(uint32_t pair) {
  uint32_t u = (pair ^ 0x8080u);
  uint32_t w;
  asm("prmt.b32 %0, %1, %2, 0x7170;" : "=r"(w) : "r"(u), "r"(0x64646464u));
  uint32_t r;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(w), "r"(0x64806480u));
  return r;
}

template <int DT>
__device__ __forceinline__ uint32_t codes_to_f16x2(uint32_t pair) {
  constexpr int F = code_format(DT);
  if constexpr (F == KVQ_FP8_E5M2) return e5m2x2_to_f16x2(pair);
  else if constexpr (F == KVQ_INT8_PER_TOKEN_HEAD) return int8x2_to_f16x2(pair);
  else return e4m3x2_to_f16x2(pair);
}

// Four codes (one 32-bit word) -> two f16x2: lo gets bytes 0-1, hi bytes
// 2-3.  The word is split into its 16-bit halves inside the asm block.
template <int DT>
__device__ __forceinline__ void word_to_f16x2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  constexpr int F = code_format(DT);
  if constexpr (F == KVQ_FP8_E5M2) {
    // E5M2 code = upper byte of the f16: place each byte above a zero byte.
    lo = prmt(w, 0u, 0x1404u);
    hi = prmt(w, 0u, 0x3424u);
  } else if constexpr (F == KVQ_INT8_PER_TOKEN_HEAD) {
    // bias to unsigned, put each byte under the f16 exponent of 1024 (0x64),
    // subtract 1024 + 128.
    const uint32_t u = w ^ 0x80808080u;
    const uint32_t a = prmt(u, 0x64646464u, 0x7170u);
    const uint32_t b = prmt(u, 0x64646464u, 0x7372u);
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(a), "r"(0x64806480u));
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(b), "r"(0x64806480u));
  } else {
    asm("{\n\t.reg .b16 l16, h16;\n\t"
        "mov.b32 {l16, h16}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, l16;\n\t"
        "cvt.rn.f16x2.e4m3x2 %1, h16;\n\t}"
        : "=r"(lo), "=r"(hi) : "r"(w));
  }
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// ---- warp MMA: D(16x8, f32) += A(16x16, f16) * B(16x8, f16) ----------------
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4],
                                              uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// The same with bf16 A and B (the "auto" cache's bf16 rows).
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4],
                                               uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Transpose an 8x8 matrix of 16-bit values held one row-pair per lane.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t r;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(r) : "r"(x));
  return r;
}

// ---- async global -> shared copies ------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
// 16-byte copy through L2 only; src_bytes = 0 writes zeros without reading.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;"
               :: "r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_8(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8, %2;"
               :: "r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" :: "n"(N) : "memory");
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

// Streaming 16-byte global load (read once, do not keep in L1).
__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

// The same without the non-coherent path: for data that other CTAs of the
// same kernel wrote before a grid barrier.
__device__ __forceinline__ uint4 ldg_stream_coherent(const void* p) {
  uint4 v;
  asm volatile("ld.global.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

__device__ __forceinline__ float fast_exp2(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// tanh(x) = 1 - 2 / (1 + e^(2x)), with e^(2x) = 2^(2 x log2 e): one exp2 and
// one reciprocal.  The absolute error stays within a few 2^-23 over the whole
// range (the result is needed to an absolute, not relative, accuracy: the
// soft cap multiplies it by the cap); +-inf give +-1.
__device__ __forceinline__ float tanh_exp(float x) {
  const float e = fast_exp2(x * 2.8853900817779268f);  // 2 log2(e)
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(1.0f + e));
  return fmaf(-2.0f, r, 1.0f);
}

}  // namespace dev
}  // namespace kvq
