// Inner arithmetic of the decode expert pass: one 16-byte unit of e2m1 codes
// (32 elements, one or two scale blocks) against FP16 activations, with the
// products formed exactly in FP32 ("Running a 133 GB MoE model on an 8 GB GPU
// at 11 tokens/s by streaming experts from NVMe", section "The engine", item
// 4: dequantise with the hardware e2m1 convert, multiply by the block scale).
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

#include "common.cuh"

namespace moe {
namespace dm {

// FP16 x FP16 -> FP32 fused multiply-add on the low halves (the product of
// two FP16 values is exact in FP32).
__device__ __forceinline__ float fma_h(uint32_t a_lo16, uint32_t b_lo16, float c) {
  float d;
  asm("fma.rn.f32.f16 %0, %1, %2, %3;"
      : "=f"(d)
      : "h"((uint16_t)(a_lo16 & 0xFFFFu)), "h"((uint16_t)(b_lo16 & 0xFFFFu)), "f"(c));
  return d;
}

// 8 e2m1 codes (one word) -> 4 f16x2; element 2i in the low half of h[i].
__device__ __forceinline__ void cvt_e2m1x8(uint32_t w, uint32_t (&h)[4]) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(w));
}

__device__ __forceinline__ __half2 as_h2(uint32_t v) { return *reinterpret_cast<const __half2*>(&v); }

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Block sums a (elements 0-15) and b (16-31) times the unit's scale(s):
// NVFP4 has one E4M3 scale per 16 elements, MXFP4 one UE8M0 per 32.
template <int FMT>
__device__ __forceinline__ float apply_scale(float a, float b, uint32_t sbits) {
  if (FMT == MOE_FMT_NVFP4) {
    const float2 s = e4m3x2_to_f32x2(sbits);
    return a * s.x + b * s.y;
  } else {
    return (a + b) * ue8m0_to_f32(sbits);
  }
}

// Scale byte(s) of one unit, from shared memory.
template <int FMT>
__device__ __forceinline__ uint32_t scale_bits(const uint8_t* sp) {
  return FMT == MOE_FMT_NVFP4 ? (uint32_t)sp[0] | ((uint32_t)sp[1] << 8) : (uint32_t)sp[0];
}

// One unit against FP16 activations held in registers (x[qq] = elements
// 8qq .. 8qq + 7 as 4 f16x2), so that one load of x serves several rows.
template <int FMT>
__device__ __forceinline__ float unit_dot_hx(uint4 q, uint32_t sbits, const uint4 (&x)[4]) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int wi = 0; wi < 4; ++wi) {
    const uint32_t xv[4] = {x[wi].x, x[wi].y, x[wi].z, x[wi].w};
    uint32_t h[4];
    cvt_e2m1x8(w[wi], h);
    const int a0 = (wi >> 1) * 2;
#pragma unroll
    for (int bi = 0; bi < 4; ++bi) {
      acc[a0] = fma_h(h[bi], xv[bi], acc[a0]);
      acc[a0 + 1] = fma_h(h[bi] >> 16, xv[bi] >> 16, acc[a0 + 1]);
    }
  }
  return apply_scale<FMT>(acc[0] + acc[1], acc[2] + acc[3], sbits);
}

// One unit against an FP32 operand stored as 4 quads of 8 floats, quad qq at
// hq + qq * qstride floats; the e2m1 values are exact in FP32 and the
// products are formed with packed FP32 FMAs.
template <int FMT>
__device__ __forceinline__ float unit_dot_f32(uint4 q, uint32_t sbits, const float* hq, int qstride) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
  float2 acc[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
  for (int wi = 0; wi < 4; ++wi) {
    const float4 h0 = *reinterpret_cast<const float4*>(hq + wi * qstride);
    const float4 h1 = *reinterpret_cast<const float4*>(hq + wi * qstride + 4);
    const float2 hv[4] = {make_float2(h0.x, h0.y), make_float2(h0.z, h0.w), make_float2(h1.x, h1.y),
                          make_float2(h1.z, h1.w)};
    uint32_t c[4];
    cvt_e2m1x8(w[wi], c);
#pragma unroll
    for (int bi = 0; bi < 4; ++bi) acc[wi >> 1] = ffma2(__half22float2(as_h2(c[bi])), hv[bi], acc[wi >> 1]);
  }
  return apply_scale<FMT>(acc[0].x + acc[0].y, acc[1].x + acc[1].y, sbits);
}

// Power-of-two exponent e with m * 2^e in [2^14, 2^15) for finite m > 0,
// clamped to [-120, 120]; 0 for zero, infinity or NaN.  Scaling FP16
// operands by 2^e and the FP32 sums by 2^-e is exact, so it changes no
// result except where unscaled FP16 would overflow or lose bits to underflow.
__device__ __forceinline__ int f16_shift(float m) {
  const int b = (__float_as_int(m) >> 23) & 0xFF;
  if (!(m > 0.f) || b == 0xFF) return 0;
  if (b == 0) return 120;
  const int e = 14 - (b - 127);
  return e < -120 ? -120 : (e > 120 ? 120 : e);
}
__device__ __forceinline__ float pow2f(int e) { return __int_as_float((127 + e) << 23); }

// Max of v over the lanes with the same key (all 32 lanes take part; lanes
// with key < 0 are ignored); true on the lowest lane of each real group.
__device__ __forceinline__ bool group_max(int key, unsigned& v) {
  const unsigned peers = __match_any_sync(0xffffffffu, key);
  v = __reduce_max_sync(peers, v);
  return key >= 0 && (int)(threadIdx.x & 31) == __ffs(peers) - 1;
}

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

// Checks one routed pair; returns the record or nullptr (and flags status).
__device__ __forceinline__ const uint8_t* checked_record(int e, int E, const void* const* ptrs,
                                                         int32_t* st) {
  if (e < 0 || e >= E) {
    status_or(st, MOE_DEV_BAD_INDEX);
    return nullptr;
  }
  const uint8_t* r = reinterpret_cast<const uint8_t*>(ptrs[e]);
  if (!r) {
    status_or(st, MOE_DEV_NULL_EXPERT);
    return nullptr;
  }
  if ((reinterpret_cast<uintptr_t>(r) & 15u) != 0) {
    status_or(st, MOE_DEV_MISALIGNED);
    return nullptr;
  }
  return r;
}

}  // namespace dm
}  // namespace moe
