// Activation quantisers of the prefill regime: FP4 for FP4 weights
// (block-scaled FP4 x FP4), MXFP8 for MXFP8 weights (W8A8).
//
// MXFP8 (OCP MX v1.0 conversion, E4M3 elements): per 32 values X =
// floor(log2(amax)) - 8, clamped to [-127, 127] (-127 for an all-zero block);
// elements v * 2^-X rounded to E4M3, nearest even, saturating at 448, sign
// kept.
//
// MXFP4 (OCP Microscaling v1.0 conversion): per 32 values along K the shared
// exponent is X = floor(log2(amax)) - 2, clamped to [-127, 127] (-127 for an
// all-zero block); elements v * 2^-X rounded to E2M1, nearest-even,
// saturating at 6.  NVFP4: per 16 values the E4M3 scale is
// RNE_sat((amax / 6) / g) with g the layer's static activation scale;
// elements v / (scale * g) rounded to E2M1 (all zero if the scale is 0).
// Quotients are IEEE fp32.  Rounding keeps the sign: a negative value that
// rounds to zero encodes as -0 (code 8).
#pragma once
#include "common.cuh"

namespace moe {

// E2M1 codes of (lo, hi), packed lo in bits 0..3, hi in bits 4..7.
MOE_DEV uint32_t e2m1_pack2(float lo, float hi) {
  uint32_t r;
  asm("{\n\t.reg .b8 q;\n\tcvt.rn.satfinite.e2m1x2.f32 q, %1, %2;\n\tcvt.u32.u8 %0, q;\n\t}"
      : "=r"(r) : "f"(hi), "f"(lo));
  // keep the sign of values that round to zero (IEEE semantics)
  r |= ((__float_as_uint(lo) >> 31) << 3) | ((__float_as_uint(hi) >> 31) << 7);
  return r & 0xffu;
}

MOE_DEV uint32_t e4m3_rn_sat(float v) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(v));
  return r & 0xffu;
}

MOE_DEV float pow2_any(int e) {  // 2^e for e in [-149, 127], exact
  if (e >= -126) return __int_as_float((127 + e) << 23);
  return __int_as_float(1 << (e + 149));
}

// 32 values -> 16 code bytes (as 4 words) + E8M0 byte.
MOE_DEV uint32_t quant_mx32(const float* v, uint32_t* words) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
  int X = -127;
  if (amax > 0.f) {
    int ex;
    frexpf(amax, &ex);          // amax = m 2^ex, m in [0.5, 1)
    X = max(-127, min(127, (ex - 1) - 2));
  }
  const float inv = pow2_any(-X);
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    uint32_t word = 0;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const int i = 8 * w + 2 * b;
      word |= e2m1_pack2(v[i] * inv, v[i + 1] * inv) << (8 * b);
    }
    words[w] = word;
  }
  return (uint32_t)(X + 127);
}

// 16 values -> 8 code bytes (2 words) + E4M3 byte.
MOE_DEV uint32_t quant_nv16(const float* v, float g, uint32_t* words) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
  const float s_raw = __fdiv_rn(__fdiv_rn(amax, 6.0f), g);
  const uint32_t sb = e4m3_rn_sat(s_raw);
  const float denom = e4m3_to_f32(sb) * g;
#pragma unroll
  for (int w = 0; w < 2; ++w) {
    uint32_t word = 0;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const int i = 8 * w + 2 * b;
      float q0 = 0.f, q1 = 0.f;
      if (denom > 0.f) { q0 = __fdiv_rn(v[i], denom); q1 = __fdiv_rn(v[i + 1], denom); }
      word |= e2m1_pack2(q0, q1) << (8 * b);
    }
    words[w] = word;
  }
  return sb;
}

// Two E4M3 bytes of (lo, hi), lo in bits 0..7, nearest even, saturating at
// 448; a negative value that rounds to zero keeps its sign (0x80).
MOE_DEV uint32_t e4m3_pack2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return ((uint32_t)r | ((__float_as_uint(lo) >> 31) << 7) | ((__float_as_uint(hi) >> 31) << 15)) & 0xffffu;
}

// 32 values -> 32 E4M3 bytes (as 8 words) + E8M0 byte.
MOE_DEV uint32_t quant_mx8_32(const float* v, uint32_t* words) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
  int X = -127;
  if (amax > 0.f) {
    int ex;
    frexpf(amax, &ex);          // amax = m 2^ex, m in [0.5, 1)
    X = max(-127, min(127, (ex - 1) - 8));
  }
  const float inv = pow2_any(-X);
#pragma unroll
  for (int w = 0; w < 8; ++w)
    words[w] = e4m3_pack2(v[4 * w] * inv, v[4 * w + 1] * inv) |
               (e4m3_pack2(v[4 * w + 2] * inv, v[4 * w + 3] * inv) << 16);
  return (uint32_t)(X + 127);
}

}  // namespace moe
