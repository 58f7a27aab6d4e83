// Exact FP4 (E2M1) / FP8 (E4M3) -> fp16 conversions for building tensor-core operands, with
// power-of-two scales applied in fp16 (E2M1 x 2^e is exact in fp16 for -23 <= e <= 13; E4M3
// values are always exact), and the fp32 -> E5M2 conversion of the 8-bit indexer operands.
#pragma once
#include <cuda_fp16.h>
#include <stdint.h>

namespace csa2 {

// Four code bytes (8 values, element 2k in the low nibble of byte k) -> four f16x2.
__device__ __forceinline__ void cvt_e2m1x8_f16x8(uint32_t w, uint32_t* o) {
  asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n cvt.rn.f16x2.e2m1x2 %0, b0;\n"
      " cvt.rn.f16x2.e2m1x2 %1, b1;\n cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3;\n}\n"
      : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3])
      : "r"(w));
}
__device__ __forceinline__ uint32_t hmul2(uint32_t x, uint32_t y) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;\n" : "=r"(r) : "r"(x), "r"(y));
  return r;
}
__device__ __forceinline__ uint32_t f2_to_h2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Both halves = 2^e as fp16 bits, built without arithmetic: normal for -14 <= e <= 15,
// subnormal down to 2^-24, 0 below, +inf above (the values an fp32 2^e rounds to in fp16).
__device__ __forceinline__ uint32_t pow2_h2(int e) {
  uint32_t h;
  if (e > 15) h = 0x7C00u;
  else if (e >= -14) h = (uint32_t)(e + 15) << 10;
  else if (e >= -24) h = 1u << (e + 24);
  else h = 0u;
  return h | (h << 16);
}

// Two fp32 values (already divided by their block scale) -> two E2M1 codes in one byte, `lo`
// in the low nibble: round to nearest with ties to the even code, saturating at +-6.
__device__ __forceinline__ uint32_t cvt_f32x2_e2m1x2(float lo, float hi) {
  uint32_t r;
  asm("{\n .reg .b8 t;\n cvt.rn.satfinite.e2m1x2.f32 t, %2, %1;\n cvt.u32.u8 %0, t;\n}\n" : "=r"(r) : "f"(lo), "f"(hi));
  return r;
}
// One code byte (two E2M1 values) -> f16x2.
__device__ __forceinline__ uint32_t cvt_e2m1x2_f16x2(uint32_t byte) {
  uint32_t r;
  asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %1;\n cvt.rn.f16x2.e2m1x2 %0, b0;\n}\n" : "=r"(r) : "r"(byte));
  return r;
}

// Two fp32 values -> two E5M2 bytes in the low 16 bits, `lo` in the low byte: round to nearest
// even, saturating at +-57344.  E2M1 x 2^e converts exactly for -15 <= e <= 13 (E5M2 has two
// mantissa bits and exponents down to 2^-16 as subnormals).
__device__ __forceinline__ uint32_t cvt_f32x2_e5m2x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e5m2x2.f32 %0, %2, %1;\n" : "=h"(r) : "f"(lo), "f"(hi));
  return r;
}

// Two E4M3 codes (low 16 bits) -> f16x2.
__device__ __forceinline__ uint32_t cvt_e4m3x2_f16x2(uint32_t two) {
  uint32_t r;
  asm("{\n .reg .b16 h0, h1;\n mov.b32 {h0, h1}, %1;\n cvt.rn.f16x2.e4m3x2 %0, h0;\n}\n" : "=r"(r) : "r"(two));
  return r;
}

}  // namespace csa2
