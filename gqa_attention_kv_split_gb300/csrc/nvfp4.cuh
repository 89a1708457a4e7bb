// nvfp4.cuh -- NVFP4 (E2M1 codes + E4M3 block scale) -> E4M3 dequantisation
// on sm_103a, the step "dequantise the NVFP4 K/V page to E4M3 in shared
// memory" of "GB300 NVFP4 Context Attention: scale slot 조기 반납과 8단 packed
// K/V ring" (introduction).
//
// value = E4M3_rne_satfinite( e2m1(code) * e4m3(scale) ).
// The product is formed in f16, where it is exact: an E2M1 value has at most
// 2 significant bits and an E4M3 value at most 4, every product lies within
// [2^-10, 2688] in magnitude (or is zero), and f16 holds 11 significant bits
// over [2^-14, 65504].  The single rounding is the hardware's f16x2 -> e4m3x2
// conversion (round to nearest even, saturating to +-448).
#pragma once
#include <cstdint>

namespace gqa {

// Two E2M1 codes (one byte; element 2i in the low nibble) -> f16x2 with the
// low nibble in the low half.
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}" : "=r"(r) : "r"(byte));
  return r;
}

// E4M3 scale byte -> f16x2 (s, s).
__device__ __forceinline__ uint32_t e4m3_to_f16x2_bcast(uint32_t sf) {
  const uint16_t two = (uint16_t)((sf & 0xffu) | ((sf & 0xffu) << 8));
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(two));
  return r;
}

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// f16x2 -> two E4M3 bytes (low half -> low byte), RNE, satfinite.
__device__ __forceinline__ uint32_t f16x2_to_e4m3x2(uint32_t h) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(r) : "r"(h));
  return r;
}

// Four packed bytes (8 E2M1 codes, element order low nibble first) sharing
// one scale (as f16x2 broadcast) -> 8 E4M3 bytes in element order.
__device__ __forceinline__ uint2 dequant8(uint32_t packed, uint32_t scale_h2) {
  const uint32_t a = f16x2_to_e4m3x2(hmul2_u32(e2m1x2_to_f16x2(packed), scale_h2));
  const uint32_t b = f16x2_to_e4m3x2(hmul2_u32(e2m1x2_to_f16x2(packed >> 8), scale_h2));
  const uint32_t c = f16x2_to_e4m3x2(hmul2_u32(e2m1x2_to_f16x2(packed >> 16), scale_h2));
  const uint32_t d = f16x2_to_e4m3x2(hmul2_u32(e2m1x2_to_f16x2(packed >> 24), scale_h2));
  return make_uint2(a | (b << 16), c | (d << 16));
}

// One 16-element block: 8 packed bytes + its scale byte -> 16 E4M3 bytes.
__device__ __forceinline__ uint4 dequant16(uint2 packed, uint32_t sf_byte) {
  const uint32_t s = e4m3_to_f16x2_bcast(sf_byte);
  const uint2 lo = dequant8(packed.x, s);
  const uint2 hi = dequant8(packed.y, s);
  return make_uint4(lo.x, lo.y, hi.x, hi.y);
}

}  // namespace gqa
