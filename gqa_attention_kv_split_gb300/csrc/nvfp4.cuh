// nvfp4.cuh -- NVFP4 (E2M1 codes + E4M3 block scale) -> E4M3 dequantisation
// on sm_103a: the conversion of packed K/V pages to E4M3 tiles in shared
// memory that the context attention of "GB300 NVFP4 Context Attention: scale
// slot 조기 반납과 8단 packed K/V ring" (introduction) performs.
//
// value = E4M3_rne_satfinite( e2m1(code) * e4m3(scale) ).
// The product is formed in f16, where it is exact: an E2M1 value has at most
// 2 significant bits and an E4M3 value at most 4, every product lies within
// [2^-10, 2688] in magnitude (or is zero), and f16 holds 11 significant bits
// over [2^-14, 65504].  The single rounding is the hardware's f16x2 -> e4m3x2
// conversion (round to nearest even, saturating to +-448).  Conversions run
// at a fraction of the ALU rate on sm_103a, so the per-element work below is
// byte permutes through a per-block table.
#pragma once
#include <cstdint>

namespace gqa {


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

// One 16-element block: 8 packed bytes + its scale byte -> 16 E4M3 bytes.
//
// A block has one scale, so its 16 possible outputs are tabulated first: the
// 8 E2M1 magnitudes {0, 0.5, 1, 1.5, 2, 3, 4, 6} (f16x2 constants) times the
// scale, rounded to E4M3 -- 4 products and 4 conversions per block instead of
// 16 + 8.  Each group of 4 codes (16 bits, element order low nibble first)
// then becomes 4 output bytes with two byte-permutes: the low 3 bits of each
// nibble index the magnitude table, and bit 3 (the E2M1 sign) selects a
// 0x80 byte that is XORed into the E4M3 sign.  Same values, bit for bit, as
// converting every element: the products are exact in f16 and each is
// rounded once, by the same conversion.
__device__ __forceinline__ uint32_t nvfp4_lookup4(uint32_t codes16, uint32_t tab_lo, uint32_t tab_hi) {
  const uint32_t mag = __byte_perm(tab_lo, tab_hi, codes16 & 0x7777u);
  const uint32_t sgn = __byte_perm(0u, 0x80808080u, (codes16 >> 1) & 0x4444u);
  return mag ^ sgn;
}

// The 8 E4M3 magnitudes of one scale: tab_lo = codes 0..3, tab_hi = codes
// 4..7, one byte each (code c in byte c & 3).
__device__ __forceinline__ uint2 nvfp4_scale_table(uint32_t sf_byte) {
  const uint32_t s = e4m3_to_f16x2_bcast(sf_byte);
  const uint32_t t01 = f16x2_to_e4m3x2(hmul2_u32(0x38000000u, s));  // (0, 0.5)
  const uint32_t t23 = f16x2_to_e4m3x2(hmul2_u32(0x3E003C00u, s));  // (1, 1.5)
  const uint32_t t45 = f16x2_to_e4m3x2(hmul2_u32(0x42004000u, s));  // (2, 3)
  const uint32_t t67 = f16x2_to_e4m3x2(hmul2_u32(0x46004400u, s));  // (4, 6)
  return make_uint2(t01 | (t23 << 16), t45 | (t67 << 16));
}

// One 16-element block through a scale table: 8 packed bytes -> 16 E4M3 bytes.
__device__ __forceinline__ uint4 dequant16_table(uint2 packed, uint2 tab) {
  return make_uint4(nvfp4_lookup4(packed.x & 0xffffu, tab.x, tab.y), nvfp4_lookup4(packed.x >> 16, tab.x, tab.y),
                    nvfp4_lookup4(packed.y & 0xffffu, tab.x, tab.y), nvfp4_lookup4(packed.y >> 16, tab.x, tab.y));
}

// One 16-element block: 8 packed bytes + its scale byte -> 16 E4M3 bytes.
__device__ __forceinline__ uint4 dequant16(uint2 packed, uint32_t sf_byte) {
  return dequant16_table(packed, nvfp4_scale_table(sf_byte));
}

}  // namespace gqa
