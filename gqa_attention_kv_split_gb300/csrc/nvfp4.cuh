// nvfp4.cuh -- NVFP4 (E2M1 codes + E4M3 block scale) -> E4M3 dequantisation
// on sm_103a: the conversion of packed K/V pages to E4M3 tiles in shared
// memory that the context attention of "GB300 NVFP4 Context Attention: scale
// slot 조기 반납과 8단 packed K/V ring" (introduction) performs.
//
// value = E4M3_rne_satfinite( e2m1(code) * e4m3(scale) ).
// A 16-element block has one scale, so its 8 possible magnitudes are
// tabulated once per scale: each product is formed in f16, where it is exact
// (an E2M1 value has at most 2 significant bits and an E4M3 value at most 4;
// every product lies within [2^-10, 2688] in magnitude or is zero, and f16
// holds 11 significant bits over [2^-14, 65504]), and rounded once by the
// hardware's f16x2 -> e4m3x2 conversion (round to nearest even, saturating to
// +-448).  The per-element work is then byte permutes: the low 3 bits of a
// code index the table of the 8 products and bit 3 (the E2M1 sign) flips the
// sign bit of the result (a flip, not a set: the scale may be negative).
//
// Two outputs per code word: E4M3 bytes (the K tile of S = Q K^T) and the
// same values widened to f16 (the V tile of the f16 P V product) by the
// hardware's exact E4M3 -> f16 conversion of those bytes, so both are the same
// E4M3 numbers bit for bit.  (A second f16 construction, straight from byte
// tables of the f16 encodings, serves as the device-side cross-check of the
// dequantisation test export.)
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

// Two E4M3 bytes (low 16 bits, first element low) -> f16x2 (exact).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t v) {
  uint32_t d;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(d) : "h"((uint16_t)v));
  return d;
}

// The 8 E4M3 magnitudes of one scale: .x = codes 0..3, .y = codes 4..7, one
// byte each (code c in byte c & 3).
__device__ __forceinline__ uint2 nvfp4_scale_table(uint32_t sf_byte) {
  const uint32_t s = e4m3_to_f16x2_bcast(sf_byte);
  const uint32_t t01 = f16x2_to_e4m3x2(hmul2_u32(0x38000000u, s));  // (0, 0.5)
  const uint32_t t23 = f16x2_to_e4m3x2(hmul2_u32(0x3E003C00u, s));  // (1, 1.5)
  const uint32_t t45 = f16x2_to_e4m3x2(hmul2_u32(0x42004000u, s));  // (2, 3)
  const uint32_t t67 = f16x2_to_e4m3x2(hmul2_u32(0x46004400u, s));  // (4, 6)
  return make_uint2(t01 | (t23 << 16), t45 | (t67 << 16));
}

// The same 8 magnitudes as f16 encodings, split into byte tables: .x/.y =
// low bytes of codes 0..3 / 4..7, .z/.w = high bytes.
__device__ __forceinline__ uint4 nvfp4_f16_table(uint2 e4m3_tab) {
  const uint32_t h01 = e4m3x2_to_f16x2(e4m3_tab.x & 0xffffu), h23 = e4m3x2_to_f16x2(e4m3_tab.x >> 16);
  const uint32_t h45 = e4m3x2_to_f16x2(e4m3_tab.y & 0xffffu), h67 = e4m3x2_to_f16x2(e4m3_tab.y >> 16);
  return make_uint4(__byte_perm(h01, h23, 0x6420), __byte_perm(h45, h67, 0x6420),
                    __byte_perm(h01, h23, 0x7531), __byte_perm(h45, h67, 0x7531));
}

// Sign bits of 8 codes (a 32-bit word, code k in bits 4k..4k+3, element
// order low nibble first) moved to bit 7 of output bytes: .x for codes 0..3,
// .y for codes 4..7.  Code 2i's sign (bit 3 of byte i) reaches bit 7 of a
// byte of w << 4; code 2i+1's sign already is bit 7 of byte i.
__device__ __forceinline__ uint2 nvfp4_sign_bytes(uint32_t w) {
  const uint32_t w4 = w << 4;
  return make_uint2(__byte_perm(w4, w, 0x5140) & 0x80808080u, __byte_perm(w4, w, 0x7362) & 0x80808080u);
}

// 8 codes -> 8 E4M3 bytes (.x = elements 0..3, .y = 4..7).
__device__ __forceinline__ uint2 nvfp4_to_e4m3_8(uint32_t w, uint2 tab) {
  const uint32_t wm = w & 0x77777777u;  // magnitude indices (a selector nibble's bit 3 must be clear)
  const uint2 sg = nvfp4_sign_bytes(w);
  return make_uint2(__byte_perm(tab.x, tab.y, wm) ^ sg.x, __byte_perm(tab.x, tab.y, wm >> 16) ^ sg.y);
}

// 8 codes -> 8 f16 values of the E4M3 results, as 4 f16x2 words (element 2i
// in the low half of word i): the E4M3 bytes, then the exact conversion.
__device__ __forceinline__ uint4 nvfp4_to_f16_8(uint32_t w, uint2 tab) {
  const uint2 e = nvfp4_to_e4m3_8(w, tab);
  return make_uint4(e4m3x2_to_f16x2(e.x & 0xffffu), e4m3x2_to_f16x2(e.x >> 16), e4m3x2_to_f16x2(e.y & 0xffffu),
                    e4m3x2_to_f16x2(e.y >> 16));
}

// The same 8 f16 values built from the f16 byte tables of nvfp4_f16_table
// (no conversion instruction): the independent construction the test export
// checks nvfp4_to_f16_8 against.
__device__ __forceinline__ uint4 nvfp4_to_f16_8_tables(uint32_t w, uint4 tab) {
  const uint32_t wm = w & 0x77777777u;
  const uint32_t wmh = wm >> 16;
  const uint2 sg = nvfp4_sign_bytes(w);
  const uint32_t h0 = __byte_perm(tab.z, tab.w, wm) ^ sg.x;
  const uint32_t h1 = __byte_perm(tab.z, tab.w, wmh) ^ sg.y;
  const uint32_t l0 = __byte_perm(tab.x, tab.y, wm);
  const uint32_t l1 = __byte_perm(tab.x, tab.y, wmh);
  return make_uint4(__byte_perm(l0, h0, 0x5140), __byte_perm(l0, h0, 0x7362), __byte_perm(l1, h1, 0x5140),
                    __byte_perm(l1, h1, 0x7362));
}

// One 16-element block (8 packed bytes) through its scale's table -> 16 E4M3 bytes.
__device__ __forceinline__ uint4 dequant16_e4m3(uint2 packed, uint2 tab) {
  const uint2 lo = nvfp4_to_e4m3_8(packed.x, tab);
  const uint2 hi = nvfp4_to_e4m3_8(packed.y, tab);
  return make_uint4(lo.x, lo.y, hi.x, hi.y);
}

}  // namespace gqa
