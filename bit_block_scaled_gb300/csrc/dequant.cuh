// 4-bit weight expansion of the grouped GEMM: bit-level E2M1 placement into
// bf16 pairs and the exact bf16 products with the block scales (the R0 weight
// operand of the layer's definition).
#pragma once

#include "common.cuh"

namespace moe4 {

// bf16x2 bits of (E2M1 codes) * 2^-126 for 8 packed codes c0..c7 (one K
// group of 8) -> 4 words (c0|c4), (c1|c5), (c2|c6), (c3|c7). The activation
// operands are stored with the same interleave within every group of 8 K
// elements (order 0,4,1,5,2,6,3,7), so the MMA pairs them correctly.
__device__ __forceinline__ void e2m1x8_raw(uint32_t x, uint32_t (&o)[4]) {
  const uint32_t y = x >> 8;
  o[0] = ((x & 0x000F000Fu) * 0x1040u) & 0x81C081C0u;  // codes 0 | 4
  o[1] = ((x & 0x00F000F0u) * 0x0104u) & 0x81C081C0u;  // codes 1 | 5
  o[2] = ((y & 0x000F000Fu) * 0x1040u) & 0x81C081C0u;  // codes 2 | 6
  o[3] = ((y & 0x00F000F0u) * 0x0104u) & 0x81C081C0u;  // codes 3 | 7
}

// a * b on bf16 pairs, one rounding (fma with a -0 addend keeps signed zeros).
__device__ __forceinline__ uint32_t bmul2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(0x80008000u));
  return d;
}

// a * b + c on bf16 pairs with a single rounding.
__device__ __forceinline__ uint32_t bfma2(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// bf16x2 (both halves) of an E4M3 scale byte times 2^118 (exact; NaN for
// 0x7F / 0xFF).
__device__ __forceinline__ uint32_t e4m3_times_2p118_x2(uint32_t b) {
  const uint32_t mag = b & 0x7Fu;
  uint32_t h;
  if (mag == 0x7Fu) {
    h = 0x7FC0u;
  } else {
    float f = __uint_as_float(mag << 20) * 0x1p120f;  // the E4M3 value
    f = f * 0x1p118f;
    if (b & 0x80u) f = -f;
    h = float_to_bf16_bits(f);
  }
  return h | (h << 16);
}

// bf16x2 of 2^(e - 1) for an E8M0 byte (the MXFP4 scale times 2^126).
__device__ __forceinline__ uint32_t e8m0_times_2p126_x2(uint32_t e8) {
  const uint32_t h = (e8 == 0xFFu) ? 0x7FC0u : ((e8 + 126u) << 7);
  return h | (h << 16);
}

// f16 operand path: f16x2 (both halves) of an E4M3 scale byte (exact; NaN for
// 0x7F / 0xFF).
__device__ __forceinline__ uint32_t e4m3_f16x2(uint32_t b) {
  const uint32_t mag = b & 0x7Fu;
  __half h;
  if (mag == 0x7Fu) {
    h = __ushort_as_half((unsigned short)0x7E00u);
  } else {
    float f = __uint_as_float(mag << 20) * 0x1p120f;  // the E4M3 value
    if (b & 0x80u) f = -f;
    h = __float2half_rn(f);
  }
  const uint32_t u = __half_as_ushort(h);
  return u | (u << 16);
}

// f16 operand path for MXFP4: f16x2 (both halves) of 2^(e8 - 115), the E8M0
// scale 2^(e8 - 127) times 2^12 (the epilogue multiplies by 2^-12). For the
// exponents the kernels accept (e8 <= 128) every E2M1 value times it stays
// below 6 * 2^13 < 65504, and is exact down to e8 = 92 (0.5 * 2^-23); e8 = 91
// is the smallest power of two f16 holds (2^-24), smaller scales give 0.
// 255 (NaN) gives NaN, exponents above 128 infinity (they are also reported).
__device__ __forceinline__ uint32_t e8m0_f16x2(uint32_t e8) {
  uint32_t h;
  if (e8 == 0xFFu) {
    h = 0x7E00u;
  } else if (e8 > 128u) {
    h = 0x7C00u;
  } else if (e8 >= 101u) {  // normal: exponent field (e8 - 115) + 15
    h = (e8 - 100u) << 10;
  } else if (e8 >= 91u) {  // subnormal: 2^(e8 - 115) = 2^(e8 - 91) * 2^-24
    h = 1u << (e8 - 91u);
  } else {
    h = 0u;
  }
  return h | (h << 16);
}

// f16x2 of the two E2M1 codes in byte `byte` of w (low nibble -> low half).
__device__ __forceinline__ uint32_t e2m1x2_f16x2(uint32_t w, int byte) {
  uint32_t d;
  switch (byte) {
    case 0:
      asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, b0;\n\t}"
          : "=r"(d) : "r"(w));
      break;
    case 1:
      asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, b1;\n\t}"
          : "=r"(d) : "r"(w));
      break;
    case 2:
      asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, b2;\n\t}"
          : "=r"(d) : "r"(w));
      break;
    default:
      asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, b3;\n\t}"
          : "=r"(d) : "r"(w));
      break;
  }
  return d;
}

// a * b on f16 pairs (exact for E2M1 x E4M3 products).
__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

}  // namespace moe4
