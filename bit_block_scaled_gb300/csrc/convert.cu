// Checkpoint-layout import (host only, runs once at load time): the expert
// weight layouts the pages' checkpoints use, rewritten into the layout the
// grouped GEMMs read (moe_qweight_t).
//
//  * GPTQ INT4, group 64 ("GPTQ INT4 ... qweight, qzeros, scales, g_idx" in
//    "Serving gpt-oss with mixed GPTQ experts", section "1. Quantize"; the
//    [K/8, N] int32 view of the [N, K/2] code bytes is the one the pages'
//    repro builds for the Marlin kernel, "Reproducer", NVFP4 Marlin issue).
//  * ModelOpt NVFP4: codes and E4M3 block scales already have this library's
//    layout; the checkpoint's weight_scale_2 is one scalar where this library
//    takes one global scale per expert ("Gap 2 ... 2b", NVFP4 gpt-oss report).
#include <stdint.h>
#include <string.h>

#include "../../include/moe4.h"

extern "C" {

moe_status_t moe_import_gptq_int4(const int32_t *qweight, const int32_t *qzeros, const uint16_t *scales,
                                  const int32_t *g_idx, int K, int N, int group_size, int zero_offset,
                                  uint8_t *q, uint16_t *scales_out, uint8_t *zeros_out) {
  if (!qweight || !qzeros || !scales || !q || !scales_out || !zeros_out) return MOE_ERR_INVALID_ARG;
  if (K <= 0 || N <= 0 || K % 64 || N % 64 || (zero_offset != 0 && zero_offset != 1)) return MOE_ERR_INVALID_ARG;
  if (group_size != 64) return MOE_ERR_UNSUPPORTED;
  if (g_idx)
    for (int k = 0; k < K; ++k)
      if (g_idx[k] != k / 64) return MOE_ERR_UNSUPPORTED;  // act-order permutations not supported
  const int G = K / 64, ZB = (G + 1) / 2, N8 = N / 8;
  // zero points first: nothing is written when one is out of range
  for (int g = 0; g < G; ++g)
    for (int n = 0; n < N; ++n) {
      const uint32_t w = (uint32_t)qzeros[(size_t)g * N8 + n / 8];
      if (((w >> (4 * (n % 8))) & 0xFu) + (uint32_t)zero_offset > 15u) return MOE_ERR_UNSUPPORTED;
    }
  // codes: qweight[i][n] holds k = 8i..8i+7 of column n, k = 8i + j in bits
  // 4j..4j+3, so its four bytes (low first) are bytes 4i..4i+3 of row n
  for (int i = 0; i < K / 8; ++i)
    for (int n = 0; n < N; ++n) {
      const uint32_t w = (uint32_t)qweight[(size_t)i * N + n];
      uint8_t *dst = q + (size_t)n * (K / 2) + 4 * i;
      for (int b = 0; b < 4; ++b) dst[b] = (uint8_t)(w >> (8 * b));
    }
  for (int n = 0; n < N; ++n) {
    for (int g = 0; g < G; ++g) scales_out[(size_t)n * G + g] = scales[(size_t)g * N + n];
    uint8_t *zr = zeros_out + (size_t)n * ZB;
    memset(zr, 0, (size_t)ZB);
    for (int g = 0; g < G; ++g) {
      const uint32_t w = (uint32_t)qzeros[(size_t)g * N8 + n / 8];
      const uint32_t z = ((w >> (4 * (n % 8))) & 0xFu) + (uint32_t)zero_offset;
      zr[g / 2] |= (uint8_t)(z << (4 * (g & 1)));
    }
  }
  return MOE_OK;
}

moe_status_t moe_import_modelopt_global_scale(float weight_scale_2, int E, float *gscale) {
  if (!gscale || E <= 0 || E > 256) return MOE_ERR_INVALID_ARG;
  for (int e = 0; e < E; ++e) gscale[e] = weight_scale_2;
  return MOE_OK;
}

}  // extern "C"
