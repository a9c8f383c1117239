// Internal launch interface between the C ABI (api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe4.h"

namespace moe4 {

struct GemmArgs {
  CUtensorMap tm_w;  // packed 4-bit weights [E][N][K/2]
  CUtensorMap tm_x;  // bf16 activations [P_max][K]
  const void *scales;
  const uint8_t *zeros;
  const float *gscale;
  const uint16_t *bias;
  const int32_t *expert_offsets;
  const int32_t *sorted_ids;
  const float *topk_w;
  const int32_t *xexp;  // f16 operand path: per-slot exponent of the activation rows (GEMM1)
  uint16_t *out;
  unsigned int *status;
  int E, N, K, P_max, num_rows, ldo, layout, I, mul, a_f16;
  float alpha, limit;
  int tile_n, stages, kpb, sc_row_bytes, z_row_bytes, m_tiles, nacc, na, xstages;
};

int choose_tile_n(int num_rows, int E);
int choose_kpb(int tile_n);

// epi: 0 = GEMM1 + swigluoai, 1 = GEMM1 + ReLU^2, 2 = GEMM2 + routing weight.
// f16 bit 0 selects the f16 operand path (NVFP4 or MXFP4 weights): the
// activations x are f16 in natural column order (GEMM1: rows scaled by
// 2^-xexp[slot]). f16 bit 1 (GEMM1 with swigluoai, when GEMM2 also runs on f16
// operands) writes a times 2^9 as f16 in natural column order (the f16 GEMM2
// undoes the 2^9 in its epilogue); otherwise GEMM1 writes a
// as bf16 with interleaved columns, as a bf16 GEMM2 reads it (ReLU^2 outputs
// are not bounded, so they always stay bf16).
moe_status_t launch_grouped_gemm(int epi, const moe_qweight_t &w, const uint16_t *x, int P_max,
                                 const int32_t *sorted_ids, const int32_t *expert_offsets, int num_rows,
                                 const float *topk_w, int mul, int layout, moe_act_t act, uint16_t *out,
                                 int ldo, unsigned int *status, cudaStream_t stream, int *launches, int f16 = 0,
                                 const int32_t *xexp = nullptr);

moe_status_t launch_route(const float *logits, const float *sel_bias, int T, int E, int k, int route,
                          int32_t *ids, float *weights, unsigned int *status, cudaStream_t stream,
                          int *launches);

// counts (optional, align_chunks(T * k) * E ints): with it, batches of many
// routed rows are aligned over many CTAs (two launches, same result).
moe_status_t launch_align(const int32_t *ids, int T, int k, int E, int block_m, int P_max,
                          int32_t *sorted_ids, int32_t *offsets, int32_t *block_ids, int32_t *row_pos,
                          unsigned int *status, cudaStream_t stream, int *launches, int32_t *counts = nullptr);
// Number of row chunks the many-CTA alignment uses for R routed rows (0: one CTA).
int align_chunks(int R);

// Token rows into the slots of their routed rows (row_pos), padding slots
// (found from offsets and sorted_ids) zeroed. f16: power-of-two scaled f16
// rows in natural column order with their exponents in xexp; else bf16 rows
// with the columns interleaved within groups of 8. tw (optional): the routing
// weight applied on the input, each slot's row rounded to bf16(x * tw[r]).
moe_status_t launch_gather(const uint16_t *x, int T, int k, int H, int E, int P_max, const int32_t *row_pos,
                           const int32_t *offsets, const int32_t *sorted_ids, uint16_t *x_out, int32_t *xexp,
                           bool f16, cudaStream_t stream, int *launches, const float *tw = nullptr);

// moe_forward with a fixed device workspace (moe_forward_static): all host
// checks before anything is enqueued, then clear the status word, run the
// layer and copy the status word to status_out (if not NULL).
moe_status_t forward_fixed_workspace(const uint16_t *x, const float *logits, const float *sel_bias, int T, int E,
                                     int k, int H, int I, int route, const moe_qweight_t *w13,
                                     const moe_qweight_t *w2, int layout, moe_act_t act, int mul, int block_m,
                                     uint16_t *out, uint32_t *status_out, void *ws, size_t ws_bytes,
                                     cudaStream_t st);

moe_status_t launch_unpermute(const uint16_t *y, const int32_t *row_pos, int T, int k, int H, int P_max,
                              uint16_t *out, unsigned int *status, cudaStream_t stream, int *launches);

}  // namespace moe4
