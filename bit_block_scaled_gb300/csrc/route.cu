// Step a1: top-k routing, one warp per token.
//
// TOPK_SOFTMAX (gpt-oss; vLLM issue "moe_wna16_marlin_gemm applies wrong
// per-row topk weights", "Minimal repro"): the k largest logits, descending,
// equal values -> lower expert id, then a softmax over the k selected.
// SIGMOID_BIAS (Nemotron-3-Nano; vLLM issue "... non-gated ReLU2 MoE
// (Nemotron-3-Nano)", Analysis item 3, n_group = 1): s = sigmoid(logit) in
// fp32, select by s + bias, weights = selected s renormalised to sum 1.
//
// Non-finite scores (the pages say nothing about them; the reading taken):
// a NaN selection score ranks as -inf, and equal scores (two -inf included)
// go to the lower expert id. The softmax weights are exp(l_j - max) when the
// largest selected logit is finite; when it is +inf or -inf, the selected
// logits equal to it share the weight equally (the limit of the softmax) and
// the rest get 0. A NaN logit weighs as -inf. Sigmoid routing weighs a NaN
// logit as s = 0; if every selected s is 0 the k weights are 1/k each.
#include "common.cuh"
#include "kernels.h"

namespace moe4 {

namespace {

constexpr int kWarps = 8;
constexpr int kMaxK = 8;

__device__ __forceinline__ float sigmoid_f32(float l) { return 1.0f / (1.0f + expf(-l)); }

// PL: expert scores per lane, ceil(E / 32) rounded up to 1, 2, 4 or 8 (E <= 256)
template <int ROUTE, int PL>
__global__ void __launch_bounds__(kWarps * 32) route_kernel(const float *__restrict__ logits,
                                                            const float *__restrict__ sel_bias, int T, int E,
                                                            int k, int32_t *__restrict__ ids,
                                                            float *__restrict__ weights) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * kWarps + (threadIdx.x >> 5);
  if (t >= T) return;
  const float *row = logits + (size_t)t * E;
  float sc[PL];
#pragma unroll
  for (int i = 0; i < PL; ++i) {
    const int e = lane + 32 * i;
    float v = -INFINITY;
    if (e < E) {
      const float l = row[e];
      v = (ROUTE == MOE_ROUTE_SIGMOID_BIAS) ? sigmoid_f32(l) + sel_bias[e] : l;
      if (v != v) v = -INFINITY;  // NaN never outranks a number
    }
    sc[i] = v;
  }
  unsigned taken = 0;
  int sel_id[kMaxK];
  float sel_v[kMaxK];
#pragma unroll
  for (int j = 0; j < kMaxK; ++j) {
    if (j >= k) break;
    float best = -INFINITY;
    int bid = 0x7FFFFFFF;
#pragma unroll
    for (int i = 0; i < PL; ++i) {
      const int e = lane + 32 * i;
      if (e < E && !((taken >> i) & 1u) && (sc[i] > best || (sc[i] == best && e < bid))) {
        best = sc[i];
        bid = e;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, best, o);
      const int oid = __shfl_xor_sync(0xffffffffu, bid, o);
      if (ov > best || (ov == best && oid < bid)) {
        best = ov;
        bid = oid;
      }
    }
    if ((bid & 31) == lane) taken |= 1u << (bid >> 5);
    sel_id[j] = bid;
    if (ROUTE == MOE_ROUTE_SIGMOID_BIAS) {
      const float sv = sigmoid_f32(row[bid]);
      sel_v[j] = sv != sv ? 0.f : sv;  // a NaN logit weighs as s = 0
    } else {
      const float l = row[bid];
      sel_v[j] = l != l ? -INFINITY : l;  // a NaN logit weighs as -inf
    }
  }
  if (lane != 0) return;
  float w[kMaxK];
  float sum = 0.f;
  if (ROUTE == MOE_ROUTE_SIGMOID_BIAS) {
#pragma unroll
    for (int j = 0; j < kMaxK; ++j)
      if (j < k) {
        w[j] = sel_v[j];
        sum += w[j];
      }
    if (sum == 0.f) {  // every selected s is 0: equal weights
#pragma unroll
      for (int j = 0; j < kMaxK; ++j) w[j] = 1.f;
      sum = (float)k;
    }
  } else {
    // the slots hold descending scores, so slot 0 has the largest logit
    float m = sel_v[0];
#pragma unroll
    for (int j = 1; j < kMaxK; ++j)
      if (j < k) m = fmaxf(m, sel_v[j]);
    const bool finite = fabsf(m) <= 3.402823466e38f;
#pragma unroll
    for (int j = 0; j < kMaxK; ++j)
      if (j < k) {
        w[j] = finite ? expf(sel_v[j] - m) : (sel_v[j] == m ? 1.f : 0.f);
        sum += w[j];
      }
  }
#pragma unroll
  for (int j = 0; j < kMaxK; ++j)
    if (j < k) {
      ids[(size_t)t * k + j] = sel_id[j];
      weights[(size_t)t * k + j] = w[j] / sum;
    }
}

}  // namespace

moe_status_t launch_route(const float *logits, const float *sel_bias, int T, int E, int k, int route,
                          int32_t *ids, float *weights, unsigned int *status, cudaStream_t stream,
                          int *launches) {
  (void)status;
  if (T == 0) return MOE_OK;
  const dim3 grid((T + kWarps - 1) / kWarps), block(kWarps * 32);
  auto go = [&](auto kern) {
    return launch_pdl(kern, grid, block, 0, stream, logits, sel_bias, T, E, k, ids, weights);
  };
  const bool sig = route == MOE_ROUTE_SIGMOID_BIAS;
  cudaError_t err;
  if (E <= 32)
    err = sig ? go(route_kernel<MOE_ROUTE_SIGMOID_BIAS, 1>) : go(route_kernel<MOE_ROUTE_TOPK_SOFTMAX, 1>);
  else if (E <= 64)
    err = sig ? go(route_kernel<MOE_ROUTE_SIGMOID_BIAS, 2>) : go(route_kernel<MOE_ROUTE_TOPK_SOFTMAX, 2>);
  else if (E <= 128)
    err = sig ? go(route_kernel<MOE_ROUTE_SIGMOID_BIAS, 4>) : go(route_kernel<MOE_ROUTE_TOPK_SOFTMAX, 4>);
  else
    err = sig ? go(route_kernel<MOE_ROUTE_SIGMOID_BIAS, 8>) : go(route_kernel<MOE_ROUTE_TOPK_SOFTMAX, 8>);
  if (launches) ++*launches;
  return err == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe4
