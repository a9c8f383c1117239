// The C ABI of libmoe4 (declared in include/moe4.h): argument checking,
// workspace carving and the step order of the fused layer.
#include <string.h>

#include "common.cuh"
#include "kernels.h"

using namespace moe4;

namespace {

thread_local int g_last_launches = 0;

inline bool aligned16(const void *p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline size_t up256(size_t v) { return (v + 255) / 256 * 256; }
inline bool valid_block_m(int bm) { return bm == 16 || bm == 32 || bm == 64 || bm == 128 || bm == 256; }
inline unsigned int *status_of(void *ws) { return static_cast<unsigned int *>(ws); }

bool valid_dims(int T, int E, int k, int H, int I) {
  if (T < 0 || E < 1 || E > 256 || k < 1 || k > 8 || k > E) return false;
  if (H < 64 || I < 64 || H % 64 || I % 64 || H > 4096 || I > 4096) return false;
  if ((int64_t)T * k >= (1 << 24)) return false;
  return true;
}

moe_status_t check_weight(const moe_qweight_t *w, int E, int N, int K) {
  if (!w) return MOE_ERR_INVALID_ARG;
  if (w->E != E || w->N != N || w->K != K) return MOE_ERR_INVALID_ARG;
  if (w->fmt < MOE_FMT_NVFP4 || w->fmt > MOE_FMT_INT4) return MOE_ERR_INVALID_ARG;
  if (!aligned16(w->q) || !aligned16(w->scales)) return MOE_ERR_INVALID_ARG;
  if (w->fmt == MOE_FMT_NVFP4 && !aligned16(w->gscale)) return MOE_ERR_INVALID_ARG;
  if (w->fmt == MOE_FMT_INT4 && !aligned16(w->zeros)) return MOE_ERR_INVALID_ARG;
  if (w->bias && !aligned16(w->bias)) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

struct Carve {
  size_t status, ids, tw, sorted, offsets, blocks, rowpos, xexp, xperm, a, xin, lin, outb, total;
};

Carve carve(int T, int E, int k, int H, int I, int bm) {
  const int64_t P = moe_padded_rows(T, k, E, bm);
  const size_t R = (size_t)T * k;
  Carve c;
  size_t o = 0;
  c.status = o; o += up256(MOE_STATUS_BYTES);
  c.ids = o; o += up256(R * 4);
  c.tw = o; o += up256(R * 4);
  c.sorted = o; o += up256((size_t)P * 4);
  c.offsets = o; o += up256((size_t)(E + 1) * 4);
  c.blocks = o; o += up256((size_t)(P / bm) * 4);
  c.rowpos = o; o += up256(R * 4);
  c.xexp = o; o += up256((size_t)P * 4);       // f16 operand path: per-slot exponents
  c.xperm = o; o += up256((size_t)P * H * 2);  // x_perm, later reused for y
  c.a = o; o += up256((size_t)P * I * 2);
  c.xin = o; o += up256((size_t)T * H * 2);    // staging for moe_forward_host
  c.lin = o; o += up256((size_t)T * E * 4);
  c.outb = o; o += up256((size_t)T * H * 2);
  c.total = o;
  return c;
}

template <typename T>
T *at(void *ws, size_t off) {
  return reinterpret_cast<T *>(static_cast<char *>(ws) + off);
}

// A bounded wait that runs out: a barrier initialised for one arrival that
// never comes. mbar_wait gives up after its cycle limit and the status word
// records the time-out, as in the layer's kernels.
__global__ void wait_selftest_kernel(unsigned int *status) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = smem_u32(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);
    fence_mbar_init();
  }
  __syncthreads();
  const bool ok = mbar_wait(b, 0);
  if (!ok && threadIdx.x == 0) raise_status(status, MOE_ERR_TIMEOUT);
}

}  // namespace

extern "C" {

int64_t moe_padded_rows(int T, int k, int E, int block_m) {
  if (T <= 0 || k <= 0 || E <= 0 || block_m <= 0) return 0;
  const int64_t R = (int64_t)T * k;
  const int64_t act = R < E ? R : E;
  return (R + act * (block_m - 1)) / block_m * block_m;
}

moe_status_t moe_workspace_size(int T, int E, int k, int H, int I, int block_m, size_t *bytes) {
  if (!bytes) return MOE_ERR_INVALID_ARG;
  if (block_m == 0) block_m = 16;
  if (!valid_dims(T, E, k, H, I) || !valid_block_m(block_m)) return MOE_ERR_INVALID_ARG;
  *bytes = carve(T, E, k, H, I, block_m).total;
  return MOE_OK;
}

moe_status_t moe_route_topk(const float *logits, const float *sel_bias, int T, int E, int k, int route,
                            int32_t *topk_ids, float *topk_weights, void *ws, moe_stream_t stream) {
  g_last_launches = 0;
  if (T < 0 || E < 1 || E > 256 || k < 1 || k > 8 || k > E) return MOE_ERR_INVALID_ARG;
  if (route != MOE_ROUTE_TOPK_SOFTMAX && route != MOE_ROUTE_SIGMOID_BIAS) return MOE_ERR_INVALID_ARG;
  if (!aligned16(ws)) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!aligned16(logits) || !aligned16(topk_ids) || !aligned16(topk_weights)) return MOE_ERR_INVALID_ARG;
  if (route == MOE_ROUTE_SIGMOID_BIAS && !aligned16(sel_bias)) return MOE_ERR_INVALID_ARG;
  return launch_route(logits, sel_bias, T, E, k, route, topk_ids, topk_weights, status_of(ws),
                      (cudaStream_t)stream, &g_last_launches);
}

moe_status_t moe_align_permute(const int32_t *topk_ids, int T, int k, int E, int block_m, const uint16_t *x,
                               int H, int32_t *sorted_token_ids, int32_t *expert_offsets,
                               int32_t *block_expert_ids, int32_t *row_pos, uint16_t *x_perm, void *ws,
                               moe_stream_t stream) {
  g_last_launches = 0;
  if (T < 0 || E < 1 || E > 256 || k < 1 || k > 8 || k > E || !valid_block_m(block_m)) return MOE_ERR_INVALID_ARG;
  if (H < 64 || H % 64 || H > 4096 || (int64_t)T * k >= (1 << 24)) return MOE_ERR_INVALID_ARG;
  if (!aligned16(ws) || !aligned16(expert_offsets)) return MOE_ERR_INVALID_ARG;
  const int P = (int)moe_padded_rows(T, k, E, block_m);
  if (T > 0 && (!aligned16(topk_ids) || !aligned16(x) || !aligned16(sorted_token_ids) ||
                !aligned16(block_expert_ids) || !aligned16(row_pos) || !aligned16(x_perm)))
    return MOE_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  // x_perm is written only by the gather, after the alignment: the many-CTA
  // alignment keeps its per-chunk counts there meanwhile
  moe_status_t s = launch_align(topk_ids, T, k, E, block_m, P, sorted_token_ids, expert_offsets,
                                block_expert_ids, row_pos, status_of(ws), st, &g_last_launches,
                                reinterpret_cast<int32_t *>(x_perm));
  if (s != MOE_OK) return s;
  return launch_gather(x, T, k, H, E, P, row_pos, expert_offsets, sorted_token_ids, x_perm, nullptr, false, st,
                       &g_last_launches);
}

moe_status_t moe_grouped_gemm1_act(const uint16_t *x_perm, const int32_t *sorted_token_ids,
                                   const int32_t *expert_offsets, int P_max, int num_rows,
                                   const moe_qweight_t *w13, int gate_up_layout, moe_act_t act, uint16_t *a_out,
                                   void *ws, moe_stream_t stream) {
  g_last_launches = 0;
  if (!w13 || !aligned16(ws) || P_max < 0 || num_rows < 0) return MOE_ERR_INVALID_ARG;
  if (act.kind != MOE_ACT_SWIGLUOAI && act.kind != MOE_ACT_RELU2) return MOE_ERR_INVALID_ARG;
  if (gate_up_layout != MOE_LAYOUT_INTERLEAVED && gate_up_layout != MOE_LAYOUT_CONCAT) return MOE_ERR_INVALID_ARG;
  const bool gated = act.kind == MOE_ACT_SWIGLUOAI;
  const int I = gated ? w13->N / 2 : w13->N;
  if (!valid_dims(0, w13->E, 1, w13->K, I)) return MOE_ERR_INVALID_ARG;
  if (gated && w13->N % 2) return MOE_ERR_INVALID_ARG;
  moe_status_t s = check_weight(w13, w13->E, w13->N, w13->K);
  if (s != MOE_OK) return s;
  if (P_max == 0 || num_rows == 0) return MOE_OK;
  if (!aligned16(x_perm) || !aligned16(sorted_token_ids) || !aligned16(expert_offsets) || !aligned16(a_out))
    return MOE_ERR_INVALID_ARG;
  return launch_grouped_gemm(gated ? 0 : 1, *w13, x_perm, P_max, sorted_token_ids, expert_offsets, num_rows,
                             nullptr, 0, gate_up_layout, act, a_out, I, status_of(ws), (cudaStream_t)stream,
                             &g_last_launches);
}

moe_status_t moe_grouped_gemm2_weighted(const uint16_t *a, const int32_t *sorted_token_ids,
                                        const int32_t *expert_offsets, int P_max, const moe_qweight_t *w2,
                                        const float *topk_weights_flat, int mul_topk_weights, int num_rows,
                                        uint16_t *y, void *ws, moe_stream_t stream) {
  g_last_launches = 0;
  if (!w2 || !aligned16(ws) || P_max < 0 || num_rows < 0) return MOE_ERR_INVALID_ARG;
  if (!valid_dims(0, w2->E, 1, w2->N, w2->K)) return MOE_ERR_INVALID_ARG;
  moe_status_t s = check_weight(w2, w2->E, w2->N, w2->K);
  if (s != MOE_OK) return s;
  if (P_max == 0 || num_rows == 0) return MOE_OK;
  if (!aligned16(a) || !aligned16(sorted_token_ids) || !aligned16(expert_offsets) || !aligned16(y))
    return MOE_ERR_INVALID_ARG;
  if (mul_topk_weights && !aligned16(topk_weights_flat)) return MOE_ERR_INVALID_ARG;
  moe_act_t none = {0, 0.f, 0.f};
  return launch_grouped_gemm(2, *w2, a, P_max, sorted_token_ids, expert_offsets, num_rows, topk_weights_flat,
                             mul_topk_weights ? 1 : 0, 0, none, y, w2->N, status_of(ws), (cudaStream_t)stream,
                             &g_last_launches);
}

moe_status_t moe_unpermute_reduce(const uint16_t *y, const int32_t *row_pos, int T, int k, int H, int P_max,
                                  uint16_t *out, void *ws, moe_stream_t stream) {
  g_last_launches = 0;
  if (T < 0 || k < 1 || k > 8 || H < 64 || H % 64 || H > 4096 || P_max < 0 || !aligned16(ws))
    return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!aligned16(y) || !aligned16(row_pos) || !aligned16(out)) return MOE_ERR_INVALID_ARG;
  return launch_unpermute(y, row_pos, T, k, H, P_max, out, status_of(ws), (cudaStream_t)stream,
                          &g_last_launches);
}

// ev (optional): 7 events recorded before the first kernel and after each of
// the six (route, align, gather, GEMM1, GEMM2, unpermute)
static moe_status_t forward_impl(const uint16_t *x, const float *logits, const float *sel_bias, int T, int E,
                                 int k, int H, int I, int route, const moe_qweight_t *w13,
                                 const moe_qweight_t *w2, int layout, moe_act_t act, int mul, int bm,
                                 uint16_t *out, void *ws, cudaStream_t st, cudaEvent_t *ev = nullptr) {
  auto mark = [&](int i) { return !ev || cudaEventRecord(ev[i], st) == cudaSuccess; };
  const Carve c = carve(T, E, k, H, I, bm);
  const int P = (int)moe_padded_rows(T, k, E, bm);
  const int R = T * k;
  unsigned int *status = status_of(ws);
  int32_t *ids = at<int32_t>(ws, c.ids);
  float *tw = at<float>(ws, c.tw);
  int32_t *sorted = at<int32_t>(ws, c.sorted);
  int32_t *offs = at<int32_t>(ws, c.offsets);
  int32_t *blocks = at<int32_t>(ws, c.blocks);
  int32_t *rowpos = at<int32_t>(ws, c.rowpos);
  uint16_t *xperm = at<uint16_t>(ws, c.xperm);
  uint16_t *abuf = at<uint16_t>(ws, c.a);
  uint16_t *ybuf = xperm;  // x_perm is dead once GEMM1 has run
  int32_t *xexp = at<int32_t>(ws, c.xexp);
  int *n = &g_last_launches;
  moe_status_t s;
  // NVFP4 layers feed the tensor cores f16 operands: E2M1 x E4M3 weights are
  // exact in f16 and expand with the hardware conversion; token rows are
  // scaled by a power of two into f16 range (undone in the GEMM1 epilogue);
  // with swigluoai, a (rounded to bf16, R1) is held as f16, which is exact.
  // ReLU^2 layers take f16 operands in GEMM1 only (its output is
  // not bounded, so a stays bf16). MXFP4 weights take the same path with their power-of-two scales folded
  // by 2^12 into f16 range. GEMM2 runs on f16 operands only when a is f16
  // (GEMM1 on f16 operands with swigluoai) and its own weights are FP4.
  auto fp4 = [](const moe_qweight_t *w) { return w->fmt == MOE_FMT_NVFP4 || w->fmt == MOE_FMT_MXFP4; };
  const int f16_1 = fp4(w13) ? 1 : 0;
  // a is held as f16 times 2^9 (exact for |a| >= 2^-26 once rounded to bf16),
  // so |a| <= (limit + 1) * max(limit, 0.2785 / alpha) must stay within 64:
  // the gpt-oss constants (alpha 1.702, limit 7) give 56
  const bool a_fits = act.alpha > 0.f && act.limit >= 0.f &&
                      (act.limit + 1.f) * fmaxf(act.limit, 0.2785f / act.alpha) <= 64.f;
  const int f16_2 = (f16_1 && fp4(w2) && act.kind == MOE_ACT_SWIGLUOAI && a_fits) ? 1 : 0;
  if (!mark(0)) return MOE_ERR_CUDA;
  if ((s = launch_route(logits, sel_bias, T, E, k, route, ids, tw, status, st, n)) != MOE_OK) return s;
  if (!mark(1)) return MOE_ERR_CUDA;
  // (the per-chunk counts of a many-CTA alignment live in x_perm until the gather)
  if ((s = launch_align(ids, T, k, E, bm, P, sorted, offs, blocks, rowpos, status, st, n,
                        reinterpret_cast<int32_t *>(xperm))) != MOE_OK)
    return s;
  if (!mark(2)) return MOE_ERR_CUDA;
  // mul: 0 no routing weight, 1 in the GEMM2 epilogue, 2 on GEMM1's input rows
  const float *tw_in = mul == 2 ? tw : nullptr;
  s = launch_gather(x, T, k, H, E, P, rowpos, offs, sorted, xperm, xexp, f16_1 != 0, st, n, tw_in);
  if (s != MOE_OK) return s;
  if (!mark(3)) return MOE_ERR_CUDA;
  const int epi1 = act.kind == MOE_ACT_SWIGLUOAI ? 0 : 1;
  if ((s = launch_grouped_gemm(epi1, *w13, xperm, P, sorted, offs, R, nullptr, 0, layout, act, abuf, I, status, st,
                               n, f16_1 | (f16_2 << 1), xexp)) != MOE_OK)
    return s;
  if (!mark(4)) return MOE_ERR_CUDA;
  moe_act_t none = {0, 0.f, 0.f};
  if ((s = launch_grouped_gemm(2, *w2, abuf, P, sorted, offs, R, tw, mul == 1 ? 1 : 0, 0, none, ybuf, H, status, st,
                               n, f16_2)) != MOE_OK)
    return s;
  if (!mark(5)) return MOE_ERR_CUDA;
  if ((s = launch_unpermute(ybuf, rowpos, T, k, H, P, out, status, st, n)) != MOE_OK) return s;
  return mark(6) ? MOE_OK : MOE_ERR_CUDA;
}

// staging: the workspace must also hold moe_forward_host's staging buffers
// for x, logits and out (they sit at its end); the device-pointer paths that
// never touch them may pass false.
static moe_status_t check_forward(const float *sel_bias, int T, int E, int k, int H, int I, int route,
                                  const moe_qweight_t *w13, const moe_qweight_t *w2, int layout, moe_act_t act,
                                  int *block_m, void *ws, size_t ws_bytes, int mul, bool staging = true) {
  if (*block_m == 0) *block_m = 16;
  if (mul < 0 || mul > 2) return MOE_ERR_INVALID_ARG;  // routing weight: none, on the output, on the input
  if (!valid_dims(T, E, k, H, I) || !valid_block_m(*block_m)) return MOE_ERR_INVALID_ARG;
  if (route != MOE_ROUTE_TOPK_SOFTMAX && route != MOE_ROUTE_SIGMOID_BIAS) return MOE_ERR_INVALID_ARG;
  if (route == MOE_ROUTE_SIGMOID_BIAS && !aligned16(sel_bias)) return MOE_ERR_INVALID_ARG;
  if (act.kind != MOE_ACT_SWIGLUOAI && act.kind != MOE_ACT_RELU2) return MOE_ERR_INVALID_ARG;
  if (layout != MOE_LAYOUT_INTERLEAVED && layout != MOE_LAYOUT_CONCAT) return MOE_ERR_INVALID_ARG;
  const int N1 = act.kind == MOE_ACT_SWIGLUOAI ? 2 * I : I;
  moe_status_t s;
  if ((s = check_weight(w13, E, N1, H)) != MOE_OK) return s;
  if ((s = check_weight(w2, E, H, I)) != MOE_OK) return s;
  if (!aligned16(ws)) return MOE_ERR_INVALID_ARG;
  const Carve c = carve(T, E, k, H, I, *block_m);
  if (ws_bytes < (staging ? c.total : c.xin)) return MOE_ERR_WORKSPACE;
  return MOE_OK;
}



moe_status_t moe_forward(const uint16_t *x, const float *logits, const float *sel_bias, int T, int E, int k, int H,
                         int I, int route, const moe_qweight_t *w13, const moe_qweight_t *w2, int gate_up_layout,
                         moe_act_t act, int mul_topk_weights, int block_m, uint16_t *out, void *ws,
                         size_t ws_bytes, moe_stream_t stream) {
  g_last_launches = 0;
  moe_status_t s = check_forward(sel_bias, T, E, k, H, I, route, w13, w2, gate_up_layout, act, &block_m, ws,
                                 ws_bytes, mul_topk_weights);
  if (s != MOE_OK) return s;
  if (T == 0) return MOE_OK;
  if (!aligned16(x) || !aligned16(logits) || !aligned16(out)) return MOE_ERR_INVALID_ARG;
  return forward_impl(x, logits, sel_bias, T, E, k, H, I, route, w13, w2, gate_up_layout, act, mul_topk_weights,
                      block_m, out, ws, (cudaStream_t)stream);
}

moe_status_t moe_forward_profile(const uint16_t *x, const float *logits, const float *sel_bias, int T, int E,
                                 int k, int H, int I, int route, const moe_qweight_t *w13, const moe_qweight_t *w2,
                                 int gate_up_layout, moe_act_t act, int mul_topk_weights, int block_m, uint16_t *out,
                                 void *ws, size_t ws_bytes, moe_stream_t stream, float *kernel_ms) {
  g_last_launches = 0;
  if (!kernel_ms) return MOE_ERR_INVALID_ARG;
  moe_status_t s = check_forward(sel_bias, T, E, k, H, I, route, w13, w2, gate_up_layout, act, &block_m, ws,
                                 ws_bytes, mul_topk_weights);
  if (s != MOE_OK) return s;
  for (int i = 0; i < 6; ++i) kernel_ms[i] = 0.f;
  if (T == 0) return MOE_OK;
  if (!aligned16(x) || !aligned16(logits) || !aligned16(out)) return MOE_ERR_INVALID_ARG;
  cudaEvent_t ev[7];
  int made = 0;
  for (; made < 7; ++made)
    if (cudaEventCreate(&ev[made]) != cudaSuccess) break;
  if (made == 7) {
    s = forward_impl(x, logits, sel_bias, T, E, k, H, I, route, w13, w2, gate_up_layout, act, mul_topk_weights,
                     block_m, out, ws, (cudaStream_t)stream, ev);
    if (s == MOE_OK && cudaEventSynchronize(ev[6]) != cudaSuccess) s = MOE_ERR_CUDA;
    for (int i = 0; s == MOE_OK && i < 6; ++i)
      if (cudaEventElapsedTime(&kernel_ms[i], ev[i], ev[i + 1]) != cudaSuccess) s = MOE_ERR_CUDA;
  } else {
    s = MOE_ERR_CUDA;
  }
  for (int i = 0; i < made; ++i) cudaEventDestroy(ev[i]);
  return s;
}

moe_status_t moe_forward_host(const uint16_t *x_host, const float *logits_host, const float *sel_bias, int T,
                              int E, int k, int H, int I, int route, const moe_qweight_t *w13,
                              const moe_qweight_t *w2, int gate_up_layout, moe_act_t act, int mul_topk_weights,
                              int block_m, uint16_t *out_host, void *ws, size_t ws_bytes, moe_stream_t stream) {
  g_last_launches = 0;
  moe_status_t s = check_forward(sel_bias, T, E, k, H, I, route, w13, w2, gate_up_layout, act, &block_m, ws,
                                 ws_bytes, mul_topk_weights);
  if (s != MOE_OK) return s;
  if (T == 0) return MOE_OK;
  if (!x_host || !logits_host || !out_host) return MOE_ERR_INVALID_ARG;
  const Carve c = carve(T, E, k, H, I, block_m);
  cudaStream_t st = (cudaStream_t)stream;
  // Page-locked host buffers are mapped into the device's address space: the
  // route and gather kernels then read x and logits, and the unpermute writes
  // out, in place over the host link (NVLink-C2C on a Grace host), with no
  // staging copies. Other host memory is staged through the workspace.
  void *xm = nullptr, *lm = nullptr, *om = nullptr;
  const bool mapped = cudaHostGetDevicePointer(&xm, const_cast<uint16_t *>(x_host), 0) == cudaSuccess &&
                      cudaHostGetDevicePointer(&lm, const_cast<float *>(logits_host), 0) == cudaSuccess &&
                      cudaHostGetDevicePointer(&om, out_host, 0) == cudaSuccess && aligned16(xm) &&
                      aligned16(lm) && aligned16(om);
  if (!mapped) (void)cudaGetLastError();  // a pageable buffer: not an error
  if (mapped)
    return forward_impl(static_cast<const uint16_t *>(xm), static_cast<const float *>(lm), sel_bias, T, E, k, H, I,
                        route, w13, w2, gate_up_layout, act, mul_topk_weights, block_m,
                        static_cast<uint16_t *>(om), ws, st);
  uint16_t *xd = at<uint16_t>(ws, c.xin);
  float *ld = at<float>(ws, c.lin);
  uint16_t *od = at<uint16_t>(ws, c.outb);
  if (cudaMemcpyAsync(xd, x_host, (size_t)T * H * 2, cudaMemcpyHostToDevice, st) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemcpyAsync(ld, logits_host, (size_t)T * E * 4, cudaMemcpyHostToDevice, st) != cudaSuccess)
    return MOE_ERR_CUDA;
  s = forward_impl(xd, ld, sel_bias, T, E, k, H, I, route, w13, w2, gate_up_layout, act, mul_topk_weights, block_m,
                   od, ws, st);
  if (s != MOE_OK) return s;
  if (cudaMemcpyAsync(out_host, od, (size_t)T * H * 2, cudaMemcpyDeviceToHost, st) != cudaSuccess) return MOE_ERR_CUDA;
  return MOE_OK;
}

moe_status_t moe_read_status(const void *ws, moe_stream_t stream, int *status) {
  if (!aligned16(ws) || !status) return MOE_ERR_INVALID_ARG;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return MOE_ERR_CUDA;
  unsigned int word = 0;
  if (cudaMemcpy(&word, ws, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  *status = MOE_OK;
  for (int code = 1; code < 32; ++code)
    if (word & (1u << (code - 1))) {
      *status = code;
      break;
    }
  return MOE_OK;
}

moe_status_t moe_clear_status(void *ws, moe_stream_t stream) {
  if (!aligned16(ws)) return MOE_ERR_INVALID_ARG;
  return cudaMemsetAsync(ws, 0, MOE_STATUS_BYTES, (cudaStream_t)stream) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status_t moe_wait_selftest(void *ws, moe_stream_t stream) {
  g_last_launches = 0;
  if (!aligned16(ws)) return MOE_ERR_INVALID_ARG;
  wait_selftest_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(status_of(ws));
  ++g_last_launches;
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

const char *moe_status_string(int status) {
  switch (status) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
    case MOE_ERR_BAD_INDEX: return "MOE_ERR_BAD_INDEX";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE";
    case MOE_ERR_SCALE_RANGE: return "MOE_ERR_SCALE_RANGE";
    default: return "MOE_ERR_UNKNOWN";
  }
}

int moe_last_launch_count(void) { return g_last_launches; }

}  // extern "C"

namespace moe4 {

// The fixed-workspace forward behind moe_forward_static: every host-side
// check that moe_forward makes comes first (against the part of the
// workspace the device-pointer path uses, without moe_forward_host's
// staging buffers), so a rejected call enqueues nothing. Only then is the
// status word cleared, the layer run and the status word copied out.
moe_status_t forward_fixed_workspace(const uint16_t *x, const float *logits, const float *sel_bias, int T, int E,
                                     int k, int H, int I, int route, const moe_qweight_t *w13,
                                     const moe_qweight_t *w2, int layout, moe_act_t act, int mul, int block_m,
                                     uint16_t *out, uint32_t *status_out, void *ws, size_t ws_bytes,
                                     cudaStream_t st) {
  g_last_launches = 0;
  moe_status_t s = check_forward(sel_bias, T, E, k, H, I, route, w13, w2, layout, act, &block_m, ws, ws_bytes, mul,
                                 /*staging=*/false);
  if (s == MOE_ERR_WORKSPACE) return MOE_ERR_UNSUPPORTED;  // past the fixed workspace's capacity
  if (s != MOE_OK) return s;
  if (T == 0) return MOE_OK;
  if (!aligned16(x) || !aligned16(logits) || !aligned16(out)) return MOE_ERR_INVALID_ARG;
  if (status_out && (reinterpret_cast<uintptr_t>(status_out) & 3u)) return MOE_ERR_INVALID_ARG;
  // the workspace keeps the previous call's contents: only the status word
  // has to start at zero (every intermediate is written before it is read)
  if (cudaMemsetAsync(ws, 0, MOE_STATUS_BYTES, st) != cudaSuccess) return MOE_ERR_CUDA;
  s = forward_impl(x, logits, sel_bias, T, E, k, H, I, route, w13, w2, layout, act, mul, block_m, out, ws, st);
  if (s != MOE_OK) return s;
  if (status_out && cudaMemcpyAsync(status_out, ws, sizeof(uint32_t), cudaMemcpyDeviceToDevice, st) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

}  // namespace moe4
