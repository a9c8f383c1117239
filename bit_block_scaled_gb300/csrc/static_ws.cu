// moe_forward_static: the whole layer for callers that cannot allocate device
// memory themselves -- code running where cudaMalloc is unavailable or not
// allowed (inside a CUDA-graph capture in a framework that forbids
// allocation during capture, a plugin whose host hands it only input and
// output buffers, or a runtime with a fixed memory budget taken up front).
//
// The workspace that moe_forward takes from its caller lives here instead, in
// a file-scope device array of MOE_STATIC_WS_BYTES. Every GPU that loads the
// library keeps that array until the process exits, and every call shares
// it: calls whose work overlaps on the GPU (different streams, no ordering
// between them) race on it and must not be issued.
#include <mutex>

#include "common.cuh"

namespace {

static __device__ __align__(256) unsigned char g_static_ws[MOE_STATIC_WS_BYTES];

constexpr int kMaxDevices = 64;
void *g_ws_ptr[kMaxDevices];
cudaError_t g_ws_err[kMaxDevices];
std::once_flag g_ws_once[kMaxDevices];

}  // namespace

extern "C" moe_status_t moe_forward_static(const uint16_t *x, const float *logits, const float *sel_bias, int T,
                                           int E, int k, int H, int I, int route, const moe_qweight_t *w13,
                                           const moe_qweight_t *w2, int gate_up_layout, moe_act_t act,
                                           int mul_topk_weights, int block_m, uint16_t *out,
                                           uint32_t *status_out, moe_stream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
  // Once per device, with that device current: the device address of the
  // array (in host code its name is only a host-side stand-in).
  std::call_once(g_ws_once[dev], [dev] {
    g_ws_err[dev] = cudaGetSymbolAddress(&g_ws_ptr[dev], g_static_ws);
  });
  if (g_ws_err[dev] != cudaSuccess || g_ws_ptr[dev] == nullptr) return MOE_ERR_CUDA;
  size_t need = 0;
  moe_status_t s = moe_workspace_size(T, E, k, H, I, block_m, &need);
  if (s != MOE_OK) return s;
  if (need > MOE_STATIC_WS_BYTES) return MOE_ERR_UNSUPPORTED;  // sizes past the array's capacity
  cudaStream_t st = (cudaStream_t)stream;
  // the array keeps the previous call's contents: only the status word has
  // to start at zero (every intermediate is written before it is read)
  if (cudaMemsetAsync(g_ws_ptr[dev], 0, MOE_STATUS_BYTES, st) != cudaSuccess) return MOE_ERR_CUDA;
  s = moe_forward(x, logits, sel_bias, T, E, k, H, I, route, w13, w2, gate_up_layout, act, mul_topk_weights,
                  block_m, out, g_ws_ptr[dev], MOE_STATIC_WS_BYTES, stream);
  if (s != MOE_OK) return s;
  if (status_out &&
      cudaMemcpyAsync(status_out, g_ws_ptr[dev], sizeof(uint32_t), cudaMemcpyDeviceToDevice, st) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}
