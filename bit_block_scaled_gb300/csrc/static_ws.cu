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
#include <atomic>
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace {

static __device__ __align__(256) unsigned char g_static_ws[MOE_STATIC_WS_BYTES];

constexpr int kMaxDevices = 64;
std::atomic<void *> g_ws_ptr[kMaxDevices];  // set once a lookup on that device has succeeded
std::mutex g_ws_mutex;

// Device address of the array on the current device `dev`. In host code the
// array's name is only a host-side stand-in, so its address is looked up with
// that device current. Only a successful lookup is kept; a failed one (for
// example made during a stream capture) is retried by the next call.
void *static_ws_address(int dev) {
  void *p = g_ws_ptr[dev].load(std::memory_order_acquire);
  if (p) return p;
  std::lock_guard<std::mutex> lock(g_ws_mutex);
  p = g_ws_ptr[dev].load(std::memory_order_relaxed);
  if (!p) {
    if (cudaGetSymbolAddress(&p, g_static_ws) != cudaSuccess || !p) {
      (void)cudaGetLastError();  // the failed lookup leaves no error behind for the next CUDA call
      return nullptr;
    }
    g_ws_ptr[dev].store(p, std::memory_order_release);
  }
  return p;
}

}  // namespace

extern "C" moe_status_t moe_forward_static(const uint16_t *x, const float *logits, const float *sel_bias, int T,
                                           int E, int k, int H, int I, int route, const moe_qweight_t *w13,
                                           const moe_qweight_t *w2, int gate_up_layout, moe_act_t act,
                                           int mul_topk_weights, int block_m, uint16_t *out,
                                           uint32_t *status_out, moe_stream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
  void *ws = static_ws_address(dev);
  if (!ws) return MOE_ERR_CUDA;
  // every argument is checked before anything is enqueued; sizes past the
  // array's capacity return MOE_ERR_UNSUPPORTED
  return moe4::forward_fixed_workspace(x, logits, sel_bias, T, E, k, H, I, route, w13, w2, gate_up_layout, act,
                                       mul_topk_weights, block_m, out, status_out, ws, MOE_STATIC_WS_BYTES,
                                       (cudaStream_t)stream);
}
