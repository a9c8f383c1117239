// Step a5: unpermute/reduce back to token order at the unpadded width H
// (vLLM issue "gpt-oss-120b MXFP4 + --enable-expert-parallel crashes", Root
// cause: the layer's output must be [T, H] at the real hidden size).
// out[t] = bf16(sum_{j<k} y[row_pos[t*k+j]]) with an fp32 running sum in
// ascending j: a gather-sum, not an atomic scatter, so results are
// bit-identical from run to run.
#include "common.cuh"
#include "kernels.h"

namespace moe4 {

namespace {

__device__ __forceinline__ void acc8(float (&a)[8], const uint4 v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    a[2 * i] += __uint_as_float(w[i] << 16);
    a[2 * i + 1] += __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

constexpr int kUnpermMaxThreads = 512;  // one 8-column vector per thread (H <= 4096)

// grid (T, ceil(H/8 / threads)): one token per CTA (a small batch, T < 256,
// splits each row over CTAs of 64 threads so that it still spreads over the SMs)
__global__ void __launch_bounds__(kUnpermMaxThreads) unpermute_kernel(const uint4 *__restrict__ y,
                                                                   const int32_t *__restrict__ row_pos, int T,
                                                                   int k, int H8, int P_max,
                                                                   uint4 *__restrict__ out, unsigned int *status) {
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.x;
  int pos[8];
  bool ok = true;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    pos[j] = -1;
    if (j < k) {
      pos[j] = row_pos[(size_t)t * k + j];
      if (pos[j] < 0 || pos[j] >= P_max) ok = false;
    }
  }
  if (!ok && threadIdx.x == 0 && blockIdx.y == 0) raise_status(status, MOE_ERR_BAD_INDEX);
  const int v = blockIdx.y * blockDim.x + threadIdx.x;
  if (v < H8) {
    // all k rows' loads first (streaming: y is read once), then the sum in
    // ascending j
    uint4 q[8];
#pragma unroll
    for (int j = 0; j < 8; ++j)
      q[j] = (j < k && pos[j] >= 0 && pos[j] < P_max) ? __ldcs(&y[(size_t)pos[j] * H8 + v]) : make_uint4(0, 0, 0, 0);
    float a[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (j < k && pos[j] >= 0 && pos[j] < P_max) acc8(a, q[j]);
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __nv_bfloat162 h = __floats2bfloat162_rn(a[2 * i], a[2 * i + 1]);
      o[i] = *reinterpret_cast<const uint32_t *>(&h);
    }
    out[(size_t)t * H8 + v] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

}  // namespace

moe_status_t launch_unpermute(const uint16_t *y, const int32_t *row_pos, int T, int k, int H, int P_max,
                              uint16_t *out, unsigned int *status, cudaStream_t stream, int *launches) {
  if (T == 0) return MOE_OK;
  const int H8 = H / 8;
  int threads = (H8 + 31) / 32 * 32;
  if (threads > kUnpermMaxThreads) return MOE_ERR_UNSUPPORTED;
  if (T < 256) threads = 64;
  const dim3 grid(T, (H8 + threads - 1) / threads);
  const cudaError_t err = launch_pdl(unpermute_kernel, grid, dim3(threads), 0, stream,
                                     reinterpret_cast<const uint4 *>(y), row_pos, T, k, H8, P_max,
                                     reinterpret_cast<uint4 *>(out), status);
  if (launches) ++*launches;
  return err == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe4
