// Step a2: align/permute routed rows into per-expert blocks, then gather the
// token rows (vLLM issue "moe_wna16_marlin_gemm applies wrong per-row topk
// weights", "Minimal repro": moe_align_block_size and the sorted_ids /
// expert_ids it produces).
//
// align_kernel is one CTA of W warps (8 up to 1024 routed rows, else 32). Warp
// w owns the contiguous flat rows [w * R / W, (w + 1) * R / W) and walks them
// in order, 32 at a time:
//   1. per-warp expert counts (__match_any_sync groups equal ids in a step);
//   2. a warp prefix sum of the block-padded totals gives expert_offsets, and
//      a per-expert prefix over the W warps gives each warp's first slot;
//   3. each warp walks its rows again and places every row at its expert's
//      running slot.
// The order inside an expert is ascending flat row id by construction, so the
// layout does not depend on thread timing.
#include "common.cuh"
#include "kernels.h"

namespace moe4 {

namespace {

constexpr int kAlignThreads = 1024;
constexpr int kMaxE = 256;
constexpr int kAlignSplitRows = 4096;  // from this many routed rows on, the alignment runs over many CTAs

__global__ void __launch_bounds__(kAlignThreads) align_kernel(const int32_t *__restrict__ ids, int R, int E,
                                                              int bm, int P_max, int32_t *__restrict__ sorted,
                                                              int32_t *__restrict__ offsets,
                                                              int32_t *__restrict__ block_ids,
                                                              int32_t *__restrict__ row_pos,
                                                              unsigned int *status) {
  __shared__ int off[kMaxE + 1];
  __shared__ int wcnt[32 * kMaxE];  // [warp][expert]: counts, then first slot
  pdl_wait();
  pdl_trigger();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nwarps = blockDim.x >> 5, nthr = blockDim.x;
  const int r_lo = (int)((long long)R * warp / nwarps), r_hi = (int)((long long)R * (warp + 1) / nwarps);

  // 1. per-warp counts, in row order
  for (int e = lane; e < E; e += 32) wcnt[warp * E + e] = 0;
  __syncwarp();
  for (int r0 = r_lo; r0 < r_hi; r0 += 32) {
    const int r = r0 + lane;
    int e = -1;
    if (r < r_hi) {
      e = ids[r];
      if (e < 0 || e >= E) {
        raise_status(status, MOE_ERR_BAD_INDEX);
        row_pos[r] = -1;
        e = -1;
      }
    }
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    if (e >= 0 && lane == __ffs(peers) - 1) wcnt[warp * E + e] += __popc(peers);
    __syncwarp();
  }
  __syncthreads();
  // 2. expert totals -> padded offsets (warp 0), then each warp's first slot
  if (warp == 0) {
    int running = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + lane;
      int c = 0;
      if (e < E)
        for (int w = 0; w < nwarps; ++w) c += wcnt[w * E + e];
      const int pc = (c + bm - 1) / bm * bm;
      int incl = pc;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      if (e < E) off[e] = running + incl - pc;
      running += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) off[E] = running;
  }
  __syncthreads();
  for (int e = tid; e < E; e += nthr) {
    int run = off[e];
    for (int w = 0; w < nwarps; ++w) {
      const int c = wcnt[w * E + e];
      wcnt[w * E + e] = run;
      run += c;
    }
  }
  for (int e = tid; e <= E; e += nthr) offsets[e] = off[e];
  for (int q = tid; q < P_max; q += nthr) sorted[q] = R;
  const int nb = P_max / bm;
  for (int b = tid; b < nb; b += nthr) {
    const int s = b * bm;
    int be = -1;
    if (s < off[E]) {
      int lo = 0, hi = E - 1;  // largest e with off[e] <= s
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (off[mid] <= s) lo = mid; else hi = mid - 1;
      }
      be = lo;
    }
    block_ids[b] = be;
  }
  __syncthreads();
  // 3. placement, in row order within each warp
  for (int r0 = r_lo; r0 < r_hi; r0 += 32) {
    const int r = r0 + lane;
    int e = -1;
    if (r < r_hi) {
      e = ids[r];
      if (e < 0 || e >= E) e = -1;
    }
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    if (e >= 0) {
      const int pos = wcnt[warp * E + e] + __popc(peers & ((1u << lane) - 1u));
      sorted[pos] = r;
      row_pos[r] = pos;
    }
    __syncwarp();
    if (e >= 0 && lane == __ffs(peers) - 1) wcnt[warp * E + e] += __popc(peers);
    __syncwarp();
  }
}

// Within every group of 8 columns, x_perm stores the elements in the order
// 0,4,1,5,2,6,3,7 (the order the GEMM's weight expansion produces them in).
__device__ __forceinline__ uint4 interleave8(uint4 v) {
  return make_uint4(__byte_perm(v.x, v.z, 0x5410), __byte_perm(v.x, v.z, 0x7632),
                    __byte_perm(v.y, v.w, 0x5410), __byte_perm(v.y, v.w, 0x7632));
}

// Routing weight applied on the input: bf16(fp32(x * w)) for both bf16 halves.
__device__ __forceinline__ uint32_t weigh_bf16x2(uint32_t pair, float w) {
  const uint32_t lo = float_to_bf16_bits(__fmul_rn(bf16_bits_to_float((uint16_t)(pair & 0xFFFFu)), w));
  const uint32_t hi = float_to_bf16_bits(__fmul_rn(bf16_bits_to_float((uint16_t)(pair >> 16)), w));
  return lo | (hi << 16);
}

__device__ __forceinline__ uint4 weigh8(uint4 q, float w) {
  return make_uint4(weigh_bf16x2(q.x, w), weigh_bf16x2(q.y, w), weigh_bf16x2(q.z, w), weigh_bf16x2(q.w, w));
}

// The same alignment for large batches, over many CTAs: the rows are cut into
// chunks of kChunkRows in row order. align_count_kernel counts each chunk's
// rows per expert; align_place_kernel then lets every CTA derive, from all the
// chunks' counts, the padded expert offsets and the first slot of its own
// chunk in each expert (the slots of the earlier chunks' rows come first), and
// place its rows exactly as the one-CTA kernel would: ascending flat row id
// within each expert, so the result is the same bytes.
constexpr int kChunkRows = kAlignThreads;  // one row per thread

__global__ void __launch_bounds__(kAlignThreads) align_count_kernel(const int32_t *__restrict__ ids, int R, int E,
                                                                    int32_t *__restrict__ counts,
                                                                    int32_t *__restrict__ row_pos,
                                                                    unsigned int *status) {
  __shared__ int cnt[kMaxE];
  pdl_wait();
  pdl_trigger();
  const int tid = threadIdx.x;
  for (int e = tid; e < E; e += kAlignThreads) cnt[e] = 0;
  __syncthreads();
  const int r = blockIdx.x * kChunkRows + tid;
  if (r < R) {
    const int e = ids[r];
    if (e < 0 || e >= E) {
      raise_status(status, MOE_ERR_BAD_INDEX);
      row_pos[r] = -1;
    } else {
      atomicAdd(&cnt[e], 1);
    }
  }
  __syncthreads();
  for (int e = tid; e < E; e += kAlignThreads) counts[(size_t)blockIdx.x * E + e] = cnt[e];
}

__global__ void __launch_bounds__(kAlignThreads) align_place_kernel(const int32_t *__restrict__ ids, int R, int E,
                                                                    int bm, int P_max, int nchunks,
                                                                    const int32_t *__restrict__ counts,
                                                                    int32_t *__restrict__ sorted,
                                                                    int32_t *__restrict__ offsets,
                                                                    int32_t *__restrict__ block_ids,
                                                                    int32_t *__restrict__ row_pos) {
  __shared__ int off[kMaxE + 1];
  __shared__ int tot[kMaxE];
  __shared__ int bef[kMaxE];        // rows of the earlier chunks, per expert
  __shared__ int wcnt[32 * kMaxE];  // [warp][expert]: counts, then first slot
  pdl_wait();
  pdl_trigger();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c = blockIdx.x;
  // each expert's total and the rows of the chunks before this one
  for (int e = tid; e < E; e += kAlignThreads) {
    int t = 0, before = 0;
    for (int q = 0; q < nchunks; ++q) {
      const int v = counts[(size_t)q * E + e];
      if (q < c) before += v;
      t += v;
    }
    tot[e] = t;
    bef[e] = before;
  }
  __syncthreads();
  if (warp == 0) {  // padded offsets
    int running = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + lane;
      const int pc = e < E ? (tot[e] + bm - 1) / bm * bm : 0;
      int incl = pc;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      if (e < E) off[e] = running + incl - pc;
      running += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) off[E] = running;
  }
  // per-warp counts of this chunk, in row order
  const int r = c * kChunkRows + tid;
  int e_r = -1;
  if (r < R) {
    e_r = ids[r];
    if (e_r < 0 || e_r >= E) e_r = -1;
  }
  for (int e = lane; e < E; e += 32) wcnt[warp * E + e] = 0;
  __syncwarp();
  const unsigned peers = __match_any_sync(0xffffffffu, e_r);
  if (e_r >= 0 && lane == __ffs(peers) - 1) wcnt[warp * E + e_r] = __popc(peers);
  __syncthreads();
  // first slot of each warp's rows in each expert
  for (int e = tid; e < E; e += kAlignThreads) {
    int run = off[e] + bef[e];
    for (int w = 0; w < 32; ++w) {
      const int cw = wcnt[w * E + e];
      wcnt[w * E + e] = run;
      run += cw;
    }
  }
  __syncthreads();
  if (e_r >= 0) {
    const int pos = wcnt[warp * E + e_r] + __popc(peers & ((1u << lane) - 1u));
    sorted[pos] = r;
    row_pos[r] = pos;
  }
  // padding slots of this CTA's share of the experts, the slots past the
  // last expert, the block -> expert table and the offsets
  for (int e = c; e < E; e += gridDim.x)
    for (int q = off[e] + tot[e] + tid; q < off[e + 1]; q += kAlignThreads) sorted[q] = R;
  if (c == 0) {
    for (int q = off[E] + tid; q < P_max; q += kAlignThreads) sorted[q] = R;
    for (int e = tid; e <= E; e += kAlignThreads) offsets[e] = off[e];
  }
  const int nb = P_max / bm;
  for (int b = c * kAlignThreads + tid; b < nb; b += gridDim.x * kAlignThreads) {
    const int s0 = b * bm;
    int be = -1;
    if (s0 < off[E]) {
      int lo = 0, hi = E - 1;  // largest e with off[e] <= s0
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (off[mid] <= s0) lo = mid; else hi = mid - 1;
      }
      be = lo;
    }
    block_ids[b] = be;
  }
}

// Gather, one CTA per token: the token's row is read once and written to the
// slots of its k routed rows (row_pos); E more CTAs zero each expert's padding
// slots (the tail of its segment whose sorted id is not a routed row). Slots
// past offsets[E] are never read by the GEMMs and are not written.
//   bf16 (F16 = false): x_perm[p] = x[t] with the columns interleaved within
//     groups of 8 (the order the GEMM's weight expansion produces them in).
//   f16 (F16 = true): x16[p] = f16(x[t] * 2^-e_p) in natural column order, with
//     e_p chosen so that the row's largest magnitude lands in [2^14, 2^15)
//     (exact for every bf16 element down to 2^-31 of it); xexp[p] = e_p, which
//     the GEMM epilogue multiplies back. Padding slots get e_p = 0.
// With tw (routing weight on the input) the row of slot p is first rounded to
// bf16(x * tw[r]), r the routed row's own flat index.
constexpr int kGatherMaxThreads = 512;  // one 8-column vector per thread (H <= 4096)

template <bool F16>
__global__ void __launch_bounds__(kGatherMaxThreads) gather_tok_kernel(
    const uint4 *__restrict__ x, int T, int k, int H8, int E, const int32_t *__restrict__ row_pos,
    const int32_t *__restrict__ offs, const int32_t *__restrict__ sorted, int P_max, uint4 *__restrict__ x_out,
    int32_t *__restrict__ xexp, const float *__restrict__ tw) {
  __shared__ float wmax[8][kGatherMaxThreads / 32];
  pdl_wait();
  pdl_trigger();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int R = T * k;
  if ((int)blockIdx.x >= T) {  // padding slots of expert e
    const int e = blockIdx.x - T;
    const int lo = offs[e], hi = offs[e + 1];
    for (int q = hi - 1; q >= lo; --q) {
      const int sid = sorted[q];
      if (sid >= 0 && sid < R) break;  // a routed row: the padding ends here
      for (int v = tid; v < H8; v += blockDim.x) x_out[(size_t)q * H8 + v] = make_uint4(0, 0, 0, 0);
      if (F16 && tid == 0) xexp[q] = 0;
    }
    return;
  }
  const int t = blockIdx.x;
  const bool has = tid < H8;
  const uint4 q = has ? x[(size_t)t * H8 + tid] : make_uint4(0, 0, 0, 0);
  // one exponent per slot with tw (each slot has its own weight), else one per token
  const int ne = F16 ? (tw ? k : 1) : 0;
  int ex[8];
  if (F16) {
    const int nw = blockDim.x >> 5;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (j < ne) {
        const uint4 u = tw ? weigh8(q, tw[(size_t)t * k + j]) : q;
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
        float m = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i)
          m = fmaxf(m, fmaxf(fabsf(__uint_as_float(w[i] << 16)), fabsf(__uint_as_float(w[i] & 0xFFFF0000u))));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (lane == 0) wmax[j][warp] = m;
      }
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (j < ne) {
        float m = 0.f;
        for (int w = 0; w < nw; ++w) m = fmaxf(m, wmax[j][w]);
        // m < 2^x (x from the fp32 exponent field); scaling by 2^-e, e = x - 15,
        // puts the largest entry in [2^14, 2^15): below the f16 maximum, and
        // every bf16 entry down to 2^-31 of it stays exact in f16 (normal down
        // to 2^-28 of it, subnormal with 8 bits below)
        const int xe = (int)((__float_as_uint(m) >> 23) & 0xFFu) - 126;
        ex[j] = max(-126, min(xe - 15, 126));
      }
    }
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    if (j >= k) break;
    const int r = t * k + j;
    const int p = row_pos[r];
    if (p < 0 || p >= P_max) continue;  // a row with a bad expert id is not placed
    const uint4 u = tw ? weigh8(q, tw[r]) : q;
    if (F16) {
      const int e = tw ? ex[j] : ex[0];
      const float sc = __uint_as_float((uint32_t)(127 - e) << 23);  // 2^-e
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
      uint32_t o[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const __half2 h = __floats2half2_rn(__uint_as_float(w[i] << 16) * sc, __uint_as_float(w[i] & 0xFFFF0000u) * sc);
        o[i] = *reinterpret_cast<const uint32_t *>(&h);
      }
      if (has) x_out[(size_t)p * H8 + tid] = make_uint4(o[0], o[1], o[2], o[3]);
      if (tid == 0) xexp[p] = e;
    } else {
      if (has) x_out[(size_t)p * H8 + tid] = interleave8(u);
    }
  }
}

}  // namespace

int align_chunks(int R) { return R >= kAlignSplitRows ? (R + kChunkRows - 1) / kChunkRows : 0; }

moe_status_t launch_align(const int32_t *ids, int T, int k, int E, int block_m, int P_max,
                          int32_t *sorted_ids, int32_t *offsets, int32_t *block_ids, int32_t *row_pos,
                          unsigned int *status, cudaStream_t stream, int *launches, int32_t *counts) {
  const int R = T * k;
  const int nchunks = align_chunks(R);
  if (counts && nchunks > 0) {  // many rows: counts per chunk, then placement over many CTAs
    cudaError_t err = launch_pdl(align_count_kernel, dim3(nchunks), dim3(kAlignThreads), 0, stream, ids, R, E, counts,
                                 row_pos, status);
    if (launches) ++*launches;
    if (err != cudaSuccess) return MOE_ERR_CUDA;
    err = launch_pdl(align_place_kernel, dim3(nchunks), dim3(kAlignThreads), 0, stream, ids, R, E, block_m, P_max,
                     nchunks, (const int32_t *)counts, sorted_ids, offsets, block_ids, row_pos);
    if (launches) ++*launches;
    return err == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
  }
  // up to 1024 rows: 8 warps (a shorter per-expert prefix over the warps)
  const int threads = R <= 1024 ? 256 : kAlignThreads;
  const cudaError_t err = launch_pdl(align_kernel, dim3(1), dim3(threads), 0, stream, ids, R, E, block_m,
                                     P_max, sorted_ids, offsets, block_ids, row_pos, status);
  if (launches) ++*launches;
  return err == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status_t launch_gather(const uint16_t *x, int T, int k, int H, int E, int P_max, const int32_t *row_pos,
                           const int32_t *offsets, const int32_t *sorted_ids, uint16_t *x_out, int32_t *xexp,
                           bool f16, cudaStream_t stream, int *launches, const float *tw) {
  if (T == 0 || P_max == 0) return MOE_OK;
  const int H8 = H / 8;
  const int threads = (H8 + 31) / 32 * 32;
  if (threads > kGatherMaxThreads || k > 8) return MOE_ERR_UNSUPPORTED;
  const auto kern = f16 ? gather_tok_kernel<true> : gather_tok_kernel<false>;
  const cudaError_t err = launch_pdl(kern, dim3(T + E), dim3(threads), 0, stream, reinterpret_cast<const uint4 *>(x),
                                     T, k, H8, E, row_pos, offsets, sorted_ids, P_max,
                                     reinterpret_cast<uint4 *>(x_out), xexp, tw);
  if (launches) ++*launches;
  return err == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe4
