// Grouped GEMMs of the MoE layer with 4-bit block-scaled weights (steps a3, a4).
//
// One CTA computes one (weight tile, token tile) pair of one expert:
//   D[128 weight rows][n tokens] = W'[rows][K] . X[tokens][K]^T   (fp32, TMEM)
// with the weights as the MMA's M side ("swap-AB"), so a handful of routed
// tokens per expert (decode) still fills the 128-row MMA. The dequantised bf16
// weights never touch shared memory: the dequant warps write them straight
// into tensor memory (tcgen05.st) and the MMA reads its A operand from there,
// while the token rows (B operand) arrive by TMA into shared memory.
//
// Warp roles (320 threads):
//   warp 0      TMA producer: packed 4-bit weight tile (SWIZZLE_32B) and the
//               token rows (SWIZZLE_128B) per 64-wide K block, and the tile's
//               block scales once (bulk copy)
//   warp 1      TMEM allocation; one thread issues tcgen05.mma (kind::f16,
//               A from TMEM, B from shared memory)
//   warps 2..9  dequantise: warp w owns TMEM lanes 32*(w%4).. (one weight row
//               per lane) and half of each K block; then the epilogue
// The epilogues: GEMM1 adds bias and applies swigluoai (gate/up pairs are
// adjacent TMEM lanes) or ReLU^2; GEMM2 adds bias and multiplies each token row
// by its own routing weight, read through that row's flat index (the failure
// in the vLLM issue "moe_wna16_marlin_gemm applies wrong per-row topk weights",
// section "Forensic", was reading another row's entry).
//
// Dequantisation (the R0 operand of the pages' formula w = E2M1 * scale):
//  * E2M1 codes are placed straight into bf16 bit fields (sign -> bit 15,
//    exponent/mantissa -> bits 8..6); that bf16 equals the code's value times
//    2^-126 (code 1 becomes the bf16 subnormal 2^-127). One bf16x2 multiply by
//    (scale * 2^(126-c)) gives the exact product times 2^-c; the epilogue
//    multiplies the fp32 accumulator by 2^c. c = 8 for NVFP4 (E4M3 up to 448),
//    c = 0 for MXFP4 (E8M0 exponents up to 128, i.e. scales up to 2). The
//    scale byte -> bf16 conversion goes through a 256-entry table in shared
//    memory.
//  * GPTQ INT4: (q - z) * s is exact in fp32, then rounded once to bf16.
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace moe4 {

namespace {

constexpr int kWarps = 10;
constexpr int kThreads = kWarps * 32;
constexpr int kDqThreads = 256;  // warps 2..9
constexpr int kTileM = 128;      // weight rows per tile (TMEM lanes)
constexpr int kBK = 64;          // K per pipeline stage (128 bytes of bf16)
constexpr int kACols = 128;      // TMEM columns for the dequantised operand:
                                 // 128 / (32 * KPB) stage-sized buffers
constexpr int kMaxStagesL = 8;

enum { EPI_SWIGLU = 0, EPI_RELU2 = 1, EPI_WEIGHTED = 2 };

struct Smem {
  uint32_t x, w, sc, z, lut, ids, tw, bar, misc, total;
};

__host__ __device__ inline uint32_t align_up(uint32_t v, uint32_t a) { return (v + a - 1) / a * a; }

// Shared-memory carve-up; identical on host (sizing) and device (addresses).
__host__ __device__ inline Smem smem_layout(int tile_n, int stages, int kpb, int sc_row_bytes,
                                            int z_row_bytes) {
  Smem s;
  uint32_t o = 0;
  s.x = o;   o += stages * kpb * tile_n * 128;
  o = align_up(o, 1024);
  s.w = o;   o += stages * kTileM * 32 * kpb;
  s.sc = o;  o += align_up(kTileM * sc_row_bytes, 128);
  s.z = o;   o += align_up(kTileM * z_row_bytes, 128);
  s.lut = o; o += 256 * 4;
  s.ids = o; o += tile_n * 4;
  s.tw = o;  o += tile_n * 4;
  o = align_up(o, 8);
  s.bar = o; o += (2 * kMaxStagesL + 2 * 4 + 4) * 8;
  s.misc = o; o += 64;
  s.total = o + 1024;  // slack for aligning the dynamic base to 1024
  return s;
}

// TMEM columns: accumulator [0, tile_n), then kACols columns of operand
// buffers, each one stage wide (32 columns = 64 bf16 of K per lane per block).
__host__ __device__ inline uint32_t tmem_a_col(int tile_n) { return align_up(tile_n, 32); }
__host__ __device__ inline uint32_t tmem_cols(int tile_n) {
  const uint32_t need = tmem_a_col(tile_n) + kACols;
  uint32_t c = 32;
  while (c < need) c <<= 1;
  return c < 256 ? 256 : c;  // >= 256 keeps at most two CTAs per SM on TMEM
}

// bf16x2 bits of (E2M1 codes) * 2^-126 for 8 packed codes -> 4 words holding
// consecutive K pairs (k, k+1).
__device__ __forceinline__ void e2m1x8_raw(uint32_t x, uint32_t (&o)[4]) {
  const uint32_t y = x >> 8;
  const uint32_t r04 = ((x & 0x000F000Fu) * 0x1040u) & 0x81C081C0u;  // codes 0 | 4
  const uint32_t r15 = ((x & 0x00F000F0u) * 0x0104u) & 0x81C081C0u;  // codes 1 | 5
  const uint32_t r26 = ((y & 0x000F000Fu) * 0x1040u) & 0x81C081C0u;  // codes 2 | 6
  const uint32_t r37 = ((y & 0x00F000F0u) * 0x0104u) & 0x81C081C0u;  // codes 3 | 7
  o[0] = __byte_perm(r04, r15, 0x5410);
  o[1] = __byte_perm(r26, r37, 0x5410);
  o[2] = __byte_perm(r04, r15, 0x7632);
  o[3] = __byte_perm(r26, r37, 0x7632);
}

// a * b on bf16 pairs, one rounding (fma with a -0 addend keeps signed zeros).
__device__ __forceinline__ uint32_t bmul2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(0x80008000u));
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

// Position in a ring of n slots plus the parity of the current lap (the
// mbarrier phase), advanced by increments so hot loops never divide.
struct Ring {
  int slot = 0, phase = 0;
  __device__ __forceinline__ void advance(int n) {
    if (++slot == n) {
      slot = 0;
      phase ^= 1;
    }
  }
};

}  // namespace

template <int FMT, int EPI, int KPB>
__global__ void __launch_bounds__(kThreads, 2) grouped_gemm_kernel(const __grid_constant__ GemmArgs p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte aligned start (pointer arithmetic on the shared array keeps the
  // compiler's knowledge that all these addresses are shared memory)
  uint8_t *base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const Smem L = smem_layout(p.tile_n, p.stages, KPB, p.sc_row_bytes, p.z_row_bytes);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t bar0 = smem_u32(base + L.bar);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (kMaxStagesL + s); };
  constexpr int NA = kACols / (32 * KPB);  // operand buffers in TMEM
  auto dq_bar = [&](int s) { return bar0 + 8u * (2 * kMaxStagesL + s); };
  auto afree_bar = [&](int s) { return bar0 + 8u * (2 * kMaxStagesL + 4 + s); };
  const uint32_t sc_bar = bar0 + 8u * (2 * kMaxStagesL + 2 * 4);
  const uint32_t acc_bar = sc_bar + 8u;
  volatile int *misc = reinterpret_cast<volatile int *>(base + L.misc);
  // misc[0] = tmem base, [1..4] = tile info, [5] = abort flag
  int *ids_s = reinterpret_cast<int *>(base + L.ids);
  float *tw_s = reinterpret_cast<float *>(base + L.tw);
  uint32_t *lut = reinterpret_cast<uint32_t *>(base + L.lut);

  // ---- locate this CTA's token tile: expert e, slots [row0, row0 + nrows)
  if (warp == 0) {
    const int t = blockIdx.y;
    int cum = 0, found = 0, fe = 0, frow = 0, fn = 0;
    for (int e0 = 0; e0 < p.E && !found; e0 += 32) {
      const int e = e0 + lane;
      int seg = 0;
      if (e < p.E) seg = p.expert_offsets[e + 1] - p.expert_offsets[e];
      const int nt = (seg + p.tile_n - 1) / p.tile_n;
      int incl = nt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      const int excl = cum + incl - nt;
      const bool mine = (t >= excl) && (t < excl + nt);
      const unsigned m = __ballot_sync(0xffffffffu, mine);
      if (m) {
        const int src = __ffs(m) - 1;
        const int le = __shfl_sync(0xffffffffu, e, src);
        const int lex = __shfl_sync(0xffffffffu, excl, src);
        const int lseg = __shfl_sync(0xffffffffu, seg, src);
        fe = le;
        frow = p.expert_offsets[le] + (t - lex) * p.tile_n;
        fn = min(p.tile_n, p.expert_offsets[le] + lseg - frow);
        found = 1;
      }
      cum += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) {
      misc[1] = fe;
      misc[2] = frow;
      misc[3] = fn;
      const bool in_range = frow >= 0 && frow + fn <= p.P_max;
      if (found && fn > 0 && !in_range) raise_status(p.status, MOE_ERR_BAD_INDEX);
      misc[4] = found && fn > 0 && in_range;
      misc[5] = 0;
    }
  }
  if (tid == 32) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int s = 0; s < NA; ++s) {
      mbar_init(dq_bar(s), kDqThreads);
      mbar_init(afree_bar(s), 1);
    }
    mbar_init(sc_bar, 1);
    mbar_init(acc_bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (!misc[4]) return;  // no tile for this CTA
  const int e = misc[1], row0 = misc[2], nrows = misc[3];
  const int n16 = (nrows + 15) & ~15;
  const int mt = blockIdx.x;
  const bool gated = (EPI == EPI_SWIGLU);
  const bool concat = gated && p.layout == MOE_LAYOUT_CONCAT;
  // packed weight rows of this tile: two 64-row halves
  const int wrow0 = concat ? mt * 64 : mt * kTileM;
  const int wrow1 = concat ? p.I + mt * 64 : mt * kTileM + 64;
  const bool half1 = wrow1 < p.N;
  const int KB = p.K / kBK;
  constexpr int kpb = KPB;                // K blocks per pipeline stage
  constexpr uint32_t rb = 32u * KPB;      // packed bytes per weight row per stage
  const int NS = (KB + kpb - 1) / kpb;    // pipeline stages of the tile
  const uint32_t ncols = tmem_cols(p.tile_n);
  const uint32_t a_col = tmem_a_col(p.tile_n);

  if (warp == 1) {
    tmem_alloc(smem_u32(const_cast<int *>(misc)), ncols);
    tmem_relinquish();
  }
  if (warp >= 2) {
    const int i0 = tid - 64;
    if (FMT == MOE_FMT_NVFP4) lut[i0] = e4m3_times_2p118_x2((uint32_t)i0);
    if (FMT == MOE_FMT_MXFP4) lut[i0] = e8m0_times_2p126_x2((uint32_t)i0);
    for (int i = i0; i < p.tile_n; i += kDqThreads) {
      int sid = p.num_rows;
      if (i < nrows) sid = p.sorted_ids[row0 + i];
      ids_s[i] = sid;
      float w = 0.f;
      if (EPI == EPI_WEIGHTED && p.mul && sid < p.num_rows) w = p.topk_w[sid];
      tw_s[i] = w;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = static_cast<uint32_t>(misc[0]);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // (the whole warp runs the loop so its control flow stays uniform; lane 0
    // issues the copies)
    const bool leader = lane == 0;
    const uint8_t *sc_g = static_cast<const uint8_t *>(p.scales);
    const size_t scb = (size_t)p.sc_row_bytes, zb = (size_t)p.z_row_bytes;
    const uint32_t rows0 = 64, rows1 = half1 ? 64 : 0;
    if (leader) {
      prefetch_tmap(&p.tm_w);
      prefetch_tmap(&p.tm_x);
      uint32_t tx = (rows0 + rows1) * (uint32_t)(scb + (FMT == MOE_FMT_INT4 ? zb : 0));
      mbar_arrive_expect_tx(sc_bar, tx);
      const uint32_t sc_s = smem_u32(base + L.sc), z_s = smem_u32(base + L.z);
      bulk_load(sc_s, sc_g + ((size_t)e * p.N + wrow0) * scb, rows0 * scb, sc_bar);
      if (rows1) bulk_load(sc_s + 64 * scb, sc_g + ((size_t)e * p.N + wrow1) * scb, rows1 * scb, sc_bar);
      if (FMT == MOE_FMT_INT4) {
        bulk_load(z_s, p.zeros + ((size_t)e * p.N + wrow0) * zb, rows0 * zb, sc_bar);
        if (rows1) bulk_load(z_s + 64 * zb, p.zeros + ((size_t)e * p.N + wrow1) * zb, rows1 * zb, sc_bar);
      }
    }
    const uint32_t w_s = smem_u32(base + L.w), x_s = smem_u32(base + L.x);
    const uint32_t xstage = (uint32_t)kpb * p.tile_n * 128;
    Ring r;
    int issued = 0;
    for (int st = 0; st < NS; ++st) {
      bool ok = st < p.stages || mbar_wait(empty_bar(r.slot), r.phase ^ 1);
      ok = __all_sync(0xffffffffu, ok && !misc[5]);
      if (!ok) {
        if (leader) {
          raise_status(p.status, MOE_ERR_TIMEOUT);
          misc[5] = 1;
        }
        break;
      }
      if (leader) {
        const int kb0 = st * kpb;
        const int nkb = min(kpb, KB - kb0);  // K blocks in this stage
        const uint32_t fb = full_bar(r.slot);
        mbar_arrive_expect_tx(fb, (rows0 + rows1) * rb + (uint32_t)(nkb * n16 * 128));
        const uint32_t ws = w_s + r.slot * (kTileM * rb);
        tma_load_3d(ws, &p.tm_w, fb, st * (int)rb, wrow0, e);
        if (rows1) tma_load_3d(ws + 64 * rb, &p.tm_w, fb, st * (int)rb, wrow1, e);
        const uint32_t xs0 = x_s + r.slot * xstage;
        for (int j = 0; j < nkb; ++j) {
          const uint32_t xs = xs0 + j * (p.tile_n * 128);
          for (int i = 0; i < n16; i += 16) tma_load_2d(xs + i * 128, &p.tm_x, fb, (kb0 + j) * kBK, row0 + i);
        }
      }
      issued = st + 1;
      r.advance(p.stages);
    }
    if (misc[5] && leader) {
      // wind down: let the copies already issued land before the CTA exits
      // (slots before r.slot were filled in the current lap, the rest in the
      // previous one if there was one)
      for (int q = 0; q < p.stages; ++q) {
        if (q < r.slot) (void)mbar_wait(full_bar(q), r.phase);
        else if (q < issued) (void)mbar_wait(full_bar(q), r.phase ^ 1);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // (whole warp in the loop, lane 0 issues the tcgen05 instructions)
    const bool leader = lane == 0;
    const uint32_t idesc = idesc_bf16(kTileM, n16);
    const uint32_t x_s = smem_u32(base + L.x);
    Ring rs, ra;
    for (int st = 0; st < NS; ++st) {
      const int kb0 = st * kpb;
      const int nkb = min(kpb, KB - kb0);
      bool ok = mbar_wait(full_bar(rs.slot), rs.phase) && mbar_wait(dq_bar(ra.slot), ra.phase);
      ok = __all_sync(0xffffffffu, ok && !misc[5]);
      if (!ok) {
        if (leader) {
          raise_status(p.status, MOE_ERR_TIMEOUT);
          misc[5] = 1;
        }
        break;
      }
      tc_fence_after();
      if (leader) {
        const uint32_t aa = tmem + a_col + (32u * kpb) * ra.slot;
        const uint32_t xb = x_s + rs.slot * kpb * (p.tile_n * 128);
#pragma unroll
        for (int j = 0; j < kpb; ++j) {
          if (j < nkb) {
            const uint64_t bd = smem_desc_sw128(xb + j * (p.tile_n * 128));
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk)
              umma_bf16_ts(tmem, aa + 32u * j + 8u * kk, bd + 2u * kk, idesc, (kb0 + j + kk) != 0);
          }
        }
        umma_commit(afree_bar(ra.slot));
        umma_commit(empty_bar(rs.slot));
      }
      __syncwarp();
      ra.advance(NA);
      rs.advance(p.stages);
    }
    if (leader) umma_commit(acc_bar);  // also covers a partial pipeline on abort
    __syncwarp();
  } else if (warp >= 2) {
    // ------------------------------------------------------ dequant + epilogue
    const int q4 = warp & 3;             // TMEM lane quarter of this warp
    const int hk = (warp >= 6) ? 1 : 0;  // which 32-wide half of each K block
    const int r = q4 * 32 + lane;        // weight row in the tile == TMEM lane
    // packed / scale row in shared memory for this operand row
    const int pr = concat ? ((r & 1) ? 64 + (r >> 1) : (r >> 1)) : r;
    const bool row_ok = pr < 64 || half1;
    const uint8_t *w_tile = base + L.w;
    const uint8_t *sc_row = base + L.sc + (size_t)pr * p.sc_row_bytes;
    const uint8_t *z_row = base + L.z + (size_t)pr * p.z_row_bytes;
    const uint32_t t_lane = tmem + ((uint32_t)(q4 * 32) << 16);
    // the packed tile arrives with the 32/64/128-byte swizzle matching its row
    // width: 16-byte chunk index ^= address bits [7, 7 + log2(kpb) + 1)
    const int sw = (int)(((uint32_t)pr * rb >> 7) & (uint32_t)(2 * kpb - 1));
    const uint8_t *w_row = w_tile + pr * rb;
    // Dequantise K block kb (held in stage slot `slot` at position j) of this
    // thread's row half into 16 bf16x2 words.
    auto dequant = [&](int kb, int slot, int j, uint32_t (&out)[16]) {
      const int chunk = 2 * j + hk;
      if (row_ok) {
        const uint4 c = *reinterpret_cast<const uint4 *>(w_row + slot * (kTileM * rb) + ((chunk ^ sw) << 4));
        const uint32_t xw[4] = {c.x, c.y, c.z, c.w};
        if (FMT == MOE_FMT_NVFP4) {
          const uint32_t sb = *reinterpret_cast<const uint16_t *>(sc_row + kb * 4 + hk * 2);
#pragma unroll
          for (int g = 0; g < 2; ++g) {
            const uint32_t s2 = lut[(sb >> (8 * g)) & 0xFFu];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              uint32_t o4[4];
              e2m1x8_raw(xw[2 * g + h], o4);
#pragma unroll
              for (int q = 0; q < 4; ++q) out[(2 * g + h) * 4 + q] = bmul2(o4[q], s2);
            }
          }
        } else if (FMT == MOE_FMT_MXFP4) {
          const uint32_t e8 = sc_row[kb * 2 + hk];
          if (e8 > 128u && e8 != 255u) raise_status(p.status, MOE_ERR_SCALE_RANGE);
          const uint32_t s2 = lut[e8];
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            uint32_t o4[4];
            e2m1x8_raw(xw[h], o4);
#pragma unroll
            for (int q = 0; q < 4; ++q) out[h * 4 + q] = bmul2(o4[q], s2);
          }
        } else {  // INT4, one group of 64 per K block
          const float sf = __half2float(*reinterpret_cast<const __half *>(sc_row + kb * 2));
          const uint32_t zz = (z_row[kb >> 1] >> ((kb & 1) * 4)) & 0xFu;
          const float cz = -(float)zz * sf;  // exact
#pragma unroll
          for (int w8 = 0; w8 < 4; ++w8) {
            const uint32_t x = xw[w8];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const float q0 = __uint_as_float(0x4B000000u | ((x >> (8 * q)) & 0xFu)) - 8388608.f;
              const float q1 = __uint_as_float(0x4B000000u | ((x >> (8 * q + 4)) & 0xFu)) - 8388608.f;
              const __nv_bfloat162 v = __floats2bfloat162_rn(fmaf(q0, sf, cz), fmaf(q1, sf, cz));
              out[w8 * 4 + q] = *reinterpret_cast<const uint32_t *>(&v);
            }
          }
        }
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) out[i] = 0u;
      }
    };
    bool ok = mbar_wait(sc_bar, 0);
    if (!ok) {
      raise_status(p.status, MOE_ERR_TIMEOUT);
      misc[5] = 1;
    }
    ok = __all_sync(0xffffffffu, ok);
    Ring cs, ca;  // stage slot / lap, operand buffer / lap
    const uint32_t t_a = t_lane + a_col + 16u * hk;
    for (int st = 0; st < NS && ok; ++st) {
      const int kb0 = st * kpb;
      const int nkb = min(kpb, KB - kb0);
      ok = mbar_wait(full_bar(cs.slot), cs.phase);
      if (ok && st >= NA) ok = mbar_wait(afree_bar(ca.slot), ca.phase ^ 1);
      ok = __all_sync(0xffffffffu, ok && !misc[5]);
      if (!ok) {
        raise_status(p.status, MOE_ERR_TIMEOUT);
        misc[5] = 1;
        break;
      }
      tc_fence_after();
#pragma unroll
      for (int j = 0; j < kpb; ++j) {
        if (j < nkb) {
          uint32_t v[16];
          dequant(kb0 + j, cs.slot, j, v);
          tmem_st16(t_a + (32u * kpb) * ca.slot + 32u * j, v);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(dq_bar(ca.slot));
      ca.advance(NA);
      cs.advance(p.stages);
    }
    // ---------------------------------------------------------------- epilogue
    const bool acc_ok = mbar_wait(acc_bar, 0);
    if (!acc_ok) raise_status(p.status, MOE_ERR_TIMEOUT);
    __syncwarp();
    tc_fence_after();
    // warp-uniform decision: tcgen05.ld is a warp-collective instruction
    if (__all_sync(0xffffffffu, acc_ok && !misc[5])) {
      // weight row / output column of this lane
      int n_w;  // row of W (for bias)
      int col;  // output column
      bool col_ok;
      if (gated) {
        col = mt * 64 + (r >> 1);
        n_w = concat ? ((r & 1) ? p.I + col : col) : mt * kTileM + r;
        col_ok = col < p.I;
      } else {
        n_w = mt * kTileM + r;
        col = n_w;
        col_ok = n_w < p.N;
      }
      float gmul = 1.f;
      if (FMT == MOE_FMT_NVFP4) gmul = p.gscale[e] * 256.f;  // undo the 2^-8 operand fold
      float bias = 0.f;
      if (p.bias && col_ok) bias = bf16_bits_to_float(p.bias[(size_t)e * p.N + n_w]);
      for (int c0 = 16 * hk; c0 < n16; c0 += 32) {
        uint32_t v[16];
        tmem_ld16(t_lane + c0, v);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int tok = c0 + j;
          const bool store = tok < nrows && ids_s[tok] < p.num_rows && col_ok;
          float h = __fadd_rn(__fmul_rn(__uint_as_float(v[j]), gmul), bias);
          uint16_t *orow = p.out + (size_t)(row0 + tok) * p.ldo;
          if (EPI == EPI_SWIGLU) {
            const float other = __shfl_xor_sync(0xffffffffu, h, 1);
            if (!(r & 1) && store) {
              const float g = fminf(h, p.limit);
              const float u = fminf(fmaxf(other, -p.limit), p.limit);
              const float sg = 1.0f / (1.0f + expf(-p.alpha * g));
              orow[col] = float_to_bf16_bits((u + 1.0f) * g * sg);
            }
          } else if (EPI == EPI_RELU2) {
            if (store) {
              const float rr = fmaxf(h, 0.f);
              orow[col] = float_to_bf16_bits(rr * rr);
            }
          } else {
            if (store) {
              if (p.mul) h = __fmul_rn(h, tw_s[tok]);
              orow[col] = float_to_bf16_bits(h);
            }
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, ncols);
  }
}

// --------------------------------------------------------------------- host
namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

template <int FMT, int EPI, int KPB>
moe_status_t launch_t(const GemmArgs &a, dim3 grid, uint32_t smem, cudaStream_t st) {
  auto kern = grouped_gemm_kernel<FMT, EPI, KPB>;
  static uint32_t configured = 0;  // per instantiation; grows monotonically
  if (smem > configured) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return MOE_ERR_CUDA;
    configured = smem;
  }
  kern<<<grid, kThreads, smem, st>>>(a);
  return cudaPeekAtLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace

// Two K blocks (64 contiguous bytes per weight row) per stage for token tiles
// up to 128 rows; one for wider tiles, whose activation rows already make each
// stage large.
int choose_kpb(int tile_n) { return tile_n <= 128 ? 2 : 1; }

int choose_tile_n(int num_rows, int E) {
  const int active = num_rows < E ? (num_rows > 0 ? num_rows : 1) : E;
  const int avg = (num_rows + active - 1) / active;
  int n = ((2 * avg + 15) / 16) * 16;
  if (n < 32) n = 32;
  if (n > 256) n = 256;
  return n;
}

moe_status_t launch_grouped_gemm(int epi, const moe_qweight_t &w, const uint16_t *x, int P_max,
                                 const int32_t *sorted_ids, const int32_t *expert_offsets, int num_rows,
                                 const float *topk_w, int mul, int layout, moe_act_t act, uint16_t *out,
                                 int ldo, unsigned int *status, cudaStream_t stream, int *launches) {
  if (P_max <= 0 || num_rows <= 0) return MOE_OK;
  auto enc = encode_fn();
  if (!enc) return MOE_ERR_CUDA;
  GemmArgs a;
  memset(&a, 0, sizeof(a));
  const int E = w.E, N = w.N, K = w.K;
  // K blocks per pipeline stage: longer contiguous runs per weight row make the
  // DRAM reads efficient (32 bytes per row per request streams poorly)
  a.tile_n = choose_tile_n(num_rows, E);
  const int kpb = choose_kpb(a.tile_n);
  // packed weights: [E][N][K/2] bytes, box (32 * kpb) B x 64 rows x 1 expert
  {
    cuuint64_t dims[3] = {(cuuint64_t)(K / 2), (cuuint64_t)N, (cuuint64_t)E};
    cuuint64_t strides[2] = {(cuuint64_t)(K / 2), (cuuint64_t)N * (K / 2)};
    cuuint32_t box[3] = {(cuuint32_t)(32 * kpb), 64, 1};
    cuuint32_t es[3] = {1, 1, 1};
    const CUtensorMapSwizzle swz = kpb == 1 ? CU_TENSOR_MAP_SWIZZLE_32B
                                   : kpb == 2 ? CU_TENSOR_MAP_SWIZZLE_64B
                                              : CU_TENSOR_MAP_SWIZZLE_128B;
    if (enc(&a.tm_w, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t *>(w.q), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return MOE_ERR_CUDA;
  }
  a.kpb = kpb;
  // activations: [P_max][K] bf16, box 64 x 16 rows, 128-byte swizzle
  {
    cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)P_max};
    cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    cuuint32_t box[2] = {64, 16};
    cuuint32_t es[2] = {1, 1};
    if (enc(&a.tm_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(x), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return MOE_ERR_CUDA;
  }
  a.scales = w.scales;
  a.zeros = w.zeros;
  a.gscale = w.gscale;
  a.bias = w.bias;
  a.expert_offsets = expert_offsets;
  a.sorted_ids = sorted_ids;
  a.topk_w = topk_w;
  a.out = out;
  a.status = status;
  a.E = E;
  a.N = N;
  a.K = K;
  a.P_max = P_max;
  a.num_rows = num_rows;
  a.ldo = ldo;
  a.layout = layout;
  a.I = (epi == 0) ? N / 2 : N;
  a.mul = mul;
  a.alpha = act.alpha;
  a.limit = act.limit;
  a.tile_n = choose_tile_n(num_rows, E);
  a.sc_row_bytes = (w.fmt == MOE_FMT_NVFP4) ? K / 16 : (w.fmt == MOE_FMT_MXFP4 ? K / 32 : (K / 64) * 2);
  a.z_row_bytes = (w.fmt == MOE_FMT_INT4) ? (K / 64 + 1) / 2 : 0;
  // stages: as many as fit; two CTAs per SM when TMEM allows it (256 columns)
  const bool two_per_sm = tmem_cols(a.tile_n) <= 256;
  const uint32_t budget = two_per_sm ? 110 * 1024 : 225 * 1024;
  int stages = kMaxStagesL;
  while (stages > 2 && smem_layout(a.tile_n, stages, kpb, a.sc_row_bytes, a.z_row_bytes).total > budget)
    --stages;
  a.stages = stages;
  uint32_t smem = smem_layout(a.tile_n, stages, kpb, a.sc_row_bytes, a.z_row_bytes).total;
  // never more CTAs per SM than TMEM holds (2 x 256 or 1 x 512 columns)
  const uint32_t min_smem = two_per_sm ? 80 * 1024 : 120 * 1024;
  if (smem < min_smem) smem = min_smem;
  if (smem > 227 * 1024) return MOE_ERR_UNSUPPORTED;
  const int m_tiles = (epi == 0) ? (N / 2 + 63) / 64 : (N + kTileM - 1) / kTileM;
  const int active = num_rows < E ? num_rows : E;
  const int max_tiles = P_max / a.tile_n + active + 1;
  dim3 grid(m_tiles, max_tiles);
  if (launches) ++*launches;
  const int f = w.fmt;
#define MOE4_DISPATCH_K(F, K)                                                  \
  if (f == F && kpb == K) {                                                    \
    if (epi == 0) return launch_t<F, EPI_SWIGLU, K>(a, grid, smem, stream);    \
    if (epi == 1) return launch_t<F, EPI_RELU2, K>(a, grid, smem, stream);     \
    return launch_t<F, EPI_WEIGHTED, K>(a, grid, smem, stream);                \
  }
#define MOE4_DISPATCH(F) MOE4_DISPATCH_K(F, 1) MOE4_DISPATCH_K(F, 2)
  MOE4_DISPATCH(MOE_FMT_NVFP4)
  MOE4_DISPATCH(MOE_FMT_MXFP4)
  MOE4_DISPATCH(MOE_FMT_INT4)
#undef MOE4_DISPATCH
#undef MOE4_DISPATCH_K
  return MOE_ERR_UNSUPPORTED;
}

}  // namespace moe4
