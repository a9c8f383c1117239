// Grouped GEMMs of the MoE layer with 4-bit block-scaled weights (steps a3, a4).
//
// A work tile is (weight tile of 128 rows of one expert, token tile of up to
// tile_n routed rows of that expert):
//   D[128 weight rows][n tokens] = W'[rows][K] . X[tokens][K]^T   (fp32, TMEM)
// with the weights as the MMA's M side ("swap-AB"), so a handful of routed
// tokens per expert (decode) still fills the 128-row MMA. The dequantised bf16
// weights never touch shared memory: the dequant warps write them straight
// into tensor memory (tcgen05.st) and the MMA reads its A operand from there,
// while the token rows (B operand) arrive by TMA into shared memory.
//
// The kernel is persistent, one CTA per SM (it takes all 512 TMEM columns):
// each CTA walks the tiles blockIdx.x, blockIdx.x + gridDim.x, ... and every
// role derives the tile coordinates by itself from expert_offsets, so roles
// synchronise on data only. Warp roles (864 threads for wide token tiles,
// 736 for the narrow tiles of decode):
//   warp 0        TMA producer: per tile the block scales (bulk copy, two
//                 buffers), then per stage the packed 4-bit weight rows into
//                 the weight ring; it runs ahead into the next tile
//   warp 26 / 22  TMA producer of the token rows, in a ring of its own. A
//                 weight slot is released as soon as the dequantisation warps
//                 have read it, not when the MMAs that read the token rows
//                 complete, so the weights run further ahead
//   warp 1        TMEM allocation; one lane issues tcgen05.mma (kind::f16, A
//                 from TMEM, B from shared memory) into one of two TMEM
//                 accumulators
//   warps 2..17   dequantise, in two groups of 8 that take alternate stages:
//                 warp w owns TMEM lanes 32*(w%4).. (one weight row per lane)
//                 and half of its group's stage K range
//   warps 18..25  epilogue of the previous tile's accumulator while the next
//   (18..21)      tile is being computed (two warps per TMEM lane quarter, one
//                 per half of the token columns; one per quarter for decode)
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
//  * GPTQ INT4: bf16_rne((q - z) * s), the exact product rounded once, built
//    from bf16-pair FMAs (the fp16 scale split into two bf16 parts).
#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>

#include "common.cuh"
#include "dequant.cuh"
#include "kernels.h"

namespace moe4 {

namespace {

constexpr int kFirstDqWarp = 2, kDqWarps = 16;
constexpr int kFirstEpiWarp = kFirstDqWarp + kDqWarps;
constexpr int kDqThreads = kDqWarps * 32;
constexpr int kDqGroupThreads = kDqThreads / 2;  // one of the two dequant groups
// Epilogue warps: 8 (two per TMEM lane quarter, one per half of the token
// columns) for the wide token tiles of prefill (KPB = 2), 4 for the narrow
// tiles of decode (KPB = 4), whose 16-32 token columns one warp per quarter
// drains in time; the smaller CTA also leaves the decode kernel more
// registers per thread (c1 GEMM1 88 -> 82 us in one comparison run). The
// token-row producer follows the epilogue warps.
__host__ __device__ constexpr int epi_warps(int kpb) { return kpb == 4 ? 4 : 8; }
__host__ __device__ constexpr int x_warp(int kpb) { return kFirstEpiWarp + epi_warps(kpb); }
__host__ __device__ constexpr int cta_threads(int kpb) { return (x_warp(kpb) + 1) * 32; }
constexpr int kTileM = 128;       // weight rows per tile (TMEM lanes)
constexpr int kBK = 64;           // K per MMA block (128 bytes of bf16)
constexpr int kTmemCols = 512;    // the whole tensor memory of the SM
constexpr int kMaxNA = 8;         // at most this many operand buffers
constexpr int kMaxStagesL = 12;
constexpr int kMaxE = 256;

// named barriers (id 0 is __syncthreads): the dequant and epilogue groups
constexpr int kBarDq0 = 1, kBarEpi = 2, kBarDq1 = 3;

enum { EPI_SWIGLU = 0, EPI_RELU2 = 1, EPI_WEIGHTED = 2 };

struct Smem {
  uint32_t x, w, sc, z, lut, offs, tfirst, ids, tw, ex, bar, misc, total;
};

__host__ __device__ inline uint32_t align_up(uint32_t v, uint32_t a) { return (v + a - 1) / a * a; }

// Shared-memory carve-up; identical on host (sizing) and device (addresses).
__host__ __device__ inline Smem smem_layout(int tile_n, int stages, int kpb, int sc_row_bytes,
                                            int z_row_bytes, int xstages) {
  Smem s;
  uint32_t o = 0;
  s.x = o;    o += xstages * kpb * tile_n * 128;
  o = align_up(o, 1024);
  s.w = o;    o += stages * kTileM * 32 * kpb;
  s.sc = o;   o += 2 * align_up(kTileM * sc_row_bytes, 128);
  s.z = o;    o += 2 * align_up(kTileM * z_row_bytes, 128);
  s.lut = o;  o += 256 * 4;
  s.offs = o; o += (kMaxE + 1) * 4;
  s.tfirst = o; o += (kMaxE + 1) * 4;
  o = align_up(o, 16);
  s.ids = o;  o += 2 * tile_n * 4;  // one buffer per TMEM accumulator
  s.tw = o;   o += 2 * tile_n * 4;
  s.ex = o;   o += 2 * tile_n * 4;
  o = align_up(o, 8);
  s.bar = o;  o += (4 * kMaxStagesL + 2 * kMaxNA + 8) * 8;
  s.misc = o; o += 64;
  s.total = o + 1024;  // slack for aligning the dynamic base to 1024
  return s;
}

// TMEM columns: nacc accumulators of tile_n columns (rounded to 32), then as
// many stage-sized operand buffers as the rest of the 512 columns hold.
__host__ __device__ inline uint32_t tmem_acc_stride(int tile_n) { return align_up(tile_n, 32); }

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

struct TokenTile {
  int e, row0, nrows;
};

// Token tiles: each expert's slot segment is split into tiles of at most
// tile_n rows; tfirst[e] is the number of the expert's first token tile
// (tfirst[E] = the count), built once per CTA by one warp.
__device__ __forceinline__ void build_tile_table(const int *offs, int E, int tile_n, int *tfirst, int lane) {
  int cum = 0;
  for (int e0 = 0; e0 < E; e0 += 32) {
    const int e = e0 + lane;
    const int seg = e < E ? offs[e + 1] - offs[e] : 0;
    const int nt = (seg + tile_n - 1) / tile_n;
    int incl = nt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (e < E) tfirst[e] = cum + incl - nt;
    cum += __shfl_sync(0xffffffffu, incl, 31);
  }
  if (lane == 0) tfirst[E] = cum;
}

// Token tile number tt (tt < tfirst[E], non-decreasing from call to call) ->
// expert and slot range; e carries the expert of the previous call.
__device__ __forceinline__ TokenTile next_token_tile(const int *offs, const int *tfirst, int tile_n, int tt,
                                                      int &e) {
  while (tfirst[e + 1] <= tt) ++e;
  TokenTile r;
  r.e = e;
  r.row0 = offs[e] + (tt - tfirst[e]) * tile_n;
  r.nrows = min(tile_n, offs[e + 1] - r.row0);
  return r;
}

}  // namespace

template <int FMT, int EPI, int KPB, bool F16>
__global__ void __launch_bounds__(cta_threads(KPB), 1) grouped_gemm_kernel(const __grid_constant__ GemmArgs p) {
  constexpr int kEpiWarps = epi_warps(KPB), kEpiThreads = kEpiWarps * 32;
  constexpr int kXWarp = x_warp(KPB), kThreads = cta_threads(KPB);
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte aligned start (pointer arithmetic on the shared array keeps the
  // compiler's knowledge that all these addresses are shared memory)
  uint8_t *base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  // weights and token rows in separate rings (kXWarp loads the token rows;
  // a weight slot is freed once it has been dequantised)
  const int NX = p.xstages;
  // INT4 (the costliest expansion): each stage is expanded and handed to the
  // MMA warp in two halves of its K blocks, so the MMAs of the first half run
  // while the second half is expanded (c2 GEMM1 498 -> 467 us). The FP4
  // expansions are fast enough that the extra TMEM-store wait costs more.
  constexpr bool HALVES = FMT == MOE_FMT_INT4;
  constexpr int NH = HALVES ? 2 : 1;
  const Smem L = smem_layout(p.tile_n, p.stages, KPB, p.sc_row_bytes, p.z_row_bytes, NX);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int NA = p.na;                     // operand buffers in TMEM
  constexpr int kpb = KPB;                 // K blocks per pipeline stage
  constexpr uint32_t rb = 32u * KPB;       // packed bytes per weight row per stage
  const uint32_t bar0 = smem_u32(base + L.bar);
  // full_bar / wempty_bar: weight ring slot loaded / read by its dequant group
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  // done_bar(slot): the MMAs of the stage in that token-row ring slot have
  // completed, so both the slot and the stage's TMEM operand buffer are free
  auto done_bar = [&](int s) { return bar0 + 8u * (kMaxStagesL + s); };
  constexpr int kB2 = 2 * kMaxStagesL, kB3 = kB2 + 2 * kMaxNA;
  // dq_bar(slot, h): the stage in operand buffer slot is expanded (h = 0), or,
  // for INT4, half h of its K blocks is
  auto dq_bar = [&](int s, int h) { return bar0 + 8u * (kB2 + 2 * s + h); };
  auto scfull_bar = [&](int s) { return bar0 + 8u * (kB3 + s); };
  auto scempty_bar = [&](int s) { return bar0 + 8u * (kB3 + 2 + s); };
  auto accfull_bar = [&](int s) { return bar0 + 8u * (kB3 + 4 + s); };
  auto accempty_bar = [&](int s) { return bar0 + 8u * (kB3 + 6 + s); };
  constexpr int kB4 = kB3 + 8;
  auto xfull_bar = [&](int s) { return bar0 + 8u * (kB4 + s); };
  auto wempty_bar = [&](int s) { return bar0 + 8u * (kB4 + kMaxStagesL + s); };
  volatile int *misc = reinterpret_cast<volatile int *>(base + L.misc);  // [0] tmem, [1] abort
  int *offs_s = reinterpret_cast<int *>(base + L.offs);
  int *tfirst_s = reinterpret_cast<int *>(base + L.tfirst);
  int *ids_s = reinterpret_cast<int *>(base + L.ids);
  float *tw_s = reinterpret_cast<float *>(base + L.tw);
  uint32_t *lut = reinterpret_cast<uint32_t *>(base + L.lut);
  const uint32_t sc_buf = align_up(kTileM * p.sc_row_bytes, 128);
  const uint32_t z_buf = align_up(kTileM * p.z_row_bytes, 128);

  // ------------------------------------------------------------------ setup
  if (tid < 256) {
    if (FMT == MOE_FMT_NVFP4) lut[tid] = F16 ? e4m3_f16x2((uint32_t)tid) : e4m3_times_2p118_x2((uint32_t)tid);
    if (FMT == MOE_FMT_MXFP4) lut[tid] = F16 ? e8m0_f16x2((uint32_t)tid) : e8m0_times_2p126_x2((uint32_t)tid);
  }
  if (tid == 32) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(wempty_bar(s), kDqGroupThreads / 32);
    }
    for (int s = 0; s < NX; ++s) {
      mbar_init(xfull_bar(s), 1);
      mbar_init(done_bar(s), 1);
    }
    for (int s = 0; s < NA; ++s) {
      mbar_init(dq_bar(s, 0), kDqGroupThreads);
      mbar_init(dq_bar(s, 1), kDqGroupThreads);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(scfull_bar(s), 1);
      mbar_init(scempty_bar(s), kDqThreads);
      mbar_init(accfull_bar(s), 1);
      mbar_init(accempty_bar(s), kEpiThreads);
    }
    misc[1] = 0;
    fence_mbar_init();
  }
  const int nacc = p.nacc;
  const uint32_t acc_stride = tmem_acc_stride(p.tile_n);
  const uint32_t a_col = nacc * acc_stride;
  const uint32_t ncols = kTmemCols;
  if (warp == 1) {
    tmem_alloc(smem_u32(const_cast<int *>(misc)), ncols);
    tmem_relinquish();
  }
  // Everything above overlaps the previous kernel on the stream. The token
  // rows (x_perm, or GEMM1's output) and the per-row exponents come from that
  // kernel: the token-row warp and the epilogue wait for it (pdl_wait) before
  // they read them. expert_offsets comes from the alignment, which completed
  // before the previous kernel (the gather, or GEMM1) passed its own wait and
  // let this grid launch, so it is read here already; the weight producer and
  // the dequantisation warps start streaming and expanding this grid's first
  // weight tiles while the previous kernel drains.
  pdl_trigger();
  for (int i = tid; i <= p.E; i += kThreads) {
    const int v = p.expert_offsets[i];
    const bool good = v >= 0 && v <= p.P_max;
    offs_s[i] = good ? v : 0;
    if (!good) raise_status(p.status, MOE_ERR_BAD_INDEX);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) build_tile_table(offs_s, p.E, p.tile_n, tfirst_s, lane);
  __syncthreads();
  const uint32_t tmem = static_cast<uint32_t>(misc[0]);

  const int KB = p.K / kBK;
  const int NS = (KB + kpb - 1) / kpb;  // pipeline stages per tile
  const bool gated = (EPI == EPI_SWIGLU);
  const bool concat = gated && p.layout == MOE_LAYOUT_CONCAT;
  const int m_tiles = p.m_tiles;
  // every role computes the same tile count and tile coordinates
  const int total = m_tiles * tfirst_s[p.E];
  auto tile_rows = [&](int mt, int &wrow0, int &wrow1) {
    wrow0 = concat ? mt * 64 : mt * kTileM;
    wrow1 = concat ? p.I + mt * 64 : mt * kTileM + 64;
  };
  auto fail = [&](bool leader) {
    if (leader) {
      raise_status(p.status, MOE_ERR_TIMEOUT);
      misc[1] = 1;
    }
  };

  if (warp == 0) {
    // ============================================================ producer
    // (the whole warp runs the loop so its control flow stays uniform; lane 0
    // issues the copies)
    const bool leader = lane == 0;
    if (leader) prefetch_tmap(&p.tm_w);
    const uint8_t *sc_g = static_cast<const uint8_t *>(p.scales);
    const size_t scb = (size_t)p.sc_row_bytes, zb = (size_t)p.z_row_bytes;
    const uint32_t w_s = smem_u32(base + L.w);
    const uint32_t sc_s = smem_u32(base + L.sc), z_s = smem_u32(base + L.z);
    Ring rst, rsc;
    int ntiles = 0, te = 0;
    uint32_t issued_mask = 0, issued_par = 0;  // stage slots with copies in flight
    bool ok = true;
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x, ++ntiles) {
      const int mt = t % m_tiles;
      const TokenTile tt = next_token_tile(offs_s, tfirst_s, p.tile_n, t / m_tiles, te);
      int wrow0, wrow1;
      tile_rows(mt, wrow0, wrow1);
      const uint32_t rows1 = wrow1 < p.N ? 64 : 0;
      // block scales of this tile into scale buffer rsc.slot
      ok = ntiles < 2 || mbar_wait_relaxed(scempty_bar(rsc.slot), rsc.phase ^ 1);
      ok = __all_sync(0xffffffffu, ok && !misc[1]);
      if (!ok) {
        fail(leader);
        break;
      }
      if (leader) {
        const uint32_t tx = (64 + rows1) * (uint32_t)(scb + (FMT == MOE_FMT_INT4 ? zb : 0));
        const uint32_t sb = scfull_bar(rsc.slot);
        mbar_arrive_expect_tx(sb, tx);
        const uint32_t ss = sc_s + rsc.slot * sc_buf;
        bulk_load(ss, sc_g + ((size_t)tt.e * p.N + wrow0) * scb, 64 * scb, sb);
        if (rows1) bulk_load(ss + 64 * scb, sc_g + ((size_t)tt.e * p.N + wrow1) * scb, rows1 * scb, sb);
        if (FMT == MOE_FMT_INT4) {
          const uint32_t zs = z_s + rsc.slot * z_buf;
          bulk_load(zs, p.zeros + ((size_t)tt.e * p.N + wrow0) * zb, 64 * zb, sb);
          if (rows1) bulk_load(zs + 64 * zb, p.zeros + ((size_t)tt.e * p.N + wrow1) * zb, rows1 * zb, sb);
        }
      }
      rsc.advance(2);
      for (int st = 0; st < NS; ++st) {
        ok = !((issued_mask >> rst.slot) & 1u) || mbar_wait_relaxed(wempty_bar(rst.slot), rst.phase ^ 1);
        ok = __all_sync(0xffffffffu, ok && !misc[1]);
        if (!ok) {
          fail(leader);
          break;
        }
        if (leader) {
          const uint32_t fb = full_bar(rst.slot);
          mbar_arrive_expect_tx(fb, (64 + rows1) * rb);
          const uint32_t ws = w_s + rst.slot * (kTileM * rb);
          tma_load_3d(ws, &p.tm_w, fb, st * (int)rb, wrow0, tt.e);
          if (rows1) tma_load_3d(ws + 64 * rb, &p.tm_w, fb, st * (int)rb, wrow1, tt.e);
        }
        issued_mask |= 1u << rst.slot;
        issued_par = (issued_par & ~(1u << rst.slot)) | ((uint32_t)rst.phase << rst.slot);
        rst.advance(p.stages);
      }
    }
    if (!ok && leader) {
      // wind down: let the copies already issued land before the CTA exits
      for (int q = 0; q < p.stages; ++q)
        if ((issued_mask >> q) & 1u) (void)mbar_wait(full_bar(q), (issued_par >> q) & 1u);
    }
  } else if (warp == 1) {
    // ============================================================ MMA issuer
    const bool leader = lane == 0;
    const uint32_t x_s = smem_u32(base + L.x);
    Ring rs, ra, rc;
    int ntiles = 0, te = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x, ++ntiles) {
      const TokenTile tt = next_token_tile(offs_s, tfirst_s, p.tile_n, t / m_tiles, te);
      const int n16 = (tt.nrows + 15) & ~15;
      const uint32_t idesc = F16 ? idesc_f16(kTileM, n16) : idesc_bf16(kTileM, n16);
      const uint32_t acc = tmem + acc_stride * rc.slot;
      // the epilogue must have drained this accumulator
      ok = ntiles < nacc || mbar_wait(accempty_bar(rc.slot), rc.phase ^ 1);
      ok = __all_sync(0xffffffffu, ok && !misc[1]);
      if (!ok) {
        fail(leader);
        break;
      }
      for (int st = 0; st < NS; ++st) {
        const int kb0 = st * kpb;
        const int nkb = min(kpb, KB - kb0);
        // operands computed by the whole warp (warp-uniform values), issued by
        // one elected lane (INT4: each half of the K blocks once expanded)
        const uint32_t aa = tmem + a_col + (32u * kpb) * ra.slot;
        const uint32_t xb = x_s + rs.slot * kpb * (p.tile_n * 128);
        const uint32_t db = done_bar(rs.slot);
#pragma unroll
        for (int h = 0; h < NH; ++h) {
          ok = (h || mbar_wait(xfull_bar(rs.slot), rs.phase)) && mbar_wait(dq_bar(ra.slot, h), ra.phase);
          ok = __all_sync(0xffffffffu, ok && !misc[1]);
          if (!ok) break;
          tc_fence_after();
          if (elect_one()) {
#pragma unroll
            for (int jj = 0; jj < kpb / NH; ++jj) {
              const int j = h * (kpb / NH) + jj;
              if (j < nkb) {
                const uint64_t bd = smem_desc_sw128(xb + j * (p.tile_n * 128));
#pragma unroll
                for (int kk = 0; kk < kBK / 16; ++kk)
                  umma_bf16_ts(acc, aa + 32u * j + 8u * kk, bd + 2u * kk, idesc, (kb0 + j + kk) != 0);
              }
            }
            if (h == NH - 1) umma_commit(db);  // one commit frees the ring slot and the operand buffer
          }
          __syncwarp();
        }
        if (!ok) {
          fail(leader);
          break;
        }
        ra.advance(NA);
        rs.advance(NX);
      }
      if (!ok) break;
      const uint32_t ab = accfull_bar(rc.slot);
      if (elect_one()) umma_commit(ab);
      __syncwarp();
      rc.advance(nacc);
    }
  } else if (warp < kFirstEpiWarp) {
    // ============================================================ dequant
    // Two groups of 8 warps take alternate K stages, so one group's barrier
    // waits overlap the other group's arithmetic. In a group, warp w owns TMEM
    // lane quarter w % 4 and one half of the stage's K range.
    const int dw = warp - kFirstDqWarp;
    const int grp = dw >> 3;                      // 0: even stages, 1: odd stages
    const int q4 = warp & 3;                      // TMEM lane quarter of this warp
    const int kq = (dw >> 2) & 1;                 // which half of the stage's K
    const bool lead = (dw & 7) == 0;              // polls the barriers for its group
    const int gbar = grp ? kBarDq1 : kBarDq0;
    constexpr int nw = KPB;                       // 32-wide K chunks per warp per stage
    const int r = q4 * 32 + lane;        // weight row in the tile == TMEM lane
    // packed / scale row in shared memory for this operand row
    const int pr = concat ? ((r & 1) ? 64 + (r >> 1) : (r >> 1)) : r;
    const uint8_t *w_row = base + L.w + pr * rb;
    // the packed tile arrives with the 32/64-byte swizzle matching its row
    // width: 16-byte chunk index ^= address bits [7, 7 + log2(kpb) + 1)
    const int sw = (int)(((uint32_t)pr * rb >> 7) & (uint32_t)(2 * kpb - 1));
    const uint32_t t_a = tmem + ((uint32_t)(q4 * 32) << 16) + a_col;
    // cl: ring position of stage kdone - NA, the previous user of this stage's
    // operand buffer (its done barrier says the buffer is free; NA <= stages,
    // so that barrier cannot have moved on by a whole lap)
    Ring cs, ca, rsc, cl;
    int kdone = 0;  // K stages dequantised so far (all tiles)
    bool ok = true;
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
      const int mt = t % m_tiles;
      int wrow0, wrow1;
      tile_rows(mt, wrow0, wrow1);
      const bool row_ok = pr < 64 || wrow1 < p.N;
      const uint8_t *sc_row = base + L.sc + rsc.slot * sc_buf + (uint32_t)pr * p.sc_row_bytes;
      const uint8_t *z_row = base + L.z + rsc.slot * z_buf + (uint32_t)pr * p.z_row_bytes;
      // the lead warp polls for the whole group; the rest block in bar.red
      bool lok = true;
      if (lead) lok = mbar_wait(scfull_bar(rsc.slot), rsc.phase) && !misc[1];
      ok = bar_and(gbar, kDqGroupThreads, lok);
      if (!ok) {
        fail(lead && lane == 0);
        break;
      }
      for (int st = 0; st < NS; ++st, ++kdone) {
        if ((kdone & 1) != grp) {  // the other group's stage
          ca.advance(NA);
          cs.advance(p.stages);
          if (kdone >= NA) cl.advance(NX);
          continue;
        }
        const int kb0 = st * kpb;
        const int nkb = min(kpb, KB - kb0);
        lok = true;
        if (lead)
          lok = mbar_wait(full_bar(cs.slot), cs.phase) &&
                (kdone < NA || mbar_wait(done_bar(cl.slot), cl.phase)) && !misc[1];
        ok = bar_and(gbar, kDqGroupThreads, lok);
        if (!ok) {
          fail(lead && lane == 0);
          break;
        }
        tc_fence_after();
        if (F16) {
          // f16 operands (NVFP4, MXFP4): hardware E2M1 -> f16 pairs in natural
          // K order, times the block scale as f16 (NVFP4: the E4M3 value;
          // MXFP4: 2^(e8 - 115)). All of this warp's shared-memory loads for
          // the stage are issued first, then the arithmetic and TMEM stores.
          uint4 cw[nw];
          uint32_t sv[nw][2];
#pragma unroll
          for (int i = 0; i < nw; ++i) {
            const int ch = kq * nw + i;
            const int j = ch >> 1, hk = ch & 1;
            const int kb = min(kb0 + j, KB - 1);
            cw[i] = *reinterpret_cast<const uint4 *>(w_row + cs.slot * (kTileM * rb) + ((ch ^ sw) << 4));
            if (FMT == MOE_FMT_NVFP4) {
              const uint32_t sb = *reinterpret_cast<const uint16_t *>(sc_row + kb * 4 + hk * 2);
              sv[i][0] = lut[sb & 0xFFu];
              sv[i][1] = lut[(sb >> 8) & 0xFFu];
            } else {
              const uint32_t e8 = sc_row[kb * 2 + hk];
              if (row_ok && j < nkb && e8 > 128u && e8 != 255u) raise_status(p.status, MOE_ERR_SCALE_RANGE);
              sv[i][0] = sv[i][1] = lut[e8];
            }
          }
#pragma unroll
          for (int i = 0; i < nw; ++i) {
            const int ch = kq * nw + i;
            const int j = ch >> 1, hk = ch & 1;
            uint32_t out[16];
            const uint32_t xw[4] = {cw[i].x, cw[i].y, cw[i].z, cw[i].w};
#pragma unroll
            for (int h = 0; h < 4; ++h)
#pragma unroll
              for (int b = 0; b < 4; ++b) out[h * 4 + b] = hmul2(e2m1x2_f16x2(xw[h], b), sv[i][h >> 1]);
            if (!row_ok) {
#pragma unroll
              for (int q = 0; q < 16; ++q) out[q] = 0u;
            }
            if (j < nkb) tmem_st16(t_a + (32u * kpb) * ca.slot + 32u * j + 16u * hk, out);
          }
        } else
#pragma unroll
        for (int i = 0; i < nw; ++i) {
          // 16-byte chunk of the row: K block ch / 2, half ch % 2. INT4: the
          // first half of the stage's chunks first, split between the lane
          // quarter's two warps, then the second half
          const int ch = HALVES ? (i / (nw / 2)) * nw + kq * (nw / 2) + i % (nw / 2) : kq * nw + i;
          const int j = ch >> 1, hk = ch & 1;
          if (HALVES && i == nw / 2) {  // the first half is in TMEM: hand it to the MMA warp
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(dq_bar(ca.slot, 0));
          }
          if (j < nkb) {
            const int kb = kb0 + j;
            uint32_t out[16];
            if (row_ok) {
              const uint4 c = *reinterpret_cast<const uint4 *>(w_row + cs.slot * (kTileM * rb) +
                                                              ((ch ^ sw) << 4));
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
                // bf16_rne((q - z) * s) with a single rounding, on bf16 pairs:
                // s (fp16, 11 significant bits) = s_hi + s_lo, both exact in
                // bf16; (q - z) * s_lo is exact in bf16 (at most 7 bits), so
                // fma(q - z, s_hi, (q - z) * s_lo) rounds the exact product once
                const float sf = __half2float(*reinterpret_cast<const __half *>(sc_row + kb * 2));
                const uint32_t zz = (z_row[kb >> 1] >> ((kb & 1) * 4)) & 0xFu;
                const uint32_t hi = float_to_bf16_bits(sf);
                const uint32_t lo = float_to_bf16_bits(sf - bf16_bits_to_float((uint16_t)hi));
                const uint32_t nz = float_to_bf16_bits(-128.f - (float)zz);  // -(128 + z), exact
                const uint32_t shi2 = hi | (hi << 16), slo2 = lo | (lo << 16), nz2 = nz | (nz << 16);
#pragma unroll
                for (int w8 = 0; w8 < 4; ++w8) {
                  const uint32_t x = xw[w8];
#pragma unroll
                  for (int q = 0; q < 4; ++q) {  // codes q and q + 4 (interleaved order)
                    // bf16 pair (128 + code): the code sits in the low mantissa bits
                    const uint32_t c128 = ((x >> (4 * q)) & 0x000F000Fu) | 0x43004300u;
                    const uint32_t d = bfma2(c128, 0x3F803F80u, nz2);  // code - z, exact
                    out[w8 * 4 + q] = bfma2(d, shi2, bmul2(d, slo2));
                  }
                }
              }
            } else {
#pragma unroll
              for (int i = 0; i < 16; ++i) out[i] = 0u;
            }
            tmem_st16(t_a + (32u * kpb) * ca.slot + 32u * j + 16u * hk, out);
          }
        }
        __syncwarp();  // this warp has read its rows of the weight slot
        if (lane == 0) mbar_arrive(wempty_bar(cs.slot));
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(dq_bar(ca.slot, NH - 1));
        ca.advance(NA);
        cs.advance(p.stages);
        if (kdone >= NA) cl.advance(NX);
      }
      if (!ok) break;
      mbar_arrive(scempty_bar(rsc.slot));  // done with this tile's scales
      rsc.advance(2);
    }
  } else if (warp == kXWarp) {
    // ============================================================ token rows
    pdl_wait();
    const bool leader = lane == 0;
    if (leader) prefetch_tmap(&p.tm_x);
    const uint32_t x_s = smem_u32(base + L.x);
    const uint32_t xstage = (uint32_t)kpb * p.tile_n * 128;
    Ring rx;
    int te = 0;
    uint32_t issued_mask = 0, issued_par = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
      const TokenTile tt = next_token_tile(offs_s, tfirst_s, p.tile_n, t / m_tiles, te);
      for (int st = 0; st < NS; ++st) {
        ok = !((issued_mask >> rx.slot) & 1u) || mbar_wait(done_bar(rx.slot), rx.phase ^ 1);
        ok = __all_sync(0xffffffffu, ok && !misc[1]);
        if (!ok) {
          fail(leader);
          break;
        }
        if (leader) {
          const int kb0 = st * kpb;
          const int nkb = min(kpb, KB - kb0);
          const uint32_t fb = xfull_bar(rx.slot);
          mbar_arrive_expect_tx(fb, (uint32_t)(nkb * p.tile_n * 128));
          const uint32_t xs0 = x_s + rx.slot * xstage;
          for (int j = 0; j < nkb; ++j)
            tma_load_2d(xs0 + j * (p.tile_n * 128), &p.tm_x, fb, (kb0 + j) * kBK, tt.row0);
        }
        issued_mask |= 1u << rx.slot;
        issued_par = (issued_par & ~(1u << rx.slot)) | ((uint32_t)rx.phase << rx.slot);
        rx.advance(NX);
      }
    }
    if (!ok && leader)
      for (int q = 0; q < NX; ++q)
        if ((issued_mask >> q) & 1u) (void)mbar_wait(xfull_bar(q), (issued_par >> q) & 1u);
  } else {
    // ============================================================ epilogue
    pdl_wait();
    const int q4 = warp & 3;
    const int eh = (warp - kFirstEpiWarp) >> 2;  // which part of the token columns
    const bool lead = warp == kFirstEpiWarp;
    const int r = q4 * 32 + lane;  // weight row in the tile == TMEM lane
    const uint32_t t_lane = tmem + ((uint32_t)(q4 * 32) << 16);
    const int etid = tid - kFirstEpiWarp * 32;  // thread index within the epilogue warps
    Ring rc;
    int te = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
      const int mt = t % m_tiles;
      const TokenTile tt = next_token_tile(offs_s, tfirst_s, p.tile_n, t / m_tiles, te);
      const int e = tt.e, row0 = tt.row0, nrows = tt.nrows;
      const int n16 = (nrows + 15) & ~15;
      float gmul = 1.f;
      // undo the operands' power-of-two folds: bf16 NVFP4 weights carry 2^-8,
      // f16 MXFP4 weights 2^12, and a f16 GEMM2 reads a scaled by 2^9
      const float afold = (F16 && EPI == EPI_WEIGHTED) ? 0x1p-9f : 1.f;
      if (FMT == MOE_FMT_NVFP4) gmul = F16 ? p.gscale[e] * afold : p.gscale[e] * 256.f;
      if (FMT == MOE_FMT_MXFP4 && F16) gmul = 0x1p-12f * afold;
      // this tile's row ids, routing weights and per-token 2^e of the f16
      // activation rows, staged by all epilogue warps into the buffer of
      // this tile's accumulator; the barrier below publishes them, and the
      // buffer's previous tile was finished by every warp before the
      // barrier of the tile in between
      int *ids_w = ids_s + rc.slot * p.tile_n;
      float *tw_w = tw_s + rc.slot * p.tile_n;
      float *gm_w = reinterpret_cast<float *>(base + L.ex) + rc.slot * p.tile_n;
      for (int i = etid; i < n16; i += kEpiThreads) {
        int sid = p.num_rows;
        if (i < nrows) sid = p.sorted_ids[row0 + i];
        ids_w[i] = sid;
        float w = 0.f;
        if (EPI == EPI_WEIGHTED && p.mul && sid >= 0 && sid < p.num_rows) w = p.topk_w[sid];
        tw_w[i] = w;
        float gm = 1.f;  // undoes the activation row's 2^-e (exact)
        if (F16 && EPI != EPI_WEIGHTED && i < nrows) gm = __uint_as_float((uint32_t)(127 + p.xexp[row0 + i]) << 23);
        gm_w[i] = gm;
      }
      int n_w, col;
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
      // GEMM1 writes its output interleaved within groups of 8 columns (the
      // layout GEMM2 reads its activations in): column c sits at 2*(c%4)+c/4
      const int col_st = (col & ~7) | ((col & 3) << 1) | ((col >> 2) & 1);
      float bias = 0.f;
      if (p.bias && col_ok) bias = bf16_bits_to_float(p.bias[(size_t)e * p.N + n_w]);
      bool lok = true;
      if (lead) lok = mbar_wait_relaxed(accfull_bar(rc.slot), rc.phase) && !misc[1];
      ok = bar_and(kBarEpi, kEpiThreads, lok);
      if (!ok) {
        fail(lead && lane == 0);
        break;
      }
      tc_fence_after();
      const uint32_t ta = t_lane + acc_stride * rc.slot;
      for (int c0 = 16 * eh; c0 < n16; c0 += 16 * (kEpiWarps / 4)) {
        uint32_t v[16];
        tmem_ld16(ta + c0, v);
        // which of these 16 tokens are stored (one shared-memory read per lane)
        const int ltok = c0 + (lane & 15);
        const int lsid = ids_w[ltok];
        const uint32_t smask =
            col_ok ? (__ballot_sync(0xffffffffu, ltok < nrows && lsid >= 0 && lsid < p.num_rows) & 0xFFFFu) : 0u;
        float gm[16];
        if (F16 && EPI != EPI_WEIGHTED) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float4 g4 = *reinterpret_cast<const float4 *>(gm_w + c0 + 4 * q);
            gm[4 * q] = g4.x;
            gm[4 * q + 1] = g4.y;
            gm[4 * q + 2] = g4.z;
            gm[4 * q + 3] = g4.w;
          }
        }
        tmem_ld_wait();
        float h[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          float acc = __uint_as_float(v[j]);
          if (F16 && EPI != EPI_WEIGHTED) acc = __fmul_rn(acc, gm[j]);
          h[j] = __fadd_rn(__fmul_rn(acc, gmul), bias);
        }
        if (EPI == EPI_SWIGLU) {
          // gate and up rows are adjacent lanes: the even lane finishes tokens
          // 0..7 of the chunk and the odd lane tokens 8..15, each after one
          // exchange per token pair, so no lane idles
          const bool odd = r & 1;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float recv = __shfl_xor_sync(0xffffffffu, odd ? h[j] : h[8 + j], 1);
            const int jt = odd ? 8 + j : j;
            if ((smask >> jt) & 1u) {
              const float g = fminf(odd ? recv : h[j], p.limit);
              const float u = fminf(fmaxf(odd ? h[8 + j] : recv, -p.limit), p.limit);
              const float sg = __fdividef(1.0f, 1.0f + __expf(-p.alpha * g));  // fast-math sigmoid
              const uint16_t ab = float_to_bf16_bits((u + 1.0f) * g * sg);  // R1
              uint16_t *orow = p.out + (size_t)(row0 + c0 + jt) * p.ldo;
              if (F16 && p.a_f16)  // the bf16 value times 2^9, held as f16 for an f16 GEMM2, natural order
                orow[col] = __half_as_ushort(__float2half_rn(bf16_bits_to_float(ab) * 512.f));
              else
                orow[col_st] = ab;
            }
          }
        } else {
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            if ((smask >> j) & 1u) {
              uint16_t *orow = p.out + (size_t)(row0 + c0 + j) * p.ldo;
              if (EPI == EPI_RELU2) {
                const float rr = fmaxf(h[j], 0.f);
                orow[col_st] = float_to_bf16_bits(rr * rr);
              } else {
                const float hw = p.mul ? __fmul_rn(h[j], tw_w[c0 + j]) : h[j];
                orow[col] = float_to_bf16_bits(hw);
              }
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(accempty_bar(rc.slot));
      rc.advance(nacc);
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

// Per-device host caches: devices are numbered below kMaxDevices.
constexpr int kMaxDevices = 64;
constexpr uint32_t kMaxSmem = 227 * 1024;  // dynamic shared memory a CTA may opt into

int current_device() {
  int dev = 0;
  return (cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < kMaxDevices) ? dev : 0;
}

// SM count of the current device (queried once per device).
int sm_count() {
  static std::atomic<int> cached[kMaxDevices];
  const int dev = current_device();
  int n = cached[dev].load(std::memory_order_relaxed);
  if (n <= 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cached[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

template <int FMT, int EPI, int KPB, bool F16>
moe_status_t launch_t(const GemmArgs &a, dim3 grid, uint32_t smem, cudaStream_t st) {
  auto kern = grouped_gemm_kernel<FMT, EPI, KPB, F16>;
  // the dynamic shared-memory limit is a per-device function attribute: set
  // it once per device to the most any launch asks for (every thread writes
  // the same value, so racing first launches agree)
  static std::atomic<int> configured[kMaxDevices];
  std::atomic<int> &done = configured[current_device()];
  if (!done.load(std::memory_order_acquire)) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kMaxSmem) != cudaSuccess)
      return MOE_ERR_CUDA;
    done.store(1, std::memory_order_release);
  }
  return launch_pdl(kern, grid, dim3(cta_threads(KPB)), smem, st, a) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace

// K blocks per pipeline stage: four (128 contiguous bytes per weight row) for
// the narrow token tiles of decode, whose stages are mostly weights; two for
// wider tiles, whose activation rows already make each stage large.
int choose_kpb(int tile_n) { return tile_n <= 32 ? 4 : 2; }

int choose_tile_n(int num_rows, int E) {
  const int active = num_rows < E ? (num_rows > 0 ? num_rows : 1) : E;
  const int avg = (num_rows + active - 1) / active;
  int n = ((2 * avg + 15) / 16) * 16;
  if (n < 16) n = 16;
  // wider tiles amortise each dequantised weight tile over more tokens: 192
  // rows (two accumulators next to two operand buffers in TMEM) when that
  // cuts the token tiles of an average expert, else 160 (three operand
  // buffers), which also keeps unevenly loaded experts of up to 160 rows in
  // one tile
  if (n > 128) n = ((avg + 159) / 160 == (avg + 191) / 192) ? 160 : 192;
  return n;
}

moe_status_t launch_grouped_gemm(int epi, const moe_qweight_t &w, const uint16_t *x, int P_max,
                                 const int32_t *sorted_ids, const int32_t *expert_offsets, int num_rows,
                                 const float *topk_w, int mul, int layout, moe_act_t act, uint16_t *out,
                                 int ldo, unsigned int *status, cudaStream_t stream, int *launches, int f16,
                                 const int32_t *xexp) {
  if (P_max <= 0 || num_rows <= 0) return MOE_OK;
  if (w.E > kMaxE) return MOE_ERR_UNSUPPORTED;
  // f16: bit 0 = f16 operands (NVFP4 / MXFP4 weights), bit 1 = GEMM1 writes a
  // as f16 in natural column order (for an f16 GEMM2) instead of bf16
  const int a_f16 = (f16 >> 1) & 1;
  f16 &= 1;
  if (f16 && ((w.fmt != MOE_FMT_NVFP4 && w.fmt != MOE_FMT_MXFP4) || (epi != 2 && !xexp)))
    return MOE_ERR_UNSUPPORTED;
  auto enc = encode_fn();
  if (!enc) return MOE_ERR_CUDA;
  GemmArgs a;
  memset(&a, 0, sizeof(a));
  const int E = w.E, N = w.N, K = w.K;
  a.tile_n = choose_tile_n(num_rows, E);
  if (a.tile_n > P_max) a.tile_n = P_max;  // the activation box never exceeds the rows (P_max % 16 == 0)
  // K blocks per pipeline stage: longer contiguous runs per weight row
  const int kpb = choose_kpb(a.tile_n);
  // packed weights: [E][N][K/2] bytes, box (32 * kpb) B x 64 rows x 1 expert
  {
    cuuint64_t dims[3] = {(cuuint64_t)(K / 2), (cuuint64_t)N, (cuuint64_t)E};
    cuuint64_t strides[2] = {(cuuint64_t)(K / 2), (cuuint64_t)N * (K / 2)};
    cuuint32_t box[3] = {(cuuint32_t)(32 * kpb), 64, 1};
    cuuint32_t es[3] = {1, 1, 1};
    const CUtensorMapSwizzle swz = kpb == 4 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    if (enc(&a.tm_w, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t *>(w.q), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return MOE_ERR_CUDA;
  }
  a.kpb = kpb;
  // activations: [P_max][K] bf16, box 64 x tile_n rows, 128-byte swizzle
  {
    cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)P_max};
    cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)a.tile_n};
    cuuint32_t es[2] = {1, 1};
    if (enc(&a.tm_x, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
            const_cast<uint16_t *>(x), dims, strides, box, es,
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
  a.xexp = xexp;
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
  a.a_f16 = a_f16;
  a.alpha = act.alpha;
  a.limit = act.limit;
  a.m_tiles = (epi == 0) ? (N / 2 + 63) / 64 : (N + kTileM - 1) / kTileM;
  a.sc_row_bytes = (w.fmt == MOE_FMT_NVFP4) ? K / 16 : (w.fmt == MOE_FMT_MXFP4 ? K / 32 : (K / 64) * 2);
  a.z_row_bytes = (w.fmt == MOE_FMT_INT4) ? (K / 64 + 1) / 2 : 0;
  // two TMEM accumulators when at least two operand buffers still fit; the
  // rest of the 512 columns holds as many stage-sized operand buffers as fit
  const int stride = (int)tmem_acc_stride(a.tile_n);
  a.nacc = (2 * stride + 2 * 32 * kpb <= kTmemCols) ? 2 : 1;
  a.na = (kTmemCols - a.nacc * stride) / (32 * kpb);
  if (a.na > kMaxNA) a.na = kMaxNA;
  // ring depths: up to four token-row slots, as many weight slots as then fit
  // in shared memory, and never fewer weight slots than token-row slots
  const uint32_t budget = 225 * 1024;
  auto smem_of = [&](int st, int xs) {
    return smem_layout(a.tile_n, st, kpb, a.sc_row_bytes, a.z_row_bytes, xs).total;
  };
  auto weight_slots = [&](int xs) {
    int st = kMaxStagesL;
    while (st > 2 && smem_of(st, xs) > budget) --st;
    return st;
  };
  int xst = 4;
  while (xst > 2 && (smem_of(weight_slots(xst), xst) > budget || weight_slots(xst) < xst)) --xst;
  a.xstages = xst;
  a.stages = weight_slots(xst);
  // an operand buffer is freed by the done barrier of its previous stage's
  // token-row slot, which must not have been reused meanwhile: NA <= xstages
  if (a.na > xst) a.na = xst;
  uint32_t smem = smem_of(a.stages, xst);
  // one CTA per SM: it allocates all of TMEM
  if (smem < 120 * 1024) smem = 120 * 1024;
  if (smem > kMaxSmem) return MOE_ERR_UNSUPPORTED;
  // persistent grid: one wave of resident CTAs, at most one per possible tile
  const int active = num_rows < E ? num_rows : E;
  const int max_tiles = a.m_tiles * (P_max / a.tile_n + active + 1);
  int ctas = sm_count();
  if (ctas > max_tiles) ctas = max_tiles;
  dim3 grid(ctas);
  if (launches) ++*launches;
  const int f = w.fmt;
  if (f16) {  // NVFP4 or MXFP4 (checked above)
#define MOE4_F16_K(F, K)                                                          \
  if (f == F && kpb == K) {                                                       \
    if (epi == 0) return launch_t<F, EPI_SWIGLU, K, true>(a, grid, smem, stream); \
    if (epi == 1) return launch_t<F, EPI_RELU2, K, true>(a, grid, smem, stream);  \
    return launch_t<F, EPI_WEIGHTED, K, true>(a, grid, smem, stream);             \
  }
    MOE4_F16_K(MOE_FMT_NVFP4, 2)
    MOE4_F16_K(MOE_FMT_NVFP4, 4)
    MOE4_F16_K(MOE_FMT_MXFP4, 2)
    MOE4_F16_K(MOE_FMT_MXFP4, 4)
#undef MOE4_F16_K
  }
#define MOE4_DISPATCH_K(F, K)                                                         \
  if (f == F && kpb == K) {                                                           \
    if (epi == 0) return launch_t<F, EPI_SWIGLU, K, false>(a, grid, smem, stream);    \
    if (epi == 1) return launch_t<F, EPI_RELU2, K, false>(a, grid, smem, stream);     \
    return launch_t<F, EPI_WEIGHTED, K, false>(a, grid, smem, stream);                \
  }
#define MOE4_DISPATCH(F) MOE4_DISPATCH_K(F, 2) MOE4_DISPATCH_K(F, 4)
  MOE4_DISPATCH(MOE_FMT_NVFP4)
  MOE4_DISPATCH(MOE_FMT_MXFP4)
  MOE4_DISPATCH(MOE_FMT_INT4)
#undef MOE4_DISPATCH
#undef MOE4_DISPATCH_K
  return MOE_ERR_UNSUPPORTED;
}

}  // namespace moe4
