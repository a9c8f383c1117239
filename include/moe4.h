/*
 * moe4.h -- C ABI of libmoe4, the fused Mixture-of-Experts layer with 4-bit
 * block-scaled expert weights, for one GB300 GPU (sm_103a).
 *
 * The layer (per token t, routed experts e_tj and weights w_tj, j < top_k):
 *     out[t] = sum_j w_tj * ( W2[e] . act( W13[e] . x[t] + b13[e] ) + b2[e] )
 * computed as five steps -- route, align/permute, grouped GEMM1 + activation,
 * grouped GEMM2 + per-row routing weight, unpermute/reduce -- or all at once
 * by moe_forward.
 *
 * Sources (web pages on the subject; cited by page title and section):
 *  [MARLIN] vLLM issue "[Bug]: moe_wna16_marlin_gemm applies wrong per-row
 *           topk weights (mul_topk_weights=True) at gpt-oss NVFP4 MoE shapes",
 *           sections "Describe the bug", "Forensic" and "Minimal repro".
 *  [NVFP4]  vLLM issue "[Bug]: gpt-oss-20b NVFP4 inference is broken",
 *           Gaps 1-3 (biases, per-expert global scale, clamped SwiGLU,
 *           interleaved gate/up).
 *  [NEMO]   vLLM issue "[Bug]: NVFP4 MoE monolithic backend
 *           (trtllm_fp4_block_scale_moe) produces semantically corrupt output
 *           for non-gated ReLU2 MoE (Nemotron-3-Nano) on SM100", Environment
 *           and Analysis.
 *  [EP]     vLLM issue "[Bug]: gpt-oss-120b MXFP4 + --enable-expert-parallel
 *           crashes at startup", Root cause (output width = unpadded hidden).
 *  [GPTQ]   OneCompression guide "GPT-OSS (mixed_gptq)", "Why GPT-OSS needs
 *           special handling" and "1. Quantize" (INT4, group_size 64).
 *
 * Conventions for every entry point:
 *  - Device pointers are caller-owned device memory; host pointers appear only
 *    in moe_forward_host. The library never allocates memory and keeps no
 *    per-call state other than cached device properties (and the fixed
 *    device array that moe_forward_static uses as its workspace).
 *  - Tensors are dense, row-major, contiguous. Integers are int32. bf16 values
 *    are passed as uint16_t bit patterns. Every device pointer must be 16-byte
 *    aligned.
 *  - Every call is asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *    default stream) and returns MOE_OK or an error code. Arguments are
 *    checked on the host first; on MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED
 *    nothing is launched.
 *  - Errors detected on the device (an expert id out of range, a bounded wait
 *    that ran out, an unsupported scale) are latched as bits in the device
 *    status word at the start of the workspace `ws`; moe_read_status reads
 *    them back (it synchronises the stream) and moe_clear_status resets them.
 *  - Kernels use no atomics on floating-point data: repeated calls with the
 *    same inputs give bit-identical outputs.
 *  - Sizes: E <= 256, 1 <= top_k <= min(E, 8), H and I multiples of 64 and
 *    at most 4096, T * top_k < 2^24.
 */
#ifndef MOE4_H
#define MOE4_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *moe_stream_t; /* == cudaStream_t */

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1, /* null / misaligned pointer, bad size or enum   */
  MOE_ERR_UNSUPPORTED = 2, /* valid but not built (format/activation/size)  */
  MOE_ERR_CUDA = 3,        /* a CUDA runtime call or launch failed          */
  MOE_ERR_TIMEOUT = 4,     /* device: a bounded wait inside a kernel ran out */
  MOE_ERR_BAD_INDEX = 5,   /* device: an expert id or row index out of range */
  MOE_ERR_WORKSPACE = 6,   /* ws_bytes smaller than moe_workspace_size      */
  MOE_ERR_SCALE_RANGE = 7  /* device: an MXFP4 exponent above 2^1 (e8m0>128) */
} moe_status_t;

/* Weight formats [MARLIN "Minimal repro"; GPTQ "1. Quantize"; EP]. */
typedef enum {
  MOE_FMT_NVFP4 = 0, /* E2M1 codes, E4M3 scale per 16 along K, fp32 gscale[E] */
  MOE_FMT_MXFP4 = 1, /* E2M1 codes, E8M0 scale per 32 along K                 */
  MOE_FMT_INT4 = 2   /* 4-bit codes q, fp16 scale + 4-bit zero per 64 along K,
                        w = bf16((q - z) * s)                                 */
} moe_format_t;

typedef enum {
  MOE_ACT_SWIGLUOAI = 0, /* gated: g = min(g, limit), u = clamp(u, -limit, limit),
                            a = (u + 1) * g * sigmoid(alpha * g) [NVFP4 Gap 3a] */
  MOE_ACT_RELU2 = 1      /* non-gated: a = max(h, 0)^2 [NEMO]                   */
} moe_act_kind_t;

/* Row order of the gated W13 [NVFP4 Gap 3c]: INTERLEAVED = gpt-oss order, row
 * 2j is gate_j and row 2j+1 is up_j; CONCAT = [gate rows; up rows]. The bias
 * follows the same order. Ignored for non-gated activations. */
typedef enum { MOE_LAYOUT_INTERLEAVED = 0, MOE_LAYOUT_CONCAT = 1 } moe_gate_up_layout_t;

/* Routing [MARLIN "Minimal repro"; NEMO Analysis item 3]. */
typedef enum {
  MOE_ROUTE_TOPK_SOFTMAX = 0, /* top-k of logits (ties -> lower id), softmax over the k */
  MOE_ROUTE_SIGMOID_BIAS = 1  /* s = sigmoid(logit) (fp32); select top-k of s + bias;
                                 weights = selected s / sum(selected s)              */
} moe_route_t;

/* One quantised projection, all experts: W13 (N = 2I gated, I non-gated; K = H)
 * or W2 (N = H; K = I). Packed codes: two 4-bit codes per byte along K, the
 * even K index in the low nibble [MARLIN "Minimal repro"]. */
typedef struct {
  int32_t fmt;            /* moe_format_t                                   */
  int32_t E, N, K;        /* experts, output rows, reduction length          */
  const uint8_t *q;       /* [E][N][K/2]                                     */
  const void *scales;     /* NVFP4: E4M3 bytes [E][N][K/16]; MXFP4: E8M0 bytes
                             [E][N][K/32]; INT4: fp16 [E][N][K/64]           */
  const uint8_t *zeros;   /* INT4 only: [E][N][ceil(K/128)] bytes, two 4-bit
                             zero points per byte, even group in the low nibble */
  const float *gscale;    /* NVFP4 only: per-expert fp32 global scale [E]
                             (a checkpoint's single scalar is broadcast by the
                             caller [NVFP4 Gap 2b]); NULL otherwise          */
  const uint16_t *bias;   /* bf16 [E][N] or NULL [NVFP4 Gap 1]                */
} moe_qweight_t;

typedef struct {
  int32_t kind; /* moe_act_kind_t */
  float alpha;  /* swigluoai: 1.702 for gpt-oss */
  float limit;  /* swigluoai: 7.0 for gpt-oss   */
} moe_act_t;

/* Bytes at the start of every workspace reserved for the status word. */
#define MOE_STATUS_BYTES 256

/* Padded slot count P_max of the aligned layout: at most min(E, T*k) experts
 * are non-empty and each pads to a multiple of block_m, so
 * P_max = floor((T*k + min(E, T*k) * (block_m - 1)) / block_m) * block_m.
 * Host only. */
int64_t moe_padded_rows(int T, int k, int E, int block_m);

/* Workspace bytes moe_forward needs for these sizes (status word, routing,
 * alignment metadata and the x_perm / a / y intermediates). Host only. */
moe_status_t moe_workspace_size(int T, int E, int k, int H, int I, int block_m,
                                size_t *bytes);

/* Step a1 -- routing. logits fp32 [T][E]; sel_bias fp32 [E] (SIGMOID_BIAS
 * only, else ignored). Out: topk_ids int32 [T][k] (descending score),
 * topk_weights fp32 [T][k]. ws: >= MOE_STATUS_BYTES. */
moe_status_t moe_route_topk(const float *logits, const float *sel_bias, int T,
                            int E, int k, int route, int32_t *topk_ids,
                            float *topk_weights, void *ws, moe_stream_t stream);

/* Step a2 -- align/permute [MARLIN "Minimal repro", moe_align_block_size].
 * Flat routed rows r = t*k + j are grouped by expert; within an expert rows
 * keep ascending r; each expert's segment is padded to a multiple of block_m
 * (16, 32, 64, 128 or 256) with the sentinel T*k; empty experts get no slots.
 * Out (P_max = moe_padded_rows(T, k, E, block_m)):
 *   sorted_token_ids int32 [P_max]   flat row of each slot (T*k = padding)
 *   expert_offsets   int32 [E+1]     first slot of each expert; [E] = used slots
 *   block_expert_ids int32 [P_max/block_m]  expert of each block, -1 unused
 *                    (the pages' moe_align_block_size output, for callers
 *                    that schedule by block; the grouped GEMMs below walk
 *                    expert_offsets instead and do not read it)
 *   row_pos          int32 [T*k]     slot of each flat row
 *   x_perm           bf16  [P_max][H] x[sorted/k] per slot, zero in padding,
 *                    columns interleaved within every group of 8 (below)
 * An expert id outside [0, E) latches MOE_ERR_BAD_INDEX and is dropped
 * (row_pos = -1). Rows of x_perm at and past expert_offsets[E] are left
 * unspecified (from 4096 routed rows on, the call keeps per-chunk expert
 * counts at the start of x_perm until it writes the rows).
 * Interleaved columns: x_perm and a_out (below) store the columns of each
 * group of 8 in the order 0,4,1,5,2,6,3,7 -- the order in which the GEMMs
 * expand the packed 4-bit weights -- so stored column 8g+q holds column
 * 8g + (0,4,1,5,2,6,3,7)[q]. Only these two intermediates use it. */
moe_status_t moe_align_permute(const int32_t *topk_ids, int T, int k, int E,
                               int block_m, const uint16_t *x, int H,
                               int32_t *sorted_token_ids, int32_t *expert_offsets,
                               int32_t *block_expert_ids, int32_t *row_pos,
                               uint16_t *x_perm, void *ws, moe_stream_t stream);

/* Step a3 -- grouped GEMM1 with bias and activation fused [NVFP4 Gaps 1, 3;
 * NEMO]. For every used slot p of expert e (sorted_token_ids[p] < num_rows):
 *   h = (x_perm[p] . W13'[e]^T) * gscale[e] + b13[e]   (fp32 accumulate)
 *   a_out[p] = bf16(act(h))                  a_out: bf16 [P_max][I]
 * x_perm is read and a_out written with interleaved columns (see
 * moe_align_permute).
 * W13' is the bf16 dequantised operand. Padding slots of a_out are not written.
 * P_max must be moe_padded_rows(...) of the align call that made the metadata.
 * Both grouped GEMMs start streaming weights while the previous kernel on the
 * stream drains (programmatic dependent launch); they wait for it before
 * reading x_perm / a, but read expert_offsets at once: it must not be written
 * by that previous kernel (moe_align_permute's last kernel is its gather, so
 * the step sequence above satisfies this). */
moe_status_t moe_grouped_gemm1_act(const uint16_t *x_perm,
                                   const int32_t *sorted_token_ids,
                                   const int32_t *expert_offsets, int P_max,
                                   int num_rows, const moe_qweight_t *w13,
                                   int gate_up_layout, moe_act_t act,
                                   uint16_t *a_out, void *ws, moe_stream_t stream);

/* Step a4 -- grouped GEMM2 with bias and the per-row routing weight fused
 * [MARLIN "Describe the bug", "Workaround"]. For every used slot p of expert e:
 *   z = (a[p] . W2'[e]^T) * gscale[e] + b2[e]
 *   if mul_topk_weights: z *= topk_weights_flat[sorted_token_ids[p]]
 *   y[p] = bf16(z)                            y: bf16 [P_max][H]
 * a is read with interleaved columns (as moe_grouped_gemm1_act writes it);
 * y has plain column order.
 * The weight is read through the slot's own flat row id (the Marlin kernel
 * read another row's entry). Padding slots of y are not written. */
moe_status_t moe_grouped_gemm2_weighted(const uint16_t *a,
                                        const int32_t *sorted_token_ids,
                                        const int32_t *expert_offsets, int P_max,
                                        const moe_qweight_t *w2,
                                        const float *topk_weights_flat,
                                        int mul_topk_weights, int num_rows,
                                        uint16_t *y, void *ws, moe_stream_t stream);

/* Step a5 -- unpermute/reduce at the unpadded width H [EP Root cause]:
 *   out[t] = bf16( sum_{j=0..k-1} fp32(y[row_pos[t*k + j]]) ), j ascending.
 * A deterministic gather-sum (no atomics). out: bf16 [T][H], stride H. */
moe_status_t moe_unpermute_reduce(const uint16_t *y, const int32_t *row_pos,
                                  int T, int k, int H, int P_max, uint16_t *out,
                                  void *ws, moe_stream_t stream);

/* Steps a1..a5 in order on one stream, intermediates in `ws` (ws_bytes >=
 * moe_workspace_size(T, E, k, H, I, block_m)). x bf16 [T][H], logits fp32
 * [T][E], out bf16 [T][H]. block_m = 0 picks 16. No host synchronisation:
 * the call can be captured in a CUDA graph.
 * mul_topk_weights selects where each routed row's own routing weight w
 * applies [MARLIN "Minimal repro": apply_router_weight_on_input]: 0 nowhere,
 * 1 in the GEMM2 epilogue (z *= w, as moe_grouped_gemm2_weighted), 2 on the
 * input (the row enters GEMM1 as bf16(x * w) and GEMM2 does not multiply);
 * other values are MOE_ERR_INVALID_ARG. The same holds for the _host,
 * _static and _profile variants. */
moe_status_t moe_forward(const uint16_t *x, const float *logits,
                         const float *sel_bias, int T, int E, int k, int H,
                         int I, int route, const moe_qweight_t *w13,
                         const moe_qweight_t *w2, int gate_up_layout,
                         moe_act_t act, int mul_topk_weights, int block_m,
                         uint16_t *out, void *ws, size_t ws_bytes,
                         moe_stream_t stream);

/* moe_forward with x, logits and out in HOST memory; weights and ws stay in
 * device memory. Page-locked (pinned, hence mapped) buffers are read and
 * written in place by the kernels over the host link, with no staging
 * copies; pageable ones are copied in through the workspace and out back on
 * `stream`. Returns after enqueueing; the caller synchronises the stream
 * before reading out. */
moe_status_t moe_forward_host(const uint16_t *x_host, const float *logits_host,
                              const float *sel_bias, int T, int E, int k, int H,
                              int I, int route, const moe_qweight_t *w13,
                              const moe_qweight_t *w2, int gate_up_layout,
                              moe_act_t act, int mul_topk_weights, int block_m,
                              uint16_t *out_host, void *ws, size_t ws_bytes,
                              moe_stream_t stream);

/* moe_forward, then the device time of each of its six kernels: kernel_ms
 * (host, 6 floats) receives route, align, gather, GEMM1, GEMM2 and unpermute
 * in milliseconds, from CUDA events recorded on `stream` around each launch.
 * Synchronises the stream. For measurement; there is no counterpart on the
 * source pages. */
moe_status_t moe_forward_profile(const uint16_t *x, const float *logits,
                                 const float *sel_bias, int T, int E, int k,
                                 int H, int I, int route, const moe_qweight_t *w13,
                                 const moe_qweight_t *w2, int gate_up_layout,
                                 moe_act_t act, int mul_topk_weights, int block_m,
                                 uint16_t *out, void *ws, size_t ws_bytes,
                                 moe_stream_t stream, float *kernel_ms);

/* The same layer with no workspace argument, for callers that cannot
 * allocate device memory (no cudaMalloc where they run: inside a graph
 * capture that forbids allocation, a plugin handed only its input and output
 * buffers, a runtime whose memory budget is fixed up front). There is no
 * counterpart on the source pages; it is a deployment convenience.
 * The workspace is a file-scope device array of MOE_STATIC_WS_BYTES inside
 * the library; every GPU that loads the library holds it until the process
 * exits. The call needs moe_workspace_size's bytes minus the staging buffers
 * of moe_forward_host (which it never uses); sizes past the array return
 * MOE_ERR_UNSUPPORTED (at H = I = 2880, E = 32, top-4, block_m 16 the
 * array holds up to T = 607 tokens, 2,428 routed rows).
 * Every argument is checked before anything is enqueued: a call that returns
 * MOE_ERR_INVALID_ARG or MOE_ERR_UNSUPPORTED leaves the stream, the array and
 * status_out untouched, and so does a call with T = 0.
 * The first call on a device looks up the array's device address, so make it
 * before any stream capture; if that lookup fails the call returns
 * MOE_ERR_CUDA and the next call tries again. All calls share the array:
 * calls that overlap on the GPU race and must not be issued. Each call clears
 * the array's status word first; status_out (device, 4-byte aligned, may be
 * NULL) receives the raw status word after the call (bit c-1 set when device
 * error code c was detected).
 * Allocates nothing: no cudaMalloc, cudaFree or allocating library call. */
#define MOE_STATIC_WS_BYTES (32u << 20)
moe_status_t moe_forward_static(const uint16_t *x, const float *logits,
                                const float *sel_bias, int T, int E, int k, int H,
                                int I, int route, const moe_qweight_t *w13,
                                const moe_qweight_t *w2, int gate_up_layout,
                                moe_act_t act, int mul_topk_weights, int block_m,
                                uint16_t *out, uint32_t *status_out,
                                moe_stream_t stream);

/* Reads the device status word of `ws` (synchronises `stream`); *status gets
 * the lowest-numbered latched error, or MOE_OK. */
moe_status_t moe_read_status(const void *ws, moe_stream_t stream, int *status);

/* Clears the device status word of `ws` (asynchronous on `stream`). */
moe_status_t moe_clear_status(void *ws, moe_stream_t stream);

/* Exercises the failure path of the kernels' bounded waits: one single-warp
 * kernel waits on a shared-memory barrier that nothing arrives on, gives up
 * after the same cycle limit the layer's waits use (about a second), latches
 * MOE_ERR_TIMEOUT in the status word of `ws` and returns; the context stays
 * usable. Asynchronous on `stream`; for tests. */
moe_status_t moe_wait_selftest(void *ws, moe_stream_t stream);

/* Readable name of a status code (static string). */
const char *moe_status_string(int status);

/* Number of kernels the last moe_forward call on this thread launched. */
int moe_last_launch_count(void);

/* ---------------------------------------------------------------------------
 * Checkpoint-layout import (host memory, host only, no CUDA calls; for load
 * time). They rewrite the expert weights of the pages' checkpoints into the
 * moe_qweight_t layout above.
 * ------------------------------------------------------------------------- */

/* One GPTQ INT4 linear layer (N outputs, K inputs, group 64) of one expert
 * [GPTQ "1. Quantize": per-expert gate_proj / up_proj / down_proj with
 * qweight, qzeros, scales, g_idx; MARLIN "Reproducer": qweight is the int32
 * [K/8][N] view of the [N][K/2] code bytes]. In:
 *   qweight int32 [K/8][N]: the code of input k = 8i + j of output n in bits
 *           4j..4j+3 of qweight[i][n]
 *   qzeros  int32 [K/64][N/8]: the zero point of output n = 8m + j, group g,
 *           in bits 4j..4j+3 of qzeros[g][m], stored as (zero - zero_offset)
 *   scales  fp16 [K/64][N]
 *   g_idx   int32 [K] or NULL: group of input k; must be k / 64
 * Out (caller-owned): q uint8 [N][K/2] (low nibble = even k), scales_out fp16
 * [N][K/64], zeros_out uint8 [N][ceil(K/128)] (low nibble = even group), i.e.
 * rows of moe_qweight_t q / scales / zeros. For W13, convert gate_proj into
 * rows 0..I-1 and up_proj into rows I..2I-1 (pointers offset by I rows) and
 * pass MOE_LAYOUT_CONCAT. zero_offset: 0 when qzeros holds the zero points
 * themselves, 1 when it holds them minus one.
 * Errors: MOE_ERR_INVALID_ARG (null pointer, K or N not a multiple of 64,
 * zero_offset not 0 or 1); MOE_ERR_UNSUPPORTED (group_size != 64, a g_idx
 * other than k / 64, a zero point outside 0..15). Nothing is written on
 * error. */
moe_status_t moe_import_gptq_int4(const int32_t *qweight, const int32_t *qzeros,
                                  const uint16_t *scales, const int32_t *g_idx,
                                  int K, int N, int group_size, int zero_offset,
                                  uint8_t *q, uint16_t *scales_out,
                                  uint8_t *zeros_out);

/* ModelOpt NVFP4 [NVFP4 "Gap 2", 2b]: the codes (two E2M1 per byte, low
 * nibble = even k) and E4M3 group-16 scales already have the moe_qweight_t
 * layout, but the checkpoint keeps weight_scale_2 as one scalar where this
 * library takes one global scale per expert: gscale[e] = weight_scale_2 for
 * e < E (host array of E floats). MOE_ERR_INVALID_ARG for a null pointer or
 * E outside 1..256. */
moe_status_t moe_import_modelopt_global_scale(float weight_scale_2, int E,
                                              float *gscale);

#ifdef __cplusplus
}
#endif

#endif /* MOE4_H */
