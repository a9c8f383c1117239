"""Dequantisation, grouped GEMMs with fused epilogues, unpermute, whole layer.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

The layer computes, per token t with routed experts e_tj and weights w_tj
(j < k), the plain definition

    out[t] = sum_j w_tj * MLP_{e_tj}(x[t])
    MLP_e(x) = W2[e] . act(W13[e] . x + b13[e]) + b2[e]

which the repro in the vLLM issue "moe_wna16_marlin_gemm applies wrong per-row
topk weights" (section "Minimal repro") writes per row as
``out[row] = (act[row] @ w[e].T + bias) * topk_w[row]``. The fused layer is an
exact reorganisation of it, with float rounding at fixed points that the CUDA
path follows as well:

  R0  the bf16 weight operand: NVFP4 E2M1*E4M3 (exact in bf16; the per-expert
      fp32 global scale multiplies the accumulator), MXFP4 E2M1*2^(e-127)
      (exact), GPTQ INT4 bf16_rne((q - z) * s_fp16);
  --  accumulation over K in float64 (rounded once to fp32; ``acc_dtype``
      float32 sums in fp32 instead, for the timed CPU baseline); then
      h = fp32(fp32(acc * gscale) + bias);
  R1  the activation output a is rounded to bf16;
  R2  GEMM2: z = fp32(fp32(acc * gscale) + b2); z = fp32(z * w_row) when the
      routing weight is applied in the epilogue; y = bf16(z);
  R3  unpermute: fp32 sum over j = 0..k-1 in that order, rounded to bf16.

Where the routing weight is applied (``mul_topk_weights``): 0 nowhere, 1 (or
True) in the GEMM2 epilogue as above, 2 on the input. The pages name the switch
(``apply_router_weight_on_input``; with it off, GEMM2 multiplies -- vLLM issue
"moe_wna16_marlin_gemm applies wrong per-row topk weights", "Minimal repro")
but do not spell out the other setting. Its plain reading, taken here: every
routed row (t, j) enters GEMM1 as  Rin  x_in = bf16(fp32(x[t] * w_tj)), and
GEMM2 does not multiply.

Formulas that the pages name but do not print, and the readings taken:
  * swigluoai (vLLM issue "gpt-oss-20b NVFP4 inference is broken", Gap 3a/3b:
    ``gemm1_alpha/beta/clamp_limit``): gate = min(gate, limit),
    up = clamp(up, -limit, limit), a = (up + 1) * gate * sigmoid(alpha * gate)
    with limit 7, alpha 1.702 and the "+1" being beta = 1; the bias is added
    before the clamp.
  * gate/up order (same issue, Gap 3c: gpt-oss stores them interleaved): in the
    INTERLEAVED layout row 2j is gate_j and row 2j+1 is up_j; CONCAT stacks
    [gate; up]. Biases follow the same order.
  * ReLU2 (vLLM issue "... non-gated ReLU2 MoE (Nemotron-3-Nano)"): a = max(h,0)^2.
  * MXFP4 / GPTQ INT4 decoding: see ``dequant_mxfp4`` / ``dequant_int4``.

Parity: pinned (tests/test_oracle_layer.py: brute force on tiny layers, the
dense per-token definition, k = 1 against a single dense MLP through
torch.nn.functional.linear, closed forms for all-zero codes and one-hot inputs,
internal vs external weight multiply, per-row applied ratio, token permutation
and unpadded output shape). Full-scale float values beyond these invariants are
parity unpinned: the pages print no reproducible numbers at those sizes.
"""
import numpy as np

from .formats import (E2M1_VALUES, E4M3_VALUES, E8M0_VALUES, bf16_rne, f32,
                      unpack_nibbles)
from . import align as _align
from . import routing as _routing

FMT_NVFP4, FMT_MXFP4, FMT_INT4 = 0, 1, 2
ACT_SWIGLUOAI, ACT_RELU2 = 0, 1
LAYOUT_INTERLEAVED, LAYOUT_CONCAT = 0, 1
MUL_NONE, MUL_OUTPUT, MUL_INPUT = 0, 1, 2


def weight_rows_on_input(x_rows, row_weights):
    """Rin: bf16(fp32(x * w)) for each routed row and its own routing weight."""
    prod = np.asarray(x_rows, np.float64) * np.asarray(row_weights, np.float64)[:, None]
    return bf16_rne(f32(prod))


# --------------------------------------------------------------------------- R0
def dequant_nvfp4(q: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """One expert. q uint8 [N, K/2], scales E4M3 bytes [N, K/16] ->
    float64 [N, K] = E2M1[code] * E4M3[scale]; exact in bf16 (pinned)."""
    codes = unpack_nibbles(q)
    vals = E2M1_VALUES[codes]
    s = E4M3_VALUES[np.asarray(scales, dtype=np.uint8)]
    return vals * np.repeat(s, 16, axis=1)


def dequant_mxfp4(q: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """One expert. q uint8 [N, K/2], scales E8M0 bytes [N, K/32] ->
    float64 [N, K] = bf16(E2M1[code] * 2^(e-127)); exact whenever the product
    is inside the bf16 range."""
    codes = unpack_nibbles(q)
    vals = E2M1_VALUES[codes]
    s = E8M0_VALUES[np.asarray(scales, dtype=np.uint8)]
    prod = vals * np.repeat(s, 32, axis=1)
    return bf16_rne(f32(prod)).astype(np.float64)


def int4_zero_codes(zeros: np.ndarray, n_groups: int) -> np.ndarray:
    """[N, ceil(G/2)] bytes, two 4-bit zero points per byte with the even group
    in the low nibble -> [N, G] codes."""
    z = unpack_nibbles(zeros)
    return z[:, :n_groups]


def dequant_int4(q: np.ndarray, scales: np.ndarray, zeros: np.ndarray) -> np.ndarray:
    """One expert, GPTQ-style asymmetric INT4 with group size 64 along K
    (OneCompression guide "GPT-OSS (mixed_gptq)", "1. Quantize": group_size=64,
    2880/64 = 45 groups). q uint8 [N, K/2] (4-bit codes 0..15, low nibble =
    even k), scales fp16 [N, K/64], zeros [N, ceil(K/128)] ->
    float64 [N, K] = bf16_rne((q - z) * s). (q - z) * s is exact in fp32."""
    codes = unpack_nibbles(q).astype(np.float64)
    G = scales.shape[1]
    s = np.asarray(scales, dtype=np.float16).astype(np.float64)
    z = int4_zero_codes(zeros, G).astype(np.float64)
    prod = (codes - np.repeat(z, 64, axis=1)) * np.repeat(s, 64, axis=1)
    return bf16_rne(f32(prod)).astype(np.float64)


def dequant(w: dict, e: int) -> np.ndarray:
    """R0 operand of expert e of a quantised projection (dict as made by
    ``synth.quantize``)."""
    fmt = w["fmt"]
    if fmt == FMT_NVFP4:
        return dequant_nvfp4(w["q"][e], w["scales"][e])
    if fmt == FMT_MXFP4:
        return dequant_mxfp4(w["q"][e], w["scales"][e])
    if fmt == FMT_INT4:
        return dequant_int4(w["q"][e], w["scales"][e], w["zeros"][e])
    raise ValueError(fmt)


def gscale_of(w: dict, e: int):
    g = w.get("gscale")
    return None if g is None else np.float32(g[e])


def bias_of(w: dict, e: int):
    b = w.get("bias")
    return None if b is None else np.asarray(b[e], dtype=np.float32)


# ------------------------------------------------------------------ GEMM pieces
def matvec_rows(W: np.ndarray, X: np.ndarray, acc_dtype=np.float64) -> np.ndarray:
    """acc[i, n] = sum_k X[i, k] * W[n, k], rounded to fp32.

    acc_dtype float64 (parity mode): summed in float64 one row at a time (the
    same call per row whatever the batching, so results do not depend on how
    rows are grouped), rounded once to fp32. acc_dtype float32 (the timed CPU
    baseline): one float32 matrix product over all rows; the operands are the
    same values (bf16 activations and R0 weights are exact in fp32), only the
    summation precision and order differ."""
    if np.dtype(acc_dtype) == np.float32:
        return np.asarray(X, dtype=np.float32) @ np.asarray(W, dtype=np.float32).T
    X = np.asarray(X, dtype=np.float64)
    out = np.empty((X.shape[0], W.shape[0]), dtype=np.float64)
    for i in range(X.shape[0]):
        out[i] = W @ X[i]
    return f32(out)


def linear_epilogue(acc32: np.ndarray, gscale, bias) -> np.ndarray:
    """h = fp32(fp32(acc * gscale) + bias), each step rounded to fp32."""
    h = acc32
    if gscale is not None:
        h = f32(h.astype(np.float64) * np.float64(gscale))
    if bias is not None:
        h = f32(h.astype(np.float64) + np.asarray(bias, dtype=np.float64)[None, :])
    return h.astype(np.float32)


def gate_up_split(h: np.ndarray, layout: int):
    """h [n, 2I] -> (gate [n, I], up [n, I])."""
    I = h.shape[1] // 2
    if layout == LAYOUT_INTERLEAVED:
        return h[:, 0::2], h[:, 1::2]
    if layout == LAYOUT_CONCAT:
        return h[:, :I], h[:, I:]
    raise ValueError(layout)


def swigluoai(gate: np.ndarray, up: np.ndarray, alpha: float, limit: float) -> np.ndarray:
    """fp32 in, fp32 out (evaluated in float64, rounded once)."""
    g = np.minimum(gate.astype(np.float64), np.float64(np.float32(limit)))
    u = np.clip(up.astype(np.float64), -np.float64(np.float32(limit)),
                np.float64(np.float32(limit)))
    a = np.float64(np.float32(alpha))
    with np.errstate(over="ignore"):  # exp overflow gives sigmoid 0, the exact limit
        return f32((u + 1.0) * g * (1.0 / (1.0 + np.exp(-a * g))))


def relu2(h: np.ndarray) -> np.ndarray:
    r = np.maximum(h.astype(np.float64), 0.0)
    return f32(r * r)


def expert_gemm1_act(x_rows, W13, gscale, bias, act, layout, alpha=1.702, limit=7.0,
                     acc_dtype=np.float64):
    """Rows routed to one expert: x_rows [n, H] (bf16 values) -> a [n, I] bf16."""
    h = linear_epilogue(matvec_rows(W13, x_rows, acc_dtype), gscale, bias)
    if act == ACT_SWIGLUOAI:
        g, u = gate_up_split(h, layout)
        a = swigluoai(g, u, alpha, limit)
    elif act == ACT_RELU2:
        a = relu2(h)
    else:
        raise ValueError(act)
    return bf16_rne(a)                                              # R1


def expert_gemm2(a_rows, W2, gscale, bias, row_weights=None, acc_dtype=np.float64):
    """Rows of one expert: a_rows [n, I] -> y [n, H] bf16; row_weights [n] fp32
    multiplies each row by its own routing weight (the epilogue multiply)."""
    z = linear_epilogue(matvec_rows(W2, a_rows, acc_dtype), gscale, bias)
    if row_weights is not None:
        z = f32(z.astype(np.float64) * np.asarray(row_weights, np.float64)[:, None])
    return bf16_rne(z)                                              # R2


def unpermute_reduce(y: np.ndarray, row_pos: np.ndarray, T: int, k: int) -> np.ndarray:
    """out[t] = bf16(sum_{j=0..k-1} y[row_pos[t*k + j]]) with an fp32 running
    sum in ascending j (no atomics: a fixed order). Width = y's width, the
    unpadded hidden size."""
    H = y.shape[1]
    acc = np.zeros((T, H), dtype=np.float32)
    rp = np.asarray(row_pos).reshape(T, k)
    for j in range(k):
        acc = (acc + y[rp[:, j]].astype(np.float32)).astype(np.float32)
    return bf16_rne(acc)                                            # R3


# ------------------------------------------------------------------- the layer
def grouped_gemm1_act(x_perm, expert_offsets, sorted_token_ids, num_rows, w13,
                      act, layout, alpha=1.702, limit=7.0, acc_dtype=np.float64):
    """Step a3b over all experts, streamed one expert at a time (each expert's
    weights are dequantised once, used for its rows and dropped). Rows of
    x_perm that hold padding (sorted id >= num_rows) are left at zero."""
    E = len(expert_offsets) - 1
    N1 = w13["q"].shape[1]
    I = N1 // 2 if act == ACT_SWIGLUOAI else N1
    a = np.zeros((x_perm.shape[0], I), dtype=np.float32)
    s = np.asarray(sorted_token_ids)
    for e in range(E):
        lo, hi = int(expert_offsets[e]), int(expert_offsets[e + 1])
        slots = np.arange(lo, hi)
        slots = slots[s[slots] < num_rows]
        if slots.size == 0:
            continue
        W = dequant(w13, e)
        a[slots] = expert_gemm1_act(x_perm[slots], W, gscale_of(w13, e),
                                    bias_of(w13, e), act, layout, alpha, limit, acc_dtype)
    return a


def grouped_gemm2_weighted(a, expert_offsets, sorted_token_ids, num_rows, w2,
                           topk_weights_flat, mul_topk_weights, acc_dtype=np.float64):
    """Step a4 over all experts, streamed one expert at a time; padding slots
    are left at zero. The routing
    weight of slot p is topk_weights_flat[sorted_token_ids[p]] -- the row's own
    flat index (the failure in the vLLM issue "moe_wna16_marlin_gemm applies
    wrong per-row topk weights" was reading another row's entry)."""
    E = len(expert_offsets) - 1
    H = w2["q"].shape[1]
    y = np.zeros((a.shape[0], H), dtype=np.float32)
    s = np.asarray(sorted_token_ids)
    tw = np.asarray(topk_weights_flat, dtype=np.float32)
    for e in range(E):
        lo, hi = int(expert_offsets[e]), int(expert_offsets[e + 1])
        slots = np.arange(lo, hi)
        slots = slots[s[slots] < num_rows]
        if slots.size == 0:
            continue
        W = dequant(w2, e)
        rw = tw[s[slots]] if mul_topk_weights == MUL_OUTPUT else None
        y[slots] = expert_gemm2(a[slots], W, gscale_of(w2, e), bias_of(w2, e), rw, acc_dtype)
    return y


def moe_forward(x, logits, w13, w2, k, route_mode=_routing.ROUTE_TOPK_SOFTMAX,
                sel_bias=None, act=ACT_SWIGLUOAI, layout=LAYOUT_INTERLEAVED,
                alpha=1.702, limit=7.0, mul_topk_weights=True, block_m=16,
                topk_ids=None, topk_weights=None, acc_dtype=np.float64):
    """Steps a1..a5 in order; returns every intermediate. ``topk_ids`` /
    ``topk_weights`` may be given to skip routing (e.g. to feed another
    implementation's routing decisions downstream). ``acc_dtype``: float64
    accumulation for parity (the default), float32 for the timed CPU
    baseline (see ``matvec_rows``)."""
    x = np.asarray(x, dtype=np.float32)
    T, H = x.shape
    E = w13["q"].shape[0]
    if topk_ids is None:
        topk_ids, topk_weights = _routing.route(logits, k, route_mode, sel_bias)
    topk_ids = np.asarray(topk_ids, dtype=np.int32)
    topk_weights = np.asarray(topk_weights, dtype=np.float32)
    meta = _align.align_permute(topk_ids, E, block_m)
    R = T * k
    x_perm = _align.gather_rows(x, meta["sorted_token_ids"], k)
    if mul_topk_weights == MUL_INPUT:
        srt = np.asarray(meta["sorted_token_ids"])
        used = np.nonzero(srt < R)[0]
        x_perm = x_perm.copy()
        x_perm[used] = weight_rows_on_input(x_perm[used], topk_weights.reshape(-1)[srt[used]])
    a = grouped_gemm1_act(x_perm, meta["expert_offsets"], meta["sorted_token_ids"],
                          R, w13, act, layout, alpha, limit, acc_dtype)
    y = grouped_gemm2_weighted(a, meta["expert_offsets"], meta["sorted_token_ids"],
                               R, w2, topk_weights.reshape(-1), mul_topk_weights, acc_dtype)
    out = unpermute_reduce(y, meta["row_pos"], T, k)
    return dict(topk_ids=topk_ids, topk_weights=topk_weights, x_perm=x_perm,
                a=a, y=y, out=out, **meta)


def moe_forward_tokens(x, topk_ids, topk_weights, w13, w2, tokens, act=ACT_SWIGLUOAI,
                       layout=LAYOUT_INTERLEAVED, alpha=1.702, limit=7.0,
                       mul_topk_weights=True):
    """The per-token definition (no permutation), for a subset of tokens:
    out[t] = bf16(sum_j y_tj) with y_tj = R2(w_tj * MLP_{e_tj}(x[t])).
    Same rounding points as ``moe_forward``; used for pins and for sampled
    parity at full sizes. Dequantised experts are computed once per call."""
    x = np.asarray(x, dtype=np.float32)
    ids = np.asarray(topk_ids)
    tw = np.asarray(topk_weights, dtype=np.float32)
    k = ids.shape[1]
    tokens = list(tokens)
    cache = {}

    def ops(e):
        if e not in cache:
            cache[e] = (dequant(w13, e), dequant(w2, e))
        return cache[e]

    out = np.zeros((len(tokens), x.shape[1]), dtype=np.float32)
    for i, t in enumerate(tokens):
        acc = np.zeros(x.shape[1], dtype=np.float32)
        for j in range(k):
            e = int(ids[t, j])
            W13, W2 = ops(e)
            xin = x[t:t + 1]
            if mul_topk_weights == MUL_INPUT:
                xin = weight_rows_on_input(xin, tw[t, j:j + 1])
            a = expert_gemm1_act(xin, W13, gscale_of(w13, e), bias_of(w13, e),
                                 act, layout, alpha, limit)
            rw = tw[t, j:j + 1] if mul_topk_weights == MUL_OUTPUT else None
            y = expert_gemm2(a, W2, gscale_of(w2, e), bias_of(w2, e), rw)
            acc = (acc + y[0]).astype(np.float32)
        out[i] = bf16_rne(acc)
    return out
