"""Top-k routing (step a1 of the layer).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

Two routing modes:

* ``topk_softmax`` (gpt-oss): per token, take the k largest router logits
  (descending; equal values -> lower expert id first), then a softmax over the
  k selected logits. The repro in the vLLM issue "moe_wna16_marlin_gemm applies
  wrong per-row topk weights", section "Minimal repro", instead takes the
  softmax over all E experts and then top-k without renormalising; both pick
  the same experts, and renormalising the repro's weights gives exactly these
  weights (a pinned invariant). The softmax is evaluated in float64 and
  rounded once to float32.

* ``sigmoid_bias_topk`` (Nemotron-3-Nano): the vLLM issue "NVFP4 MoE monolithic
  backend ... Nemotron-3-Nano", section Environment and Analysis item 3, names
  fp32 sigmoid + per-expert bias grouped top-k with n_group = 1 (a plain
  top-k over all experts). Reading taken: s = sigmoid(logit) rounded to fp32;
  the selection score is the fp32 sum s + bias; the weights are the selected
  s renormalised to sum 1 (the bias never enters the weights); no extra
  routed scaling factor.

Non-finite scores (the pages say nothing about them; the reading taken, the
same on both sides): a NaN selection score ranks as -inf, and equal scores
(two -inf included) go to the lower expert id. The softmax over the selected
logits is exp(l_j - max) / sum when the largest selected logit is finite; when
it is +inf or -inf, the selected logits equal to it share the weight equally
(the limit of the softmax as those logits grow or fall together) and the rest
get 0; a NaN logit weighs as -inf. Sigmoid routing weighs a NaN logit as
s = 0 (the sigmoid of -inf); if every selected s is 0, each of the k weights
is 1/k.

Parity: pinned (invariants, brute force and the non-finite limits in
tests/test_oracle_routing_align.py).
"""
import numpy as np

from .formats import f32


def _nan_as_neg_inf(v: np.ndarray) -> np.ndarray:
    v = np.asarray(v, dtype=np.float64).copy()
    v[np.isnan(v)] = -np.inf
    return v


def _topk_desc(scores: np.ndarray, k: int) -> np.ndarray:
    """Indices of the k largest entries per row, descending; ties -> lower id;
    a NaN score ranks as -inf."""
    T, E = scores.shape
    # lexsort sorts ascending by the last key first: primary key -score, then id
    ids = np.empty((T, k), dtype=np.int32)
    col = np.arange(E)
    for t in range(T):
        order = np.lexsort((col, -_nan_as_neg_inf(scores[t])))
        ids[t] = order[:k]
    return ids


def _softmax_selected(sel: np.ndarray) -> np.ndarray:
    """Softmax of each row of selected logits (float64), with the limits
    above for a non-finite maximum and NaN weighed as -inf."""
    sel = _nan_as_neg_inf(sel)
    m = sel.max(axis=1, keepdims=True)
    finite = np.isfinite(m)
    with np.errstate(invalid="ignore"):
        ex = np.where(finite, np.exp(np.where(finite, sel - m, 0.0)), (sel == m).astype(np.float64))
    return ex / ex.sum(axis=1, keepdims=True)


def topk_softmax(logits: np.ndarray, k: int):
    """logits fp32 [T, E] -> (topk_ids int32 [T, k], topk_weights fp32 [T, k])."""
    logits = np.asarray(logits, dtype=np.float32)
    ids = _topk_desc(logits, k)
    sel = np.take_along_axis(logits, ids, axis=1).astype(np.float64)
    w = f32(_softmax_selected(sel))
    return ids, w


def sigmoid_f32(logits: np.ndarray) -> np.ndarray:
    """fp32 sigmoid, evaluated in float64 and rounded once."""
    l64 = np.asarray(logits, dtype=np.float32).astype(np.float64)
    with np.errstate(over="ignore", invalid="ignore"):
        return f32(1.0 / (1.0 + np.exp(-l64)))


def selection_scores(logits: np.ndarray, sel_bias: np.ndarray) -> np.ndarray:
    """fp32 selection score s + bias used by ``sigmoid_bias_topk``."""
    s = sigmoid_f32(logits)
    return (s + np.asarray(sel_bias, dtype=np.float32)[None, :]).astype(np.float32)


def sigmoid_bias_topk(logits: np.ndarray, sel_bias: np.ndarray, k: int):
    """logits fp32 [T, E], sel_bias fp32 [E] -> (ids int32 [T,k], weights fp32 [T,k])."""
    s = sigmoid_f32(logits)
    score = selection_scores(logits, sel_bias)
    ids = _topk_desc(score, k)
    s_sel = np.take_along_axis(s, ids, axis=1).astype(np.float64)
    s_sel[np.isnan(s_sel)] = 0.0                      # a NaN logit weighs as s = 0
    tot = s_sel.sum(axis=1, keepdims=True)
    s_sel = np.where(tot == 0.0, 1.0, s_sel)          # all zero: equal weights
    w = f32(s_sel / s_sel.sum(axis=1, keepdims=True))
    return ids, w


ROUTE_TOPK_SOFTMAX = 0
ROUTE_SIGMOID_BIAS = 1


def route(logits, k, mode=ROUTE_TOPK_SOFTMAX, sel_bias=None):
    if mode == ROUTE_TOPK_SOFTMAX:
        return topk_softmax(logits, k)
    if mode == ROUTE_SIGMOID_BIAS:
        return sigmoid_bias_topk(logits, sel_bias, k)
    raise ValueError(f"unknown routing mode {mode}")
