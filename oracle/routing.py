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

Parity: pinned (invariants and brute force in tests/test_oracle_routing.py).
"""
import numpy as np

from .formats import f32


def _topk_desc(scores: np.ndarray, k: int) -> np.ndarray:
    """Indices of the k largest entries per row, descending; ties -> lower id."""
    T, E = scores.shape
    # lexsort sorts ascending by the last key first: primary key -score, then id
    ids = np.empty((T, k), dtype=np.int32)
    col = np.arange(E)
    for t in range(T):
        order = np.lexsort((col, -scores[t].astype(np.float64)))
        ids[t] = order[:k]
    return ids


def topk_softmax(logits: np.ndarray, k: int):
    """logits fp32 [T, E] -> (topk_ids int32 [T, k], topk_weights fp32 [T, k])."""
    logits = np.asarray(logits, dtype=np.float32)
    ids = _topk_desc(logits, k)
    sel = np.take_along_axis(logits, ids, axis=1).astype(np.float64)
    m = sel.max(axis=1, keepdims=True)
    ex = np.exp(sel - m)
    w = f32(ex / ex.sum(axis=1, keepdims=True))
    return ids, w


def sigmoid_f32(logits: np.ndarray) -> np.ndarray:
    """fp32 sigmoid, evaluated in float64 and rounded once."""
    l64 = np.asarray(logits, dtype=np.float32).astype(np.float64)
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
