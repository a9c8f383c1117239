"""Routing edge cases on the GPU against the oracle, through the C ABI:
exactly tied logits (integer-valued fp32, so both sides see equal scores) and
rows with NaN, +inf and -inf logits, for both routing modes. The ids must be
bit-exact; the weights follow the oracle's non-finite reading (a NaN score
ranks as -inf, a non-finite maximum shares the weight among the logits equal
to it, all-zero sigmoid scores give 1/k each) within fp32 rounding."""
import numpy as np
import pytest
import torch

import bit_block_scaled_gb300 as moe
from gpu_helpers import OR, act_of, assert_close, built, get_config, gpu_forward, make, oracle_full, ws_status

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    return built()


def _route_gpu(logits, sel_bias, k, mode):
    T, E = logits.shape
    dev = "cuda"
    lg = torch.from_numpy(np.ascontiguousarray(logits)).to(dev)
    sb = None if sel_bias is None else torch.from_numpy(np.ascontiguousarray(sel_bias)).to(dev)
    ids = torch.empty(T, k, dtype=torch.int32, device=dev)
    tw = torch.empty(T, k, dtype=torch.float32, device=dev)
    ws = ws_status()
    moe.moe_route_topk(lg, sb, k, mode, ids, tw, ws)
    assert moe.moe_read_status(ws) == 0
    return ids.cpu().numpy(), tw.cpu().numpy()


def _edge_rows(E, rng):
    nan, inf = np.float32(np.nan), np.float32(np.inf)
    rows = [np.full(E, nan, np.float32), np.full(E, -inf, np.float32), np.zeros(E, np.float32)]
    r = rng.integers(-2, 3, E).astype(np.float32)
    r[rng.choice(E, E // 3, replace=False)] = nan
    rows.append(r)
    r = rng.integers(-2, 3, E).astype(np.float32)
    r[rng.choice(E, 2, replace=False)] = inf
    rows.append(r)
    r = rng.integers(-2, 3, E).astype(np.float32)
    r[rng.choice(E, E - 2, replace=False)] = -inf
    rows.append(r)
    r = np.full(E, nan, np.float32)
    r[rng.choice(E, 1)] = 1.0
    rows.append(r)
    return np.stack(rows)


@pytest.mark.parametrize("E,k", [(8, 2), (32, 4), (128, 4), (128, 6), (256, 8)])
def test_topk_softmax_ties_and_non_finite(E, k):
    rng = np.random.default_rng(E * 10 + k)
    ties = rng.integers(-3, 4, size=(300, E)).astype(np.float32)   # many exact ties
    logits = np.concatenate([ties, _edge_rows(E, rng)])
    ids, tw = _route_gpu(logits, None, k, OR.ROUTE_TOPK_SOFTMAX)
    rid, rw = OR.topk_softmax(logits, k)
    assert np.array_equal(ids, rid)
    assert np.all(np.isfinite(tw))
    np.testing.assert_allclose(tw, rw, rtol=2e-6, atol=1e-7)


@pytest.mark.parametrize("E,k", [(8, 2), (128, 6), (256, 8)])
def test_sigmoid_bias_ties_and_non_finite(E, k):
    rng = np.random.default_rng(E * 7 + k)
    ties = rng.integers(-3, 4, size=(300, E)).astype(np.float32)
    logits = np.concatenate([ties, _edge_rows(E, rng)])
    # zero bias and an integer-spaced bias both keep the ties exact: equal
    # logits give equal sigmoid values on both sides, and s + 0 / s + 1 are
    # the same fp32 sums on both sides
    for bias in (np.zeros(E, np.float32), rng.integers(0, 2, E).astype(np.float32)):
        ids, tw = _route_gpu(logits, bias, k, OR.ROUTE_SIGMOID_BIAS)
        rid, rw = OR.sigmoid_bias_topk(logits, bias, k)
        scores = OR.selection_scores(logits, bias)
        # exact ties are decided by id on both sides; scores closer than 2
        # ulps (different exp roundings) may swap, as in the near-tie rule
        from gpu_helpers import near_tie_ok
        assert near_tie_ok(np.nan_to_num(scores, nan=-np.inf), ids, rid) == []
        same = (ids == rid).all(axis=1)
        assert same[-7:].all()                       # the hand-made edge rows match exactly
        assert np.all(np.isfinite(tw))
        np.testing.assert_allclose(tw[same], rw[same], rtol=2e-6, atol=1e-7)


def test_forward_with_non_finite_logits_stays_finite():
    """A layer whose router logits hold NaN and +-inf rows: the fused forward
    routes them by the same reading as the oracle and the output is finite and
    within tolerance."""
    cfg = get_config("c0")
    L, N = make(cfg)
    rng = np.random.default_rng(5)
    logits = N["logits"].copy()
    logits[:7] = _edge_rows(cfg.E, rng)
    L = dict(L)
    N = dict(N)
    L["logits"] = torch.from_numpy(logits).to("cuda")
    N["logits"] = logits
    out, ws = gpu_forward(L, cfg)
    assert moe.moe_read_status(ws) == 0
    got = out.float().cpu().numpy()
    assert_close(got, oracle_full(N, cfg)["out"], "out with non-finite logits")
