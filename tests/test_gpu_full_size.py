"""Parity at the full sizes of every workload, through the C ABI, in the launch
configuration the benchmark uses (block_m 16, one stream).

* Integer steps, whole problem, bit-exact against the oracle:
  - routing ids (sigmoid routing: up to the documented 2-ulp near-tie rule);
  - sorted_token_ids, expert_offsets, block_expert_ids and row_pos.
* Routing weights, whole problem: within fp32 rounding of the oracle.
* Float steps, expert by expert: the GEMM1 + activation row `a` and the
  GEMM2 + weight row `y` of the first and last routed row of every active
  expert (its first and last token tile), a middle row of the largest expert,
  and every routed row of a few sampled tokens, whose output rows from
  moe_forward are checked too. Bound: |gpu - oracle| <= 1e-2 + 1e-2 |oracle|.
* Properties at any size:
  - moe_forward's output is finite everywhere;
  - it equals the step-by-step path bit for bit;
  - sampled x_perm rows are exact copies of their token rows.
"""
import numpy as np
import pytest
import torch

import bit_block_scaled_gb300 as moe
from gpu_helpers import (OA, OL, OR, act_of, assert_close, built, deinterleave8, get_config,
                         near_tie_ok)

pytestmark = pytest.mark.gpu

BLOCK_M = 16
# (workload, number of sampled tokens); the first and last token are always in
FULL = [("c1", 6), ("c2", 6), ("c3_t1", 1), ("c3_t32", 4), ("c3_t8192", 4), ("c4", 4)]


@pytest.fixture(scope="module", autouse=True)
def lib():
    return built()


_WEIGHTS = {}


def _layer(cfg):
    """The workload's layer on the device; the c3 sweep's token counts share
    one set of expert weights (drawn once per module)."""
    from synth.gen import make_activations, make_projection
    d = make_activations(cfg, 0, "cuda")
    base = cfg.name.split("_t")[0]
    if _WEIGHTS.get("base") != base:
        _WEIGHTS.clear()
        _WEIGHTS["base"] = base
        _WEIGHTS["w13"] = make_projection(cfg, "w13", cfg.N1, cfg.H, 0, "cuda", cfg.bias)
        _WEIGHTS["w2"] = make_projection(cfg, "w2", cfg.H, cfg.I, 0, "cuda", cfg.bias)
    d["w13"], d["w2"], d["cfg"] = _WEIGHTS["w13"], _WEIGHTS["w2"], cfg
    return d


def _host(t):
    t = t.detach().cpu()
    return t.float().numpy() if t.dtype == torch.bfloat16 else t.numpy()


def _expert_view(w, experts):
    """NumPy copy of the routed experts of one projection only (the oracle's
    dequant/gscale_of/bias_of index by expert id)."""
    v = dict(fmt=w["fmt"], E=w["E"], N=w["N"], K=w["K"], q={}, scales={}, zeros=None,
             gscale=None, bias=None)
    if w.get("zeros") is not None:
        v["zeros"] = {}
    if w.get("gscale") is not None:
        v["gscale"] = {}
    if w.get("bias") is not None:
        v["bias"] = {}
    for e in experts:
        v["q"][e] = _host(w["q"][e])
        v["scales"][e] = _host(w["scales"][e])
        if v["zeros"] is not None:
            v["zeros"][e] = _host(w["zeros"][e])
        if v["gscale"] is not None:
            v["gscale"][e] = float(w["gscale"][e])
        if v["bias"] is not None:
            v["bias"][e] = _host(w["bias"][e])
    return v


def _run_steps(L, cfg):
    """The five step entry points on device buffers (nothing copied back)."""
    T, E, k, H, I = cfg.T, cfg.E, cfg.k, cfg.H, cfg.I
    dev = "cuda"
    ws = torch.zeros(moe._lib.STATUS_BYTES, dtype=torch.uint8, device=dev)
    ids = torch.empty(T, k, dtype=torch.int32, device=dev)
    tw = torch.empty(T, k, dtype=torch.float32, device=dev)
    moe.moe_route_topk(L["logits"], L["sel_bias"], k, moe.ROUTE[cfg.route], ids, tw, ws)
    P = moe.moe_padded_rows(T, k, E, BLOCK_M)
    sorted_ids = torch.empty(P, dtype=torch.int32, device=dev)
    offs = torch.empty(E + 1, dtype=torch.int32, device=dev)
    blocks = torch.empty(P // BLOCK_M, dtype=torch.int32, device=dev)
    row_pos = torch.empty(T * k, dtype=torch.int32, device=dev)
    x_perm = torch.empty(P, H, dtype=torch.bfloat16, device=dev)
    moe.moe_align_permute(ids, E, BLOCK_M, L["x"], sorted_ids, offs, blocks, row_pos, x_perm, ws)
    a = torch.empty(P, I, dtype=torch.bfloat16, device=dev)
    moe.moe_grouped_gemm1_act(x_perm, sorted_ids, offs, T * k, L["w13"], 0, act_of(cfg), a, ws)
    y = torch.empty(P, H, dtype=torch.bfloat16, device=dev)
    moe.moe_grouped_gemm2_weighted(a, sorted_ids, offs, L["w2"], tw.reshape(-1), True, T * k, y, ws)
    out = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    moe.moe_unpermute_reduce(y, row_pos, T, k, out, ws)
    return dict(ids=ids, tw=tw, sorted=sorted_ids, offs=offs, blocks=blocks, row_pos=row_pos,
                x_perm=x_perm, a=a, y=y, out=out, status=moe.moe_read_status(ws))


@pytest.mark.parametrize("key,n_sample", FULL)
def test_full_size_workload(key, n_sample):
    cfg = get_config(key)
    T, E, k, H, I = cfg.T, cfg.E, cfg.k, cfg.H, cfg.I
    L = _layer(cfg)
    g = _run_steps(L, cfg)
    assert g["status"] == 0

    # fused entry point: same bytes as the steps, finite everywhere
    ws = torch.zeros(moe.moe_workspace_size(T, E, k, H, I, BLOCK_M), dtype=torch.uint8, device="cuda")
    out = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
    moe.moe_forward(L["x"], L["logits"], L["sel_bias"], k, moe.ROUTE[cfg.route], L["w13"], L["w2"], 0,
                    act_of(cfg), True, BLOCK_M, out, ws)
    assert moe.moe_read_status(ws) == 0
    assert torch.isfinite(out.float()).all()
    assert torch.equal(out.view(torch.int16), g["out"].view(torch.int16))

    # routing, whole problem
    logits = _host(L["logits"])
    ids = _host(g["ids"]).astype(np.int32)
    tw = _host(g["tw"])
    if cfg.route == "topk_softmax":
        rid, rw = OR.topk_softmax(logits, k)
        assert np.array_equal(ids, rid)
    else:
        sel_bias = _host(L["sel_bias"])
        rid, rw = OR.sigmoid_bias_topk(logits, sel_bias, k)
        assert near_tie_ok(OR.selection_scores(logits, sel_bias), ids, rid) == []
    same = (ids == rid).all(axis=1)
    np.testing.assert_allclose(tw[same], rw[same], rtol=2e-6, atol=1e-7)

    # alignment, whole problem, from the GPU's own ids
    o = OA.align_permute(ids, E, BLOCK_M)
    assert np.array_equal(_host(g["sorted"]), o["sorted_token_ids"])
    assert np.array_equal(_host(g["offs"]), o["expert_offsets"])
    assert np.array_equal(_host(g["blocks"]), o["block_expert_ids"])
    row_pos = _host(g["row_pos"])
    assert np.array_equal(row_pos, o["row_pos"])

    # Float steps against the oracle, expert by expert (each expert's weights
    # are copied to the host and dequantised once). Checked slots: the first
    # and the last routed row of every active expert (so every expert's first
    # and last token tile), a middle row of the largest expert, and every
    # routed row of the sampled tokens (whose output rows are checked too).
    rng = np.random.default_rng(1234)
    tokens = sorted(set([0, T - 1] + rng.choice(T, size=max(n_sample - 2, 0), replace=False).tolist()))
    srt = _host(g["sorted"])
    offs = _host(g["offs"])
    R = T * k
    real = lambda lo, hi: [p for p in range(lo, hi) if srt[p] < R]
    picked = {}
    sizes = []
    for e in range(E):
        rows = real(int(offs[e]), int(offs[e + 1]))
        if rows:
            picked.setdefault(e, set()).update({rows[0], rows[-1]})
            sizes.append((len(rows), e, rows))
    n_big, e_big, rows_big = max(sizes)
    picked[e_big].add(rows_big[len(rows_big) // 2])
    for t in tokens:
        for j in range(k):
            p = int(row_pos[t * k + j])
            picked.setdefault(int(ids[t, j]), set()).add(p)
    x = _host(L["x"])
    act = OL.ACT_SWIGLUOAI if cfg.act == "swigluoai" else OL.ACT_RELU2
    twf = tw.reshape(-1)
    y_ref_of = {}
    checked = 0
    for e, slots in sorted(picked.items()):
        slots = sorted(slots)
        w13 = _expert_view(L["w13"], [e])
        w2 = _expert_view(L["w2"], [e])
        rows = srt[slots]
        xin = x[rows // k]
        W13 = OL.dequant(w13, e)
        a_ref = OL.expert_gemm1_act(xin, W13, OL.gscale_of(w13, e), OL.bias_of(w13, e), act,
                                    OL.LAYOUT_INTERLEAVED, cfg.alpha, cfg.limit)
        del W13
        W2 = OL.dequant(w2, e)
        y_ref = OL.expert_gemm2(a_ref, W2, OL.gscale_of(w2, e), OL.bias_of(w2, e), twf[rows])
        del W2
        a_g = deinterleave8(_host(g["a"][slots]))
        y_g = _host(g["y"][slots])
        assert np.array_equal(deinterleave8(_host(g["x_perm"][slots])), xin), f"{key} x_perm rows of expert {e}"
        assert_close(a_g, a_ref, f"{key} a, expert {e}, slots {slots[:4]}")
        assert_close(y_g, y_ref, f"{key} y, expert {e}, slots {slots[:4]}")
        for p, yr in zip(slots, y_ref):
            y_ref_of[p] = yr
        checked += len(slots)
    assert len(picked) == len({int(e) for e in ids.reshape(-1)})   # every active expert
    out_g = _host(out[tokens])
    steps_g = _host(g["out"][tokens])
    for n, t in enumerate(tokens):
        y_tok = np.stack([y_ref_of[int(row_pos[t * k + j])] for j in range(k)])
        o_ref = OL.unpermute_reduce(y_tok, np.arange(k), 1, k)[0]
        assert_close(out_g[n], o_ref, f"{key} out (moe_forward), token {t}")
        assert_close(steps_g[n], o_ref, f"{key} out (steps), token {t}")
