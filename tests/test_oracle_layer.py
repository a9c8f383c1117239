"""Pins for the oracle's layer steps a3..a6 (CPU only).

A plausible mistake anywhere in the oracle (a dropped bias, a wrong sign, a
transposed operand, the wrong routing weight, the gate/up order, the nibble
order) fails at least one of these.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as Fnn

from oracle import formats as F
from oracle import layer as L
from oracle import routing as R
from synth import get_config, make_layer, to_numpy


def tiny_layer(fmt="nvfp4", act="swigluoai", T=4, E=4, k=2, H=64, I=64, seed=0,
               bias=True, route="topk_softmax"):
    cfg = get_config("c0", T=T, E=E, k=k, H=H, I=I, fmt=fmt, act=act, bias=bias,
                     route=route, sel_bias_std=0.1 if route == "sigmoid_bias" else 0.0,
                     name=f"tiny_{fmt}_{act}")
    return cfg, to_numpy(make_layer(cfg, seed))


# ----------------------------------------------------------- brute force
def _bf16(v):
    return float(F.bf16_rne(np.array([v], np.float32))[0])


def _f32(v):
    return float(np.float32(v))


def _brute_dequant(w, e):
    """Independent pure-Python decode of one expert."""
    fmt = w["fmt"]
    q = w["q"][e]
    N, K2 = q.shape
    K = 2 * K2
    lut = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    out = [[0.0] * K for _ in range(N)]
    for n in range(N):
        for kk in range(K):
            byte = int(q[n, kk // 2])
            code = (byte >> 4) if kk % 2 else (byte & 15)
            if fmt == 2:
                g = kk // 64
                zb = int(w["zeros"][e][n, g // 2])
                z = (zb >> 4) if g % 2 else (zb & 15)
                s = float(w["scales"][e][n, g])
                out[n][kk] = _bf16(_f32((code - z) * s))
                continue
            v = lut[code & 7] * (-1.0 if code & 8 else 1.0)
            if fmt == 0:
                sb = int(w["scales"][e][n, kk // 16])
                ex, m = (sb >> 3) & 15, sb & 7
                sv = (m / 8) * 2.0 ** -6 if ex == 0 else (1 + m / 8) * 2.0 ** (ex - 7)
                out[n][kk] = v * sv
            else:
                out[n][kk] = _bf16(_f32(v * 2.0 ** (int(w["scales"][e][n, kk // 32]) - 127)))
    return out


def _brute_layer(Lr, cfg, ids, tw, mul=True):
    """mul: False/0 no routing weight, True/1 on the output (GEMM2 epilogue),
    2 on the input (each routed row bf16(fp32(x * w)) before GEMM1)."""
    x = Lr["x"]
    w13, w2 = Lr["w13"], Lr["w2"]
    T, k = ids.shape
    out = []
    cache = {}
    for t in range(T):
        acc = 0.0
        row_out = [0.0] * cfg.H
        for j in range(k):
            e = int(ids[t, j])
            if e not in cache:
                cache[e] = (_brute_dequant(w13, e), _brute_dequant(w2, e))
            W13, W2 = cache[e]
            xr = [float(x[t, i]) for i in range(cfg.H)]
            if mul == 2:
                xr = [_bf16(_f32(v * float(tw[t, j]))) for v in xr]
            h = []
            for n in range(cfg.N1):
                s = _f32(math.fsum(xr[i] * W13[n][i] for i in range(cfg.H)))
                if w13["gscale"] is not None:
                    s = _f32(s * float(w13["gscale"][e]))
                if w13["bias"] is not None:
                    s = _f32(s + float(w13["bias"][e][n]))
                h.append(s)
            a = []
            for i in range(cfg.I):
                if cfg.act == "swigluoai":
                    g, u = h[2 * i], h[2 * i + 1]
                    g = min(g, 7.0)
                    u = max(-7.0, min(u, 7.0))
                    al = float(np.float32(1.702))
                    a.append(_bf16(_f32((u + 1) * g * (1 / (1 + math.exp(-al * g))))))
                else:
                    r = max(h[i], 0.0)
                    a.append(_bf16(_f32(r * r)))
            for n in range(cfg.H):
                z = _f32(math.fsum(a[i] * W2[n][i] for i in range(cfg.I)))
                if w2["gscale"] is not None:
                    z = _f32(z * float(w2["gscale"][e]))
                if w2["bias"] is not None:
                    z = _f32(z + float(w2["bias"][e][n]))
                if mul is True or mul == 1:
                    z = _f32(z * float(tw[t, j]))
                row_out[n] = _f32(row_out[n] + _bf16(z)) if j else _bf16(z)
        out.append([_bf16(v) for v in row_out])
    return np.array(out, np.float32)


@pytest.mark.parametrize("fmt,act,H,I", [
    ("nvfp4", "swigluoai", 64, 64),
    ("nvfp4", "relu2", 192, 64),
    ("mxfp4", "swigluoai", 64, 192),
    ("int4", "swigluoai", 128, 64),
    ("int4", "relu2", 64, 64),
])
def test_brute_force_tiny_layer_bit_exact(fmt, act, H, I):
    cfg, Lr = tiny_layer(fmt, act, T=3, E=4, k=2, H=H, I=I)
    r = L.moe_forward(Lr["x"], Lr["logits"], Lr["w13"], Lr["w2"], cfg.k,
                      act=L.ACT_SWIGLUOAI if act == "swigluoai" else L.ACT_RELU2)
    bf = _brute_layer(Lr, cfg, r["topk_ids"], r["topk_weights"])
    assert r["out"].shape == (cfg.T, cfg.H)
    assert np.array_equal(r["out"].view(np.uint32), bf.view(np.uint32))


# ----------------------------------------------------------- definitions
@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4", "int4"])
def test_permuted_path_equals_per_token_definition(fmt):
    cfg, Lr = tiny_layer(fmt, T=12, E=6, k=3, H=128, I=192, seed=1)
    r = L.moe_forward(Lr["x"], Lr["logits"], Lr["w13"], Lr["w2"], cfg.k, block_m=4)
    d = L.moe_forward_tokens(Lr["x"], r["topk_ids"], r["topk_weights"], Lr["w13"],
                             Lr["w2"], range(cfg.T))
    assert np.array_equal(r["out"].view(np.uint32), d.view(np.uint32))


def test_block_m_does_not_change_results():
    cfg, Lr = tiny_layer("nvfp4", T=9, E=5, k=2, H=64, I=64, seed=2)
    outs = [L.moe_forward(Lr["x"], Lr["logits"], Lr["w13"], Lr["w2"], cfg.k,
                          block_m=bm)["out"] for bm in (1, 4, 16, 64)]
    for o in outs[1:]:
        assert np.array_equal(o.view(np.uint32), outs[0].view(np.uint32))


def _dense_mlp_torch(x, W13, b13, gs13, W2, b2, gs2, I, act):
    """An expert MLP through torch.nn.functional.linear in float64."""
    xt = torch.from_numpy(x.astype(np.float64))
    W = torch.from_numpy(W13) * (1.0 if gs13 is None else float(gs13))
    h = Fnn.linear(xt, W, None if b13 is None else torch.from_numpy(b13.astype(np.float64)))
    if act == "swigluoai":
        g, u = h[:, 0::2].clamp(max=7.0), h[:, 1::2].clamp(-7.0, 7.0)
        a = (u + 1) * g * torch.sigmoid(1.702 * g)
    else:
        a = torch.relu(h) ** 2
    W2t = torch.from_numpy(W2) * (1.0 if gs2 is None else float(gs2))
    return Fnn.linear(a, W2t, None if b2 is None else torch.from_numpy(b2.astype(np.float64))).numpy()


@pytest.mark.parametrize("fmt,act", [("nvfp4", "swigluoai"), ("int4", "relu2")])
def test_top1_equals_single_dense_expert(fmt, act):
    cfg, Lr = tiny_layer(fmt, act, T=8, E=3, k=1, H=128, I=64, seed=3)
    r = L.moe_forward(Lr["x"], Lr["logits"], Lr["w13"], Lr["w2"], 1,
                      act=L.ACT_SWIGLUOAI if act == "swigluoai" else L.ACT_RELU2)
    assert np.all(r["topk_weights"] == 1.0)
    for t in range(cfg.T):
        e = int(r["topk_ids"][t, 0])
        w13, w2 = Lr["w13"], Lr["w2"]
        ref = _dense_mlp_torch(Lr["x"][t:t + 1], L.dequant(w13, e), L.bias_of(w13, e),
                               L.gscale_of(w13, e), L.dequant(w2, e), L.bias_of(w2, e),
                               L.gscale_of(w2, e), cfg.I, act)
        np.testing.assert_allclose(r["out"][t], ref[0], rtol=1.6e-2, atol=1e-3)


def test_internal_vs_external_multiply():
    cfg, Lr = tiny_layer("nvfp4", T=16, E=4, k=2, H=64, I=64, seed=4)
    ids, _ = R.topk_softmax(Lr["logits"], 2)
    n = ids.size
    # powers of two: scaling commutes with rounding -> bit-identical
    tw = np.float32(2.0) ** (-(np.arange(n) % 5) - 1).astype(np.float32).reshape(ids.shape)
    ri = L.moe_forward(Lr["x"], None, Lr["w13"], Lr["w2"], 2, topk_ids=ids,
                       topk_weights=tw, mul_topk_weights=True)
    rn = L.moe_forward(Lr["x"], None, Lr["w13"], Lr["w2"], 2, topk_ids=ids,
                       topk_weights=tw, mul_topk_weights=False)
    valid = ri["sorted_token_ids"] < n
    tw_slot = tw.reshape(-1)[ri["sorted_token_ids"][valid]]
    ext = F.bf16_rne(rn["y"][valid] * tw_slot[:, None])
    assert np.array_equal(ext.view(np.uint32), ri["y"][valid].view(np.uint32))
    # general weights: within one bf16 ulp
    _, tw2 = R.topk_softmax(Lr["logits"], 2)
    ri = L.moe_forward(Lr["x"], None, Lr["w13"], Lr["w2"], 2, topk_ids=ids,
                       topk_weights=tw2, mul_topk_weights=True)
    tw_slot = tw2.reshape(-1)[ri["sorted_token_ids"][valid]]
    ext = F.bf16_rne(rn["y"][valid] * tw_slot[:, None])
    ulp = np.abs(ri["y"][valid]) * 2.0 ** -7
    assert np.all(np.abs(ext - ri["y"][valid]) <= ulp + 1e-30)


def test_per_row_applied_ratio_is_own_weight():
    """The forensic of the Marlin bug report: y_mul / y_nomul per row must be the
    row's own routing weight; every row gets a distinct weight."""
    cfg, Lr = tiny_layer("nvfp4", T=32, E=8, k=4, H=64, I=64, seed=5)
    ids, _ = R.topk_softmax(Lr["logits"], 4)
    n = ids.size
    tw = np.linspace(0.05, 0.95, n).astype(np.float32)
    np.random.default_rng(0).shuffle(tw)
    tw = tw.reshape(ids.shape)
    ri = L.moe_forward(Lr["x"], None, Lr["w13"], Lr["w2"], 4, topk_ids=ids,
                       topk_weights=tw, mul_topk_weights=True)
    rn = L.moe_forward(Lr["x"], None, Lr["w13"], Lr["w2"], 4, topk_ids=ids,
                       topk_weights=tw, mul_topk_weights=False)
    for p, row in enumerate(ri["sorted_token_ids"]):
        if row >= n:
            continue
        m = np.abs(rn["y"][p]) > 1e-3
        ratio = np.median(ri["y"][p][m] / rn["y"][p][m])
        own = tw.reshape(-1)[row]
        assert abs(ratio - own) <= own * 2.0 ** -7
        others = np.delete(tw.reshape(-1), row)
        assert np.min(np.abs(others - ratio)) > abs(ratio - own) or np.sum(m) == 0


def test_token_permutation_permutes_output():
    cfg, Lr = tiny_layer("mxfp4", T=10, E=5, k=2, H=64, I=64, seed=6)
    r = L.moe_forward(Lr["x"], Lr["logits"], Lr["w13"], Lr["w2"], 2)
    perm = np.random.default_rng(1).permutation(cfg.T)
    rp = L.moe_forward(Lr["x"][perm], Lr["logits"][perm], Lr["w13"], Lr["w2"], 2)
    assert np.array_equal(rp["out"].view(np.uint32), r["out"][perm].view(np.uint32))


def test_all_zero_codes_closed_form():
    cfg, Lr = tiny_layer("nvfp4", T=6, E=3, k=2, H=64, I=64, seed=7)
    for w in (Lr["w13"], Lr["w2"]):
        w["q"][:] = 0
    r = L.moe_forward(Lr["x"], Lr["logits"], Lr["w13"], Lr["w2"], 2)
    b2 = Lr["w2"]["bias"]
    for t in range(cfg.T):
        acc = np.zeros(cfg.H, np.float32)
        for j in range(2):
            e = r["topk_ids"][t, j]
            acc = (acc + F.bf16_rne(b2[e] * r["topk_weights"][t, j])).astype(np.float32)
        assert np.array_equal(r["out"][t], F.bf16_rne(acc))


def test_one_hot_input_reads_one_weight_column():
    """x = e_k makes the GEMM1 pre-activation column k of W13 times the global
    scale plus the bias: pins nibble order, scale indexing and row order."""
    H, N = 32, 4
    q = np.zeros((N, H // 2), np.uint8)
    q[:, 5] = [0x71, 0x17, 0xF9, 0x2A]           # even k=10 -> low nibble, odd k=11 -> high
    scales = np.full((N, H // 16), 0x38, np.uint8)   # 1.0
    scales[2, 0] = 0x40                                # 2.0 for row 2, k < 16
    w = dict(fmt=L.FMT_NVFP4, q=q[None], scales=scales[None],
             gscale=np.array([0.5], np.float32), bias=np.array([[1, 2, 3, 4]], np.float32))
    W = L.dequant(w, 0)
    # byte -> (even k, odd k) codes: 0x71 -> (1, 7), 0x17 -> (7, 1), 0xF9 -> (9, 15),
    # 0x2A -> (10, 2); values from the printed table, row 2 carries scale 2.0
    for kk, expect in ((10, [0.5, 6.0, -0.5 * 2, -1.0]), (11, [6.0, 0.5, -6.0 * 2, 1.0])):
        x = np.zeros((1, H), np.float32)
        x[0, kk] = 1.0
        h = L.linear_epilogue(L.matvec_rows(W, x), w["gscale"][0], w["bias"][0])
        assert h[0].tolist() == [e * 0.5 + b for e, b in zip(expect, [1, 2, 3, 4])], kk


def test_gate_up_layouts_agree():
    cfg, Lr = tiny_layer("nvfp4", T=8, E=2, k=1, H=64, I=64, seed=8)
    w13 = Lr["w13"]
    conc = dict(w13)
    # INTERLEAVED rows (g0,u0,g1,u1,..) -> CONCAT rows (g0,g1,..,u0,u1,..)
    order = np.concatenate([np.arange(0, 2 * cfg.I, 2), np.arange(1, 2 * cfg.I, 2)])
    conc["q"] = w13["q"][:, order]
    conc["scales"] = w13["scales"][:, order]
    conc["bias"] = w13["bias"][:, order]
    ri = L.moe_forward(Lr["x"], Lr["logits"], w13, Lr["w2"], 1, layout=L.LAYOUT_INTERLEAVED)
    rc = L.moe_forward(Lr["x"], Lr["logits"], conc, Lr["w2"], 1, layout=L.LAYOUT_CONCAT)
    assert np.array_equal(ri["out"].view(np.uint32), rc["out"].view(np.uint32))
    # the layouts really differ: reading interleaved weights as CONCAT changes the output
    rx = L.moe_forward(Lr["x"], Lr["logits"], w13, Lr["w2"], 1, layout=L.LAYOUT_CONCAT)
    assert not np.array_equal(rx["out"], ri["out"])


def test_swigluoai_values():
    g = np.array([-1.0, 0.0, 1.0, 7.5, 100.0], np.float32)
    u = np.array([2.0, 3.0, -9.0, 0.5, 8.0], np.float32)
    a = L.swigluoai(g, u, 1.702, 7.0)
    sig = lambda z: 1.0 / (1.0 + math.exp(-z))
    al = float(np.float32(1.702))
    expect = [3 * -1 * sig(-al), 0.0, -6 * 1 * sig(al), 1.5 * 7 * sig(al * 7), 8 * 7 * sig(al * 7)]
    np.testing.assert_allclose(a, np.array(expect, np.float32), rtol=1e-7)


def test_unpadded_output_shape():
    cfg, Lr = tiny_layer("nvfp4", T=5, E=3, k=2, H=192, I=64, seed=9)
    r = L.moe_forward(Lr["x"], Lr["logits"], Lr["w13"], Lr["w2"], 2)
    assert r["out"].shape == (5, 192) and r["y"].shape[1] == 192
    assert r["out"].strides == (192 * 4, 4)


@pytest.mark.parametrize("fmt,act,H,I", [
    ("nvfp4", "swigluoai", 64, 64),
    ("mxfp4", "relu2", 64, 128),
    ("int4", "swigluoai", 128, 64),
])
def test_brute_force_routing_weight_on_input(fmt, act, H, I):
    """mul_topk_weights = 2 (the weight applied to each routed row's input)
    against the pure-Python loops, bit for bit; and the mode differs from the
    output multiply (swigluoai and ReLU^2 are not linear)."""
    cfg, Lr = tiny_layer(fmt, act, T=3, E=4, k=2, H=H, I=I)
    a = L.ACT_SWIGLUOAI if act == "swigluoai" else L.ACT_RELU2
    r = L.moe_forward(Lr["x"], Lr["logits"], Lr["w13"], Lr["w2"], cfg.k, act=a, mul_topk_weights=2)
    bf = _brute_layer(Lr, cfg, r["topk_ids"], r["topk_weights"], mul=2)
    assert np.array_equal(r["out"].view(np.uint32), bf.view(np.uint32))
    r1 = L.moe_forward(Lr["x"], Lr["logits"], Lr["w13"], Lr["w2"], cfg.k, act=a, mul_topk_weights=True)
    assert not np.array_equal(r["out"], r1["out"])
    toks = L.moe_forward_tokens(Lr["x"], r["topk_ids"], r["topk_weights"], Lr["w13"], Lr["w2"],
                                range(cfg.T), act=a, mul_topk_weights=2)
    assert np.array_equal(toks.view(np.uint32), r["out"].view(np.uint32))


def test_unit_weights_on_input_equal_no_weight():
    """With every routing weight exactly 1 the input multiply is the identity:
    on-input, on-output and no weighting give the same bits."""
    cfg, Lr = tiny_layer("nvfp4", "swigluoai", T=4, E=4, k=2, H=64, I=64)
    r0 = L.moe_forward(Lr["x"], Lr["logits"], Lr["w13"], Lr["w2"], cfg.k, mul_topk_weights=False)
    ones = np.ones_like(r0["topk_weights"])
    outs = [L.moe_forward(Lr["x"], None, Lr["w13"], Lr["w2"], cfg.k, mul_topk_weights=m,
                          topk_ids=r0["topk_ids"], topk_weights=ones)["out"] for m in (0, 1, 2)]
    assert all(np.array_equal(o.view(np.uint32), outs[0].view(np.uint32)) for o in outs)


@pytest.mark.parametrize("fmt,act", [("nvfp4", "swigluoai"), ("mxfp4", "swigluoai"), ("int4", "relu2")])
def test_float32_accumulation_mode_within_tolerance_of_float64(fmt, act):
    """The timed CPU baseline runs the oracle with float32 accumulation. It
    computes the same layer: integer outputs are identical, and every float
    output is within the layer's tolerance |d| <= 1e-2 + 1e-2 |ref| of the
    float64 parity mode (fp32 sums over K = 512 differ from the float64 sum by
    far less than one bf16 ulp of the result, so R1..R3 flip an ulp at most)."""
    cfg, N = tiny_layer(fmt=fmt, act=act, T=48, E=6, k=2, H=512, I=384, seed=21)
    args = (N["x"], N["logits"], N["w13"], N["w2"], cfg.k)
    kw = dict(act=L.ACT_SWIGLUOAI if act == "swigluoai" else L.ACT_RELU2)
    r64 = L.moe_forward(*args, **kw)
    r32 = L.moe_forward(*args, acc_dtype=np.float32, **kw)
    for key in ("topk_ids", "sorted_token_ids", "expert_offsets", "row_pos"):
        assert np.array_equal(r32[key], r64[key])
    for key in ("a", "y", "out"):
        err = np.abs(r32[key] - r64[key])
        assert np.all(err <= 1e-2 + 1e-2 * np.abs(r64[key])), key
    # not a silent copy of the float64 path: the sums really are fp32
    acc64 = L.matvec_rows(L.dequant(N["w13"], 0), N["x"][:8])
    acc32 = L.matvec_rows(L.dequant(N["w13"], 0), N["x"][:8], np.float32)
    assert acc32.dtype == np.float32 and not np.array_equal(acc32, acc64)
    np.testing.assert_allclose(acc32, acc64, rtol=1e-4, atol=1e-4)
