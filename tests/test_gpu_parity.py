"""GPU parity: every step of the CUDA path through the C ABI against the oracle.

Integer work (routing ids, sorted ids, offsets, block ids, row positions, the
x_perm gather) must be bit-exact; floating-point outputs must satisfy
|gpu - oracle| <= 1e-2 + 1e-2 |oracle| with no NaN/Inf.
"""
import numpy as np
import pytest
import torch

from gpu_helpers import (OR, act_of, assert_close, built, get_config, gpu_forward, gpu_steps, interleave8,
                         make, near_tie_ok, oracle_full, ws_status)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    return built()


def _check_steps(g, o, cfg, exact_routing=True):
    if exact_routing:
        assert np.array_equal(g["topk_ids"], o["topk_ids"])
    np.testing.assert_allclose(g["topk_weights"], o["topk_weights"], rtol=2e-6, atol=1e-7)
    assert np.array_equal(g["sorted_token_ids"], o["sorted_token_ids"])
    assert np.array_equal(g["expert_offsets"], o["expert_offsets"])
    assert np.array_equal(g["block_expert_ids"], o["block_expert_ids"])
    assert np.array_equal(g["row_pos"], o["row_pos"])
    used = int(o["expert_offsets"][-1])
    assert np.array_equal(g["x_perm"][:used], o["x_perm"][:used])
    valid = o["sorted_token_ids"] < cfg.T * cfg.k
    assert_close(g["a"][valid], o["a"][valid], "a (GEMM1 + act)")
    assert_close(g["y"][valid], o["y"][valid], "y (GEMM2 + weight)")
    assert_close(g["out"], o["out"], "out")
    assert g["status"] == 0


def test_c0_tiny_layer_steps():
    cfg = get_config("c0")
    L, N = make(cfg)
    g = gpu_steps(L, cfg)
    o = oracle_full(N, cfg)
    _check_steps(g, o, cfg)


def test_c0_forward_matches_steps_bit_exact():
    cfg = get_config("c0")
    L, N = make(cfg)
    g = gpu_steps(L, cfg)
    out, ws = gpu_forward(L, cfg)
    assert np.array_equal(out.float().cpu().numpy(), g["out"])


def test_gemm2_from_oracle_intermediates():
    """The minimum slice: GEMM2 fed with the oracle's own a and metadata."""
    import bit_block_scaled_gb300 as moe
    cfg = get_config("c0")
    L, N = make(cfg)
    o = oracle_full(N, cfg)
    dev = "cuda"
    # the library stores a with the columns of each group of 8 interleaved
    a = torch.from_numpy(np.ascontiguousarray(interleave8(o["a"]))).to(torch.bfloat16).to(dev)
    sorted_ids = torch.from_numpy(o["sorted_token_ids"]).to(dev)
    offs = torch.from_numpy(o["expert_offsets"]).to(dev)
    tw = torch.from_numpy(o["topk_weights"].reshape(-1)).to(dev)
    y = torch.zeros(a.shape[0], cfg.H, dtype=torch.bfloat16, device=dev)
    ws = ws_status()
    moe.moe_grouped_gemm2_weighted(a, sorted_ids, offs, L["w2"], tw, 1, cfg.T * cfg.k, y, ws)
    valid = o["sorted_token_ids"] < cfg.T * cfg.k
    assert_close(y.float().cpu().numpy()[valid], o["y"][valid], "y")
    assert moe.moe_read_status(ws) == 0


FORMATS = [
    # fmt, act, H, I, E, T, k, layout
    ("nvfp4", "swigluoai", 320, 192, 5, 37, 2, 0),
    ("nvfp4", "swigluoai", 320, 192, 5, 37, 2, 1),
    ("nvfp4", "relu2", 192, 320, 6, 29, 3, 0),
    ("mxfp4", "swigluoai", 384, 256, 4, 41, 2, 0),
    ("mxfp4", "swigluoai", 384, 256, 4, 41, 2, 1),
    ("mxfp4", "relu2", 256, 192, 7, 23, 2, 0),
    ("int4", "swigluoai", 320, 256, 5, 33, 2, 0),
    ("int4", "relu2", 448, 192, 4, 19, 3, 0),
]


@pytest.mark.parametrize("fmt,act,H,I,E,T,k,layout", FORMATS)
def test_formats_and_activations(fmt, act, H, I, E, T, k, layout):
    import bit_block_scaled_gb300 as moe
    route = "sigmoid_bias" if act == "relu2" else "topk_softmax"
    cfg = get_config("c0", name=f"fmt_{fmt}_{act}_{H}_{I}", fmt=fmt, act=act, H=H, I=I, E=E, T=T,
                     k=k, route=route, sel_bias_std=0.1 if route == "sigmoid_bias" else 0.0,
                     bias=(act == "swigluoai"))
    L, N = make(cfg, seed=3)
    if layout == 1:
        # the same weights stored [gate; up]
        idx = torch.cat([torch.arange(0, 2 * I, 2), torch.arange(1, 2 * I, 2)]).cuda()
        w = dict(L["w13"])
        for key in ("q", "scales", "zeros", "bias"):
            if w.get(key) is not None:
                w[key] = w[key][:, idx].contiguous()
        L = dict(L)
        L["w13"] = w
    g = gpu_steps(L, cfg, layout=layout)
    ids = g["topk_ids"].astype(np.int32)
    o = oracle_full(N, cfg, ids=ids, tw=g["topk_weights"])
    oref = oracle_full(N, cfg)
    if cfg.route == "sigmoid_bias":
        scores = OR.selection_scores(N["logits"], N["sel_bias"])
        assert near_tie_ok(scores, ids, oref["topk_ids"]) == []
    else:
        assert np.array_equal(ids, oref["topk_ids"])
    np.testing.assert_allclose(g["topk_weights"], oref["topk_weights"], rtol=2e-6, atol=1e-7) \
        if np.array_equal(ids, oref["topk_ids"]) else None
    _check_steps(g, o, cfg, exact_routing=False)
    # the fused forward (f16 operands for NVFP4 / MXFP4) in the same layout
    out, ws = gpu_forward(L, cfg, layout=layout)
    assert moe.moe_read_status(ws) == 0
    assert_close(out.float().cpu().numpy(), o["out"], f"fused out ({fmt}, {act}, layout {layout})")


def test_c1_decode_layer_full():
    cfg = get_config("c1")
    L, N = make(cfg)
    g = gpu_steps(L, cfg)
    o = oracle_full(N, cfg)
    _check_steps(g, o, cfg)


@pytest.mark.parametrize("block_m", [16, 32, 64, 128, 256])
def test_block_m_sweep_same_output(block_m):
    cfg = get_config("c0", name="bm_sweep", T=40, E=6, k=2, H=192, I=128)
    L, N = make(cfg, seed=5)
    out, ws = gpu_forward(L, cfg, block_m=block_m)
    ref, _ = gpu_forward(L, cfg, block_m=16)
    assert np.array_equal(out.float().cpu().numpy(), ref.float().cpu().numpy())


def test_determinism_bit_identical():
    cfg = get_config("c0", name="det", T=300, E=8, k=2, H=256, I=192)
    L, N = make(cfg, seed=6)
    a, _ = gpu_forward(L, cfg)
    b, _ = gpu_forward(L, cfg)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_one_expert_takes_all_rows_spans_tiles():
    """All 600 routed rows on expert 2: the token dimension splits into several
    tiles of at most 256 rows with a ragged last tile."""
    cfg = get_config("c0", name="hot", T=300, E=4, k=2, H=192, I=128)
    L, N = make(cfg, seed=7)
    L["logits"][:, 2] += 100.0
    N["logits"][:, 2] += 100.0
    g = gpu_steps(L, cfg)
    o = oracle_full(N, cfg)
    _check_steps(g, o, cfg)


def test_top1_and_top8():
    for k, E in ((1, 4), (8, 16)):
        cfg = get_config("c0", name=f"k{k}", T=21, E=E, k=k, H=128, I=128)
        L, N = make(cfg, seed=8)
        g = gpu_steps(L, cfg)
        o = oracle_full(N, cfg)
        _check_steps(g, o, cfg)
        if k == 1:
            assert np.all(g["topk_weights"] == 1.0)


def test_external_multiply_and_applied_ratio():
    """mul_topk_weights=False + external multiply agrees with the fused
    multiply within one bf16 ulp, and the ratio y_mul / y_nomul of every row is
    that row's own routing weight (the Marlin forensic)."""
    cfg = get_config("c0", name="ratio", T=32, E=32, k=4, H=2880, I=256)
    L, N = make(cfg, seed=9)
    gm = gpu_steps(L, cfg, mul=True)
    gn = gpu_steps(L, cfg, mul=False)
    R = cfg.T * cfg.k
    tw = gm["topk_weights"].reshape(-1)
    for p, row in enumerate(gm["sorted_token_ids"]):
        if row >= R:
            continue
        ym, yn = gm["y"][p], gn["y"][p]
        ext = (yn * tw[row]).astype(np.float32)
        assert np.all(np.abs(ext - ym) <= np.abs(ym) * 2.0 ** -7 + 1e-6)
        m = np.abs(yn) > 1e-3
        ratio = np.median(ym[m] / yn[m])
        assert abs(ratio - tw[row]) <= tw[row] * 2.0 ** -7


def test_output_shape_stride_and_canary():
    import bit_block_scaled_gb300 as moe
    cfg = get_config("c0", name="canary", T=9, E=4, k=2, H=2880, I=128)
    L, N = make(cfg, seed=10)
    nbytes = moe.moe_workspace_size(cfg.T, cfg.E, cfg.k, cfg.H, cfg.I, 16)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    buf = torch.full((cfg.T * cfg.H + 4096,), -7.0, dtype=torch.bfloat16, device="cuda")
    out = buf[:cfg.T * cfg.H].view(cfg.T, cfg.H)
    moe.moe_forward(L["x"], L["logits"], None, cfg.k, 0, L["w13"], L["w2"], 0,
                    moe.act("swigluoai"), 1, 16, out, ws)
    torch.cuda.synchronize()
    assert out.shape == (9, 2880) and out.stride() == (2880, 1)
    assert torch.all(buf[cfg.T * cfg.H:] == -7.0)
    o = oracle_full(N, cfg)
    assert_close(out.float().cpu().numpy(), o["out"], "out")


def test_empty_batch_is_a_no_op():
    import bit_block_scaled_gb300 as moe
    cfg = get_config("c0", name="empty", T=0, E=4, k=2, H=128, I=128)
    L, N = make(cfg)
    nbytes = moe.moe_workspace_size(0, 4, 2, 128, 128, 16)
    ws = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device="cuda")
    out = torch.empty(0, 128, dtype=torch.bfloat16, device="cuda")
    moe.moe_forward(L["x"], L["logits"], None, 2, 0, L["w13"], L["w2"], 0, moe.act(), 1, 16, out, ws)
    assert moe.moe_last_launch_count() == 0
    assert moe.moe_read_status(ws) == 0


def test_bad_expert_id_latches_status():
    import bit_block_scaled_gb300 as moe
    T, k, E, H = 8, 2, 4, 128
    ids = torch.tensor([[0, 1]] * T, dtype=torch.int32, device="cuda")
    ids[3, 1] = 9                       # out of range
    ids[5, 0] = -2
    x = torch.randn(T, H, device="cuda").to(torch.bfloat16)
    P = moe.moe_padded_rows(T, k, E, 16)
    sorted_ids = torch.empty(P, dtype=torch.int32, device="cuda")
    offs = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    blocks = torch.empty(P // 16, dtype=torch.int32, device="cuda")
    row_pos = torch.empty(T * k, dtype=torch.int32, device="cuda")
    x_perm = torch.empty(P, H, dtype=torch.bfloat16, device="cuda")
    ws = ws_status()
    moe.moe_align_permute(ids, E, 16, x, sorted_ids, offs, blocks, row_pos, x_perm, ws)
    st = moe.moe_read_status(ws)
    assert st == 5, moe.moe_status_string(st)
    rp = row_pos.cpu().numpy()
    assert rp[3 * 2 + 1] == -1 and rp[5 * 2] == -1
    # the valid rows are still placed
    assert int(offs[-1]) == 32
    moe.moe_clear_status(ws)
    assert moe.moe_read_status(ws) == 0


def test_invalid_arguments_rejected_on_host():
    import bit_block_scaled_gb300 as moe
    cfg = get_config("c0")
    L, N = make(cfg)
    out = torch.empty(cfg.T, cfg.H, dtype=torch.bfloat16, device="cuda")
    ws = torch.zeros(moe.moe_workspace_size(cfg.T, cfg.E, cfg.k, cfg.H, cfg.I, 16), dtype=torch.uint8,
                     device="cuda")
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_forward(L["x"], L["logits"], None, cfg.k, 0, L["w13"], L["w2"], 0, moe.act(), 1, 24,
                        out, ws)
    assert ei.value.code == 1
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_forward(L["x"], L["logits"], None, cfg.k, 0, L["w13"], L["w2"], 0, moe.act(), 1, 16,
                        out, ws[:1024])
    assert ei.value.code == 6
    big = torch.empty(cfg.T * cfg.H + 8, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(moe.MoeError) as ei:   # output 2 bytes off a 16-byte boundary
        moe.moe_forward(L["x"], L["logits"], None, cfg.k, 0, L["w13"], L["w2"], 0, moe.act(), 1, 16,
                        big[1:1 + cfg.T * cfg.H].view(cfg.T, cfg.H), ws)
    assert ei.value.code == 1


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4", "int4"])
def test_dequantised_weights_bit_exact(fmt):
    """GEMM2 with one-hot activation rows, no bias and no routing weight reads
    single dequantised weights out of the kernel: y[p, n] = W2'[e, n, k_p]
    (one exact product, then a bf16 value rounded to bf16 again). Every value
    must equal the oracle's R0 operand bit for bit."""
    import bit_block_scaled_gb300 as moe
    from oracle import layer as OLm
    cfg = get_config("c0", name=f"onehot_{fmt}", fmt=fmt, T=64, E=2, k=1, H=320, I=192, bias=False)
    L, N = make(cfg, seed=11)
    E, H, I = cfg.E, cfg.H, cfg.I
    rows = 64
    ks = (np.arange(rows) * 37) % I                 # column picked by each row
    a = np.zeros((rows, I), np.float32)
    a[np.arange(rows), ks] = 1.0
    experts = np.arange(rows) % E
    order = np.argsort(experts, kind="stable")      # group rows by expert
    a, ks, experts = a[order], ks[order], experts[order]
    offs = np.zeros(E + 1, np.int32)
    offs[1:] = np.cumsum(np.bincount(experts, minlength=E))
    dev = "cuda"
    a_dev = torch.from_numpy(np.ascontiguousarray(interleave8(a))).to(torch.bfloat16).to(dev)
    sorted_ids = torch.arange(rows, dtype=torch.int32, device=dev)
    offs_dev = torch.from_numpy(offs).to(dev)
    tw = torch.ones(rows, dtype=torch.float32, device=dev)
    y = torch.zeros(rows, H, dtype=torch.bfloat16, device=dev)
    ws = ws_status()
    moe.moe_grouped_gemm2_weighted(a_dev, sorted_ids, offs_dev, L["w2"], tw, False, rows, y, ws)
    assert moe.moe_read_status(ws) == 0
    got = y.float().cpu().numpy()
    for e in range(E):
        W = OLm.dequant(N["w2"], e).astype(np.float32)          # [H, I]
        gs = OLm.gscale_of(N["w2"], e)
        for p in np.nonzero(experts == e)[0]:
            ref = W[:, ks[p]]
            if gs is not None:   # NVFP4: the per-expert global scale multiplies the accumulator
                ref = OLm.bf16_rne((ref.astype(np.float32) * np.float32(gs)).astype(np.float32))
            assert np.array_equal(got[p], ref), (fmt, e, p, np.nonzero(got[p] != ref)[0][:5])


# few routed rows spread over many experts (mostly one or two rows per
# expert): narrow token tiles, many experts with no rows at all
SMALL = [
    # fmt, act, H, I, E, T, k, layout
    ("nvfp4", "swigluoai", 320, 192, 32, 3, 2, 0),
    ("nvfp4", "swigluoai", 320, 192, 32, 3, 2, 1),
    ("nvfp4", "relu2", 192, 320, 24, 5, 3, 0),
    ("mxfp4", "swigluoai", 384, 256, 64, 1, 4, 0),
    ("mxfp4", "relu2", 256, 192, 16, 4, 2, 0),
    ("int4", "swigluoai", 320, 256, 40, 6, 4, 0),
    ("int4", "relu2", 448, 192, 20, 2, 3, 0),
]


@pytest.mark.parametrize("fmt,act,H,I,E,T,k,layout", SMALL)
def test_small_batch_many_experts(fmt, act, H, I, E, T, k, layout):
    test_formats_and_activations(fmt, act, H, I, E, T, k, layout)


def test_fused_f16_operands_large_activation_rows():
    """moe_forward feeds NVFP4 swigluoai layers to the tensor cores as f16
    operands, each token row scaled by a power of two into f16 range. Rows far
    outside f16 range (|x| up to 1e9) must still match the oracle."""
    cfg = get_config("c0", name="bigx", T=24, E=8, k=2, H=256, I=256)
    L, N = make(cfg, seed=12)
    scale = torch.ones(cfg.T, 1, device="cuda")
    scale[3] = 1e9
    scale[7] = 7e4
    scale[11] = 3e-3
    L = dict(L)
    L["x"] = (L["x"].float() * scale).to(torch.bfloat16)
    N = dict(N)
    N["x"] = L["x"].float().cpu().numpy()
    out, ws = gpu_forward(L, cfg)
    import bit_block_scaled_gb300 as moe
    assert moe.moe_read_status(ws) == 0
    o = oracle_full(N, cfg)
    assert_close(out.float().cpu().numpy(), o["out"], "out with large rows")


def test_forward_profile_matches_forward():
    """moe_forward_profile runs the same kernels as moe_forward (same output
    bytes) and reports a positive device time for each of the six."""
    import bit_block_scaled_gb300 as moe
    cfg = get_config("c0")
    L, N = make(cfg)
    ref, _ = gpu_forward(L, cfg)
    ws = torch.zeros(moe.moe_workspace_size(cfg.T, cfg.E, cfg.k, cfg.H, cfg.I, 16), dtype=torch.uint8,
                     device="cuda")
    out = torch.empty(cfg.T, cfg.H, dtype=torch.bfloat16, device="cuda")
    ms = moe.moe_forward_profile(L["x"], L["logits"], L["sel_bias"], cfg.k, moe.ROUTE[cfg.route], L["w13"],
                                 L["w2"], 0, act_of(cfg), True, 16, out, ws)
    assert set(ms) == {"route", "align", "gather", "gemm1", "gemm2", "unpermute"}
    assert all(v > 0 for v in ms.values())
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    assert moe.moe_read_status(ws) == 0


def test_fused_nvfp4_relu2_matches_oracle():
    """moe_forward on an NVFP4 ReLU^2 layer (f16 operands in GEMM1 only, a
    kept in bf16) against the oracle, with sigmoid + bias routing."""
    cfg = get_config("c0", name="relu2_fused", fmt="nvfp4", act="relu2", H=192, I=320, E=6, T=29, k=3,
                     route="sigmoid_bias", sel_bias_std=0.1, bias=False)
    L, N = make(cfg, seed=13)
    g = gpu_steps(L, cfg)
    out, ws = gpu_forward(L, cfg)
    import bit_block_scaled_gb300 as moe
    assert moe.moe_read_status(ws) == 0
    o = oracle_full(N, cfg, ids=g["topk_ids"].astype(np.int32), tw=g["topk_weights"])
    assert_close(out.float().cpu().numpy(), o["out"], "fused relu2 out")
    assert_close(out.float().cpu().numpy(), g["out"], "fused vs steps", atol=1e-3, rtol=1e-3)


# w13 and w2 in different formats: GEMM2 runs on f16 operands only when GEMM1
# wrote a as f16, so every combination must hand a over in the layout the
# second GEMM reads
MIXED = [
    # fmt of w13, fmt of w2, act
    ("nvfp4", "int4", "swigluoai"),
    ("nvfp4", "mxfp4", "swigluoai"),
    ("mxfp4", "nvfp4", "swigluoai"),
    ("int4", "mxfp4", "swigluoai"),
    ("mxfp4", "int4", "relu2"),
]


@pytest.mark.parametrize("f13,f2,act", MIXED)
def test_fused_mixed_weight_formats(f13, f2, act):
    import bit_block_scaled_gb300 as moe
    from synth import make_layer, to_numpy
    base = dict(name=f"mixed_{f13}_{f2}", act=act, H=320, I=256, E=6, T=21, k=2)
    cfg13 = get_config("c0", fmt=f13, **base)
    cfg2 = get_config("c0", fmt=f2, **base)
    L = dict(make_layer(cfg13, 17, device="cuda"))
    L["w2"] = make_layer(cfg2, 17, device="cuda")["w2"]
    N = to_numpy(L)
    g = gpu_steps(L, cfg13)
    out, ws = gpu_forward(L, cfg13)
    assert moe.moe_read_status(ws) == 0
    o = oracle_full(N, cfg13, ids=g["topk_ids"].astype(np.int32), tw=g["topk_weights"])
    assert_close(out.float().cpu().numpy(), o["out"], f"fused out, w13 {f13}, w2 {f2}")
    assert_close(g["out"], o["out"], f"steps out, w13 {f13}, w2 {f2}")


def test_fused_mxfp4_f16_scale_range():
    """The fused forward runs MXFP4 layers on f16 operands, each E8M0 scale
    folded by 2^12 into f16 range: the largest accepted exponent (128, a scale
    of 2) must not overflow, and exponents down to 92 stay exact; 91 and below
    lose bits or vanish, which is far inside the tolerance."""
    import bit_block_scaled_gb300 as moe
    from synth import make_layer, to_numpy
    cfg = get_config("c0", name="mx_range", fmt="mxfp4", H=256, I=192, E=4, T=12, k=2)
    L = dict(make_layer(cfg, 3, device="cuda"))
    for key in ("w13", "w2"):
        w = dict(L[key])
        sc = w["scales"].clone()
        sc[0, :16, 0] = 128
        sc[1, :16, 1] = 127
        sc[1, 16:32, 0] = 92
        sc[2, :16, 2] = 91
        sc[3, :16, 1] = 60
        w["scales"] = sc
        L[key] = w
    N = to_numpy(L)
    out, ws = gpu_forward(L, cfg)
    assert moe.moe_read_status(ws) == 0
    o = oracle_full(N, cfg)
    assert_close(out.float().cpu().numpy(), o["out"], "mxfp4 f16 path, extreme scales")


@pytest.mark.parametrize("fmt,act", [("nvfp4", "swigluoai"), ("mxfp4", "relu2"), ("int4", "swigluoai"),
                                     ("mxfp4", "swigluoai")])
def test_routing_weight_on_input(fmt, act):
    """mul_topk_weights = 2: each routed row enters GEMM1 as bf16(x * w) with
    its own routing weight and GEMM2 does not multiply (bf16 and f16 gathers)."""
    import bit_block_scaled_gb300 as moe
    cfg = get_config("c0", name=f"on_input_{fmt}_{act}", fmt=fmt, act=act, H=320, I=256, E=8, T=37, k=3)
    L, N = make(cfg, seed=31)
    g = gpu_steps(L, cfg)
    ws = torch.zeros(moe.moe_workspace_size(cfg.T, cfg.E, cfg.k, cfg.H, cfg.I, 16), dtype=torch.uint8,
                     device="cuda")
    out = torch.empty(cfg.T, cfg.H, dtype=torch.bfloat16, device="cuda")
    moe.moe_forward(L["x"], L["logits"], L["sel_bias"], cfg.k, moe.ROUTE[cfg.route], L["w13"], L["w2"], 0,
                    act_of(cfg), 2, 16, out, ws)
    assert moe.moe_read_status(ws) == 0
    o = oracle_full(N, cfg, ids=g["topk_ids"].astype(np.int32), tw=g["topk_weights"], mul=2)
    assert_close(out.float().cpu().numpy(), o["out"], f"on-input out ({fmt}, {act})")
    o1 = oracle_full(N, cfg, ids=g["topk_ids"].astype(np.int32), tw=g["topk_weights"], mul=True)
    assert not np.allclose(o["out"], o1["out"])  # the two settings really differ here
    with pytest.raises(moe.MoeError) as e:
        moe.moe_forward(L["x"], L["logits"], L["sel_bias"], cfg.k, moe.ROUTE[cfg.route], L["w13"], L["w2"], 0,
                        act_of(cfg), 3, 16, out, ws)
    assert e.value.code == 1


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4", "int4"])
def test_maximum_sizes(fmt):
    """The largest sizes the ABI accepts: 256 experts with top-8 routing, and
    H = I = 4096 (256-byte NVFP4 scale rows, 16 K stages of 256 per tile),
    each through the steps and the fused forward."""
    import bit_block_scaled_gb300 as moe
    for name, T, E, k, H, I in (("maxE", 40, 256, 8, 128, 128), ("maxH", 9, 2, 2, 4096, 4096)):
        cfg = get_config("c0", name=f"{name}_{fmt}", fmt=fmt, T=T, E=E, k=k, H=H, I=I)
        L, N = make(cfg, seed=41)
        g = gpu_steps(L, cfg)
        o = oracle_full(N, cfg)
        _check_steps(g, o, cfg)
        out, ws = gpu_forward(L, cfg)
        assert moe.moe_read_status(ws) == 0
        assert_close(out.float().cpu().numpy(), o["out"], f"fused out {name} {fmt}")
