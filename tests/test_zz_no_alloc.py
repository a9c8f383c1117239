"""moe_forward_static (the entry point with the library's own fixed device
workspace) against moe_forward on the same inputs, through the C ABI.

Collected last on purpose: it must pass both in a fresh process and after
every other GPU test has used the device."""
import ctypes

import numpy as np
import pytest
import torch

import bit_block_scaled_gb300 as moe
from gpu_helpers import act_of, assert_close, built, get_config, gpu_forward, make, oracle_full

pytestmark = pytest.mark.gpu

CODE = {name: code for code, name in moe.STATUS.items()}


@pytest.fixture(scope="module", autouse=True)
def lib():
    return built()


def _static(L, cfg, block_m=16):
    out = torch.full((cfg.T, cfg.H), float("nan"), dtype=torch.bfloat16, device="cuda")
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    moe.moe_forward_static(L["x"], L["logits"], L["sel_bias"], cfg.k, moe.ROUTE[cfg.route], L["w13"], L["w2"],
                           0, act_of(cfg), True, block_m, out, status)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), int(status.item())


@pytest.mark.parametrize("key", ["c0", "c1"])
def test_static_matches_forward_twice_in_a_row(key):
    cfg = get_config(key)
    L, N = make(cfg)
    ref, ws = gpu_forward(L, cfg)
    ref = ref.float().cpu().numpy()
    assert moe.moe_read_status(ws) == 0
    for _ in range(2):  # the second call reuses the array the first one left behind
        got, status = _static(L, cfg)
        assert status == 0
        assert_close(got, ref, f"{key} static vs moe_forward")
    if key == "c0":
        assert_close(got, oracle_full(N, cfg)["out"], "c0 static vs oracle")


def test_static_status_word_is_per_call():
    """An MXFP4 scale exponent past the supported range latches
    MOE_ERR_SCALE_RANGE in the call that reads it; the next call, on valid
    weights, starts from a cleared status word."""
    cfg = get_config("c0", fmt="mxfp4")
    L, _ = make(cfg)
    bad = dict(L["w13"])
    bad["scales"] = L["w13"]["scales"].clone()
    bad["scales"][:, 0, 0] = 200  # E8M0 exponent 200 = 2^73 in every expert: out of range
    Lb = dict(L)
    Lb["w13"] = bad
    _, status = _static(Lb, cfg)
    assert status == 1 << (CODE["MOE_ERR_SCALE_RANGE"] - 1)
    _, status = _static(L, cfg)
    assert status == 0


def test_static_rejects_sizes_past_its_capacity():
    cfg = get_config("c1", T=4096)
    T, E, k, H, I = cfg.T, cfg.E, cfg.k, cfg.H, cfg.I
    assert moe.moe_workspace_size(T, E, k, H, I, 16) > 32 << 20
    L, _ = make(get_config("c1"))
    x = torch.zeros(T, H, dtype=torch.bfloat16, device="cuda")
    logits = torch.zeros(T, E, dtype=torch.float32, device="cuda")
    out = torch.zeros(T, H, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_forward_static(x, logits, None, k, moe.ROUTE[cfg.route], L["w13"], L["w2"], 0, act_of(cfg),
                               True, 16, out)
    assert ei.value.code == CODE["MOE_ERR_UNSUPPORTED"]
    assert np.all(out.float().cpu().numpy() == 0)  # nothing launched


def test_static_call_allocates_nothing():
    """After a first call (which may load the library's device code), a second
    call leaves the device's free memory and torch's allocator unchanged."""
    cfg = get_config("c1")
    L, _ = make(cfg)
    out = torch.empty(cfg.T, cfg.H, dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")

    def call():
        moe.moe_forward_static(L["x"], L["logits"], L["sel_bias"], cfg.k, moe.ROUTE[cfg.route], L["w13"],
                               L["w2"], 0, act_of(cfg), True, 16, out, status)
        torch.cuda.synchronize()

    call()
    free0, _ = torch.cuda.mem_get_info()
    alloc0 = torch.cuda.memory_allocated()
    call()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    assert torch.cuda.memory_allocated() == alloc0
    assert int(status.item()) == 0


def _captured_node_count(stream, fn):
    """Runs fn while `stream` is being captured (driver API, relaxed mode) and
    returns how many nodes the capture recorded."""
    cu = ctypes.CDLL("libcuda.so.1")
    h = ctypes.c_void_p(stream.cuda_stream)
    assert cu.cuStreamBeginCapture_v2(h, 2) == 0          # CU_STREAM_CAPTURE_MODE_RELAXED
    try:
        fn()
    finally:
        graph = ctypes.c_void_p()
        assert cu.cuStreamEndCapture(h, ctypes.byref(graph)) == 0
    n = ctypes.c_size_t(0)
    assert cu.cuGraphGetNodes(graph, None, ctypes.byref(n)) == 0
    cu.cuGraphDestroy(graph)
    return n.value


def test_rejected_static_call_enqueues_nothing():
    """A call rejected by the host checks (an unknown activation kind, sizes
    past the array) puts no work on the stream: a stream capture around it
    records no node, and the status word a previous call left stays as it was
    (the next accepted call, which clears it, still reports its own status)."""
    cfg = get_config("c0", fmt="mxfp4")
    L, _ = make(cfg)
    bad = dict(L["w13"])
    bad["scales"] = L["w13"]["scales"].clone()
    bad["scales"][:, 0, 0] = 200                          # latches MOE_ERR_SCALE_RANGE
    out = torch.zeros(cfg.T, cfg.H, dtype=torch.bfloat16, device="cuda")
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.Stream()
    moe.moe_forward_static(L["x"], L["logits"], None, cfg.k, moe.ROUTE[cfg.route], bad, L["w2"], 0,
                           act_of(cfg), True, 16, out, status, stream)
    torch.cuda.synchronize()
    assert int(status.item()) == 1 << (CODE["MOE_ERR_SCALE_RANGE"] - 1)
    status.fill_(-1)
    out.zero_()
    torch.cuda.synchronize()
    wrong_act = moe.act("swigluoai", cfg.alpha, cfg.limit)
    wrong_act.kind = 7

    def rejected():
        with pytest.raises(moe.MoeError) as ei:
            moe.moe_forward_static(L["x"], L["logits"], None, cfg.k, moe.ROUTE[cfg.route], L["w13"], L["w2"],
                                   0, wrong_act, True, 16, out, status, stream)
        assert ei.value.code == CODE["MOE_ERR_INVALID_ARG"]

    assert _captured_node_count(stream, rejected) == 0
    torch.cuda.synchronize()
    assert int(status.item()) == -1                       # status_out untouched
    assert torch.count_nonzero(out).item() == 0          # nothing launched
