"""moe_forward_static (the entry point with the library's own fixed device
workspace) against moe_forward on the same inputs, through the C ABI.

Collected last on purpose: it must pass both in a fresh process and after
every other GPU test has used the device."""
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
