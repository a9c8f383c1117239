"""moe_forward_host against moe_forward, bit for bit: with page-locked host
buffers (read and written in place by the kernels) and with pageable ones
(staged through the workspace), for a decode and a prefill-shaped batch."""
import numpy as np
import pytest
import torch

from gpu_helpers import act_of, built, get_config, make

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    return built()


@pytest.mark.parametrize("T,pinned", [(5, True), (5, False), (700, True), (700, False)])
def test_host_forward_matches_device_forward(T, pinned):
    import bit_block_scaled_gb300 as moe
    cfg = get_config("c0", name=f"host_{T}", H=256, I=256, E=16, T=T, k=4)
    L, _ = make(cfg, seed=17)
    route = moe.ROUTE[cfg.route]
    nbytes = moe.moe_workspace_size(cfg.T, cfg.E, cfg.k, cfg.H, cfg.I, 16)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    ref = torch.empty(cfg.T, cfg.H, dtype=torch.bfloat16, device="cuda")
    moe.moe_forward(L["x"], L["logits"], L["sel_bias"], cfg.k, route, L["w13"], L["w2"], 0, act_of(cfg), 1, 16,
                    ref, ws)
    xh, lh = L["x"].cpu(), L["logits"].cpu()
    oh = torch.full((cfg.T, cfg.H), float("nan"), dtype=torch.bfloat16)
    if pinned:
        xh, lh, oh = xh.pin_memory(), lh.pin_memory(), oh.pin_memory()
    ws2 = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    moe.moe_forward_host(xh, lh, L["sel_bias"], cfg.k, route, L["w13"], L["w2"], 0, act_of(cfg), 1, 16, oh, ws2)
    torch.cuda.synchronize()
    assert moe.moe_read_status(ws2) == 0
    assert torch.equal(oh.view(torch.int16), ref.cpu().view(torch.int16))
