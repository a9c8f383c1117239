"""Host-side argument checks of the C ABI (include/moe4.h: "Arguments are
checked on the host first; on MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED nothing
is launched"). Every call here is rejected, or has nothing to do, before its
first CUDA call, so the tests run on the CPU with host buffers standing in for
device pointers; a missing check would surface as a CUDA error code instead."""
import pytest
import torch

import bit_block_scaled_gb300 as moe
from bit_block_scaled_gb300 import build as B
from synth import get_config, make_layer

INVALID, WORKSPACE = 1, 6


@pytest.fixture(scope="module")
def layer():
    B.build()
    moe.load()
    cfg = get_config("c0")  # T16 E8 k2 H256 I256 NVFP4 swigluoai
    return cfg, make_layer(cfg, 0, device="cpu")


def _ws(cfg, T=None):
    n = moe.moe_workspace_size(cfg.T if T is None else T, cfg.E, cfg.k, cfg.H, cfg.I, 16)
    return torch.zeros(n, dtype=torch.uint8)


def _forward(cfg, L, fn=moe.moe_forward, **kw):
    a = dict(x=L["x"], logits=L["logits"], k=cfg.k, route=moe.ROUTE[cfg.route], w13=L["w13"], w2=L["w2"],
             layout=0, act=moe.act(cfg.act, cfg.alpha, cfg.limit), mul=1, block_m=16,
             out=torch.empty(L["x"].shape[0], cfg.H, dtype=torch.bfloat16), ws=None)
    a.update(kw)
    ws = _ws(cfg, a["x"].shape[0]) if a["ws"] is None else a["ws"]
    fn(a["x"], a["logits"], None, a["k"], a["route"], a["w13"], a["w2"], a["layout"], a["act"], a["mul"],
       a["block_m"], a["out"], ws, 0)


def _code(fn):
    with pytest.raises(moe.MoeError) as e:
        fn()
    return e.value.code


def _misaligned(t):
    """The same shape and dtype, 2 bytes past a 16-byte boundary."""
    raw = torch.empty(t.numel() * t.element_size() + 16, dtype=torch.uint8)
    return raw[2:2 + t.numel() * t.element_size()].view(t.dtype).view(t.shape)


@pytest.mark.parametrize("fn", [moe.moe_forward, moe.moe_forward_host])
def test_forward_rejections(layer, fn):
    cfg, L = layer
    assert _code(lambda: _forward(cfg, L, fn, mul=3)) == INVALID          # routing-weight placement
    assert _code(lambda: _forward(cfg, L, fn, mul=-1)) == INVALID
    assert _code(lambda: _forward(cfg, L, fn, block_m=48)) == INVALID     # block_m not a power of two >= 16
    assert _code(lambda: _forward(cfg, L, fn, route=7)) == INVALID
    assert _code(lambda: _forward(cfg, L, fn, act=moe.Act(9, 1.702, 7.0))) == INVALID
    assert _code(lambda: _forward(cfg, L, fn, layout=2)) == INVALID
    assert _code(lambda: _forward(cfg, L, fn, k=9)) == INVALID            # k > 8
    assert _code(lambda: _forward(cfg, L, fn, w13=L["w2"])) == INVALID    # W13 of the wrong shape
    assert _code(lambda: _forward(cfg, L, fn, ws=torch.zeros(4096, dtype=torch.uint8))) == WORKSPACE
    assert _code(lambda: _forward(cfg, L, fn, ws=_misaligned(_ws(cfg)))) == INVALID
    logits300 = torch.zeros(cfg.T, 300)
    assert _code(lambda: _forward(cfg, L, fn, logits=logits300)) == INVALID  # E > 256


def test_forward_misaligned_device_pointers(layer):
    cfg, L = layer
    assert _code(lambda: _forward(cfg, L, x=_misaligned(L["x"]))) == INVALID
    assert _code(lambda: _forward(cfg, L, out=_misaligned(torch.empty(cfg.T, cfg.H, dtype=torch.bfloat16)))) \
        == INVALID


def test_empty_batch_launches_nothing(layer):
    cfg, L = layer
    x0 = L["x"][:0].contiguous()
    _forward(cfg, L, x=x0, logits=L["logits"][:0].contiguous(), out=torch.empty(0, cfg.H, dtype=torch.bfloat16))
    assert moe.moe_last_launch_count() == 0


def test_step_rejections(layer):
    cfg, L = layer
    ws = _ws(cfg)
    ids = torch.zeros(cfg.T, cfg.k, dtype=torch.int32)
    tw = torch.zeros(cfg.T, cfg.k)
    assert _code(lambda: moe.moe_route_topk(L["logits"], None, 0, 0, ids, tw, ws, 0)) == INVALID  # k = 0
    assert _code(lambda: moe.moe_route_topk(L["logits"], None, cfg.k, 9, ids, tw, ws, 0)) == INVALID
    moe.moe_route_topk(L["logits"][:0].contiguous(), None, cfg.k, 0, ids[:0], tw[:0], ws, 0)  # T = 0: nothing to do
    P = moe.moe_padded_rows(cfg.T, cfg.k, cfg.E, 16)
    srt = torch.zeros(P, dtype=torch.int32)
    offs = torch.zeros(cfg.E + 1, dtype=torch.int32)
    blk = torch.zeros(P // 16, dtype=torch.int32)
    rp = torch.zeros(cfg.T * cfg.k, dtype=torch.int32)
    xp = torch.zeros(P, cfg.H, dtype=torch.bfloat16)
    assert _code(lambda: moe.moe_align_permute(ids, cfg.E, 8, L["x"], srt, offs, blk, rp, xp, ws, 0)) == INVALID
    x100 = torch.zeros(cfg.T, 100, dtype=torch.bfloat16)                      # H not a multiple of 64
    assert _code(lambda: moe.moe_align_permute(ids, cfg.E, 16, x100, srt, offs, blk, rp, xp, ws, 0)) == INVALID
