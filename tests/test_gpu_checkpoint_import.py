"""Checkpoint layouts through the whole layer on the GPU.

GPTQ INT4 ("Serving gpt-oss with mixed GPTQ experts", section "1. Quantize":
per-expert gate, up and down projections as qweight / qzeros / scales /
g_idx, group size 64): each projection's GPTQ tensors are imported with
moe_import_gptq_int4, gate and up are stacked into W13 in the CONCAT layout,
and moe_forward runs the layer. The reference is the oracle's per-token
definition evaluated on weights decoded straight from the GPTQ tensors by the
GPTQ formula bf16((code - zero) * scale), so the import and the kernel are
checked together against the checkpoint itself.

ModelOpt NVFP4 (NVFP4 gpt-oss report, "Gap 2"): one scalar weight_scale_2
broadcast by moe_import_modelopt_global_scale to every expert's global scale.
"""
import numpy as np
import pytest
import torch

import bit_block_scaled_gb300 as moe
from gpu_helpers import act_of, assert_close, built, get_config, make, oracle_full
from oracle import formats as OF
from oracle import layer as OL
from oracle import routing as OR
from synth.quantize import quantize_int4
from test_checkpoint_import import _gptq_tensors

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    return built()


def _gptq_linear(N, K, seed):
    """One GPTQ-quantised linear layer [N, K]: its checkpoint tensors."""
    g = torch.Generator().manual_seed(seed)
    w = torch.randn(N, K, generator=g) * 0.02
    q, s, z = quantize_int4(w)
    return _gptq_tensors(q.numpy(), s.numpy(), z.numpy(), K)


def _gptq_formula(qweight, qzeros, scales):
    """bf16((code - zero) * scale) [N, K], read straight from the GPTQ tensors."""
    K = qweight.shape[0] * 8
    N = qweight.shape[1]
    u = qweight.view(np.uint32).astype(np.int64)
    codes = np.stack([(u >> (4 * j)) & 0xF for j in range(8)], axis=1).reshape(K, N)
    uz = qzeros.view(np.uint32).astype(np.int64)
    zeros = np.stack([(uz >> (4 * j)) & 0xF for j in range(8)], axis=2).reshape(K // 64, N)
    ref = (codes - np.repeat(zeros, 64, axis=0)) * np.repeat(scales.astype(np.float64), 64, axis=0)
    return OF.bf16_rne(ref.T).astype(np.float64)


@pytest.mark.parametrize("E,k,T,H,I", [(4, 2, 40, 320, 192), (8, 4, 24, 576, 320)])
def test_gptq_checkpoint_through_the_fused_forward(E, k, T, H, I):
    rng = np.random.default_rng(E * 100 + H)
    parts = {"gate": [], "up": [], "down": []}
    for e in range(E):
        parts["gate"].append(_gptq_linear(I, H, 1000 * e + 1))
        parts["up"].append(_gptq_linear(I, H, 1000 * e + 2))
        parts["down"].append(_gptq_linear(H, I, 1000 * e + 3))
    imp = {name: [moe.moe_import_gptq_int4(qw, qz, sc, gi) for (qw, qz, sc, gi) in lst]
           for name, lst in parts.items()}
    dev = "cuda"
    cat = lambda a, b: np.concatenate([a, b], axis=0)
    b13 = (rng.standard_normal((E, 2 * I)) * 0.01).astype(np.float32)
    b2 = (rng.standard_normal((E, H)) * 0.01).astype(np.float32)
    w13 = dict(fmt=2, E=E, N=2 * I, K=H, gscale=None,
               q=torch.from_numpy(np.stack([cat(imp["gate"][e][0], imp["up"][e][0]) for e in range(E)])).to(dev),
               scales=torch.from_numpy(np.stack([cat(imp["gate"][e][1], imp["up"][e][1])
                                                 for e in range(E)])).to(dev),
               zeros=torch.from_numpy(np.stack([cat(imp["gate"][e][2], imp["up"][e][2])
                                                for e in range(E)])).to(dev),
               bias=torch.from_numpy(b13).to(torch.bfloat16).to(dev))
    w2 = dict(fmt=2, E=E, N=H, K=I, gscale=None,
              q=torch.from_numpy(np.stack([imp["down"][e][0] for e in range(E)])).to(dev),
              scales=torch.from_numpy(np.stack([imp["down"][e][1] for e in range(E)])).to(dev),
              zeros=torch.from_numpy(np.stack([imp["down"][e][2] for e in range(E)])).to(dev),
              bias=torch.from_numpy(b2).to(torch.bfloat16).to(dev))
    x = torch.from_numpy(rng.standard_normal((T, H)).astype(np.float32)).to(torch.bfloat16).to(dev)
    logits = torch.from_numpy(rng.standard_normal((T, E)).astype(np.float32)).to(dev)
    act = moe.act("swigluoai", 1.702, 7.0)
    out = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    ws = torch.zeros(moe.moe_workspace_size(T, E, k, H, I, 16), dtype=torch.uint8, device=dev)
    moe.moe_forward(x, logits, None, k, moe.ROUTE["topk_softmax"], w13, w2, moe.LAYOUT["concat"], act, 1, 16,
                    out, ws)
    assert moe.moe_read_status(ws) == 0
    got = out.cpu().float().numpy()

    # reference: the per-token definition on weights decoded from the GPTQ tensors
    xh = x.cpu().float().numpy()
    ids, tw = OR.topk_softmax(logits.cpu().numpy(), k)
    b13h = w13["bias"].cpu().float().numpy()
    b2h = w2["bias"].cpu().float().numpy()
    ref = np.zeros((T, H), np.float32)
    for t in range(T):
        acc = np.zeros(H, np.float32)
        for j in range(k):
            e = int(ids[t, j])
            W13 = np.concatenate([_gptq_formula(*parts["gate"][e][:3]), _gptq_formula(*parts["up"][e][:3])])
            a = OL.expert_gemm1_act(xh[t:t + 1], W13, None, b13h[e], OL.ACT_SWIGLUOAI, OL.LAYOUT_CONCAT)
            y = OL.expert_gemm2(a, _gptq_formula(*parts["down"][e][:3]), None, b2h[e], tw[t, j:j + 1])
            acc = (acc + y[0]).astype(np.float32)
        ref[t] = OF.bf16_rne(acc)
    assert_close(got, ref, f"GPTQ checkpoint E{E} k{k} T{T} H{H} I{I}")


def test_modelopt_scalar_global_scale_through_the_fused_forward():
    """NVFP4 weights with one ModelOpt weight_scale_2 per projection: the
    broadcast global scales give the layer the oracle computes with that
    scalar in every expert."""
    cfg = get_config("c0")
    L, N = make(cfg, seed=23)
    for proj in ("w13", "w2"):
        gs = float(N[proj]["gscale"][0])
        g = moe.moe_import_modelopt_global_scale(gs, cfg.E)
        L[proj] = dict(L[proj])
        L[proj]["gscale"] = torch.from_numpy(g).to("cuda")
        N[proj] = dict(N[proj])
        N[proj]["gscale"] = np.full(cfg.E, np.float32(gs), np.float32)
    out = torch.empty(cfg.T, cfg.H, dtype=torch.bfloat16, device="cuda")
    ws = torch.zeros(moe.moe_workspace_size(cfg.T, cfg.E, cfg.k, cfg.H, cfg.I, 16), dtype=torch.uint8,
                     device="cuda")
    moe.moe_forward(L["x"], L["logits"], None, cfg.k, 0, L["w13"], L["w2"], 0, act_of(cfg), 1, 16, out, ws)
    assert moe.moe_read_status(ws) == 0
    assert_close(out.cpu().float().numpy(), oracle_full(N, cfg)["out"], "ModelOpt scalar global scale")
