"""Seeded generation of one MoE layer's inputs.

Every tensor has its own generator seeded from (seed, workload, tensor name,
expert), so generation is order-independent and can be streamed per expert.
Distributions follow the stated workloads: activations bf16 N(0, 1); router
logits fp32 N(0, 1) (plus -zipf * ln(e + 1) for the skewed workload); expert
weights fp32 N(0, 0.02) quantised to the workload's 4-bit format; biases bf16
N(0, 0.01); the selection bias of sigmoid routing fp32 N(0, 0.1).

Every tensor is drawn by a torch CPU generator and quantised on the CPU;
only the finished bytes are copied to ``device``. The layer is therefore the
same bytes whichever device it is made for, and making it launches no GPU
work beyond the copies.
"""
import os
import zlib
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

from .configs import FMT, LayerConfig
from . import quantize as qz


def _seed(*parts) -> int:
    return zlib.crc32("|".join(str(p) for p in parts).encode()) & 0x7FFFFFFF


def _gen(*parts) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(_seed(*parts))
    return g


def randn(shape, std, device, *parts) -> torch.Tensor:
    """N(0, std^2) fp32 drawn on the CPU from the generator of ``parts``, then
    copied to ``device``."""
    t = torch.randn(shape, generator=_gen(*parts), dtype=torch.float32) * std
    return t.to(device)


def make_projection(cfg: LayerConfig, which: str, N: int, K: int, seed: int,
                    device="cpu", with_bias=True, experts=None) -> dict:
    """Quantised weights of one projection ("w13" [E, N, K] or "w2")."""
    E = cfg.E
    fmt = FMT[cfg.fmt]
    q = torch.empty((E, N, K // 2), dtype=torch.uint8, device=device)
    out = dict(fmt=fmt, E=E, N=N, K=K, q=q, zeros=None, gscale=None, bias=None)
    if fmt == 0:
        out["scales"] = torch.empty((E, N, K // 16), dtype=torch.uint8, device=device)
        out["gscale"] = torch.empty((E,), dtype=torch.float32, device=device)
    elif fmt == 1:
        out["scales"] = torch.empty((E, N, K // 32), dtype=torch.uint8, device=device)
    else:
        out["scales"] = torch.empty((E, N, K // 64), dtype=torch.float16, device=device)
        out["zeros"] = torch.empty((E, N, (K // 64 + 1) // 2), dtype=torch.uint8, device=device)
    def draw(e):
        # drawn and quantised on the host (one generator per expert, so the
        # bytes do not depend on the order or the thread that makes them)
        w = randn((N, K), cfg.w_std, "cpu", seed, cfg.name.split("_t")[0], which, e)
        if fmt == 0:
            return qz.quantize_nvfp4(w)
        if fmt == 1:
            return qz.quantize_mxfp4(w)
        return qz.quantize_int4(w)

    todo = list(range(E) if experts is None else experts)
    with ThreadPoolExecutor(max(1, min(8, os.cpu_count() or 1))) as pool:
        for e, res in zip(todo, pool.map(draw, todo)):
            # the finished bytes go to the device
            if fmt == 0:
                pq, sc, gs = res
                out["gscale"][e] = gs
            elif fmt == 1:
                pq, sc = res
            else:
                pq, sc, zz = res
                out["zeros"][e] = zz
            q[e] = pq
            out["scales"][e] = sc
    if with_bias:
        out["bias"] = randn((E, N), cfg.bias_std, "cpu", seed, cfg.name.split("_t")[0],
                            which + "_bias").to(torch.bfloat16).to(device)
    return out


def make_activations(cfg: LayerConfig, seed: int, device="cpu") -> dict:
    base = cfg.name.split("_t")[0]
    x = randn((cfg.T, cfg.H), cfg.x_std, "cpu", seed, cfg.name, "x").to(torch.bfloat16)
    logits = randn((cfg.T, cfg.E), 1.0, "cpu", seed, cfg.name, "logits")
    if cfg.zipf:
        prior = -cfg.zipf * torch.log(torch.arange(1, cfg.E + 1, dtype=torch.float32))
        logits = logits + prior[None, :]
    sel_bias = None
    if cfg.route == "sigmoid_bias":
        sel_bias = randn((cfg.E,), cfg.sel_bias_std, "cpu", seed, base, "sel_bias").to(device)
    return dict(x=x.to(device), logits=logits.contiguous().to(device), sel_bias=sel_bias)


def make_layer(cfg: LayerConfig, seed: int = 0, device="cpu", weights=True) -> dict:
    """All inputs of one layer as torch tensors on ``device``."""
    d = make_activations(cfg, seed, device)
    if weights:
        d["w13"] = make_projection(cfg, "w13", cfg.N1, cfg.H, seed, device, cfg.bias)
        d["w2"] = make_projection(cfg, "w2", cfg.H, cfg.I, seed, device, cfg.bias)
    d["cfg"] = cfg
    return d


def _np(t):
    if t is None:
        return None
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return t.to(torch.float32).numpy()
    return t.numpy()


def to_numpy(layer: dict) -> dict:
    """Host NumPy copy (bf16 tensors become float32 holding the bf16 values)."""
    out = {}
    for key, v in layer.items():
        if isinstance(v, dict):
            out[key] = {kk: (_np(vv) if isinstance(vv, torch.Tensor) else vv)
                        for kk, vv in v.items()}
        elif isinstance(v, torch.Tensor):
            out[key] = _np(v)
        else:
            out[key] = v
    return out


__all__ = ["make_layer", "make_projection", "make_activations", "to_numpy", "randn", "np"]
