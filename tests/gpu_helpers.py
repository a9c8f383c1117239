"""Shared helpers for the GPU parity tests: run the layer step by step through
the C ABI and compare with the oracle."""
import numpy as np
import torch

import bit_block_scaled_gb300 as moe
from oracle import align as OA
from oracle import layer as OL
from oracle import routing as OR
from synth import get_config, make_layer, to_numpy

ATOL = 1e-2
RTOL = 1e-2

# x_perm and a are stored with the columns of every group of 8 interleaved:
# stored position q holds column STORE_ORDER[q] (see include/moe4.h)
STORE_ORDER = np.array([0, 4, 1, 5, 2, 6, 3, 7])
LOGICAL_POS = np.argsort(STORE_ORDER)          # column c sits at LOGICAL_POS[c]


def deinterleave8(a):
    a = np.asarray(a)
    n = a.shape[-1]
    idx = (np.arange(n) // 8) * 8 + LOGICAL_POS[np.arange(n) % 8]
    return a[..., idx]


def interleave8(a):
    a = np.asarray(a)
    n = a.shape[-1]
    idx = (np.arange(n) // 8) * 8 + STORE_ORDER[np.arange(n) % 8]
    return a[..., idx]


def built():
    from bit_block_scaled_gb300 import build
    build.build()
    return moe.load()


def make(cfg, seed=0, device="cuda"):
    L = make_layer(cfg, seed, device=device)
    return L, to_numpy(L)


def ws_status(nbytes=0):
    return torch.zeros(max(nbytes, moe._lib.STATUS_BYTES), dtype=torch.uint8, device="cuda")


def act_of(cfg):
    return moe.act(cfg.act, cfg.alpha, cfg.limit)


def gpu_steps(L, cfg, block_m=16, layout=0, mul=True, ids=None, tw=None):
    """Runs a1..a5 as separate C-ABI calls; returns host copies of every output."""
    T, E, k, H, I = cfg.T, cfg.E, cfg.k, cfg.H, cfg.I
    dev = "cuda"
    ws = ws_status()
    route = moe.ROUTE[cfg.route]
    if ids is None:
        ids = torch.empty(T, k, dtype=torch.int32, device=dev)
        tw = torch.empty(T, k, dtype=torch.float32, device=dev)
        moe.moe_route_topk(L["logits"], L["sel_bias"], k, route, ids, tw, ws)
    P = moe.moe_padded_rows(T, k, E, block_m)
    sorted_ids = torch.empty(max(P, 1), dtype=torch.int32, device=dev)
    offs = torch.empty(E + 1, dtype=torch.int32, device=dev)
    blocks = torch.empty(max(P // block_m, 1), dtype=torch.int32, device=dev)
    row_pos = torch.empty(max(T * k, 1), dtype=torch.int32, device=dev)
    x_perm = torch.zeros(max(P, 1), H, dtype=torch.bfloat16, device=dev)
    moe.moe_align_permute(ids, E, block_m, L["x"], sorted_ids, offs, blocks, row_pos, x_perm, ws)
    a = torch.zeros(max(P, 1), I, dtype=torch.bfloat16, device=dev)
    moe.moe_grouped_gemm1_act(x_perm[:P], sorted_ids, offs, T * k, L["w13"], layout, act_of(cfg), a, ws)
    y = torch.zeros(max(P, 1), H, dtype=torch.bfloat16, device=dev)
    moe.moe_grouped_gemm2_weighted(a[:P], sorted_ids, offs, L["w2"], tw.reshape(-1), mul, T * k, y, ws)
    out = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    moe.moe_unpermute_reduce(y[:P], row_pos, T, k, out, ws)
    status = moe.moe_read_status(ws)
    f = lambda t: t.detach().float().cpu().numpy() if t.dtype == torch.bfloat16 else t.cpu().numpy()
    return dict(topk_ids=f(ids), topk_weights=f(tw), sorted_token_ids=f(sorted_ids)[:P],
                expert_offsets=f(offs), block_expert_ids=f(blocks)[:P // block_m],
                row_pos=f(row_pos)[:T * k], x_perm=deinterleave8(f(x_perm)[:P]),
                a=deinterleave8(f(a)[:P]), y=f(y)[:P], out=f(out), status=status, P=P)


def gpu_forward(L, cfg, block_m=16, layout=0, mul=True, stream=None):
    """One moe_forward call; returns the output tensor (device) and the workspace."""
    T, E, k, H, I = cfg.T, cfg.E, cfg.k, cfg.H, cfg.I
    nbytes = moe.moe_workspace_size(T, E, k, H, I, block_m)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    out = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
    moe.moe_forward(L["x"], L["logits"], L["sel_bias"], k, moe.ROUTE[cfg.route], L["w13"], L["w2"],
                    layout, act_of(cfg), mul, block_m, out, ws, stream)
    return out, ws


def oracle_full(N, cfg, block_m=16, ids=None, tw=None, layout=0, mul=True):
    return OL.moe_forward(N["x"], N["logits"], N["w13"], N["w2"], cfg.k,
                          route_mode=OR.ROUTE_TOPK_SOFTMAX if cfg.route == "topk_softmax"
                          else OR.ROUTE_SIGMOID_BIAS, sel_bias=N.get("sel_bias"),
                          act=OL.ACT_SWIGLUOAI if cfg.act == "swigluoai" else OL.ACT_RELU2,
                          layout=layout, alpha=cfg.alpha, limit=cfg.limit,
                          mul_topk_weights=mul, block_m=block_m, topk_ids=ids, topk_weights=tw)


def assert_close(got, ref, what, atol=ATOL, rtol=RTOL):
    got = np.asarray(got, np.float32)
    ref = np.asarray(ref, np.float32)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    err = np.abs(got - ref)
    bound = atol + rtol * np.abs(ref)
    bad = err > bound
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} / {bad.size} outside |d| <= {atol} + {rtol}|ref|; "
                             f"first at {tuple(i)}: got {got[tuple(i)]} ref {ref[tuple(i)]}; "
                             f"max err {err.max():.3e}")


def near_tie_ok(scores, got_ids, ref_ids, ulps=2):
    """Routing ids must match exactly except where two competing selection
    scores are within `ulps` float32 ulps (the two sides evaluate exp with
    different roundings)."""
    bad = []
    for t in np.nonzero((got_ids != ref_ids).any(axis=1))[0]:
        s = scores[t].astype(np.float32)
        g = set(got_ids[t].tolist())
        r = set(ref_ids[t].tolist())
        diff = (g ^ r)
        vals = s[list(diff)] if diff else s[got_ids[t]]
        kth = np.sort(s)[::-1][len(ref_ids[t]) - 1]
        spacing = np.spacing(np.float32(abs(kth))) * ulps
        if diff and np.all(np.abs(vals - kth) <= spacing):
            # same set up to a near-tie swap at the boundary
            continue
        if not diff:
            # same set, different order: only allowed between near-equal scores
            o = s[got_ids[t]]
            if np.all(np.diff(o) <= spacing):
                continue
        bad.append(int(t))
    return bad


__all__ = ["deinterleave8", "interleave8", "built", "make", "gpu_steps", "gpu_forward", "oracle_full", "assert_close", "get_config",
           "near_tie_ok", "OA", "OL", "OR", "ws_status", "act_of"]
