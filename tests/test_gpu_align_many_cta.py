"""GPU parity of the alignment step (a2) on batches large enough for the
many-CTA alignment (per-chunk counts, then placement over many CTAs), and on
the last size below it: sorted ids, expert offsets, block ids and row
positions bit-exact against the oracle's stable counting sort, and the
gathered rows bit-exact, for ragged chunk tails, skewed and sparse expert
use, every block size and a single expert.
"""
import numpy as np
import pytest
import torch

from gpu_helpers import built, deinterleave8, ws_status
from oracle import align as OA

pytestmark = pytest.mark.gpu

H = 64


@pytest.fixture(scope="module", autouse=True)
def lib():
    return built()


def _ids(T, k, E, dist, seed):
    g = torch.Generator().manual_seed(seed)
    if dist == "uniform":
        return torch.randint(0, E, (T, k), generator=g, dtype=torch.int32)
    if dist == "skew":                  # expert 3 takes about half the rows
        ids = torch.randint(0, E, (T, k), generator=g, dtype=torch.int32)
        ids[torch.rand(T, k, generator=g) < 0.5] = 3
        return ids
    if dist == "sparse":                # three experts of E in use
        pick = torch.tensor([1, E // 2, E - 1], dtype=torch.int32)
        return pick[torch.randint(0, 3, (T, k), generator=g)]
    if dist == "cyclic":                # row r goes to expert r mod E
        return (torch.arange(T * k, dtype=torch.int32) % E).reshape(T, k)
    raise ValueError(dist)


def _run(ids, E, bm, seed=0):
    import bit_block_scaled_gb300 as moe
    T, k = ids.shape
    P = moe.moe_padded_rows(T, k, E, bm)
    x = (torch.randn(T, H, generator=torch.Generator().manual_seed(seed + 1)) * 0.5).to(torch.bfloat16)
    d_ids, d_x = ids.cuda(), x.cuda()
    sorted_ids = torch.empty(P, dtype=torch.int32, device="cuda")
    offs = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    blocks = torch.empty(P // bm, dtype=torch.int32, device="cuda")
    row_pos = torch.empty(T * k, dtype=torch.int32, device="cuda")
    x_perm = torch.full((P, H), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = ws_status()
    moe.moe_align_permute(d_ids, E, bm, d_x, sorted_ids, offs, blocks, row_pos, x_perm, ws)
    launches = moe.moe_last_launch_count()
    st = moe.moe_read_status(ws)
    return dict(sorted=sorted_ids.cpu().numpy(), offs=offs.cpu().numpy(), blocks=blocks.cpu().numpy(),
                row_pos=row_pos.cpu().numpy(), x_perm=deinterleave8(x_perm.float().cpu().numpy()),
                x=x.float().numpy(), status=st, launches=launches)


@pytest.mark.parametrize("T,k,E,bm,dist", [
    (4095, 1, 128, 16, "uniform"),      # one routed row below the many-CTA size
    (1024, 4, 128, 16, "uniform"),      # exactly four chunks
    (2049, 4, 128, 32, "uniform"),      # nine chunks, the last holding four rows
    (8192, 8, 128, 16, "uniform"),      # 65,536 rows, the largest prefill batch
    (5000, 8, 256, 64, "skew"),
    (3001, 2, 256, 128, "sparse"),
    (4100, 1, 1, 256, "uniform"),       # one expert
    (700, 8, 64, 16, "cyclic"),
])
def test_alignment_bit_exact(T, k, E, bm, dist):
    ids = _ids(T, k, E, dist, seed=T + E)
    g = _run(ids, E, bm)
    o = OA.align_permute(ids.numpy(), E, bm)
    assert g["status"] == 0
    assert np.array_equal(g["offs"], o["expert_offsets"])
    assert np.array_equal(g["sorted"], o["sorted_token_ids"])
    assert np.array_equal(g["blocks"], o["block_expert_ids"])
    assert np.array_equal(g["row_pos"], o["row_pos"])
    used = int(o["expert_offsets"][-1])
    ref = OA.gather_rows(g["x"], o["sorted_token_ids"], k)
    assert np.array_equal(g["x_perm"][:used], ref[:used])      # padding slots zero, rows bit-exact
    # two launches for the alignment from 4096 routed rows on, one below, then the gather
    assert g["launches"] == (3 if T * k >= 4096 else 2)


def test_bad_ids_in_a_large_batch_latch_status_and_skip_the_row():
    T, k, E, bm = 1500, 4, 64, 16
    ids = _ids(T, k, E, "uniform", seed=5)
    bad = [(0, 0), (777, 3), (1499, 1)]
    for t, j in bad:
        ids[t, j] = E if t != 777 else -1
    g = _run(ids, E, bm)
    assert g["status"] == 5
    flat = ids.numpy().reshape(-1)
    valid = (flat >= 0) & (flat < E)
    R = T * k
    assert np.all(g["row_pos"][~valid] == -1)
    # the valid rows: offsets from their own counts, each expert's rows in
    # ascending order at its segment's start, the rest of the segment padding
    cnt = np.bincount(flat[valid], minlength=E)
    pad = (cnt + bm - 1) // bm * bm
    assert np.array_equal(g["offs"], np.concatenate([[0], np.cumsum(pad)]))
    for e in range(E):
        rows = np.nonzero(flat == e)[0]
        seg = g["sorted"][g["offs"][e]:g["offs"][e + 1]]
        assert np.array_equal(seg[:rows.size], rows)
        assert np.all(seg[rows.size:] == R)
        assert np.array_equal(g["row_pos"][rows], g["offs"][e] + np.arange(rows.size))
    assert np.all(g["sorted"][g["offs"][-1]:] == R)


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4", "int4"])
@pytest.mark.parametrize("mul,T", [(1, 1500), (2, 1500), (1, 800)])
def test_forward_large_batch_matches_oracle(fmt, mul, T):
    """moe_forward over 6,000 routed rows (the many-CTA alignment, the
    per-token gather with the routing weight on the input rows or in the
    GEMM2 epilogue; 192-row token tiles) and over 3,200 (160-row tiles),
    every output element against the oracle."""
    import bit_block_scaled_gb300 as moe
    from gpu_helpers import act_of, assert_close, get_config, gpu_steps, make, oracle_full
    cfg = get_config("c0", name=f"large_{fmt}_{mul}_{T}", fmt=fmt, H=256, I=256, E=32, T=T, k=4)
    L, N = make(cfg, seed=41)
    g = gpu_steps(L, cfg)
    ws = torch.zeros(moe.moe_workspace_size(cfg.T, cfg.E, cfg.k, cfg.H, cfg.I, 16), dtype=torch.uint8,
                     device="cuda")
    out = torch.empty(cfg.T, cfg.H, dtype=torch.bfloat16, device="cuda")
    moe.moe_forward(L["x"], L["logits"], L["sel_bias"], cfg.k, moe.ROUTE[cfg.route], L["w13"], L["w2"], 0,
                    act_of(cfg), mul, 16, out, ws)
    assert moe.moe_read_status(ws) == 0
    o = oracle_full(N, cfg, ids=g["topk_ids"].astype(np.int32), tw=g["topk_weights"], mul=mul)
    assert_close(out.float().cpu().numpy(), o["out"], f"large batch out ({fmt}, mul {mul})")


def test_forward_widest_rows_one_cta_per_token():
    """H = 4096 (512 vectors of 8 columns, the widest row) at 300 tokens: the
    gather and the unpermute each run one 512-thread CTA per token."""
    import bit_block_scaled_gb300 as moe
    from gpu_helpers import act_of, assert_close, get_config, gpu_steps, make, oracle_full
    cfg = get_config("c0", name="wide_rows", fmt="nvfp4", H=4096, I=128, E=8, T=300, k=2)
    L, N = make(cfg, seed=43)
    g = gpu_steps(L, cfg)
    ws = torch.zeros(moe.moe_workspace_size(cfg.T, cfg.E, cfg.k, cfg.H, cfg.I, 16), dtype=torch.uint8,
                     device="cuda")
    out = torch.empty(cfg.T, cfg.H, dtype=torch.bfloat16, device="cuda")
    moe.moe_forward(L["x"], L["logits"], L["sel_bias"], cfg.k, moe.ROUTE[cfg.route], L["w13"], L["w2"], 0,
                    act_of(cfg), 1, 16, out, ws)
    assert moe.moe_read_status(ws) == 0
    o = oracle_full(N, cfg, ids=g["topk_ids"].astype(np.int32), tw=g["topk_weights"])
    assert_close(g["out"], o["out"], "wide rows, steps")
    assert_close(out.float().cpu().numpy(), o["out"], "wide rows, forward")
