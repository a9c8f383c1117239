"""Alignment / permutation of routed rows into per-expert blocks (step a2).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

Follows the metadata the repro in the vLLM issue "moe_wna16_marlin_gemm applies
wrong per-row topk weights" (section "Minimal repro") builds with
``moe_align_block_size(topk_ids, BLOCK_M, E)`` and then reads back: flat row
ids ``row = t*k + j`` are grouped by expert in blocks of ``block_m`` slots;
``expert_ids[b]`` names the expert of block ``b`` (negative = unused); slots
holding a value >= T*k are padding (the repro keeps ``blk[blk < M*TOPK]``).

Readings taken where the page is silent: within an expert the flat rows are in
ascending order (a stable counting sort); the padding sentinel is exactly T*k;
each expert's segment is padded up to a multiple of block_m and empty experts
get no block; the inverse map ``row_pos[r]`` gives the slot of flat row r.

Parity: pinned (brute force and invariants in tests/test_oracle_align.py).
"""
import numpy as np


def padded_rows_max(T: int, k: int, E: int, block_m: int) -> int:
    """Upper bound on the padded slot count, rounded to whole blocks.

    At most min(E, T*k) experts are non-empty and each wastes at most
    block_m - 1 slots, so the block count is at most
    floor((T*k + min(E, T*k) * (block_m - 1)) / block_m).
    """
    R = T * k
    if R == 0:
        return 0
    nblk = (R + min(E, R) * (block_m - 1)) // block_m
    return nblk * block_m


def align_permute(topk_ids: np.ndarray, E: int, block_m: int):
    """topk_ids int32 [T, k] -> dict with

    sorted_token_ids int32 [P_max]   flat row id per slot, T*k in padding slots
    expert_offsets   int32 [E+1]     start slot of each expert's segment
    block_expert_ids int32 [P_max/block_m]  expert of each block, -1 if unused
    row_pos          int32 [T*k]     slot of each flat row
    """
    topk_ids = np.asarray(topk_ids, dtype=np.int32)
    T, k = topk_ids.shape
    R = T * k
    flat = topk_ids.reshape(-1)
    P_max = padded_rows_max(T, k, E, block_m)
    counts = np.bincount(flat, minlength=E).astype(np.int64)
    padded = (counts + block_m - 1) // block_m * block_m
    offsets = np.zeros(E + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(padded)
    assert offsets[E] <= P_max
    sorted_ids = np.full(P_max, R, dtype=np.int32)
    row_pos = np.empty(R, dtype=np.int32)
    block_ids = np.full(P_max // block_m if block_m else 0, -1, dtype=np.int32)
    for e in range(E):
        rows = np.nonzero(flat == e)[0]              # ascending flat row ids
        start = offsets[e]
        sorted_ids[start:start + rows.size] = rows
        row_pos[rows] = start + np.arange(rows.size)
        block_ids[offsets[e] // block_m: offsets[e + 1] // block_m] = e
    return dict(sorted_token_ids=sorted_ids,
                expert_offsets=offsets.astype(np.int32),
                block_expert_ids=block_ids,
                row_pos=row_pos)


def gather_rows(x: np.ndarray, sorted_token_ids: np.ndarray, k: int) -> np.ndarray:
    """x [T, H] -> x_perm [P_max, H]: slot p holds token sorted[p] // k, padding
    slots are zero."""
    T, H = x.shape
    R = T * k
    s = np.asarray(sorted_token_ids)
    out = np.zeros((s.size, H), dtype=x.dtype)
    valid = s < R
    out[valid] = x[s[valid] // k]
    return out
