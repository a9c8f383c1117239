"""Pins for the oracle's routing (a1) and alignment (a2) steps (CPU only)."""
import numpy as np
import torch

from oracle import align as A
from oracle import routing as R


def _brute_topk(row, k):
    # pure-Python selection: repeatedly take the max, lower id on ties
    remaining = list(range(len(row)))
    out = []
    for _ in range(k):
        best = remaining[0]
        for e in remaining[1:]:
            if row[e] > row[best]:
                best = e
        out.append(best)
        remaining.remove(best)
    return out


def test_topk_softmax_matches_softmax_then_topk_renormalised():
    # the repro does softmax over all experts then top-k (no renorm); renormalising
    # its weights must give top-k-then-softmax exactly up to fp rounding
    rng = np.random.default_rng(0)
    logits = rng.standard_normal((200, 32)).astype(np.float32)
    ids, w = R.topk_softmax(logits, 4)
    lt = torch.from_numpy(logits).double()
    pw, pids = torch.topk(torch.softmax(lt, -1), 4, dim=-1)
    assert np.array_equal(ids, pids.numpy())
    ren = (pw / pw.sum(-1, keepdim=True)).numpy()
    np.testing.assert_allclose(w, ren, rtol=2e-7, atol=0)
    np.testing.assert_allclose(w.astype(np.float64).sum(1), 1.0, atol=1e-6)
    assert np.all(np.diff(w, axis=1) <= 0)


def test_topk_brute_force_and_ties():
    rng = np.random.default_rng(1)
    logits = rng.integers(-3, 3, size=(50, 8)).astype(np.float32)   # many ties
    ids, _ = R.topk_softmax(logits, 3)
    for t in range(50):
        assert ids[t].tolist() == _brute_topk(logits[t].tolist(), 3)
    # literal case: equal logits -> lower expert id first
    ids, w = R.topk_softmax(np.array([[1.0, 2.0, 2.0, 0.5]], np.float32), 2)
    assert ids.tolist() == [[1, 2]]
    assert w.tolist() == [[0.5, 0.5]]


def test_sigmoid_routing_invariants():
    rng = np.random.default_rng(2)
    logits = rng.standard_normal((300, 128)).astype(np.float32)
    # zero bias: selection equals plain top-k of the logits (sigmoid is monotone)
    ids0, w0 = R.sigmoid_bias_topk(logits, np.zeros(128, np.float32), 6)
    ref = torch.topk(torch.sigmoid(torch.from_numpy(logits).double()), 6, dim=-1)
    assert np.array_equal(ids0, ref.indices.numpy())
    np.testing.assert_allclose(w0.astype(np.float64).sum(1), 1.0, atol=1e-6)
    # with a bias: weights are the selected sigmoid scores renormalised (bias-free)
    bias = (rng.standard_normal(128) * 0.1).astype(np.float32)
    ids, w = R.sigmoid_bias_topk(logits, bias, 6)
    s = torch.sigmoid(torch.from_numpy(logits).double()).numpy()
    sel = np.take_along_axis(s, ids, 1)
    np.testing.assert_allclose(w, sel / sel.sum(1, keepdims=True), rtol=2e-7)
    score = R.selection_scores(logits, bias)
    for t in range(300):
        assert ids[t].tolist() == _brute_topk(score[t].tolist(), 6)
    # the bias changes the selection for some tokens
    assert not np.array_equal(ids, ids0)


def test_sigmoid_f32_matches_library():
    x = np.linspace(-30, 30, 10001).astype(np.float32)
    ours = R.sigmoid_f32(x)
    ref = torch.sigmoid(torch.from_numpy(x).double()).float().numpy()
    assert np.array_equal(ours, ref)


def _brute_align(ids, E, bm):
    T, k = len(ids), len(ids[0])
    Rr = T * k
    flat = [ids[t][j] for t in range(T) for j in range(k)]
    slots = []
    offsets = [0]
    blocks = []
    for e in range(E):
        rows = [r for r in range(Rr) if flat[r] == e]
        pad = (-len(rows)) % bm
        slots += rows + [Rr] * pad
        blocks += [e] * ((len(rows) + pad) // bm)
        offsets.append(len(slots))
    return slots, offsets, blocks


def test_align_literal_example():
    # T=3, k=2, E=3, block_m=4 -> flat rows 0..5 with experts [1,0,1,2,0,1]
    ids = np.array([[1, 0], [1, 2], [0, 1]], np.int32)
    m = A.align_permute(ids, 3, 4)
    R6 = 6
    assert m["expert_offsets"].tolist() == [0, 4, 8, 12]
    assert m["sorted_token_ids"][:12].tolist() == [1, 4, R6, R6, 0, 2, 5, R6, 3, R6, R6, R6]
    assert m["block_expert_ids"][:3].tolist() == [0, 1, 2]
    assert m["row_pos"].tolist() == [4, 0, 5, 8, 1, 6]
    # P_max = floor((6 + 3*3) / 4) * 4 = 12
    assert A.padded_rows_max(3, 2, 3, 4) == 12


def test_align_brute_force_and_invariants():
    rng = np.random.default_rng(3)
    for trial in range(30):
        T = int(rng.integers(0, 40))
        E = int(rng.integers(1, 20))
        k = int(rng.integers(1, min(E, 6) + 1))
        bm = int(rng.choice([1, 4, 16, 32]))
        ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32) \
            if T else np.zeros((0, k), np.int32)
        m = A.align_permute(ids, E, bm)
        slots, offsets, blocks = _brute_align(ids.tolist(), E, bm)
        P = A.padded_rows_max(T, k, E, bm)
        assert len(slots) <= P and m["sorted_token_ids"].size == P
        assert m["sorted_token_ids"][:len(slots)].tolist() == slots
        assert np.all(m["sorted_token_ids"][len(slots):] == T * k)
        assert m["expert_offsets"].tolist() == offsets
        assert m["block_expert_ids"][:len(blocks)].tolist() == blocks
        assert np.all(m["block_expert_ids"][len(blocks):] == -1)
        sorted_ids = m["sorted_token_ids"]
        assert np.array_equal(sorted_ids[m["row_pos"]], np.arange(T * k))


def test_gather_rows_pads_with_zero():
    x = np.arange(12, dtype=np.float32).reshape(3, 4)
    ids = np.array([[1, 0], [1, 2], [0, 1]], np.int32)
    m = A.align_permute(ids, 3, 4)
    xp = A.gather_rows(x, m["sorted_token_ids"], 2)
    assert xp.shape == (12, 4)
    assert np.array_equal(xp[0], x[0]) and np.array_equal(xp[1], x[2])
    assert np.all(xp[2] == 0) and np.array_equal(xp[8], x[1])


def test_non_finite_logits_rank_and_weigh_by_their_limits():
    """Closed forms of the non-finite reading: NaN ranks as -inf (ties with
    -inf go to the lower id); a +inf or -inf maximum splits the weight equally
    among the selected logits equal to it; a NaN logit weighs as -inf."""
    nan, inf = np.nan, np.inf
    logits = np.array([[nan, -inf, 0.0, 1.0],      # NaN and -inf tie at -inf: id 0 first
                       [nan, nan, nan, nan],       # all NaN: ids 0, 1, 2; equal weights
                       [inf, 0.0, inf, 1.0],       # two +inf share the weight
                       [-inf, -inf, -inf, -inf],   # all -inf: equal weights
                       [2.0, nan, 2.0, -inf]], np.float32)
    ids, w = R.topk_softmax(logits, 3)
    assert ids.tolist() == [[3, 2, 0], [0, 1, 2], [0, 2, 3], [0, 1, 2], [0, 2, 1]]
    e = np.exp(1.0)
    np.testing.assert_array_equal(w[0], np.float32([e / (e + 1), 1 / (e + 1), 0.0]))
    assert w[1].tolist() == [np.float32(1 / 3)] * 3
    assert w[2].tolist() == [0.5, 0.5, 0.0]
    assert w[3].tolist() == [np.float32(1 / 3)] * 3
    assert w[4].tolist() == [0.5, 0.5, 0.0]
    assert np.all(np.isfinite(w))


def test_non_finite_logits_sigmoid_routing():
    """Sigmoid routing: NaN scores rank as -inf; a NaN logit weighs as s = 0
    (sigmoid(-inf)); selected scores that are all 0 give equal weights."""
    nan, inf = np.nan, np.inf
    logits = np.array([[nan, 0.0, -inf, inf],
                       [nan, nan, -inf, -inf],
                       [-inf, -inf, -inf, -inf]], np.float32)
    bias = np.zeros(4, np.float32)
    ids, w = R.sigmoid_bias_topk(logits, bias, 2)
    # row 0: scores [-inf(NaN), 0.5, 0, 1] -> ids 3, 1; weights 1/(1+0.5), 0.5/1.5
    assert ids.tolist() == [[3, 1], [2, 3], [0, 1]]
    np.testing.assert_array_equal(w[0], np.float32([1 / 1.5, 0.5 / 1.5]))
    assert w[1].tolist() == [0.5, 0.5]
    assert w[2].tolist() == [0.5, 0.5]
