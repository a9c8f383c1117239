"""Pins for the synthetic-input quantisers, decoded through the oracle's tables
(CPU only). The quantisers make inputs; these check they follow the stated
recipe so the workloads have the intended value distributions."""
import numpy as np
import torch

from oracle import formats as F
from oracle import layer as L
from synth import quantize as Q


def test_e2m1_encode_ties_to_even():
    x = torch.tensor([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 7.0, 100.0, -0.25, -0.3, -5.0])
    codes = Q.e2m1_encode(x).tolist()
    vals = F.E2M1_VALUES[np.array(codes)]
    assert vals.tolist() == [0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0, 6.0, 6.0, -0.0, -0.5, -4.0]


def test_e4m3_encode_matches_torch_cast():
    x = torch.rand(20000, dtype=torch.float32) * 440
    x = torch.cat([x, torch.rand(2000) * 2 ** -6, torch.tensor([0.0, 448.0, 2 ** -9, 2 ** -10])])
    ours = Q.e4m3_encode_pos(x)
    ref = x.to(torch.float8_e4m3fn).view(torch.uint8)
    assert torch.equal(ours, ref)
    assert int(Q.e4m3_encode_pos(torch.tensor([1000.0]))[0]) == 0x7E      # saturates


def test_nvfp4_quantiser_invariants():
    g = torch.Generator().manual_seed(0)
    w = torch.randn(64, 256, generator=g) * 0.02
    q, s, gs = Q.quantize_nvfp4(w)
    assert q.shape == (64, 128) and s.shape == (64, 16)
    assert float(gs) == float(w.abs().max() / 2688.0)
    # the block holding the tensor amax gets the largest scale, 448 (0x7E)
    blk = w.reshape(64, 16, 16).abs().amax(-1)
    i = int(torch.argmax(blk))
    assert int(s.reshape(-1)[i]) == 0x7E
    deq = L.dequant_nvfp4(q.numpy(), s.numpy()) * float(gs)
    step = F.E4M3_VALUES[s.numpy()].repeat(16, 1) * float(gs)
    # round-trip error at most half the widest E2M1 grid gap (2, between 4 and 6) x scale
    err = np.abs(deq - w.double().numpy())
    assert np.all(err <= step * 1.0 + 1e-12)
    rel = np.linalg.norm(deq - w.double().numpy()) / np.linalg.norm(w.double().numpy())
    assert rel < 0.15


def test_mxfp4_quantiser_invariants():
    g = torch.Generator().manual_seed(1)
    w = torch.randn(32, 256, generator=g) * 0.02
    w[0, :32] = 0.0
    w[1, :32] = 0.0
    w[1, 5] = 3.0                                   # amax/6 = 0.5: exact power of two
    q, s = Q.quantize_mxfp4(w)
    sv = F.E8M0_VALUES[s.numpy()]
    assert int(s[0, 0]) == 0                        # amax 0 -> exponent byte 0
    assert sv[1, 0] == 0.5                          # ceil(log2(0.5)) = -1, not 0
    codes = F.unpack_nibbles(q.numpy())
    # no saturation: |w| / 2^e <= 6 for every block
    ratio = np.abs(w.double().numpy()) / np.repeat(sv, 32, axis=1)
    assert np.all(ratio <= 6.0)
    deq = L.dequant_mxfp4(q.numpy(), s.numpy())
    assert deq[1, 5] == 3.0
    assert np.all(np.abs(deq - w.double().numpy()) <= np.repeat(sv, 32, axis=1) * 1.0)
    assert codes.max() <= 15


def test_int4_quantiser_invariants():
    g = torch.Generator().manual_seed(2)
    w = torch.randn(16, 192, generator=g) * 0.02
    w[3, 64:128] = 0.0                              # constant group: scale 0 -> 1
    q, s, z = Q.quantize_int4(w)
    assert q.shape == (16, 96) and s.shape == (16, 3) and z.shape == (16, 2)
    assert float(s[3, 1]) == 1.0
    deq = L.dequant_int4(q.numpy(), s.numpy(), z.numpy())
    sv = s.to(torch.float64).numpy().repeat(64, 1)
    err = np.abs(deq - w.double().numpy())
    assert np.all(err <= sv * 0.5 + np.abs(w.double().numpy()) * 2 ** -8 + 1e-12)
    assert np.all(deq[3, 64:128] == 0.0)


def test_e2m1_encode_comparisons_equal_grid_search():
    """The comparison form of the E2M1 encoder takes the same decisions as the
    nearest-value grid search with ties to the even code, on every exact
    midpoint, its neighbours one fp32 ulp away, and random magnitudes."""
    mids = torch.tensor([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], dtype=torch.float32)
    pts = torch.cat([mids, torch.nextafter(mids, torch.tensor(0.0)), torch.nextafter(mids, torch.tensor(10.0)),
                     torch.tensor([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, 6.5, 1e30, float("inf")]),
                     torch.rand(50000, generator=torch.Generator().manual_seed(3)) * 8])
    x = torch.cat([pts, -pts])
    ref = Q._nearest_even_code(x.abs(), Q._E2M1_POS) | (torch.signbit(x).to(torch.uint8) << 3)
    assert torch.equal(Q.e2m1_encode(x), ref)
