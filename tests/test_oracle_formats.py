"""Pins for the oracle's format tables (CPU only)."""
import math
import os

import numpy as np
import pytest
import torch

from oracle import formats as F
from oracle import layer as L

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(name):
    vals = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                vals.append(float(line))
    return np.array(vals)


def test_e2m1_table_matches_printed_lut():
    lut = _read_golden("e2m1_lut.txt")
    assert lut.shape == (16,)
    assert np.array_equal(F.E2M1_VALUES, lut)
    # code 8 is negative zero, as printed
    assert math.copysign(1.0, F.E2M1_VALUES[8]) == -1.0


def test_e4m3_closed_form_spot_values():
    v = F.E4M3_VALUES
    assert v[0x7E] == 448.0                  # largest finite
    assert v[0x08] == 2.0 ** -6              # smallest normal
    assert v[0x01] == 2.0 ** -9              # smallest subnormal
    assert v[0x07] == 7 * 2.0 ** -9          # largest subnormal
    assert v[0x38] == 1.0                    # exponent field 7 = bias
    assert v[0x39] == 1.125
    assert v[0xB8] == -1.0
    assert np.isnan(v[0x7F]) and np.isnan(v[0xFF])
    assert np.sum(np.isnan(v)) == 2


def test_e4m3_matches_torch_float8():
    b = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = b.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = F.E4M3_VALUES
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(ours))
    assert np.array_equal(ref[~nan], ours[~nan])


def test_e8m0_spot_values():
    v = F.E8M0_VALUES
    assert v[127] == 1.0 and v[128] == 2.0 and v[126] == 0.5
    assert v[0] == 2.0 ** -127 and v[254] == 2.0 ** 127
    assert np.isnan(v[255])


def test_e8m0_matches_torch_if_available():
    if not hasattr(torch, "float8_e8m0fnu"):
        pytest.skip("torch has no float8_e8m0fnu")
    b = torch.arange(255, dtype=torch.int32).to(torch.uint8)
    ref = b.view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    assert np.array_equal(ref, F.E8M0_VALUES[:255])


def test_nibble_order_low_is_even():
    # "two E2M1 nibbles per byte along K (low nibble = even index)":
    # byte 0x71 holds code 1 (0.5) at the even index and code 7 (6.0) at the odd one
    codes = F.unpack_nibbles(np.array([[0x71, 0xF8]], dtype=np.uint8))
    assert codes.tolist() == [[1, 7, 8, 15]]
    vals = F.E2M1_VALUES[codes]
    assert vals[0, 0] == 0.5 and vals[0, 1] == 6.0 and vals[0, 3] == -6.0


def test_bf16_rne_matches_torch():
    rng = np.random.default_rng(1)
    x = np.concatenate([
        rng.standard_normal(20000).astype(np.float32),
        (rng.standard_normal(2000) * 1e-39).astype(np.float32),      # subnormals
        (rng.standard_normal(2000) * 1e38).astype(np.float32),
        np.array([0.0, -0.0, np.inf, -np.inf, 3.3895314e38, 3.4e38,
                  1.00390625, 1.01171875, -1.00390625], dtype=np.float32),
    ])
    # exact ties: bf16 value + half an ulp
    base = rng.standard_normal(1000).astype(np.float32)
    bb = (base.view(np.uint32) & 0xFFFF0000) | 0x8000
    x = np.concatenate([x, bb.astype(np.uint32).view(np.float32)])
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    ours = F.bf16_rne(x)
    assert np.array_equal(ref.view(np.uint32), ours.view(np.uint32))
    assert np.isnan(F.bf16_rne(np.array([np.nan], np.float32))[0])


def test_e2m1_times_e4m3_exact_in_bf16():
    # every product of an E2M1 value and a finite E4M3 scale is a bf16 value
    s = F.E4M3_VALUES[:0x7F]
    prod = F.E2M1_VALUES[:, None] * s[None, :]
    assert np.all(np.isfinite(prod))
    assert np.array_equal(F.bf16_rne(prod.astype(np.float32)).astype(np.float64), prod)
    assert np.array_equal(prod.astype(np.float32).astype(np.float64), prod)


def test_nvfp4_dequant_worked_example():
    # w = E2M1[code] * E4M3(scale) * gscale, the repro's dequant formula.
    # Row 0: bytes 0x21 repeated -> codes (1, 2) = (0.5, 1.0); block scale 0x40
    # = 2.0 (exponent 8 -> 2^1). Row 1: bytes 0x9F -> codes (15, 9) = (-6, -0.5)
    # with block scale 0x30 = 0.5.
    q = np.array([[0x21] * 8, [0x9F] * 8], dtype=np.uint8)
    s = np.array([[0x40], [0x30]], dtype=np.uint8)
    w = L.dequant_nvfp4(q, s)
    assert w.shape == (2, 16)
    assert np.all(w[0, 0::2] == 1.0) and np.all(w[0, 1::2] == 2.0)
    assert np.all(w[1, 0::2] == -3.0) and np.all(w[1, 1::2] == -0.25)


def test_mxfp4_dequant_worked_example():
    q = np.array([[0x73] * 16], dtype=np.uint8)        # codes 3 (1.5), 7 (6.0)
    s = np.array([[130]], dtype=np.uint8)               # 2^3
    w = L.dequant_mxfp4(q, s)
    assert np.all(w[0, 0::2] == 12.0) and np.all(w[0, 1::2] == 48.0)


def test_int4_dequant_worked_example():
    # codes 0x5A -> q = (10, 5) at (even, odd); zero 8 for group 0, scale 0.25
    q = np.array([[0x5A] * 32], dtype=np.uint8)
    s = np.array([[0.25]], dtype=np.float16)
    z = np.array([[0x08]], dtype=np.uint8)
    w = L.dequant_int4(q, s, z)
    assert np.all(w[0, 0::2] == 0.5) and np.all(w[0, 1::2] == -0.75)
    # q == z gives exactly zero
    w0 = L.dequant_int4(np.full((1, 32), 0x88, np.uint8), s, z)
    assert np.all(w0 == 0.0)
