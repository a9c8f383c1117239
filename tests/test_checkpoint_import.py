"""Checkpoint-layout import (host functions of the C ABI, CPU only).

GPTQ INT4: the pages name the per-expert tensors (qweight, qzeros, scales,
g_idx; "Serving gpt-oss with mixed GPTQ experts", section "1. Quantize") and
print what qweight is: the int32 [K/8, N] view of the [N, K/2] code bytes
(NVFP4 Marlin issue, "Reproducer"). The converter is pinned to that
definition, and its output, dequantised by the oracle, to the GPTQ formula
(code - zero) * scale evaluated on the GPTQ tensors themselves.
ModelOpt NVFP4: weight_scale_2 is one scalar broadcast to every expert
(NVFP4 gpt-oss report, "Gap 2", 2b).
"""
import ctypes

import numpy as np
import pytest
import torch

import bit_block_scaled_gb300 as moe
from bit_block_scaled_gb300 import build as B
from oracle import formats as OF
from oracle import layer as OL
from synth.quantize import quantize_int4


@pytest.fixture(scope="module", autouse=True)
def lib():
    B.build()
    return moe.load()


def _layer(N, K, seed, min_zero=0):
    g = torch.Generator().manual_seed(seed)
    w = torch.randn(N, K, generator=g) * 0.02
    q, s, z = quantize_int4(w)
    q, s, z = q.numpy(), s.numpy(), z.numpy()
    if min_zero:  # zero points of at least min_zero (for the "minus one" storage)
        zc = OL.int4_zero_codes(z, K // 64).astype(np.uint8)
        zc = np.maximum(zc, min_zero)
        if zc.shape[1] % 2:
            zc = np.concatenate([zc, np.zeros((N, 1), np.uint8)], axis=1)
        z = (zc[:, 0::2] | (zc[:, 1::2] << 4)).astype(np.uint8)
    return q, s, z


def _gptq_tensors(q, s, z, K, zero_offset=0):
    """The GPTQ tensors of a layer given in this library's layout."""
    N = q.shape[0]
    G = K // 64
    # qweight: the int32 view of the [N, K/2] code bytes, transposed (as printed)
    qweight = np.ascontiguousarray(q.view("<i4").T)
    # qzeros: eight 4-bit zero points along N per int32, output 8m + j in bits 4j
    zc = OL.int4_zero_codes(z, G).astype(np.int64) - zero_offset  # [N, G]
    assert zc.min() >= 0
    qzeros = np.zeros((G, N // 8), dtype=np.int64)
    for j in range(8):
        qzeros |= zc[j::8, :].T << (4 * j)
    qzeros = qzeros.astype(np.uint32).view(np.int32)
    return qweight, qzeros, np.ascontiguousarray(s.T), np.arange(K, dtype=np.int32) // 64


@pytest.mark.parametrize("N,K", [(64, 64), (128, 192), (192, 2880)])
def test_gptq_import_restores_the_layout(N, K):
    q, s, z = _layer(N, K, seed=N + K)
    qw, qz, sc, gi = _gptq_tensors(q, s, z, K)
    q2, s2, z2 = moe.moe_import_gptq_int4(qw, qz, sc, gi)
    assert np.array_equal(q2, q)
    assert np.array_equal(s2.view(np.uint16), s.view(np.uint16))
    assert np.array_equal(z2, z)


def test_gptq_import_zero_offset_one():
    N, K = 128, 256
    q, s, z = _layer(N, K, seed=4, min_zero=1)
    qw, qz, sc, _ = _gptq_tensors(q, s, z, K, zero_offset=1)
    q2, s2, z2 = moe.moe_import_gptq_int4(qw, qz, sc, None, zero_offset=1)
    assert np.array_equal(q2, q) and np.array_equal(z2, z)
    assert np.array_equal(s2.view(np.uint16), s.view(np.uint16))


def test_gptq_import_dequantises_to_the_gptq_formula():
    """Oracle dequantisation of the imported layer equals bf16((code - zero) *
    scale) computed straight from the GPTQ tensors (codes read from qweight's
    nibbles, zeros from qzeros', scales from the [K/64, N] table)."""
    N, K = 128, 320
    q, s, z = _layer(N, K, seed=9)
    qw, qz, sc, gi = _gptq_tensors(q, s, z, K)
    q2, s2, z2 = moe.moe_import_gptq_int4(qw, qz, sc, gi)
    got = OL.dequant_int4(q2, s2, z2)
    u = qw.view(np.uint32).astype(np.int64)                      # [K/8, N]
    codes = np.stack([(u >> (4 * j)) & 0xF for j in range(8)], axis=1).reshape(K, N)
    uz = qz.view(np.uint32).astype(np.int64)                     # [K/64, N/8]
    zeros = np.stack([(uz >> (4 * j)) & 0xF for j in range(8)], axis=2).reshape(K // 64, N)
    scales = sc.astype(np.float64)                               # [K/64, N]
    ref = (codes - np.repeat(zeros, 64, axis=0)) * np.repeat(scales, 64, axis=0)
    assert np.array_equal(got, OF.bf16_rne(ref.T))


def test_gptq_import_rejections():
    N, K = 64, 128
    q, s, z = _layer(N, K, seed=1)
    qw, qz, sc, gi = _gptq_tensors(q, s, z, K)
    with pytest.raises(moe.MoeError) as e:
        moe.moe_import_gptq_int4(qw, qz, sc, gi, group_size=128)
    assert e.value.code == 2
    perm = gi.copy()
    perm[[0, 64]] = perm[[64, 0]]
    with pytest.raises(moe.MoeError) as e:                      # act-order g_idx
        moe.moe_import_gptq_int4(qw, qz, sc, perm)
    assert e.value.code == 2
    qz15 = qz.copy()
    qz15[0, 0] |= 0xF
    with pytest.raises(moe.MoeError) as e:                      # 15 + 1 is no 4-bit zero
        moe.moe_import_gptq_int4(qw, qz15, sc, None, zero_offset=1)
    assert e.value.code == 2
    with pytest.raises(moe.MoeError) as e:
        moe.moe_import_gptq_int4(qw, qz, sc, None, zero_offset=2)
    assert e.value.code == 1


def test_gptq_import_writes_nothing_on_error():
    N, K = 64, 128
    q, s, z = _layer(N, K, seed=2)
    qw, qz, sc, _ = _gptq_tensors(q, s, z, K)
    qz[1, 2] |= 0xF << 4
    outs = [np.full((N, K // 2), 0xAB, np.uint8), np.full((N, K // 64), 0x1234, np.uint16),
            np.full((N, 1), 0xCD, np.uint8)]
    before = [o.copy() for o in outs]
    p = lambda a: ctypes.c_void_p(a.ctypes.data)
    rc = moe.load().moe_import_gptq_int4(p(qw), p(qz), p(sc), None, K, N, 64, 1, *[p(o) for o in outs])
    assert rc == 2
    assert all(np.array_equal(a, b) for a, b in zip(outs, before))


def test_modelopt_global_scale_broadcast():
    g = moe.moe_import_modelopt_global_scale(3.0517578125e-05, 32)
    assert g.dtype == np.float32 and g.shape == (32,)
    assert np.all(g == np.float32(3.0517578125e-05))
    with pytest.raises(moe.MoeError) as e:
        moe.moe_import_modelopt_global_scale(1.0, 0)
    assert e.value.code == 1
