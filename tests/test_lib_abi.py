"""The C-ABI library builds, loads and exports every symbol include/moe4.h
declares; host-only sizing functions agree with the oracle (CPU only)."""
import os
import re

import pytest

import bit_block_scaled_gb300 as moe
from bit_block_scaled_gb300 import build as B
from oracle import align as OA

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    B.build()
    return moe.load()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "moe4.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", src))


def test_exports_every_declared_symbol(lib):
    declared = declared_functions()
    assert declared == set(moe._lib.EXPORTS)
    for name in declared:
        assert hasattr(lib, name), name


def test_padded_rows_matches_oracle(lib):
    for T, k, E, bm in [(16, 2, 8, 16), (64, 4, 32, 16), (1, 4, 128, 16), (4096, 4, 32, 256),
                        (2048, 6, 128, 32), (3, 2, 3, 4 * 4), (0, 2, 4, 16)]:
        assert moe.moe_padded_rows(T, k, E, bm) == OA.padded_rows_max(T, k, E, bm)


def test_workspace_size_and_validation(lib):
    n = moe.moe_workspace_size(64, 32, 4, 2880, 2880, 16)
    P = OA.padded_rows_max(64, 4, 32, 16)
    assert n >= P * 2880 * 2 * 2
    with pytest.raises(moe.MoeError) as e:
        moe.moe_workspace_size(64, 32, 4, 2880 + 32, 2880, 16)      # H % 64 != 0
    assert e.value.code == 1
    with pytest.raises(moe.MoeError):
        moe.moe_workspace_size(64, 300, 4, 2880, 2880, 16)          # E > 256
    with pytest.raises(moe.MoeError):
        moe.moe_workspace_size(64, 32, 9, 2880, 2880, 16)           # k > 8
    with pytest.raises(moe.MoeError):
        moe.moe_workspace_size(64, 32, 4, 2880, 2880, 48)           # block_m


def test_status_strings(lib):
    assert moe.moe_status_string(0) == "MOE_OK"
    assert moe.moe_status_string(4) == "MOE_ERR_TIMEOUT"
    assert moe.moe_status_string(99) == "MOE_ERR_UNKNOWN"


def test_build_entry_point_compiles_for_sm103a():
    assert "arch=compute_103a,code=sm_103a" in " ".join(B.ARCH)
    assert os.path.exists(B.build())


def test_binding_arity_matches_header():
    src = open(os.path.join(ROOT, "include", "moe4.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    for m in re.finditer(r"\b(moe_[a-z0-9_]+)\s*\(([^)]*)\)\s*;", src):
        name, args = m.group(1), m.group(2).strip()
        n = 0 if args in ("", "void") else args.count(",") + 1
        assert len(moe._lib._SIGS[name][1]) == n, name
