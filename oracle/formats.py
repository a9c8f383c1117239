"""Number formats used by the 4-bit expert weights, decoded by explicit tables.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

Every table below is generated from the format's definition (sign, exponent
field, mantissa field, bias) and then pinned by tests against values the pages
print or against an independent library routine:

* E2M1 (FP4): 1 sign, 2 exponent bits (bias 1), 1 mantissa bit. The repro in
  the vLLM issue "moe_wna16_marlin_gemm applies wrong per-row topk weights",
  section "Minimal repro", prints the 16-entry value table
  (0, .5, 1, 1.5, 2, 3, 4, 6 and their negatives). Pinned: all 16 codes.
* E4M3 ("fn" variant, the NVFP4 block scale, "group 16" in the same issue):
  1 sign, 4 exponent bits (bias 7), 3 mantissa bits, no infinities, 0x7F and
  0xFF are NaN, largest finite 448. Pinned: closed-form spot values and the
  library decode of ``torch.float8_e4m3fn``.
* E8M0 (the MXFP4 group-32 scale): 8-bit biased exponent, value 2^(b-127),
  255 is NaN. Pinned: spot values.
* bf16 round-to-nearest-even from float32 by the textbook bit method.
  Pinned: ``torch.Tensor.to(torch.bfloat16)`` on random and edge values.
"""
import numpy as np


def _e2m1_value(code: int) -> float:
    sign = -1.0 if (code >> 3) & 1 else 1.0
    exp_field = (code >> 1) & 0x3
    man = code & 0x1
    if exp_field == 0:                       # subnormal: m/2 * 2^(1-bias)
        mag = man * 0.5
    else:                                    # normal: (1 + m/2) * 2^(e-bias)
        mag = (1.0 + man / 2.0) * 2.0 ** (exp_field - 1)
    return sign * mag


def _e4m3_value(b: int) -> float:
    sign = -1.0 if (b >> 7) & 1 else 1.0
    exp_field = (b >> 3) & 0xF
    man = b & 0x7
    if exp_field == 0xF and man == 0x7:      # the only NaN encodings
        return float("nan")
    if exp_field == 0:                        # subnormal: m/8 * 2^(1-7)
        mag = (man / 8.0) * 2.0 ** -6
    else:
        mag = (1.0 + man / 8.0) * 2.0 ** (exp_field - 7)
    return sign * mag


def _e8m0_value(b: int) -> float:
    if b == 0xFF:
        return float("nan")
    return 2.0 ** (b - 127)


#: value of each 4-bit E2M1 code, index = code (bit 3 = sign)
E2M1_VALUES = np.array([_e2m1_value(c) for c in range(16)], dtype=np.float64)
#: value of each E4M3 byte
E4M3_VALUES = np.array([_e4m3_value(b) for b in range(256)], dtype=np.float64)
#: value of each E8M0 byte
E8M0_VALUES = np.array([_e8m0_value(b) for b in range(256)], dtype=np.float64)


def unpack_nibbles(packed: np.ndarray) -> np.ndarray:
    """[..., K/2] uint8 -> [..., K] codes. The low nibble holds the even K index
    (the repro's comment "two E2M1 nibbles per byte along K (low nibble = even
    index)")."""
    packed = np.asarray(packed, dtype=np.uint8)
    lo = packed & 0x0F
    hi = packed >> 4
    out = np.empty(packed.shape[:-1] + (packed.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = lo
    out[..., 1::2] = hi
    return out


def bf16_rne(x) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even); returns
    float32 holding the bf16 value. NaN stays NaN (made quiet), infinities
    stay infinite, overflow past the largest bf16 goes to infinity."""
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    u = x.view(np.uint32).astype(np.uint64)
    nan = np.isnan(x)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) & 0xFFFF0000).astype(np.uint32)
    r = np.where(nan, (u.astype(np.uint32) | 0x00400000) & 0xFFFF0000, r)
    return r.astype(np.uint32).view(np.float32)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """uint16 bf16 bit patterns -> float32 values (exact)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32)


def f32_to_bf16_bits(x) -> np.ndarray:
    """float32 values that are already bf16-exact -> uint16 bit patterns."""
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    return (x.view(np.uint32) >> 16).astype(np.uint16)


def f32(x) -> np.ndarray:
    """Round (float64) values to float32 (round to nearest even)."""
    return np.asarray(x, dtype=np.float64).astype(np.float32)
