"""Quantisers that turn drawn fp32 expert weights into the layer's 4-bit inputs.

These produce inputs; they are not part of the layer. Each follows the stated
workload recipe, with the readings noted where the recipe leaves a step open:

* NVFP4: global scale gs = amax / (6*448) over the expert's projection; block
  scale s = (block_amax / 6) / gs, rounded to E4M3 (nearest, ties to the even
  code, saturating at 448); codes = E2M1 nearest-even of w / (s_q * gs)
  (saturating at 6); s_q == 0 gives all-zero codes; the sign bit follows w.
* MXFP4: per 32 weights the shared exponent is ceil(log2(amax / 6)), taken
  from frexp so exact powers of two do not move, clamped to [-127, 127];
  codes = E2M1 nearest-even of w / 2^e; amax == 0 gives exponent byte 0.
* GPTQ INT4 (asymmetric min/max, group 64 along K): s = fp16((max-min)/15)
  (0 becomes 1), z = clamp(rne(-min/s), 0, 15), q = clamp(rne(w/s) + z, 0, 15).

All arithmetic is fp32 torch ops on the CPU: the layer generator draws and
quantises every tensor on the host and copies the bytes to the device, so the
GPU runs, the oracle and the timed CPU baseline all read the same bytes.
"""
import torch

# positive E2M1 magnitudes by code 0..7 (1 sign, 2 exponent bits bias 1, 1 mantissa bit)
_E2M1_POS = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def _e4m3_pos_grid():
    vals = []
    for code in range(0x7F):                  # 0x00..0x7E, 0x7F is NaN
        e, m = code >> 3, code & 7
        vals.append((m / 8.0) * 2.0 ** -6 if e == 0 else (1 + m / 8.0) * 2.0 ** (e - 7))
    return vals


_E4M3_POS = _e4m3_pos_grid()


def _nearest_even_code(mag: torch.Tensor, grid) -> torch.Tensor:
    """mag >= 0 (fp32) -> index into the increasing grid of the nearest value;
    ties go to the even index; values past the end saturate to the last."""
    g = torch.tensor(grid, dtype=torch.float32, device=mag.device)
    hi = torch.searchsorted(g, mag.contiguous()).clamp(max=len(grid) - 1)
    lo = (hi - 1).clamp(min=0)
    d_lo = mag - g[lo]
    d_hi = g[hi] - mag
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    idx = torch.where(pick_hi, hi, lo)
    idx = torch.where(mag >= g[-1], torch.full_like(idx, len(grid) - 1), idx)
    return idx.to(torch.uint8)


# E2M1 decision points between neighbouring magnitudes (0, .5, 1, 1.5, 2, 3,
# 4, 6): the midpoints, each with the side an exact tie goes to (the even
# code). A magnitude takes the code equal to the number of points it passes.
_E2M1_MIDS = [(0.25, False), (0.75, True), (1.25, False), (1.75, True), (2.5, False),
              (3.5, True), (5.0, False)]  # (midpoint, tie goes up)


def e2m1_encode(x: torch.Tensor) -> torch.Tensor:
    """fp32 -> E2M1 code (nearest, ties to the even code, saturating at 6;
    the sign bit follows x). Same decisions as the grid search of
    ``_nearest_even_code`` (pinned by a test), as seven comparisons."""
    mag = x.abs()
    code = torch.zeros(x.shape, dtype=torch.uint8)
    for mid, up in _E2M1_MIDS:
        code += (mag >= mid) if up else (mag > mid)
    return code | (torch.signbit(x).to(torch.uint8) << 3)


def e4m3_encode_pos(x: torch.Tensor) -> torch.Tensor:
    """x >= 0 -> E4M3 byte (nearest, ties to even, saturating at 448)."""
    return _nearest_even_code(x, _E4M3_POS)


def e4m3_decode_pos(code: torch.Tensor) -> torch.Tensor:
    g = torch.tensor(_E4M3_POS, dtype=torch.float32, device=code.device)
    return g[code.long()]


def pack_nibbles(codes: torch.Tensor) -> torch.Tensor:
    """[..., K] codes 0..15 -> [..., K/2] bytes, even K index in the low nibble."""
    return (codes[..., 0::2] | (codes[..., 1::2] << 4)).to(torch.uint8)


def quantize_nvfp4(w: torch.Tensor):
    """w fp32 [N, K] -> (packed [N, K/2] u8, scales [N, K/16] E4M3 bytes, gscale fp32 scalar)."""
    N, K = w.shape
    amax = w.abs().max()
    gs = amax / 2688.0                         # 6 * 448
    blk = w.reshape(N, K // 16, 16)
    bamax = blk.abs().amax(dim=-1)
    if float(gs) > 0:
        s = (bamax / 6.0) / gs
    else:
        s = torch.zeros_like(bamax)
    s_code = e4m3_encode_pos(s)
    s_val = e4m3_decode_pos(s_code)
    denom = (s_val * gs).unsqueeze(-1)
    safe = torch.where(denom > 0, denom, torch.ones_like(denom))
    xs = torch.where(denom > 0, blk / safe, torch.zeros_like(blk))
    codes = e2m1_encode(xs).reshape(N, K)
    return pack_nibbles(codes), s_code, gs.to(torch.float32)


def quantize_mxfp4(w: torch.Tensor):
    """w fp32 [N, K] -> (packed [N, K/2] u8, scales [N, K/32] E8M0 bytes)."""
    N, K = w.shape
    blk = w.reshape(N, K // 32, 32)
    amax = blk.abs().amax(dim=-1)
    m, ex = torch.frexp(amax / 6.0)
    e = torch.where(m == 0.5, ex - 1, ex).clamp(-127, 127)
    zero = amax == 0
    e = torch.where(zero, torch.full_like(e, -127), e)
    xs = torch.ldexp(blk, (-e).to(torch.float32).unsqueeze(-1))
    xs = torch.where(zero.unsqueeze(-1), torch.zeros_like(xs), xs)
    codes = e2m1_encode(xs).reshape(N, K)
    return pack_nibbles(codes), (e + 127).to(torch.uint8)


def quantize_int4(w: torch.Tensor):
    """w fp32 [N, K] -> (packed [N, K/2] u8, scales fp16 [N, K/64], zeros [N, ceil(K/128)] u8)."""
    N, K = w.shape
    G = K // 64
    blk = w.reshape(N, G, 64)
    mn = blk.amin(dim=-1)
    mx = blk.amax(dim=-1)
    s = ((mx - mn) / 15.0).to(torch.float16)
    s = torch.where(s == 0, torch.ones_like(s), s)
    s32 = s.to(torch.float32)
    z = torch.round(-mn / s32).clamp(0, 15)
    q = (torch.round(blk / s32.unsqueeze(-1)) + z.unsqueeze(-1)).clamp(0, 15)
    codes = q.to(torch.uint8).reshape(N, K)
    zc = z.to(torch.uint8)
    if G % 2:
        zc = torch.cat([zc, torch.zeros(N, 1, dtype=torch.uint8, device=w.device)], dim=1)
    return pack_nibbles(codes), s, pack_nibbles(zc)
