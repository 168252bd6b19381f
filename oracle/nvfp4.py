"""NVFP4 weight format oracle: e2m1 values, 16-element e4m3 block scales and a
float32 per-tensor scale.

TEST INFRASTRUCTURE ONLY (see the package docstring).

The pages name the format only ("nvfp4" single-file checkpoints with fast
kernels on Blackwell: "Welcome FLUX.3 Image Klein in Diffusers", section
"Single-file format checkpoints").  The element and scale encodings below are
the published OCP/NVIDIA definitions of FP4 E2M1 and FP8 E4M3; the
quantisation recipe is a reading (blocks of 16 along the input dimension,
per-tensor scale amax / (6 * 448), round-to-nearest-even with saturation).

Canonical byte layout (both sides must agree on it):
  codes  uint8 [rows, cols/2]   element 2i in the low nibble, 2i+1 in the high
  scales uint8 [rows, cols/16]  e4m3 bit patterns, block b covers cols 16b..16b+15
  global float32 scalar
"""

import numpy as np

__all__ = ["e2m1_value", "e4m3_value", "E2M1_TABLE", "E4M3_TABLE",
           "round_to_e2m1", "round_to_e4m3", "quantize", "dequantize", "BLOCK"]

BLOCK = 16
E2M1_MAX = 6.0
E4M3_MAX = 448.0


def e2m1_value(code):
    """FP4 E2M1: sign bit 3, exponent bits 2..1 (bias 1), mantissa bit 0.
    Exponent field 0 is subnormal (0.5 * m); no infinities or NaNs."""
    s = -1.0 if (code >> 3) & 1 else 1.0
    e = (code >> 1) & 3
    m = code & 1
    if e == 0:
        return s * 0.5 * m
    return s * 2.0 ** (e - 1) * (1.0 + 0.5 * m)


def e4m3_value(code):
    """FP8 E4M3 (the "FN" variant): sign bit 7, exponent bits 6..3 (bias 7),
    mantissa bits 2..0.  Exponent 0 is subnormal (2^-6 * m/8); exponent 15 with
    mantissa 7 is NaN; there are no infinities (largest finite 448)."""
    s = -1.0 if (code >> 7) & 1 else 1.0
    e = (code >> 3) & 15
    m = code & 7
    if e == 15 and m == 7:
        return float("nan")
    if e == 0:
        return s * 2.0 ** -6 * (m / 8.0)
    return s * 2.0 ** (e - 7) * (1.0 + m / 8.0)


E2M1_TABLE = np.array([e2m1_value(c) for c in range(16)], dtype=np.float64)
E4M3_TABLE = np.array([e4m3_value(c) for c in range(256)], dtype=np.float64)


def _round_to_grid_brute(mag, grid_vals, grid_codes):
    """Nearest grid value for non-negative ``mag`` (already clamped to the grid
    maximum); ties go to the code with an even mantissa LSB.  Brute force over
    the grid: slow but evidently the definition (pins ``_round_to_grid``)."""
    mag = np.asarray(mag, np.float64)
    d = np.abs(mag[..., None] - grid_vals)                  # [..., G]
    best = d.min(axis=-1, keepdims=True)
    tie_ok = d == best
    # among the tied candidates prefer an even code
    even = (grid_codes % 2 == 0)
    pick_even = tie_ok & even
    has_even = pick_even.any(axis=-1, keepdims=True)
    choose = np.where(has_even, pick_even, tie_ok)
    idx = np.argmax(choose, axis=-1)
    return grid_codes[idx]


def _round_to_grid(mag, grid_vals, grid_codes):
    """Same result as ``_round_to_grid_brute`` in O(log G) per value: the
    grid is increasing, so the nearest value is found by locating ``mag``
    among the midpoints of neighbouring grid values (exact in float64); a
    value equal to a midpoint is a tie and takes the even code of the two."""
    mag = np.asarray(mag, np.float64)
    mid = 0.5 * (grid_vals[:-1] + grid_vals[1:])
    i = np.searchsorted(mid, mag, side="left")          # first midpoint >= mag
    tie = (i < len(mid)) & (mid[np.minimum(i, len(mid) - 1)] == mag)
    lo_code = grid_codes[i]
    hi_code = grid_codes[np.minimum(i + 1, len(grid_codes) - 1)]
    return np.where(tie & (lo_code % 2 != 0), hi_code, lo_code)


_E2M1_POS_CODES = np.arange(8)
_E2M1_POS_VALS = E2M1_TABLE[:8]
_E4M3_POS_CODES = np.arange(127)                             # 0x00..0x7E, finite
_E4M3_POS_VALS = E4M3_TABLE[:127]


def round_to_e2m1(v):
    """Encode values to E2M1 codes, round to nearest even, saturating at +-6."""
    v = np.asarray(v, np.float64)
    sign = (v < 0) | ((v == 0) & np.signbit(v))
    mag = np.minimum(np.abs(v), E2M1_MAX)
    code = _round_to_grid(mag, _E2M1_POS_VALS, _E2M1_POS_CODES)
    code = np.where(code == 0, 0, code)                      # no negative zero
    return (code | np.where(sign & (code != 0), 8, 0)).astype(np.uint8)


def round_to_e4m3(v):
    """Encode non-negative values to E4M3 codes, round to nearest even,
    saturating at 448."""
    mag = np.minimum(np.abs(np.asarray(v, np.float64)), E4M3_MAX)
    return _round_to_grid(mag, _E4M3_POS_VALS, _E4M3_POS_CODES).astype(np.uint8)


def quantize(w):
    """Quantise a [rows, cols] weight (cols % 16 == 0) to NVFP4.

    global g = amax(|W|) / (6 * 448) (float32); block scale
    s_b = e4m3(amax_b / (6 g)); element code q = e2m1(w / (s_b g)); a block
    whose scale encodes to 0 stores zeros.  Returns (codes, scales, g) in the
    canonical layout of the module docstring."""
    w = np.asarray(w, np.float64)
    rows, cols = w.shape
    assert cols % BLOCK == 0
    amax = np.abs(w).max()
    g = np.float32(amax / (E2M1_MAX * E4M3_MAX)) if amax > 0 else np.float32(1.0)
    g64 = float(g)
    blocks = w.reshape(rows, cols // BLOCK, BLOCK)
    amax_b = np.abs(blocks).max(axis=-1)
    s_code = round_to_e4m3(amax_b / (E2M1_MAX * g64))
    s_val = E4M3_TABLE[s_code]
    denom = (s_val * g64)[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(denom > 0, blocks / np.where(denom > 0, denom, 1.0), 0.0)
    q = round_to_e2m1(ratio).reshape(rows, cols)
    codes = (q[:, 0::2] & 0xF) | ((q[:, 1::2] & 0xF) << 4)
    return codes.astype(np.uint8), s_code.astype(np.uint8), g


def dequantize(codes, scales, g):
    """Inverse of the canonical layout: w = e2m1(q) * e4m3(s_b) * g."""
    codes = np.asarray(codes, np.uint8)
    rows = codes.shape[0]
    lo = codes & 0xF
    hi = codes >> 4
    q = np.empty((rows, codes.shape[1] * 2), dtype=np.uint8)
    q[:, 0::2] = lo
    q[:, 1::2] = hi
    vals = E2M1_TABLE[q]
    s = E4M3_TABLE[np.asarray(scales, np.uint8)]
    return vals * np.repeat(s, BLOCK, axis=1) * float(g)
