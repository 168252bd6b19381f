"""Row-wise FP8 ("fp8r") weight format oracle: E4M3 elements with one float32
scale per output row.

TEST INFRASTRUCTURE ONLY (see the package docstring).

The pages name the variant only ("fp8r" single-file checkpoints, row-wise
FP8, with fast kernels on compute capability 8.9 and up: "Welcome FLUX.3 Image
Klein in Diffusers", section "Single-file format checkpoints"; "FLUX.3 Image
Klein support" lists the same variants).  The element encoding is the
published OCP FP8 E4M3 definition (``nvfp4.e4m3_value``).  The recipe is a
reading: for each row r (output feature) the scale s_r = amax_r / 448 rounded
to float32 (1 for an all-zero row); each element is the E4M3 code of w / s_r,
round to nearest even, saturating at +-448, no negative zero; every rounding
decision on the float64 quotient.

Canonical layout (both sides must agree on it):
  codes  uint8 [rows, cols]  E4M3 bit patterns (0x7F / 0xFF, the NaNs, never used)
  scales float32 [rows]
"""

import numpy as np

from .nvfp4 import E4M3_MAX, E4M3_TABLE, _E4M3_POS_CODES, _E4M3_POS_VALS, _round_to_grid

__all__ = ["round_to_e4m3_signed", "quantize", "dequantize"]


def round_to_e4m3_signed(v):
    """Encode values to E4M3 codes (sign bit 7), round to nearest even,
    saturating at +-448; zero (of either sign) encodes to 0x00."""
    v = np.asarray(v, np.float64)
    mag = np.minimum(np.abs(v), E4M3_MAX)
    code = _round_to_grid(mag, _E4M3_POS_VALS, _E4M3_POS_CODES)
    return (code | np.where((v < 0) & (code != 0), 0x80, 0)).astype(np.uint8)


def quantize(w):
    """Quantise a [rows, cols] weight to fp8r: (codes uint8 [rows, cols],
    scales float32 [rows])."""
    w = np.asarray(w, np.float64)
    amax = np.abs(w).max(axis=1)
    scales = np.where(amax > 0, (amax / E4M3_MAX).astype(np.float32), np.float32(1.0)).astype(np.float32)
    codes = round_to_e4m3_signed(w / scales.astype(np.float64)[:, None])
    return codes, scales


def dequantize(codes, scales):
    """w = e4m3(code) * s_row, exact in float64."""
    return E4M3_TABLE[np.asarray(codes, np.uint8)] * np.asarray(scales, np.float64)[:, None]
