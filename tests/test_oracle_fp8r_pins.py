"""Pins of the row-wise FP8 ("fp8r") oracle: signed E4M3 rounding against
torch's float8 cast and against brute force, saturation and signed zeros, the
per-row scale definition, and the quantisation error bound."""

import numpy as np
import torch

from oracle import fp8r as R
from oracle import nvfp4 as Q


def test_signed_e4m3_rounding_matches_torch_cast_in_range():
    rng = np.random.default_rng(3)
    mag = np.concatenate([rng.uniform(0, 448, 2000), 2.0 ** rng.uniform(-12, 8.8, 2000),
                          Q.E4M3_TABLE[1:126] * 0.5 + Q.E4M3_TABLE[2:127] * 0.5])   # exact midpoints (ties)
    v = np.minimum(mag, 448.0) * np.where(rng.random(mag.size) < 0.5, -1.0, 1.0)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = R.round_to_e4m3_signed(v)
    nz = Q.E4M3_TABLE[ref] != 0                       # torch keeps the sign of a value rounding to zero
    assert np.array_equal(got[nz], ref[nz])
    assert np.all(got[~nz] == 0)


def test_signed_e4m3_rounding_equals_brute_force_nearest():
    rng = np.random.default_rng(4)
    v = rng.standard_normal(3000) * 2.0 ** rng.uniform(-12, 9, 3000)
    got = R.round_to_e4m3_signed(v)
    mag = np.minimum(np.abs(v), 448.0)
    brute = Q._round_to_grid_brute(mag, Q._E4M3_POS_VALS, Q._E4M3_POS_CODES)
    want = np.where((v < 0) & (brute != 0), brute | 0x80, brute)
    assert np.array_equal(got, want.astype(np.uint8))


def test_saturation_and_zeros():
    got = R.round_to_e4m3_signed(np.array([1e9, -1e9, 448.0, -448.0, 0.0, -0.0, 2.0 ** -11, -(2.0 ** -11)]))
    assert list(got) == [0x7E, 0xFE, 0x7E, 0xFE, 0x00, 0x00, 0x00, 0x00]


def test_row_scale_is_amax_over_448_and_error_bound():
    rng = np.random.default_rng(5)
    w = rng.standard_normal((16, 96)) * 0.02
    w[3] = 0.0                                        # all-zero row: scale 1, codes 0
    codes, scales = R.quantize(w)
    assert codes.shape == w.shape and codes.dtype == np.uint8 and scales.dtype == np.float32
    amax = np.abs(w).max(axis=1)
    for r in range(16):
        if r == 3:
            assert scales[r] == 1.0 and not codes[r].any()
        else:
            assert scales[r] == np.float32(amax[r] / 448.0)
            # the row's largest element lands on (or next to) 448
            assert 0x7D <= int(codes[r][np.argmax(np.abs(w[r]))]) & 0x7F <= 0x7E
    dq = R.dequantize(codes, scales)
    # normal range: relative error <= 2^-4 (half a unit of the 3-bit mantissa);
    # below the smallest normal (2^-6 * s): absolute error <= 2^-10 * s
    s = scales.astype(np.float64)[:, None]
    err = np.abs(dq - w)
    normal = np.abs(w) >= 2.0 ** -6 * s
    assert np.all(err[normal] <= 2.0 ** -4 * np.abs(w[normal]) * (1 + 1e-12))
    assert np.all(err[~normal] <= 2.0 ** -10 * np.broadcast_to(s, w.shape)[~normal] * (1 + 1e-12))
    assert not np.any((codes == 0x7F) | (codes == 0xFF))
