"""Pins of the NVFP4 oracle: the E2M1 and E4M3 code tables against their
format definitions and against torch's float8 type, rounding ties, saturation,
and the quantisation error bound."""

import numpy as np
import torch

from oracle import nvfp4 as Q


def test_e2m1_table_is_the_format_grid():
    assert list(Q.E2M1_TABLE[:8]) == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    assert list(Q.E2M1_TABLE[8:]) == [-0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]


def test_e4m3_table_matches_torch_float8_e4m3fn():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(Q.E4M3_TABLE))
    assert np.array_equal(Q.E4M3_TABLE[~nan], ref[~nan])
    assert Q.E4M3_TABLE[0x7E] == 448.0 and Q.E4M3_TABLE[0x01] == 2.0 ** -9
    assert np.sum(np.isfinite(Q.E4M3_TABLE)) == 254


def test_e2m1_rounding_ties_to_even_and_saturates():
    vals = np.array([0.24, 0.25, 0.26, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 7.0, 100.0, -0.75, -5.0, -0.1])
    want = [0.0, 0.0, 0.5, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0, 6.0, 6.0, -1.0, -4.0, 0.0]
    got = Q.E2M1_TABLE[Q.round_to_e2m1(vals)]
    assert list(got) == want


def test_e4m3_rounding_matches_torch_cast_in_range():
    rng = np.random.default_rng(0)
    v = np.concatenate([rng.uniform(0, 448, 2000), 2.0 ** rng.uniform(-12, 8.8, 2000),
                        Q.E4M3_TABLE[1:126] * 0.5 + Q.E4M3_TABLE[2:127] * 0.5])   # exact midpoints
    v = np.minimum(v, 448.0)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(Q.round_to_e4m3(v), ref)
    assert Q.round_to_e4m3(np.array([1e6]))[0] == 0x7E        # saturates to 448


def test_quantise_dequantise_error_bound_and_layout():
    rng = np.random.default_rng(1)
    w = rng.standard_normal((8, 64)) * 0.02
    w[3, 16:32] = 0.0                                           # an all-zero block
    codes, scales, g = Q.quantize(w)
    assert codes.shape == (8, 32) and scales.shape == (8, 4) and codes.dtype == np.uint8
    assert np.float32(g) == np.float32(np.abs(w).max() / (6 * 448))
    wq = Q.dequantize(codes, scales, g)
    s = Q.E4M3_TABLE[scales] * float(g)
    # largest grid step is 2 (between 4 and 6): error <= half a local step * s_b * g,
    # bounded by 1 * s_b * g; for |q| <= 2 the step is 0.5 -> error <= 0.25 s_b g
    err = np.abs(wq - w).reshape(8, 4, 16)
    assert np.all(err <= 1.0 * s[..., None] + 1e-18)
    small = np.abs(w).reshape(8, 4, 16) <= 2 * s[..., None]
    assert np.all(err[small] <= 0.25 * np.broadcast_to(s[..., None], err.shape)[small] * (1 + 1e-12))
    assert np.all(wq[3, 16:32] == 0.0)
    # nibble order: element 2i low nibble, 2i+1 high nibble
    e0 = Q.E2M1_TABLE[codes[0, 0] & 0xF] * Q.E4M3_TABLE[scales[0, 0]] * float(g)
    e1 = Q.E2M1_TABLE[codes[0, 0] >> 4] * Q.E4M3_TABLE[scales[0, 0]] * float(g)
    assert (e0, e1) == (wq[0, 0], wq[0, 1])
    # the block maximum maps to the top of the grid (6) up to the scale rounding
    blk = np.abs(w[0, :16]).max()
    assert abs(blk / (Q.E4M3_TABLE[scales[0, 0]] * float(g)) - 6.0) < 6.0 * 2 ** -3


def test_fast_grid_rounding_equals_brute_force_definition():
    """The searchsorted rounding used by quantize() picks exactly what the
    brute-force nearest-value search (ties to the even code) picks: on random
    values, on every grid value, on every midpoint (a tie) and one ulp either
    side of it, for both the E2M1 and the E4M3 grids."""
    rng = np.random.default_rng(5)
    for vals, codes in ((Q._E2M1_POS_VALS, Q._E2M1_POS_CODES), (Q._E4M3_POS_VALS, Q._E4M3_POS_CODES)):
        mid = 0.5 * (vals[:-1] + vals[1:])
        x = np.concatenate([rng.uniform(0, vals[-1], 50000), vals, mid, np.nextafter(mid, 0),
                            np.nextafter(mid, np.inf), vals[-1] * 2.0 ** rng.uniform(-16, 0, 5000)])
        x = np.minimum(x, vals[-1])
        assert np.array_equal(Q._round_to_grid(x, vals, codes), Q._round_to_grid_brute(x, vals, codes))
