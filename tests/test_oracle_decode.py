"""Pins for the oracle's decode tables (CPU only).

E2M1: the value list of the OCP Microscaling (MX) v1.0 FP4 E2M1 element type
(magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6; bit 3 is the sign) plus invariants.
E4M3: exhaustive comparison with torch's float8_e4m3fn conversion (a library
routine), NaN only at 0x7F / 0xFF, largest finite 448.
"""
import math

import numpy as np
import torch

import oracle

# OCP MX v1.0, FP4 E2M1: codes 0..7 in order.
E2M1_MAGNITUDES = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_e2m1_matches_published_value_list():
    t = oracle.e2m1_table()
    for code in range(8):
        assert t[code] == E2M1_MAGNITUDES[code]
        assert t[code + 8] == -E2M1_MAGNITUDES[code]


def test_e2m1_sign_and_zero():
    t = oracle.e2m1_table()
    assert math.copysign(1.0, t[0]) == 1.0
    assert math.copysign(1.0, t[8]) == -1.0          # 0x8 is -0
    for code in range(16):
        assert t[code] == -t[code ^ 8]
    assert np.all(np.diff(t[:8]) > 0)                 # magnitudes strictly increase
    assert np.all(np.isfinite(t))                     # no Inf / NaN codes


def test_e4m3_exhaustive_against_torch():
    t = oracle.e4m3_table()
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(t), nan)
    assert np.array_equal(np.nonzero(nan)[0], [0x7F, 0xFF])
    assert np.array_equal(t[~nan], ref[~nan])
    # signed zeros
    assert math.copysign(1.0, t[0x80]) == -1.0 and t[0x80] == 0.0


def test_e4m3_extremes():
    t = oracle.e4m3_table()
    finite = t[np.isfinite(t)]
    assert finite.max() == 448.0 and finite.min() == -448.0
    assert t[0x01] == 2.0 ** -9                        # smallest subnormal
    assert t[0x08] == 2.0 ** -6                        # smallest normal
    assert t[0x38] == 1.0
