"""Pins for the oracle's NVFP4 quantizer (CPU only).

The pages take A, B and their scales already quantized and print no quantizer;
the recipe (stated in oracle/nvfp4_oracle.c) is the plainest reading of the
formats they name: one E4M3 scale per 16 consecutive values equal to the
block's amax / 6 rounded to nearest-even, and each value divided by the decoded
scale and rounded to nearest-even on the E2M1 grid, saturating at 6.  These
tests pin the encoders against the formats' value lists (closed forms), against
torch's float8_e4m3fn conversion, and the whole quantizer against a block worked
by hand and against invariants (block independence, error bound, exact grid
values).
"""
import numpy as np
import pytest
import torch

import oracle

# E2M1: 1 sign bit, 2 exponent bits (bias 1), 1 mantissa bit; codes 0..7.
E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def f32(x):
    return np.float32(x)


def test_e2m1_encode_round_trips_every_code():
    for c, v in enumerate(E2M1):
        assert oracle.e2m1_encode(v)[()] == c
        assert oracle.e2m1_encode(-v)[()] == (c | 8)   # sign bit, -0.0 included


def test_e2m1_midpoints_go_to_the_even_code():
    for c in range(7):
        mid = f32((E2M1[c] + E2M1[c + 1]) / 2)
        assert oracle.e2m1_encode(mid)[()] == (c if c % 2 == 0 else c + 1), mid
        below = np.nextafter(mid, f32(0))
        above = np.nextafter(mid, f32(10))
        assert oracle.e2m1_encode(below)[()] == c
        assert oracle.e2m1_encode(above)[()] == c + 1
        assert oracle.e2m1_encode(-above)[()] == (c + 1) | 8


def test_e2m1_saturates_at_six():
    for v in (6.0, 6.5, 7.0, 1e30, np.inf):
        assert oracle.e2m1_encode(v)[()] == 7
        assert oracle.e2m1_encode(-v)[()] == 15


def test_e4m3_encode_round_trips_every_finite_code():
    table = oracle.e4m3_table()
    for c in range(256):
        if c in (0x7F, 0xFF):
            continue
        assert oracle.e4m3_encode(f32(table[c]))[()] == c, hex(c)


def test_e4m3_midpoints_saturation_and_underflow():
    table = oracle.e4m3_table()
    for c in range(0x7E):
        mid = (table[c] + table[c + 1]) / 2          # exact in fp32: both are short binary fractions
        assert f32(mid) == mid
        assert oracle.e4m3_encode(f32(mid))[()] == (c if c % 2 == 0 else c + 1), hex(c)
        assert oracle.e4m3_encode(np.nextafter(f32(mid), f32(0)))[()] == c
        assert oracle.e4m3_encode(np.nextafter(f32(mid), f32(1e9)))[()] == c + 1
    for v in (448.0, 449.0, 464.0, 480.0, 1e9, np.inf):
        assert oracle.e4m3_encode(v)[()] == 0x7E      # largest finite, 1.75 * 2^8
    assert oracle.e4m3_encode(2.0 ** -10)[()] == 0    # half the smallest subnormal: tie -> even (0)
    assert oracle.e4m3_encode(np.nextafter(f32(2.0 ** -10), f32(1)))[()] == 1
    assert oracle.e4m3_encode(0.0)[()] == 0


def test_e4m3_encode_matches_torch_in_range():
    rng = np.random.default_rng(5)
    v = np.exp2(rng.uniform(-12, np.log2(440), 200000)).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.e4m3_encode(v), ref)


def test_worked_block():
    """amax 6 -> scale 6/6 = 1.0 = E4M3 0x38; 1.5 -> code 3; -3.0 -> 8|5; 0.7 is
    0.2 from 0.5 and 0.3 from 1.0 -> code 1; 6.0 -> 7; low nibble = even k."""
    x = np.zeros((1, 1, 32), np.float32)
    x[0, 0, :4] = [1.5, -3.0, 0.7, 6.0]
    x[0, 0, 16:20] = [0.1, 0.2, -0.05, 0.0]      # second block: amax 0.2 -> 0.2/6 -> E4M3
    codes, sf = oracle.quantize(x, 1, 32)
    assert codes[0, 0, :8].tolist() == [0xD3, 0x71, 0, 0, 0, 0, 0, 0]
    assert sf[0, 0, 0] == 0x38
    # 0.2/6 = 0.03333 lies between 0.03125 (2^-5, code 0x10) and 0.03515625 (0x11);
    # it is 0.00208 above the first and 0.00182 below the second -> 0x11.
    assert sf[0, 0, 1] == 0x11
    d = 0.03515625
    # 0.1/d = 2.844 -> 3 (code 5); 0.2/d = 5.689 -> 6 (code 7); -0.05/d = -1.422 -> -1.5 (8|3); 0 -> 0
    assert codes[0, 0, 8:10].tolist() == [0x75, 0x0B]


def test_zero_and_underflowing_blocks_give_zero():
    x = np.zeros((1, 2, 16), np.float32)
    x[0, 1, :] = 1e-4                             # amax/6 below half the smallest E4M3 subnormal
    codes, sf = oracle.quantize(x, 2, 16)
    assert not sf.any() and not codes.any()


def test_blocks_rows_and_batches_are_independent():
    rng = np.random.default_rng(1)
    L, rows, K = 2, 5, 64
    x = rng.standard_normal((L, rows, K)).astype(np.float32)
    codes, sf = oracle.quantize(x, rows, K, L)
    for l in range(L):
        for r in range(rows):
            for b in range(K // 16):
                cb, sb = oracle.quantize(x[l, r, b * 16:(b + 1) * 16].copy(), 1, 16)
                assert sb[0, 0, 0] == sf[l, r, b]
                assert np.array_equal(cb[0, 0], codes[l, r, b * 8:(b + 1) * 8])


def _dequant(codes, sf, K):
    e2m1 = oracle.e2m1_table()
    e4m3 = oracle.e4m3_table()
    lo = codes & 0xF
    hi = codes >> 4
    q = np.stack([lo, hi], axis=-1).reshape(codes.shape[:-1] + (K,))
    d = np.repeat(e4m3[sf], 16, axis=-1)
    return e2m1[q] * d, d


def test_dequantization_error_bound():
    """Each value lands within half a grid step of d*code: d/4 below 2, d/2
    below 4, and at most d above (step 2 between 4 and 6, plus saturation of
    at most 6 * 2^-4 when a normal scale rounded down).  Subnormal scales
    (codes below 0x08) round more coarsely; there the values beyond 6 d
    saturate to 6 d exactly."""
    rng = np.random.default_rng(2)
    x = (rng.standard_normal((3, 64, 256)) * np.exp2(rng.integers(-6, 6, (3, 64, 1)))).astype(np.float32)
    x = torch.from_numpy(x).to(torch.bfloat16).float().numpy()      # bf16-representable inputs
    codes, sf = oracle.quantize(x, 64, 256, 3)
    deq, d = _dequant(codes, sf, 256)
    err = np.abs(x - deq)
    r = np.abs(x) / d
    bound = np.where(r <= 2, d / 4, np.where(r <= 4, d / 2, d))
    normal = np.repeat(sf >= 0x08, 16, axis=-1)
    assert normal.mean() > 0.5 and (~normal).any()            # both kinds of block occur
    assert (err[normal] <= bound[normal] * (1 + 1e-6)).all()
    sat = ~normal & (r > 6)
    assert (np.abs(deq[sat]) == 6 * d[sat]).all() and (np.sign(deq[sat]) == np.sign(x[sat])).all()
    assert (err[~normal & ~sat] <= bound[~normal & ~sat] * (1 + 1e-6)).all()


def test_exact_grid_values_round_trip():
    """Blocks whose values are d * (E2M1 grid) with amax = 6 d and d an E4M3
    value quantize exactly: scale code of d, codes of the grid values."""
    rng = np.random.default_rng(3)
    table = oracle.e4m3_table()
    for _ in range(50):
        sc = int(rng.integers(0x20, 0x60))
        d = table[sc]
        codes_in = rng.integers(0, 16, 16)
        codes_in[0] = 7                           # amax = 6 d
        vals = np.array([(-1 if c & 8 else 1) * E2M1[c & 7] * d for c in codes_in], np.float32)
        codes, sf = oracle.quantize(vals, 1, 16)
        assert sf[0, 0, 0] == sc
        got = np.stack([codes[0, 0] & 0xF, codes[0, 0] >> 4], -1).ravel()
        want = np.where(np.array([E2M1[c & 7] for c in codes_in]) == 0, codes_in & 8, codes_in)
        assert np.array_equal(got, want)
