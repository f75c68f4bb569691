"""Pins of the parity checker itself (``oracle.tolerance`` / ``oracle.compare``),
which decides every GPU parity test.

The bound is the one the problem statement fixes for the GPU output:
|gpu - ref| <= 1e-3 * sum_k |a_k b_k| + 1 fp16 ulp of ref, elementwise, with
ulp(x) = 2^(max(floor(log2|x|), -14) - 10) (fp16 spacing at x; subnormal
spacing 2^-24 below 2^-14) and ulp(0) = 2^-24.  Infinities must match exactly
and NaN never passes.

The values below come from the fp16 format (10 fraction bits, minimum normal
exponent -14), not from the checker's own formula: each test shows that the
checker accepts the last representable value inside the bound and rejects the
first one outside it.  The mutation tests at the full workload shapes show that
the bound, at K up to 16384, still rejects the plausible mistakes of a GEMM
kernel: a dropped scale block, swapped nibbles, SFA and SFB exchanged.
"""
import numpy as np
import pytest
import torch

import oracle
from block_scaled_fp4_nvfp4_gb300 import workloads


def f16(x):
    return np.float16(x)


@pytest.mark.parametrize("ref,ulp", [
    (0.0, 2.0 ** -24),               # zero: smallest subnormal spacing
    (2.0 ** -24, 2.0 ** -24),        # smallest subnormal
    (3 * 2.0 ** -20, 2.0 ** -24),    # a subnormal: fixed spacing 2^-24
    (2.0 ** -14, 2.0 ** -24),        # smallest normal: spacing 2^-14 * 2^-10
    (1.0, 2.0 ** -10),
    (1.5, 2.0 ** -10),
    (-1.999, 2.0 ** -10),
    (2.0, 2.0 ** -9),
    (1000.0, 0.5),                   # [512, 1024): spacing 2^-1
    (65504.0, 32.0),                 # largest finite fp16: spacing 2^5
])
def test_ulp_term_equals_fp16_spacing(ref, ulp):
    r = f16(ref)
    tol = oracle.tolerance(np.array([r]), np.array([0.0]))[0]
    assert tol == ulp
    # the same spacing, read off the format: distance to the next fp16 away from zero
    if r != 0:
        a = np.abs(r)
        with np.errstate(over="ignore"):
            up = np.nextafter(a, np.float16(np.inf))
        if np.isfinite(up):
            assert float(up) - float(a) == ulp
        else:   # the largest finite value: the spacing below it (not a power of two)
            assert float(a) - float(np.nextafter(a, np.float16(0))) == ulp


@pytest.mark.parametrize("ref,absacc", [(1.0, 0.0), (1.0, 10.0), (-37.25, 3.0e4), (0.0, 0.0), (0.0, 0.5),
                                        (2.0 ** -20, 2.0 ** -10), (60000.0, 1.0e5), (-0.5, 123.0)])
@pytest.mark.parametrize("side", [1, -1])
def test_last_value_inside_is_accepted_first_outside_rejected(ref, absacc, side):
    r = f16(ref)
    tol = 1e-3 * absacc + float(oracle.tolerance(np.array([r]), np.array([0.0]))[0])
    # walk fp16 values away from ref on one side until the bound is crossed
    g = r
    direction = np.float16(np.inf) if side > 0 else np.float16(-np.inf)
    inside = r
    while True:
        nxt = np.nextafter(g, direction)
        if not np.isfinite(nxt):
            break
        if abs(float(nxt) - float(r)) <= tol:
            inside = nxt
            g = nxt
            continue
        outside = nxt
        break
    ok_in, ratio_in, _ = oracle.compare(np.array([inside]), np.array([r]), np.array([absacc]))
    ok_out, ratio_out, _ = oracle.compare(np.array([outside]), np.array([r]), np.array([absacc]))
    assert ok_in and ratio_in <= 1.0
    assert not ok_out and ratio_out > 1.0


def test_error_exactly_at_the_bound_passes():
    # ref 1.0, absacc 1000: bound = 1.0 + 2^-10; 2.0 is at distance 1.0, inside
    ok, ratio, _ = oracle.compare(np.array([f16(2.0)]), np.array([f16(1.0)]), np.array([1000.0]))
    assert ok and ratio <= 1.0
    # absacc 999: bound = 0.999 + 2^-10 < 1.0
    ok, ratio, _ = oracle.compare(np.array([f16(2.0)]), np.array([f16(1.0)]), np.array([999.0]))
    assert not ok and ratio > 1.0


def test_infinities_must_match_exactly():
    inf = np.float16(np.inf)
    big = np.array([1e12])
    assert oracle.compare(np.array([inf]), np.array([inf]), big)[0]
    assert oracle.compare(np.array([-inf]), np.array([-inf]), big)[0]
    assert not oracle.compare(np.array([-inf]), np.array([inf]), big)[0]      # wrong sign
    assert not oracle.compare(np.array([f16(65504.0)]), np.array([inf]), big)[0]  # finite vs Inf
    assert not oracle.compare(np.array([inf]), np.array([f16(65504.0)]), big)[0]  # Inf vs finite
    assert not oracle.compare(np.array([inf]), np.array([f16(1.0)]), big)[0]


def test_nan_never_passes():
    nan = np.float16(np.nan)
    huge = np.array([1e30])
    for g, r in [(nan, f16(1.0)), (f16(1.0), nan), (nan, nan), (nan, f16(0.0)), (nan, np.float16(np.inf))]:
        ok, ratio, _ = oracle.compare(np.array([g]), np.array([r]), huge)
        assert not ok and ratio == np.inf


def test_worst_element_is_reported_among_many():
    ref = np.full(1000, f16(1.0))
    gpu = ref.copy()
    gpu[437] = f16(1.0 + 2.0 ** -8)        # 4 ulp off with absacc 0: ratio 4
    ok, ratio, idx = oracle.compare(gpu, ref, np.zeros(1000))
    assert not ok and idx == 437 and ratio == pytest.approx(4.0)
    ok, ratio, idx = oracle.compare(ref, ref, np.zeros(1000))
    assert ok and ratio == 0.0
    assert oracle.compare(np.zeros(0, np.float16), np.zeros(0, np.float16), np.zeros(0))[0]


# ------------------------------------------------------------------ mutations at full size
def _points(M, N, L, n, seed):
    rng = np.random.default_rng(seed)
    return rng.integers(0, L, n), rng.integers(0, M, n), rng.integers(0, N, n)


def _mutants(p):
    M = p["M"]
    A, SFA, SFB = p["A"], p["SFA"], p["SFB"]
    drop = SFA.clone()
    drop[:, :, 5] = 0                                   # one 16-wide scale block of every row of A
    swapped = ((A >> 4) | (A << 4)).to(torch.uint8)     # high and low nibble exchanged
    sfa_x = SFB[:, :M].clone()                          # SFA and SFB exchanged (first M rows of B)
    sfb_x = SFB.clone()
    sfb_x[:, :M] = SFA
    return {"scale block dropped": dict(SFA=drop), "nibbles swapped": dict(A=swapped),
            "SFA and SFB exchanged": dict(SFA=sfa_x, SFB=sfb_x)}


@pytest.mark.parametrize("name", ["skinny_128x7168x16384", "dense_8192x8192x8192", "grouped2", "moe8"])
def test_checker_rejects_mutated_oracle_at_full_size(name):
    """The oracle's own C for mutated inputs, compared with the true C on 2000
    sampled points of every group: the checker must reject every mutant."""
    for gi, p in enumerate(workloads.make_inputs(name, seed=0)):
        M, N, K, L = p["M"], p["N"], p["K"], p["L"]
        ls, ms, ns = _points(M, N, L, 2000, gi)
        ref, absacc = oracle.gemm_points(p["A"], p["B"], p["SFA"], p["SFB"], M, N, K, ls, ms, ns, L=L)
        ok, worst, _ = oracle.compare(ref, ref, absacc)
        assert ok and worst == 0.0
        for what, change in _mutants(p).items():
            q = dict(p, **change)
            c, _ = oracle.gemm_points(q["A"], q["B"], q["SFA"], q["SFB"], M, N, K, ls, ms, ns, L=L)
            ok, worst, _ = oracle.compare(c, ref, absacc)
            assert not ok, "%s group %d: '%s' passed the checker (worst ratio %.3g)" % (name, gi, what, worst)


def test_one_dropped_block_in_one_row_is_rejected_at_k16384():
    """The smallest mutation: one 16-wide block of one row of A (its largest
    scale) set to zero in the 128 x 7168 x 16384 problem -- 16 of 16384 terms
    of that row's 7168 outputs.  The bound 1e-3 * sum|a_k b_k| still rejects
    the row."""
    p = workloads.make_inputs("skinny_128x7168x16384", seed=0)[0]
    M, N, K = p["M"], p["N"], p["K"]
    m0 = 3
    j = int(np.argmax(p["SFA"][0, m0].numpy()))
    sfa = p["SFA"].clone()
    sfa[0, m0, j] = 0
    ls, ms, ns = np.zeros(N, np.int64), np.full(N, m0), np.arange(N)
    ref, absacc = oracle.gemm_points(p["A"], p["B"], p["SFA"], p["SFB"], M, N, K, ls, ms, ns)
    c, _ = oracle.gemm_points(p["A"], p["B"], sfa, p["SFB"], M, N, K, ls, ms, ns)
    ok, worst, _ = oracle.compare(c, ref, absacc)
    assert not ok and worst > 2.0
