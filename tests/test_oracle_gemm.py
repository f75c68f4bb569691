"""Pins for the oracle GEMM (CPU only).

1. Tiny GEMMs against exact rational arithmetic (Fractions), with decode values
   taken from the published E2M1 list and torch's float8_e4m3fn conversion and
   the rounding done by exact rational RNE.
2. Unit scales (all 0x38 = 1.0) reproduce the plain decoded matmul rounded to
   fp16 by numpy.
3. Grouped output equals single-problem runs; L > 1 equals separate batches;
   selected points equal the full run.
4. On every workload's distribution the fp64 sum equals an int64 fixed-point sum
   (each term is a multiple of 2^-20), so the oracle's only rounding is the
   final one.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from block_scaled_fp4_nvfp4_gb300 import workloads
from test_oracle_rounding import rne_fraction_to_f16_bits

E2M1_MAG = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
E2M1_FRAC = [Fraction(v).limit_denominator(2) for v in E2M1_MAG]
E2M1_FRAC = E2M1_FRAC + [-v for v in E2M1_FRAC]
E4M3_F64 = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def e4m3_frac(code):
    return Fraction(float(E4M3_F64[code]))


def unpack_nibbles(packed):
    """[..., K/2] bytes -> [..., K] codes, low nibble = even k (float4_e2m1fn_x2)."""
    packed = np.asarray(packed, np.uint8)
    out = np.empty(packed.shape[:-1] + (packed.shape[-1] * 2,), np.uint8)
    out[..., 0::2] = packed & 0xF
    out[..., 1::2] = packed >> 4
    return out


def exact_reference(A, B, SFA, SFB, M, N, K):
    a = unpack_nibbles(A.reshape(M, K // 2))
    b = unpack_nibbles(B.reshape(N, K // 2))
    sfa = SFA.reshape(M, K // 16)
    sfb = SFB.reshape(N, K // 16)
    out = np.zeros((M, N), np.uint16)
    sums = {}
    for m in range(M):
        for n in range(N):
            s = Fraction(0)
            for k in range(K):
                s += (E2M1_FRAC[a[m, k]] * e4m3_frac(sfa[m, k // 16])
                      * E2M1_FRAC[b[n, k]] * e4m3_frac(sfb[n, k // 16]))
            sums[(m, n)] = s
            out[m, n] = rne_fraction_to_f16_bits(s)
    return out, sums


def random_bytes(rng, shape, exclude_nan=False):
    x = rng.integers(0, 256, shape, dtype=np.uint8)
    if exclude_nan:
        x[(x & 0x7F) == 0x7F] = 0x38
    return x


@pytest.mark.parametrize("M,N,K,seed", [(1, 1, 16, 0), (3, 5, 32, 1), (8, 8, 64, 2), (7, 4, 48, 3)])
def test_tiny_gemm_exact_rationals(M, N, K, seed):
    rng = np.random.default_rng(seed)
    A = random_bytes(rng, (M, K // 2))
    B = random_bytes(rng, (N, K // 2))
    # full signed E4M3 range except NaN (the oracle decodes every code)
    SFA = random_bytes(rng, (M, K // 16), exclude_nan=True)
    SFB = random_bytes(rng, (N, K // 16), exclude_nan=True)
    C, absacc, acc = oracle.gemm(A, B, SFA, SFB, M, N, K, want_acc=True)
    ref, sums = exact_reference(A, B, SFA, SFB, M, N, K)
    assert np.array_equal(C.view(np.uint16)[0], ref)
    for (m, n), s in sums.items():
        assert Fraction(float(acc[0, m, n])) == s          # the fp64 sum is exact here


def test_tiny_gemm_one_hot_scale_blocks():
    """Each scale block scales exactly its 16 k-elements (dropped/shifted index
    in k/16 would fail)."""
    M, N, K = 2, 3, 64
    rng = np.random.default_rng(7)
    A = random_bytes(rng, (M, K // 2))
    B = random_bytes(rng, (N, K // 2))
    for blk in range(K // 16):
        SFA = np.full((M, K // 16), 0x38, np.uint8)
        SFB = np.full((N, K // 16), 0x38, np.uint8)
        SFA[:, blk] = 0x48          # 4.0
        SFB[1, blk] = 0x30          # 0.5
        C, _ = oracle.gemm(A, B, SFA, SFB, M, N, K)
        ref, _ = exact_reference(A, B, SFA, SFB, M, N, K)
        assert np.array_equal(C.view(np.uint16)[0], ref)


def test_unit_scales_equal_plain_decoded_matmul():
    M, N, K = 64, 48, 512
    rng = np.random.default_rng(11)
    A = random_bytes(rng, (M, K // 2))
    B = random_bytes(rng, (N, K // 2))
    SFA = np.full((M, K // 16), 0x38, np.uint8)
    SFB = np.full((N, K // 16), 0x38, np.uint8)
    C, _ = oracle.gemm(A, B, SFA, SFB, M, N, K)
    table = np.array(E2M1_MAG + [-v for v in E2M1_MAG])
    da = table[unpack_nibbles(A)]
    db = table[unpack_nibbles(B)]
    ref = (da @ db.T).astype(np.float16)     # half-integer products: exact in fp64
    assert np.array_equal(C[0].view(np.uint16), ref.view(np.uint16))


def test_transposed_operand_would_fail():
    """A != B^T guard: C must not be symmetric in its operands' roles."""
    M = N = 16
    K = 64
    p = workloads.make_random_problem(5, M, N, K)
    C1, _ = oracle.gemm(p["A"], p["B"], p["SFA"], p["SFB"], M, N, K)
    C2, _ = oracle.gemm(p["B"], p["A"], p["SFB"], p["SFA"], N, M, K)
    assert np.array_equal(C1[0], C2[0].T)
    C3, _ = oracle.gemm(p["A"], p["B"], p["SFB"], p["SFA"], M, N, K)
    assert not np.array_equal(C1, C3)


def test_grouped_equals_single_runs():
    shapes = [(5, 24, 64, 1), (33, 8, 256, 2), (1, 40, 32, 1), (17, 16, 128, 3)]
    probs = []
    for i, (M, N, K, L) in enumerate(shapes):
        probs.append(workloads.make_random_problem(100 + i, M, N, K, L))
    outs = oracle.gemm_grouped(probs)
    for p, c in zip(probs, outs):
        ref, _ = oracle.gemm(p["A"], p["B"], p["SFA"], p["SFB"], p["M"], p["N"], p["K"], p["L"])
        assert np.array_equal(c.view(np.uint16), ref.view(np.uint16))


def test_batches_are_independent_problems():
    M, N, K, L = 9, 12, 128, 3
    p = workloads.make_random_problem(3, M, N, K, L)
    C, _ = oracle.gemm(p["A"], p["B"], p["SFA"], p["SFB"], M, N, K, L)
    for l in range(L):
        Cl, _ = oracle.gemm(p["A"][l], p["B"][l], p["SFA"][l], p["SFB"][l], M, N, K, 1)
        assert np.array_equal(C[l].view(np.uint16), Cl[0].view(np.uint16))


def test_points_equal_full_run():
    M, N, K, L = 20, 36, 256, 2
    p = workloads.make_random_problem(9, M, N, K, L)
    C, absacc = oracle.gemm(p["A"], p["B"], p["SFA"], p["SFB"], M, N, K, L)
    rng = np.random.default_rng(0)
    ls = rng.integers(0, L, 300)
    ms = rng.integers(0, M, 300)
    ns = rng.integers(0, N, 300)
    Cp, ap = oracle.gemm_points(p["A"], p["B"], p["SFA"], p["SFB"], M, N, K, ls, ms, ns, L=L)
    assert np.array_equal(Cp.view(np.uint16), C[ls, ms, ns].view(np.uint16))
    assert np.array_equal(ap, absacc[ls, ms, ns])


def fixed_point_sums(p, ls, ms, ns):
    """Exact sums scaled by 2^20 as int64: 2*e2m1 and 2^9*e4m3 are integers
    for every code the workloads draw."""
    two_e2m1 = np.array([0, 1, 2, 3, 4, 6, 8, 12, 0, -1, -2, -3, -4, -6, -8, -12], np.int64)
    sf512 = E4M3_F64 * 512.0
    out = []
    for l, m, n in zip(ls, ms, ns):
        a = two_e2m1[unpack_nibbles(p["A"][l, m].numpy())]
        b = two_e2m1[unpack_nibbles(p["B"][l, n].numpy())]
        sa = np.repeat(sf512[p["SFA"][l, m].numpy()], 16)
        sb = np.repeat(sf512[p["SFB"][l, n].numpy()], 16)
        assert np.all(sa == np.round(sa)) and np.all(sb == np.round(sb))
        out.append(int(np.sum(a * sa.astype(np.int64) * b * sb.astype(np.int64))))
    return out


@pytest.mark.parametrize("name", workloads.WORKLOAD_ORDER)
def test_fp64_sum_is_exact_on_workload_distributions(name):
    probs = workloads.make_inputs(name, seed=0)
    rng = np.random.default_rng(42)
    for p in probs:
        M, N, K, L = p["M"], p["N"], p["K"], p["L"]
        npts = 24
        ls = rng.integers(0, L, npts)
        ms = rng.integers(0, M, npts)
        ns = rng.integers(0, N, npts)
        _, _, acc = oracle.gemm_points(p["A"], p["B"], p["SFA"], p["SFB"], M, N, K, ls, ms, ns,
                                       L=L, want_acc=True)
        exact = fixed_point_sums(p, ls, ms, ns)
        for a, e in zip(acc, exact):
            assert Fraction(float(a)) == Fraction(e, 2 ** 20)
