"""CPU oracle for the NVFP4 block-scaled GEMM -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The library itself never calls it and
shares no code with it: the oracle is plain C (``nvfp4_oracle.c``) wrapped here
with ctypes and numpy marshalling only.

Every routine states the definition it follows (see the C source):
decode by table (16 E2M1 codes, 256 E4M3 codes), accumulate in fp64 in k order,
round once to fp16 (round to nearest, ties to even).

Pins (tests marked ``not gpu``): decode tables against the format's published
value list and ``torch.float8_e4m3fn``; tiny GEMMs against exact rational
arithmetic; unit scales against the plain decoded matmul; grouped output against
single-problem runs; fp64->fp16 rounding by brute force; the repack layout
against the pages' logical shape and address arithmetic; the NVFP4 quantizer's
encoders against the decode tables (exact round trips, midpoints to the even
code, saturation) and ``torch.float8_e4m3fn``, and a hand-worked block.
"""
import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        u8p = ctypes.POINTER(ctypes.c_uint8)
        u16p = ctypes.POINTER(ctypes.c_uint16)
        dp = ctypes.POINTER(ctypes.c_double)
        ip = ctypes.POINTER(ctypes.c_int)
        lib.oracle_e2m1_table.argtypes = [dp]
        lib.oracle_e4m3_table.argtypes = [dp]
        lib.oracle_f64_to_f16.argtypes = [ctypes.c_double]
        lib.oracle_f64_to_f16.restype = ctypes.c_uint16
        lib.oracle_f64_to_f16_array.argtypes = [dp, u16p, ctypes.c_int64]
        lib.oracle_gemm.argtypes = [u8p, u8p, u8p, u8p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                    ctypes.c_int, u16p, dp, dp, ctypes.c_int]
        lib.oracle_gemm.restype = ctypes.c_int
        lib.oracle_gemm_points.argtypes = [u8p, u8p, u8p, u8p, ctypes.c_int, ctypes.c_int,
                                           ctypes.c_int, ctypes.c_int, ctypes.c_int64, ip, ip, ip,
                                           u16p, dp, dp, ctypes.c_int]
        lib.oracle_gemm_points.restype = ctypes.c_int
        pp = ctypes.POINTER(u8p)
        lib.oracle_gemm_grouped.argtypes = [ctypes.c_int, pp, pp, pp, pp, ip, ip, ip, ip,
                                            ctypes.POINTER(u16p), ctypes.c_int]
        lib.oracle_gemm_grouped.restype = ctypes.c_int
        lib.oracle_repacked_bytes.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int]
        lib.oracle_repacked_bytes.restype = ctypes.c_int64
        lib.oracle_repack_scales.argtypes = [u8p, ctypes.c_int, ctypes.c_int, ctypes.c_int, u8p]
        lib.oracle_repack_scales.restype = ctypes.c_int
        lib.oracle_max_threads.restype = ctypes.c_int
        fp = ctypes.POINTER(ctypes.c_float)
        lib.oracle_e4m3_encode_array.argtypes = [fp, u8p, ctypes.c_int64]
        lib.oracle_e2m1_encode_array.argtypes = [fp, u8p, ctypes.c_int64]
        lib.oracle_quantize.argtypes = [fp, ctypes.c_int, ctypes.c_int, ctypes.c_int, u8p, u8p]
        lib.oracle_quantize.restype = ctypes.c_int
        _lib = lib
    return _lib


def _np(x, dtype):
    """numpy view of an array-like (numpy or CPU torch tensor), C-contiguous."""
    if hasattr(x, "detach"):
        x = x.detach().cpu().contiguous().numpy()
    a = np.ascontiguousarray(x)
    if a.dtype != dtype:
        a = a.view(dtype) if a.dtype.itemsize == np.dtype(dtype).itemsize else a.astype(dtype)
    return a


def _ptr(a, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def e2m1_table() -> np.ndarray:
    out = np.zeros(16, np.float64)
    _load().oracle_e2m1_table(_ptr(out, ctypes.c_double))
    return out


def e4m3_table() -> np.ndarray:
    out = np.zeros(256, np.float64)
    _load().oracle_e4m3_table(_ptr(out, ctypes.c_double))
    return out


def f64_to_f16(x) -> np.ndarray:
    """fp64 -> fp16 (returned as np.float16), RNE, overflow to Inf."""
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    out = np.zeros(a.shape, np.uint16)
    _load().oracle_f64_to_f16_array(_ptr(a, ctypes.c_double), _ptr(out, ctypes.c_uint16), a.size)
    return out.view(np.float16)


def gemm(A, B, SFA, SFB, M, N, K, L=1, nthreads=0, want_acc=False):
    """Whole problem.  A [L,M,K/2] u8, B [L,N,K/2] u8, SFA [L,M,K/16] u8,
    SFB [L,N,K/16] u8 (row-major scales).  Returns C [L,M,N] float16 and
    absacc [L,M,N] (sum of |products|), plus the exact fp64 sum if want_acc."""
    A, B, SFA, SFB = (_np(t, np.uint8) for t in (A, B, SFA, SFB))
    assert A.size == L * M * (K // 2) and B.size == L * N * (K // 2)
    assert SFA.size == L * M * (K // 16) and SFB.size == L * N * (K // 16)
    C = np.zeros((L, M, N), np.uint16)
    absacc = np.zeros((L, M, N), np.float64)
    acc = np.zeros((L, M, N), np.float64) if want_acc else None
    rc = _load().oracle_gemm(_ptr(A, ctypes.c_uint8), _ptr(B, ctypes.c_uint8),
                             _ptr(SFA, ctypes.c_uint8), _ptr(SFB, ctypes.c_uint8),
                             M, N, K, L, _ptr(C, ctypes.c_uint16),
                             _ptr(acc, ctypes.c_double) if want_acc else None,
                             _ptr(absacc, ctypes.c_double), nthreads)
    if rc != 0:
        raise RuntimeError("oracle_gemm failed: %d" % rc)
    if want_acc:
        return C.view(np.float16), absacc, acc
    return C.view(np.float16), absacc


def gemm_points(A, B, SFA, SFB, M, N, K, ls, ms, ns, L=1, nthreads=0, want_acc=False):
    """Selected outputs C[l,m,n] of a problem laid out as in ``gemm``."""
    A, B, SFA, SFB = (_np(t, np.uint8) for t in (A, B, SFA, SFB))
    ls = np.ascontiguousarray(ls, np.int32)
    ms = np.ascontiguousarray(ms, np.int32)
    ns = np.ascontiguousarray(ns, np.int32)
    n = ms.size
    assert ls.size == n and ns.size == n
    C = np.zeros(n, np.uint16)
    absacc = np.zeros(n, np.float64)
    acc = np.zeros(n, np.float64)
    rc = _load().oracle_gemm_points(_ptr(A, ctypes.c_uint8), _ptr(B, ctypes.c_uint8),
                                    _ptr(SFA, ctypes.c_uint8), _ptr(SFB, ctypes.c_uint8),
                                    M, N, K, L, n, _ptr(ls, ctypes.c_int), _ptr(ms, ctypes.c_int),
                                    _ptr(ns, ctypes.c_int), _ptr(C, ctypes.c_uint16),
                                    _ptr(acc, ctypes.c_double), _ptr(absacc, ctypes.c_double),
                                    nthreads)
    if rc != 0:
        raise RuntimeError("oracle_gemm_points failed: %d" % rc)
    if want_acc:
        return C.view(np.float16), absacc, acc
    return C.view(np.float16), absacc


def gemm_grouped(problems, nthreads=0):
    """problems: list of dicts with A, B, SFA, SFB (row-major scales), M, N, K, L.
    Returns the list of C [L,M,N] float16 arrays."""
    G = len(problems)
    keep = []
    u8p = ctypes.POINTER(ctypes.c_uint8)
    arrs = {k: (u8p * max(G, 1))() for k in ("A", "B", "SFA", "SFB")}
    Cs = []
    Cptr = (ctypes.POINTER(ctypes.c_uint16) * max(G, 1))()
    dims = {k: (ctypes.c_int * max(G, 1))() for k in ("M", "N", "K", "L")}
    for g, p in enumerate(problems):
        for k in ("A", "B", "SFA", "SFB"):
            a = _np(p[k], np.uint8)
            keep.append(a)
            arrs[k][g] = _ptr(a, ctypes.c_uint8)
        for k in ("M", "N", "K"):
            dims[k][g] = int(p[k])
        dims["L"][g] = int(p.get("L", 1))
        c = np.zeros((dims["L"][g], p["M"], p["N"]), np.uint16)
        Cs.append(c)
        Cptr[g] = _ptr(c, ctypes.c_uint16)
    rc = _load().oracle_gemm_grouped(G, arrs["A"], arrs["B"], arrs["SFA"], arrs["SFB"],
                                     dims["M"], dims["N"], dims["K"], dims["L"], Cptr, nthreads)
    if rc != 0:
        raise RuntimeError("oracle_gemm_grouped failed: %d" % rc)
    return [c.view(np.float16) for c in Cs]


def repacked_bytes(rows, K, L=1) -> int:
    return int(_load().oracle_repacked_bytes(rows, K, L))


def repack_scales(sf, rows, K, L=1) -> np.ndarray:
    """Row-major scales [L,rows,K/16] -> the tensor-core atom layout (flat u8)."""
    sf = _np(sf, np.uint8)
    assert sf.size == L * rows * (K // 16)
    out = np.zeros(repacked_bytes(rows, K, L), np.uint8)
    rc = _load().oracle_repack_scales(_ptr(sf, ctypes.c_uint8), rows, K, L, _ptr(out, ctypes.c_uint8))
    if rc != 0:
        raise RuntimeError("oracle_repack_scales failed: %d" % rc)
    return out


def e4m3_encode(v) -> np.ndarray:
    """fp32 -> E4M3 code (RNE, ties to the even code, finite values above 448 -> 448)."""
    a = np.ascontiguousarray(np.asarray(v, dtype=np.float32))
    out = np.zeros(a.shape, np.uint8)
    _load().oracle_e4m3_encode_array(_ptr(a, ctypes.c_float), _ptr(out, ctypes.c_uint8), a.size)
    return out


def e2m1_encode(v) -> np.ndarray:
    """fp32 -> E2M1 code (RNE on the value grid, ties to the even code,
    magnitudes above 6 -> 6, sign bit = sign bit of v)."""
    a = np.ascontiguousarray(np.asarray(v, dtype=np.float32))
    out = np.zeros(a.shape, np.uint8)
    _load().oracle_e2m1_encode_array(_ptr(a, ctypes.c_float), _ptr(out, ctypes.c_uint8), a.size)
    return out


def quantize(x, rows, K, L=1):
    """x [L, rows, K] (float32, or a bf16/fp16 torch tensor: converted exactly)
    -> (codes u8 [L, rows, K/2], row-major scales u8 [L, rows, K/16]).
    The recipe is stated in nvfp4_oracle.c (amax/6 as E4M3, codes RNE)."""
    if hasattr(x, "detach"):
        x = x.detach().cpu().float().contiguous().numpy()
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    assert x.size == L * rows * K and K % 16 == 0
    codes = np.zeros((L, rows, K // 2), np.uint8)
    sf = np.zeros((L, rows, K // 16), np.uint8)
    rc = _load().oracle_quantize(_ptr(x, ctypes.c_float), rows, K, L, _ptr(codes, ctypes.c_uint8),
                                 _ptr(sf, ctypes.c_uint8))
    if rc != 0:
        raise RuntimeError("oracle_quantize failed: %d" % rc)
    return codes, sf


def tolerance(ref_f16, absacc):
    """Elementwise bound |gpu - ref| <= 1e-3 * sum_k |a_k b_k| + 1 fp16 ulp(ref),
    with ulp(x) = 2^(max(floor(log2|x|), -14) - 10) and ulp(0) = 2^-24."""
    r = np.abs(np.asarray(ref_f16, np.float64))
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(r > 0, r, 1.0)))
    e = np.maximum(e, -14.0)
    ulp = np.where(r > 0, np.exp2(e - 10.0), 2.0 ** -24)
    return 1e-3 * np.asarray(absacc, np.float64) + ulp


def compare(gpu_f16, ref_f16, absacc):
    """Return (ok, worst_ratio, index) for the elementwise tolerance check.
    Infinities must match exactly; NaN never passes."""
    g = np.asarray(gpu_f16, np.float64).ravel()
    r = np.asarray(ref_f16, np.float64).ravel()
    tol = tolerance(ref_f16, absacc).ravel()
    inf = np.isinf(r)
    bad_inf = inf & (g != r)
    with np.errstate(invalid="ignore"):
        err = np.where(inf, 0.0, np.abs(g - r))
    err = np.where(np.isnan(g) | np.isnan(r), np.inf, err)
    ratio = err / tol
    ratio[bad_inf] = np.inf
    if ratio.size == 0:
        return True, 0.0, -1
    i = int(np.argmax(ratio))
    return bool(ratio[i] <= 1.0), float(ratio[i]), i
