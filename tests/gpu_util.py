"""Helpers shared by the GPU tests: build/load the library once, move a seeded
problem to the device, run it through the C ABI, compare with the oracle.

Every oracle comparison records the worst |gpu - ref| / tolerance it saw, per
test; the session summary (tests/conftest.py) prints the largest ones, so a
kernel drifting towards the bound shows before it crosses it."""
import os

import numpy as np
import pytest
import torch

import oracle

_built = False

# (test id, what was compared, elements, worst ratio) of every comparison
WORST_RATIOS = []


def record_worst(worst, n, what):
    test = os.environ.get("PYTEST_CURRENT_TEST", "?").rsplit(" (", 1)[0]
    WORST_RATIOS.append((test, what, int(n), float(worst)))


def ensure_built():
    global _built
    if not _built:
        import __graft_entry__
        __graft_entry__.build()
        _built = True
    from block_scaled_fp4_nvfp4_gb300 import binding
    return binding


def require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return ensure_built()


def to_device(p, dev="cuda"):
    """Problem dict (CPU tensors, row-major scales) -> device tensors with
    repacked scales."""
    binding = ensure_built()
    M, N, K, L = p["M"], p["N"], p["K"], p["L"]
    d = dict(M=M, N=N, K=K, L=L)
    d["A"] = p["A"].to(dev).contiguous()
    d["B"] = p["B"].to(dev).contiguous()
    d["SFA"] = binding.repack_scales(p["SFA"].to(dev).contiguous(), M, K, L)
    d["SFB"] = binding.repack_scales(p["SFB"].to(dev).contiguous(), N, K, L)
    return d


def alloc_c(M, N, L, dev="cuda", canary=4096):
    """C with a guard band after it, filled with NaN so unwritten elements show."""
    buf = torch.full((L * M * N + canary,), float("nan"), dtype=torch.float16, device=dev)
    return buf, buf[:L * M * N].view(L, M, N)


def check_canary(buf, M, N, L):
    tail = buf[L * M * N:]
    assert torch.isnan(tail).all(), "write past the end of C"


def run_single(d, C):
    binding = ensure_built()
    binding.nvfp4_gemm_run(d["A"], d["B"], d["SFA"], d["SFB"], C, d["M"], d["N"], d["K"], d["L"])


def assert_close_full(gpu_c, p):
    ref, absacc = oracle.gemm(p["A"], p["B"], p["SFA"], p["SFB"], p["M"], p["N"], p["K"], p["L"])
    g = gpu_c.detach().cpu().numpy()
    assert not np.isnan(g).any(), "unwritten output elements"
    ok, worst, idx = oracle.compare(g, ref, absacc)
    record_worst(worst, g.size, "full")
    assert ok, "worst |err|/tol = %.4g at flat index %d (gpu %r ref %r)" % (
        worst, idx, g.ravel()[idx], ref.ravel()[idx])
    return worst


def sample_points(M, N, L, n, seed=0, tile_m=128, tile_n=128):
    """Random points plus every tile's corners and the last row/column."""
    rng = np.random.default_rng(seed)
    ls = list(rng.integers(0, L, n))
    ms = list(rng.integers(0, M, n))
    ns = list(rng.integers(0, N, n))
    for l in range(L):
        for m0 in range(0, M, tile_m):
            for n0 in range(0, N, tile_n):
                for dm, dn in ((0, 0), (min(tile_m, M - m0) - 1, min(tile_n, N - n0) - 1)):
                    ls.append(l)
                    ms.append(m0 + dm)
                    ns.append(n0 + dn)
    ls += [L - 1, L - 1]
    ms += [M - 1, 0]
    ns += [0, N - 1]
    return np.array(ls), np.array(ms), np.array(ns)


def assert_close_points(gpu_c, p, ls, ms, ns):
    ref, absacc = oracle.gemm_points(p["A"], p["B"], p["SFA"], p["SFB"], p["M"], p["N"], p["K"],
                                     ls, ms, ns, L=p["L"])
    g = gpu_c.detach()[torch.as_tensor(ls), torch.as_tensor(ms), torch.as_tensor(ns)].cpu().numpy()
    assert not np.isnan(g).any(), "unwritten output elements"
    ok, worst, idx = oracle.compare(g, ref, absacc)
    record_worst(worst, g.size, "points")
    assert ok, "worst |err|/tol = %.4g at point (%d,%d,%d): gpu %r ref %r" % (
        worst, ls[idx], ms[idx], ns[idx], g[idx], ref[idx])
    return worst
