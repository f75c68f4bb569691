"""nvfp4_gemm_run_noalloc: the GEMM variant for callers that cannot allocate
device memory (its split-K scratch is a static device array inside the
library).  Its output must match nvfp4_gemm_run's on the same inputs, call
after call, although every call reuses the same scratch area.

This file is collected last so that a failure here leaves every other test
already run."""
import os

import numpy as np
import pytest
import torch

import oracle
from block_scaled_fp4_nvfp4_gb300 import workloads
from gpu_util import alloc_c, require_gpu, to_device

pytestmark = pytest.mark.gpu


def _both(binding, p):
    d = to_device(p)
    M, N, K, L = p["M"], p["N"], p["K"], p["L"]
    _, ref = alloc_c(M, N, L)
    binding.nvfp4_gemm_run(d["A"], d["B"], d["SFA"], d["SFB"], ref, M, N, K, L)
    _, got = alloc_c(M, N, L)
    binding.nvfp4_gemm_run_noalloc(d["A"], d["B"], d["SFA"], d["SFB"], got, M, N, K, L)
    torch.cuda.synchronize()
    binding.nvfp4_gemm_check_device_status()
    return ref, got


def _check_against_existing(p, ref, got):
    """|noalloc - existing| within the suite's elementwise tolerance
    (1e-3 * sum_k |a_k b_k| + 1 fp16 ulp), sum taken from the oracle."""
    _, absacc = oracle.gemm(p["A"], p["B"], p["SFA"], p["SFB"], p["M"], p["N"], p["K"], p["L"])
    g = got.cpu().numpy()
    r = ref.cpu().numpy()
    assert not np.isnan(g).any(), "unwritten output elements"
    ok, worst, idx = oracle.compare(g, r, absacc)
    assert ok, "worst |err|/tol = %.4g at flat index %d" % (worst, idx)


def test_noalloc_matches_existing_entry_point_call_after_call():
    binding = require_gpu()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    # stream-K problems, so the static scratch (partials + counters) is used
    shapes = [(128, 7168, 16384, 1), (256, 2048, 4096, 1), (128, 7168, 16384, 1)]
    for i, shape in enumerate(shapes):
        plan = binding.nvfp4_gemm_plan([shape[0]], [shape[1]], [shape[2]], [shape[3]], sms)
        assert plan["sk_max_segs"] > 1
        p = workloads.make_random_problem(900 + i, *shape)
        ref, got = _both(binding, p)
        _check_against_existing(p, ref, got)


def test_noalloc_rejects_plans_beyond_the_static_area():
    binding = require_gpu()
    p = workloads.make_random_problem(7, 2048, 2048, 2048)
    d = to_device(p)
    _, C = alloc_c(2048, 2048, 1)
    # all 256 tiles as stream-K, two segments each: 32 MiB of partials
    os.environ["NVFP4_SCHEDULE"] = "sk"
    try:
        with pytest.raises(binding.Nvfp4Error) as e:
            binding.nvfp4_gemm_run_noalloc(d["A"], d["B"], d["SFA"], d["SFB"], C, 2048, 2048, 2048, 1)
        assert e.value.code == -2
        assert "static" in str(e.value)
    finally:
        del os.environ["NVFP4_SCHEDULE"]
