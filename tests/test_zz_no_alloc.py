"""nvfp4_gemm_run_noalloc: the GEMM variant for callers that cannot allocate
device memory (code inside a host callback or a custom allocator, runtimes that
own the whole device heap, processes held to a fixed memory budget).  Its
split-K scratch is a static device array inside the library, so every call
reuses the same area; its output must still match the oracle call after call,
and equal nvfp4_gemm_run's, and a device timeout in it must be reported.

This file is collected last so that a failure here leaves every other test
already run."""
import numpy as np
import pytest
import torch

import oracle
from block_scaled_fp4_nvfp4_gb300 import workloads
from gpu_util import alloc_c, assert_close_full, check_canary, require_gpu, to_device

pytestmark = pytest.mark.gpu


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def test_noalloc_matches_oracle_and_existing_entry_point_call_after_call():
    binding = require_gpu()
    # stream-K problems, so the static scratch (partials + counters) is used
    shapes = [(128, 7168, 16384, 1), (256, 2048, 4096, 1), (128, 7168, 16384, 1)]
    for i, (M, N, K, L) in enumerate(shapes):
        p = workloads.make_random_problem(900 + i, M, N, K, L)
        d = to_device(p)
        buf, got = alloc_c(M, N, L)
        binding.nvfp4_gemm_run_noalloc(d["A"], d["B"], d["SFA"], d["SFB"], got, M, N, K, L)
        launched = binding.nvfp4_gemm_last_launch()
        tiles = binding.nvfp4_gemm_plan([M], [N], [K], [L], _sms())["tiles"]
        # one CTA per tile, no clusters: more CTAs than tiles means stream-K
        # segments summed through the static workspace and counters
        assert launched["variant"] == "single" and launched["cluster"] == 1
        assert launched["grid"] > tiles, launched
        binding.nvfp4_gemm_check_device_status()
        check_canary(buf, M, N, L)
        assert_close_full(got, p)
        _, ref = alloc_c(M, N, L)
        binding.nvfp4_gemm_run(d["A"], d["B"], d["SFA"], d["SFB"], ref, M, N, K, L)
        binding.nvfp4_gemm_check_device_status()
        _, absacc = oracle.gemm(p["A"], p["B"], p["SFA"], p["SFB"], M, N, K, L)
        ok, worst, idx = oracle.compare(got.cpu().numpy(), ref.cpu().numpy(), absacc)
        assert ok, "noalloc vs nvfp4_gemm_run: worst |err|/tol = %.4g at %d" % (worst, idx)


def test_noalloc_timeout_is_reported_and_next_call_is_right():
    """A skipped k-tile arrival (host-side injection, nothing in flight) with a
    short wait limit: the no-allocation launch gives up, the status query
    reports NVFP4_ERR_DEVICE_TIMEOUT from the static area's own word, and the
    next call on the same context is correct."""
    binding = require_gpu()
    M, N, K = 128, 2048, 4096
    p = workloads.make_random_problem(31, M, N, K)
    d = to_device(p)
    try:
        binding.nvfp4_gemm_set_wait_timeout_ns(50_000_000)
        binding.nvfp4_gemm_debug_inject_skip(2)
        _, C = alloc_c(M, N, 1)
        binding.nvfp4_gemm_run_noalloc(d["A"], d["B"], d["SFA"], d["SFB"], C, M, N, K, 1)
        with pytest.raises(binding.Nvfp4Error) as e:
            binding.nvfp4_gemm_check_device_status()
        assert e.value.code == -4
    finally:
        binding.nvfp4_gemm_debug_inject_skip(-1)
        binding.nvfp4_gemm_set_wait_timeout_ns(2_000_000_000)
    binding.nvfp4_gemm_check_device_status()   # the word was cleared by the report
    buf, C = alloc_c(M, N, 1)
    binding.nvfp4_gemm_run_noalloc(d["A"], d["B"], d["SFA"], d["SFB"], C, M, N, K, 1)
    binding.nvfp4_gemm_check_device_status()
    check_canary(buf, M, N, 1)
    assert_close_full(C, p)


def test_noalloc_rejects_plans_beyond_the_static_area(monkeypatch):
    binding = require_gpu()
    p = workloads.make_random_problem(7, 2048, 2048, 2048)
    d = to_device(p)
    _, C = alloc_c(2048, 2048, 1)
    # all 256 tiles as stream-K, two segments each: 32 MiB of partials
    monkeypatch.setenv("NVFP4_SCHEDULE", "sk")
    with pytest.raises(binding.Nvfp4Error) as e:
        binding.nvfp4_gemm_run_noalloc(d["A"], d["B"], d["SFA"], d["SFB"], C, 2048, 2048, 2048, 1)
    assert e.value.code == -2
    assert "static" in str(e.value)
    assert np.isnan(C.cpu().numpy()).all(), "a refused call wrote C"
