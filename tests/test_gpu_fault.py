"""Bounded device waits: a wait that can never be satisfied (the producer skips
one k-tile's arrival, so nothing is in flight for it) must end with
NVFP4_ERR_DEVICE_TIMEOUT reported on the host and leave the context usable.
No trap, no bad address, no endless loop."""
import pytest
import torch

from block_scaled_fp4_nvfp4_gb300 import workloads
from gpu_util import alloc_c, assert_close_full, require_gpu, run_single, to_device

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("shape,skip", [((128, 128, 256, 1), 0), ((128, 512, 4096, 1), 2)])
def test_timeout_is_reported_and_context_survives(shape, skip):
    binding = require_gpu()
    p = workloads.make_random_problem(77, *shape)
    d = to_device(p)
    M, N, K, L = shape
    try:
        binding.nvfp4_gemm_set_wait_timeout_ns(50_000_000)   # 50 ms
        binding.nvfp4_gemm_debug_inject_skip(skip)
        _, C = alloc_c(M, N, L)
        run_single(d, C)
        with pytest.raises(binding.Nvfp4Error) as e:
            binding.nvfp4_gemm_check_device_status()
        assert e.value.code == -4
    finally:
        binding.nvfp4_gemm_debug_inject_skip(-1)
        binding.nvfp4_gemm_set_wait_timeout_ns(2_000_000_000)
    # the next launch on the same context is correct and reports no error
    _, C = alloc_c(M, N, L)
    run_single(d, C)
    binding.nvfp4_gemm_check_device_status()
    assert_close_full(C, p)
