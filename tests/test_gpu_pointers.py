"""The C ABI accepts only memory of the current device: pinned host memory and
pageable host memory are refused with NVFP4_ERR_INVALID_ARG before anything is
encoded or launched, by every entry point that takes a buffer."""
import numpy as np
import pytest
import torch

from block_scaled_fp4_nvfp4_gb300 import workloads
from gpu_util import alloc_c, require_gpu, to_device

pytestmark = pytest.mark.gpu

M, N, K = 128, 256, 512


@pytest.fixture
def problem():
    binding = require_gpu()
    p = workloads.make_random_problem(41, M, N, K)
    return binding, p, to_device(p)


def _host_buffers(d):
    pinned = {k: d[k].cpu().pin_memory() for k in ("A", "B", "SFA", "SFB")}
    pageable = {k: np.ascontiguousarray(d[k].cpu().numpy()) for k in ("A", "B", "SFA", "SFB")}
    return pinned, pageable


@pytest.mark.parametrize("which", ["A", "B", "SFA", "SFB", "C"])
@pytest.mark.parametrize("kind", ["pinned", "pageable"])
def test_gemm_entry_points_refuse_host_memory(problem, which, kind):
    binding, p, d = problem
    pinned, pageable = _host_buffers(d)
    host_c = {"pinned": torch.empty((1, M, N), dtype=torch.float16).pin_memory(),
              "pageable": np.zeros((1, M, N), np.float16)}[kind]
    _, C = alloc_c(M, N, 1)
    args = dict(A=d["A"], B=d["B"], SFA=d["SFA"], SFB=d["SFB"], C=C)
    if which == "C":
        args["C"] = host_c
    else:
        args[which] = pinned[which] if kind == "pinned" else pageable[which]
    if kind == "pageable":
        args[which] = args[which].ctypes.data   # a plain host address
    calls = [
        lambda: binding.nvfp4_gemm_run(args["A"], args["B"], args["SFA"], args["SFB"], args["C"], M, N, K, 1),
        lambda: binding.nvfp4_gemm_run_grouped(1, [args["A"]], [args["B"]], [args["SFA"]], [args["SFB"]],
                                               [args["C"]], [M], [N], [K], [1]),
        lambda: binding.nvfp4_gemm_run_noalloc(args["A"], args["B"], args["SFA"], args["SFB"], args["C"],
                                               M, N, K, 1),
    ]
    for call in calls:
        with pytest.raises(binding.Nvfp4Error) as e:
            call()
        assert e.value.code == -1, str(e.value)
        assert which in str(e.value)
    torch.cuda.synchronize()
    assert torch.isnan(C).all(), "a refused call wrote C"
    binding.nvfp4_gemm_check_device_status()


def test_repack_and_quantize_refuse_host_memory(problem):
    binding, p, d = problem
    sf_host = p["SFA"].contiguous().pin_memory()
    out = torch.empty(binding.nvfp4_gemm_repacked_scales_bytes(M, K, 1), dtype=torch.uint8, device="cuda")
    with pytest.raises(binding.Nvfp4Error) as e:
        binding.nvfp4_gemm_repack_scales(sf_host, out, M, K, 1)
    assert e.value.code == -1
    out_host = torch.empty(out.numel(), dtype=torch.uint8).pin_memory()
    with pytest.raises(binding.Nvfp4Error) as e:
        binding.nvfp4_gemm_repack_scales(p["SFA"].cuda(), out_host, M, K, 1)
    assert e.value.code == -1
    x_host = torch.zeros((1, M, K), dtype=torch.bfloat16).pin_memory()
    codes = torch.empty((1, M, K // 2), dtype=torch.uint8, device="cuda")
    with pytest.raises(binding.Nvfp4Error) as e:
        binding.nvfp4_quantize(x_host, binding.DTYPE_BF16, codes, out, M, K, 1)
    assert e.value.code == -1
    # the same calls on device memory go through
    binding.nvfp4_gemm_repack_scales(p["SFA"].cuda(), out, M, K, 1)
    binding.nvfp4_quantize(x_host.cuda(), binding.DTYPE_BF16, codes, out, M, K, 1)
    torch.cuda.synchronize()
    binding.nvfp4_gemm_check_device_status()
