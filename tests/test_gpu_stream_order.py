"""Stream order across the library's kernels.  The repack, quantize and GEMM
kernels are launched as programmatic dependents of the kernel before them on
the stream and may be scheduled while it drains, so each must wait for its
predecessor before it touches global memory.  These tests queue rounds that
overwrite the buffers the previous GEMM reads (scales, codes) on one stream,
with no synchronisation in between, and check every round's C against the
oracle."""
import numpy as np
import pytest
import torch

import oracle
from block_scaled_fp4_nvfp4_gb300 import workloads
from gpu_util import alloc_c, assert_close_full, check_canary, require_gpu

pytestmark = pytest.mark.gpu

M, N, K = 512, 1024, 4096


def test_repack_overwrites_scales_the_previous_gemm_reads():
    binding = require_gpu()
    base = workloads.make_random_problem(11, M, N, K)
    scale_sets = [workloads.make_random_problem(20 + i, M, N, K) for i in range(3)]
    stream = torch.cuda.Stream()
    A, B = base["A"].cuda(), base["B"].cuda()
    raw = [(p["SFA"].cuda(), p["SFB"].cuda()) for p in scale_sets]
    sfa = torch.empty(binding.nvfp4_gemm_repacked_scales_bytes(M, K, 1), dtype=torch.uint8, device="cuda")
    sfb = torch.empty(binding.nvfp4_gemm_repacked_scales_bytes(N, K, 1), dtype=torch.uint8, device="cuda")
    outs = [alloc_c(M, N, 1) for _ in scale_sets]
    torch.cuda.synchronize()
    for (ra, rb), (_, C) in zip(raw, outs):
        binding.nvfp4_gemm_repack_scales(ra, sfa, M, K, 1, stream)
        binding.nvfp4_gemm_repack_scales(rb, sfb, N, K, 1, stream)
        binding.nvfp4_gemm_run(A, B, sfa, sfb, C, M, N, K, 1, stream)
    binding.nvfp4_gemm_check_device_status(stream)
    for p, (buf, C) in zip(scale_sets, outs):
        assert_close_full(C, dict(A=base["A"], B=base["B"], SFA=p["SFA"], SFB=p["SFB"], M=M, N=N, K=K, L=1))
        check_canary(buf, M, N, 1)


def test_quantize_overwrites_codes_the_previous_gemm_reads():
    binding = require_gpu()
    g = torch.Generator().manual_seed(5)
    xs = [torch.randn((1, M, K), generator=g).to(torch.bfloat16) for _ in range(3)]
    xb = torch.randn((1, N, K), generator=g).to(torch.bfloat16)
    stream = torch.cuda.Stream()
    codes_b, sf_b = binding.quantize(xb.cuda())
    codes_a = torch.empty((1, M, K // 2), dtype=torch.uint8, device="cuda")
    sf_a = torch.empty(binding.nvfp4_gemm_repacked_scales_bytes(M, K, 1), dtype=torch.uint8, device="cuda")
    xs_dev = [x.cuda() for x in xs]
    outs = [alloc_c(M, N, 1) for _ in xs]
    torch.cuda.synchronize()
    for x, (_, C) in zip(xs_dev, outs):
        binding.nvfp4_quantize(x, binding.DTYPE_BF16, codes_a, sf_a, M, K, 1, stream)
        binding.nvfp4_gemm_run(codes_a, codes_b, sf_a, sf_b, C, M, N, K, 1, stream)
    binding.nvfp4_gemm_check_device_status(stream)
    cb, sb = oracle.quantize(xb, N, K)
    for x, (buf, C) in zip(xs, outs):
        ca, sa = oracle.quantize(x, M, K)
        assert_close_full(C, dict(A=ca, B=cb, SFA=sa, SFB=sb, M=M, N=N, K=K, L=1))
        check_canary(buf, M, N, 1)
    # the last round's operands are what the buffers hold now
    ca, sa = oracle.quantize(xs[-1], M, K)
    assert np.array_equal(codes_a.cpu().numpy(), ca)
