"""GPU scale repack against the oracle's repack, byte for byte."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import require_gpu

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("rows,K,L", [
    (128, 256, 1), (1, 256, 1), (200, 512, 1), (7168, 16384, 1), (130, 768, 3),
    (64, 320, 2), (1000, 1024, 1), (96, 48, 1), (300, 1088, 2), (7, 8192, 1), (129, 4352, 1),
    (100, 1040, 2), (257, 33024, 1),
])
def test_repack_matches_oracle(rows, K, L):
    binding = require_gpu()
    g = torch.Generator().manual_seed(rows * 31 + K)
    sf = torch.randint(0, 256, (L, rows, K // 16), dtype=torch.uint8, generator=g)
    out = binding.repack_scales(sf.cuda(), rows, K, L)
    torch.cuda.synchronize()
    ref = oracle.repack_scales(sf, rows, K, L)
    assert out.numel() == ref.size
    assert np.array_equal(out.cpu().numpy(), ref)


def test_repack_padding_is_written_zero():
    binding = require_gpu()
    rows, K = 70, 320
    sf = torch.randint(1, 256, (1, rows, K // 16), dtype=torch.uint8)
    out = torch.full((binding.nvfp4_gemm_repacked_scales_bytes(rows, K, 1),), 0xAB, dtype=torch.uint8,
                     device="cuda")
    binding.nvfp4_gemm_repack_scales(sf.cuda(), out, rows, K, 1)
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy(), oracle.repack_scales(sf, rows, K, 1))
