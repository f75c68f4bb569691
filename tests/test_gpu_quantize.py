"""GPU NVFP4 quantizer (nvfp4_quantize) against the oracle's quantizer: codes
and repacked scales byte for byte, then the quantized operands through the
GEMM against the oracle GEMM of the oracle's quantization."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import alloc_c, assert_close_full, check_canary, require_gpu

pytestmark = pytest.mark.gpu


def _inputs(seed, L, rows, K, dtype):
    g = torch.Generator().manual_seed(seed)
    # per-row magnitudes over 2^-8 .. 2^8 so scales span subnormal to large E4M3 values
    x = torch.randn((L, rows, K), generator=g) * torch.exp2(torch.randint(-8, 9, (L, rows, 1), generator=g).float())
    return x.to(dtype)


def _check(x, rows, K, L):
    binding = require_gpu()
    codes, sf = binding.quantize(x.cuda())
    torch.cuda.synchronize()
    ref_codes, ref_sf = oracle.quantize(x, rows, K, L)
    assert np.array_equal(codes.cpu().numpy(), ref_codes), "codes differ"
    assert np.array_equal(sf.cpu().numpy(), oracle.repack_scales(ref_sf, rows, K, L)), "scales differ"
    return codes, sf


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("L,rows,K", [(1, 1, 16), (1, 128, 256), (2, 130, 272), (1, 300, 1088), (1, 64, 4160),
                                      (3, 33, 48), (1, 1000, 7168)])
def test_quantize_matches_oracle(dtype, L, rows, K):
    x = _inputs(rows * 7 + K + L, L, rows, K, dtype)
    if dtype == torch.float16:
        x = x.clamp(-60000, 60000)
    _check(x, rows, K, L)


def test_quantize_special_values():
    """Zeros and negative zeros, values at E2M1 midpoints of a unit scale
    (ties to even), blocks whose scale saturates at 448, blocks whose scale
    underflows to zero, and subnormal scales."""
    rows, K = 8, 64
    x = torch.zeros((1, rows, K), dtype=torch.float32)
    x[0, 1, :16] = -0.0
    mids = torch.tensor([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0])
    x[0, 2, :8] = mids
    x[0, 2, 8:16] = -mids
    x[0, 3, :16] = torch.linspace(-5000, 5000, 16)          # amax/6 > 448: scale saturates, codes saturate
    x[0, 4, :16] = 1e-5                                      # amax/6 far below the smallest scale: all zero
    x[0, 5, :16] = torch.linspace(-0.01, 0.01, 16)           # subnormal scale
    x[0, 6, :] = torch.randn(64) * 1e3
    x[0, 7, 16:32] = 448 * 6                                 # exactly the largest scale
    x[0, 0, :16] = torch.linspace(-3, 4, 16)                 # a normal block holding signed zeros and
    x[0, 0, 3] = -0.0                                        # values far below a quarter of its scale
    x[0, 0, 5] = 0.0
    x[0, 0, 7] = -1e-30
    x[0, 0, 9] = 1e-30
    _check(x.to(torch.bfloat16), rows, K, 1)


def test_quantized_operands_through_the_gemm():
    """bf16 A and B quantized on the GPU, multiplied by the GEMM: equals the
    oracle GEMM of the oracle's quantization (the inputs are identical bits)."""
    binding = require_gpu()
    M, N, K = 256, 384, 1024
    a = _inputs(1, 1, M, K, torch.bfloat16)
    b = _inputs(2, 1, N, K, torch.bfloat16)
    A, SFA = _check(a, M, K, 1)
    B, SFB = _check(b, N, K, 1)
    buf, C = alloc_c(M, N, 1)
    binding.nvfp4_gemm_run(A, B, SFA, SFB, C, M, N, K, 1)
    binding.nvfp4_gemm_check_device_status()
    ca, sa = oracle.quantize(a, M, K)
    cb, sb = oracle.quantize(b, N, K)
    assert_close_full(C, dict(A=ca, B=cb, SFA=sa, SFB=sb, M=M, N=N, K=K, L=1))
    check_canary(buf, M, N, 1)


def test_quantize_full_size_sampled_rows():
    """The bench's quantize leg at full size (7168 x 16384 bf16, one launch in
    the launch configuration bench.py times): codes and scales of 48 sampled
    rows (block edges, the last row, random ones) byte for byte against the
    oracle's quantization of those rows.  Scales are read back from the atom
    layout by its definition: byte (r, c) of the row-major scales sits at
    ((r/128)*(K/64) + c/4)*512 + (r%32)*16 + ((r%128)/32)*4 + c%4."""
    binding = require_gpu()
    L, rows, K = 1, 7168, 16384
    g = torch.Generator().manual_seed(20261203)
    x = (torch.randn((L, rows, K), generator=g) *
         torch.exp2(torch.randint(-8, 9, (L, rows, 1), generator=g).float())).to(torch.bfloat16)
    codes, sf = binding.quantize(x.cuda())
    torch.cuda.synchronize()
    pick = sorted(set([0, 1, 31, 32, 127, 128, 129, 3583, 3584, 7039, 7040, 7167] +
                      torch.randint(0, rows, (36,), generator=g).tolist()))
    sel = torch.tensor(pick)
    ref_codes, ref_sf = oracle.quantize(x[:, sel, :], len(pick), K, L)
    got_codes = codes[0, sel.cuda(), :].cpu().numpy()
    assert np.array_equal(got_codes, ref_codes[0]), "codes differ"
    flat = sf.cpu().numpy()
    r = np.asarray(pick)[:, None]
    c = np.arange(K // 16)[None, :]
    off = ((r // 128) * (K // 64) + c // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + c % 4
    assert np.array_equal(flat[off], ref_sf[0]), "scales differ"
