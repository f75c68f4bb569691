"""GEMM parity on the edge cases of the two formats, under every kernel variant.

The scales are float8_e4m3fn ("nvfp4 gemm, submission 125598", custom_kernel
docstring) and C is rounded to fp16 with round-to-nearest-even
(__floats2half2_rn, "nvfp4 group gemm, submission 407526", grouped_kernel
epilogue).  The cases:

  * scale bytes over the whole finite non-negative E4M3 range 0x00..0x7E --
    zero, the subnormals 0x01..0x07 (m * 2^-9) and the largest value 0x7E
    (448) -- for SFA, with SFB drawn from the subnormals and the smallest
    normals (so every product of two scales is exercised and C stays finite),
    and the same with the roles of SFA and SFB exchanged;
  * C past the fp16 range: rows of A of value +-1 with scale 448 against
    non-negative B, so those outputs round to +-Inf (the oracle's Inf must be
    matched exactly), while every other output stays far below 65504;
  * rows of A and B that are all +0 codes or all -0 codes.

Every case runs under each variant the planner can choose (one CTA per tile
at 64, 128 and 256 columns, B shared by multicast, 2-SM pair tiles,
stream-K summed in a cluster's shared memory, stream-K through the device
workspace) and is compared element by element with the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
from block_scaled_fp4_nvfp4_gb300 import workloads
from gpu_util import alloc_c, assert_close_full, check_canary, require_gpu, to_device

pytestmark = pytest.mark.gpu

_DP = (256, 512, 1024)       # two m-tiles: clusters of two CTAs are possible
_SK = (128, 1024, 4096)      # 8 tiles of 128 x 128 with 16 k-tiles: stream-K plans

VARIANTS = {
    "single128": (_DP, {"NVFP4_BN": "128", "NVFP4_SCHEDULE": "dp", "NVFP4_CLUSTER": "1"}, "single"),
    "narrow64": (_DP, {"NVFP4_BN": "64", "NVFP4_SCHEDULE": "dp"}, "single"),
    "wide256": (_DP, {"NVFP4_BN": "256", "NVFP4_SCHEDULE": "dp", "NVFP4_CLUSTER": "1"}, "single"),
    "multicast": (_DP, {"NVFP4_BN": "256", "NVFP4_SCHEDULE": "dp", "NVFP4_CLUSTER": "2", "NVFP4_PAIR": "0"},
                  "multicast"),
    "pair": (_DP, {"NVFP4_BN": "256", "NVFP4_SCHEDULE": "dp", "NVFP4_CLUSTER": "2", "NVFP4_PAIR": "1"}, "pair"),
    "cluster_reduce": (_SK, {}, "cluster_reduce"),
    "workspace_sk": (_SK, {"NVFP4_SCHEDULE": "sk", "NVFP4_SKRED": "0"}, "single"),
}
_KEYS = ("NVFP4_BN", "NVFP4_SCHEDULE", "NVFP4_CLUSTER", "NVFP4_PAIR", "NVFP4_SKRED", "NVFP4_PAD_PAIRS")

FP16_OVERFLOW = 65520.0   # RNE to fp16 gives Inf from here on


def _uniform_bytes(gen, shape, lo, hi):
    return torch.randint(lo, hi + 1, shape, dtype=torch.int32, generator=gen).to(torch.uint8)


def _case(name, M, N, K, seed):
    gen = torch.Generator().manual_seed(seed)
    p = workloads.make_problem(gen, M, N, K, 1)
    sf_shape_a, sf_shape_b = (1, M, K // 16), (1, N, K // 16)
    if name == "sfa_full_range":
        p["SFA"] = _uniform_bytes(gen, sf_shape_a, 0x00, 0x7E)
        p["SFB"] = _uniform_bytes(gen, sf_shape_b, 0x00, 0x0F)   # subnormals and 2^-6 .. 2^-6 * 1.875
    elif name == "sfb_full_range":
        p["SFA"] = _uniform_bytes(gen, sf_shape_a, 0x00, 0x0F)
        p["SFB"] = _uniform_bytes(gen, sf_shape_b, 0x00, 0x7E)
    elif name == "overflow_inf":
        p["B"] = p["B"] & 0x77                                   # every B value >= 0
        p["A"][0, 0:16] = 0x22                                   # +1.0, +1.0
        p["A"][0, 16:32] = 0xAA                                  # -1.0, -1.0
        p["SFA"][0, 0:32] = 0x7E                                 # 448
    elif name == "zero_rows":
        p["A"][0, 0:16] = 0x00                                   # +0 codes
        p["A"][0, 16:32] = 0x88                                  # -0 codes
        p["B"][0, 0:16] = 0x88
        p["B"][0, 16:32] = 0x00
    else:
        raise ValueError(name)
    return p


CASES = ["sfa_full_range", "sfb_full_range", "overflow_inf", "zero_rows"]


@pytest.mark.parametrize("case", CASES)
@pytest.mark.parametrize("variant", sorted(VARIANTS))
def test_format_edge_cases(variant, case, monkeypatch):
    binding = require_gpu()
    (M, N, K), env, expect = VARIANTS[variant]
    for k in _KEYS:
        monkeypatch.delenv(k, raising=False)
    for k, v in env.items():
        monkeypatch.setenv(k, v)
    p = _case(case, M, N, K, seed=100 * sorted(VARIANTS).index(variant) + CASES.index(case))
    ref, absacc, acc = oracle.gemm(p["A"], p["B"], p["SFA"], p["SFB"], M, N, K, 1, want_acc=True)
    # The data must keep every exact sum away from the fp16 overflow threshold
    # (an fp32 accumulator within its tolerance of 65520 could round either way).
    a = np.abs(acc)
    assert not ((a > 0.99 * 65504.0) & (a < 1.01 * FP16_OVERFLOW)).any(), "test data too close to overflow"
    if case == "overflow_inf":
        assert np.isinf(ref[0, 0:16]).all() and (ref[0, 0:16] > 0).all()
        assert np.isinf(ref[0, 16:32]).all() and (ref[0, 16:32] < 0).all()
        assert np.isfinite(ref[0, 32:]).all()
    if case.endswith("full_range"):
        sf = p["SFA"] if case.startswith("sfa") else p["SFB"]
        assert {0x00, 0x01, 0x07, 0x08, 0x7E} <= set(np.unique(sf.numpy()).tolist())
        assert np.isfinite(ref).all()
    d = to_device(p)
    buf, C = alloc_c(M, N, 1)
    binding.nvfp4_gemm_run(d["A"], d["B"], d["SFA"], d["SFB"], C, M, N, K, 1)
    assert binding.nvfp4_gemm_last_launch()["variant"] == expect
    binding.nvfp4_gemm_check_device_status()
    check_canary(buf, M, N, 1)
    assert_close_full(C, p)
    g = C.cpu().numpy()
    if case == "overflow_inf":
        assert np.array_equal(g[0, :32], ref[0, :32])     # +-Inf bit for bit
    if case == "zero_rows":
        assert (g[0, 0:32] == 0).all() and (g[0, :, 0:32] == 0).all()
