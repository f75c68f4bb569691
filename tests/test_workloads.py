"""The seeded input generators: shapes, determinism, value distributions and
the derived FLOP / byte counts (CPU only)."""
import numpy as np
import torch

from block_scaled_fp4_nvfp4_gb300 import workloads


def test_moe_group_order():
    assert workloads.moe_m_order(0) == [384, 64, 1024, 256, 192, 512, 128, 768]
    assert [s[0] for s in workloads.WORKLOADS["moe8"].shapes] == [384, 64, 1024, 256, 192, 512, 128, 768]


def test_shapes_and_determinism():
    a = workloads.make_inputs("single_128x128x256", seed=0)
    b = workloads.make_inputs("single_128x128x256", seed=0)
    c = workloads.make_inputs("single_128x128x256", seed=1)
    p = a[0]
    assert p["A"].shape == (1, 128, 128) and p["A"].dtype == torch.uint8
    assert p["SFA"].shape == (1, 128, 16) and p["SFB"].shape == (1, 128, 16)
    for k in ("A", "B", "SFA", "SFB"):
        assert torch.equal(a[0][k], b[0][k])
    assert not torch.equal(a[0]["A"], c[0]["A"])


def test_scale_distribution():
    p = workloads.make_random_problem(0, 256, 256, 4096)
    v = p["SFA"].view(torch.float8_e4m3fn).to(torch.float64).numpy().ravel()
    e = np.floor(np.log2(v))
    assert e.min() == -4 and e.max() == 1
    f = v / np.exp2(e) - 1.0
    assert np.all(f * 8 == np.round(f * 8)) and f.min() == 0.0 and f.max() == 0.875
    q = workloads.make_random_problem(0, 64, 64, 1024, j_range=(-3, 0))
    w = q["SFB"].view(torch.float8_e4m3fn).to(torch.float64).numpy().ravel()
    assert np.floor(np.log2(w)).min() == -3 and np.floor(np.log2(w)).max() == 0


def test_code_distribution_uniform():
    p = workloads.make_random_problem(1, 512, 8, 4096)
    a = p["A"].numpy().ravel()
    lo = np.bincount(a & 0xF, minlength=16)
    hi = np.bincount(a >> 4, minlength=16)
    exp = a.size / 16
    assert np.all(np.abs(lo - exp) < 0.05 * exp) and np.all(np.abs(hi - exp) < 0.05 * exp)


def test_flop_and_byte_counts():
    W = workloads.WORKLOADS
    assert W["single_128x128x256"].bytes == 69632
    assert abs(W["skinny_128x7168x16384"].flops / 1e9 - 30.06) < 0.01
    assert abs(W["skinny_128x7168x16384"].bytes / 1e6 - 69.07) < 0.01
    assert abs(W["dense_8192x8192x8192"].flops / 1e9 - 1099.5) < 0.1
    assert abs(W["grouped2"].flops / 1e9 - 120.26) < 0.01
    assert abs(W["moe8"].flops / 1e9 - 195.42) < 0.01
    assert abs(W["moe8"].bytes / 1e6 - 172.8) < 0.1
