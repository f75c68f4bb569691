"""GPU GEMM parity against the CPU oracle, through the C ABI.

Tolerance (elementwise): |gpu - ref| <= 1e-3 * sum_k |a_k b_k| + 1 ulp_fp16(ref).
Small problems are compared whole; the five workloads at full size are
compared on sampled outputs (random points plus every tile's corners).
"""
import numpy as np
import pytest
import torch

import oracle
from block_scaled_fp4_nvfp4_gb300 import workloads
from gpu_util import (alloc_c, assert_close_full, assert_close_points, check_canary, require_gpu,
                      run_single, sample_points, to_device)

pytestmark = pytest.mark.gpu


def test_single_tile_workload():
    binding = require_gpu()
    p = workloads.make_inputs("single_128x128x256", seed=0)[0]
    d = to_device(p)
    buf, C = alloc_c(128, 128, 1)
    run_single(d, C)
    binding.nvfp4_gemm_check_device_status()
    assert_close_full(C, p)
    check_canary(buf, 128, 128, 1)


@pytest.mark.parametrize("M,N,K,L", [
    (128, 128, 512, 1),
    (256, 256, 1024, 1),
    (1, 8, 256, 1),          # smallest legal problem
    (64, 128, 256, 1),       # half an M tile
    (192, 128, 768, 1),      # ragged M tile
    (200, 136, 512, 1),      # ragged M and N tiles
    (129, 264, 256, 2),      # batches, ragged everywhere
    (384, 384, 2048, 1),     # several tiles, deeper K than the stage ring
    (128, 1024, 8192, 1),    # skinny: split-K path
    (64, 2048, 4096, 1),     # skinny, partial M tile, split-K
])
def test_parity_small(M, N, K, L):
    binding = require_gpu()
    p = workloads.make_random_problem(M * 7 + N * 3 + K + L, M, N, K, L)
    d = to_device(p)
    buf, C = alloc_c(M, N, L)
    run_single(d, C)
    binding.nvfp4_gemm_check_device_status()
    assert_close_full(C, p)
    check_canary(buf, M, N, L)


ONE_HOT_CONFIGS = {
    "auto": {},
    "wide": {"NVFP4_BN": "256", "NVFP4_SCHEDULE": "dp", "NVFP4_CLUSTER": "1"},
    "pair": {"NVFP4_BN": "256", "NVFP4_SCHEDULE": "dp", "NVFP4_CLUSTER": "2", "NVFP4_PAIR": "1"},
}


@pytest.mark.parametrize("config", sorted(ONE_HOT_CONFIGS))
def test_one_hot_scales_pin_the_atom_layout(config, monkeypatch):
    """Unit scales except one (row, k-block) per operand: a misplaced scale
    byte changes exactly the rows/columns it lands in.  Run for 128-wide
    tiles, 256-wide tiles and 2-SM pair tiles (whose scales both CTAs copy)."""
    binding = require_gpu()
    for k, v in ONE_HOT_CONFIGS[config].items():
        monkeypatch.setenv(k, v)
    M, N, K = 256, 256, 512
    rng = np.random.default_rng(3)
    for trial in range(4):
        p = workloads.make_random_problem(50 + trial, M, N, K)
        p["SFA"].fill_(0x38)
        p["SFB"].fill_(0x38)
        ra, ca = int(rng.integers(0, M)), int(rng.integers(0, K // 16))
        rb, cb = int(rng.integers(0, N)), int(rng.integers(0, K // 16))
        p["SFA"][0, ra, ca] = 0x50   # 16.0
        p["SFB"][0, rb, cb] = 0x28   # 0.25
        d = to_device(p)
        _, C = alloc_c(M, N, 1)
        run_single(d, C)
        if config == "pair":
            assert binding.nvfp4_gemm_last_launch()["variant"] == "pair"
        binding.nvfp4_gemm_check_device_status()
        assert_close_full(C, p)


def test_stream_k_is_deterministic():
    binding = require_gpu()
    p = workloads.make_random_problem(11, 128, 2048, 8192)
    plan = binding.nvfp4_gemm_plan([128], [2048], [8192], [1], torch.cuda.get_device_properties(0).multi_processor_count)
    assert plan["sk_max_segs"] > 1
    d = to_device(p)
    outs = []
    for _ in range(3):
        _, C = alloc_c(128, 2048, 1)
        run_single(d, C)
        torch.cuda.synchronize()
        outs.append(C.clone())
    binding.nvfp4_gemm_check_device_status()
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    assert torch.equal(outs[0].view(torch.int16), outs[2].view(torch.int16))
    assert_close_full(outs[0], p)


def _grouped(binding, devs, probs, Cs):
    binding.nvfp4_gemm_run_grouped(
        len(probs), [d["A"] for d in devs], [d["B"] for d in devs], [d["SFA"] for d in devs],
        [d["SFB"] for d in devs], [c for _, c in Cs], [p["M"] for p in probs], [p["N"] for p in probs],
        [p["K"] for p in probs], [p["L"] for p in probs])
    binding.nvfp4_gemm_check_device_status()


def test_grouped_small_equals_oracle_and_singles(monkeypatch):
    binding = require_gpu()
    shapes = [(128, 256, 512, 1), (64, 136, 256, 1), (300, 128, 1024, 2), (128, 1024, 4096, 1)]
    probs = [workloads.make_random_problem(200 + i, *s) for i, s in enumerate(shapes)]
    devs = [to_device(p) for p in probs]
    Cs = [alloc_c(p["M"], p["N"], p["L"]) for p in probs]
    _grouped(binding, devs, probs, Cs)
    refs = oracle.gemm_grouped(probs)
    for p, (buf, c), ref in zip(probs, Cs, refs):
        check_canary(buf, p["M"], p["N"], p["L"])
        assert_close_full(c, p)
    # With whole-tile (data-parallel) decomposition every tile is summed in
    # k order by one CTA, so the grouped launch equals single launches bit for bit.
    monkeypatch.setenv("NVFP4_SCHEDULE", "dp")
    Cg = [alloc_c(p["M"], p["N"], p["L"]) for p in probs]
    _grouped(binding, devs, probs, Cg)
    for p, d, (_, c) in zip(probs, devs, Cg):
        _, c1 = alloc_c(p["M"], p["N"], p["L"])
        run_single(d, c1)
        torch.cuda.synchronize()
        assert torch.equal(c.view(torch.int16), c1.view(torch.int16))


def _run_workload(name):
    binding = require_gpu()
    probs = workloads.make_inputs(name, seed=0)
    devs = [to_device(p) for p in probs]
    Cs = [alloc_c(p["M"], p["N"], p["L"]) for p in probs]
    if len(probs) == 1:
        run_single(devs[0], Cs[0][1])
    else:
        binding.nvfp4_gemm_run_grouped(
            len(probs), [d["A"] for d in devs], [d["B"] for d in devs], [d["SFA"] for d in devs],
            [d["SFB"] for d in devs], [c for _, c in Cs], [p["M"] for p in probs],
            [p["N"] for p in probs], [p["K"] for p in probs], [p["L"] for p in probs])
    binding.nvfp4_gemm_check_device_status()
    return probs, Cs


@pytest.mark.parametrize("name", ["skinny_128x7168x16384", "dense_8192x8192x8192", "grouped2", "moe8"])
def test_workload_full_size_sampled(name):
    probs, Cs = _run_workload(name)
    for i, (p, (buf, C)) in enumerate(zip(probs, Cs)):
        check_canary(buf, p["M"], p["N"], p["L"])
        assert not torch.isnan(C).any(), "unwritten output elements"
        ls, ms, ns = sample_points(p["M"], p["N"], p["L"], 1500, seed=i)
        assert_close_points(C, p, ls, ms, ns)


def test_skinny_workload_whole_output():
    """The bench workload compared on every output element."""
    probs, Cs = _run_workload("skinny_128x7168x16384")
    assert_close_full(Cs[0][1], probs[0])


@pytest.mark.parametrize("mode", ["dp", "sk"])
@pytest.mark.parametrize("M,N,K,L", [(256, 512, 2048, 1), (200, 136, 1024, 2), (128, 7168, 4096, 1)])
def test_parity_forced_schedules(mode, M, N, K, L, monkeypatch):
    """The same problem decomposed data-parallel and fully stream-K."""
    binding = require_gpu()
    monkeypatch.setenv("NVFP4_SCHEDULE", mode)
    p = workloads.make_random_problem(M + N + K + (mode == "sk"), M, N, K, L)
    d = to_device(p)
    buf, C = alloc_c(M, N, L)
    run_single(d, C)
    binding.nvfp4_gemm_check_device_status()
    assert_close_full(C, p)
    check_canary(buf, M, N, L)


def test_parity_grouped_stream_k_across_groups(monkeypatch):
    """Stream-K ranges that cross group boundaries (groups with different K)."""
    binding = require_gpu()
    monkeypatch.setenv("NVFP4_SCHEDULE", "sk")
    shapes = [(128, 1024, 4096, 1), (256, 512, 1024, 2), (64, 256, 8192, 1)]
    probs = [workloads.make_random_problem(300 + i, *s) for i, s in enumerate(shapes)]
    devs = [to_device(p) for p in probs]
    Cs = [alloc_c(p["M"], p["N"], p["L"]) for p in probs]
    binding.nvfp4_gemm_run_grouped(
        len(probs), [d["A"] for d in devs], [d["B"] for d in devs], [d["SFA"] for d in devs],
        [d["SFB"] for d in devs], [c for _, c in Cs], [p["M"] for p in probs], [p["N"] for p in probs],
        [p["K"] for p in probs], [p["L"] for p in probs])
    binding.nvfp4_gemm_check_device_status()
    for p, (buf, c) in zip(probs, Cs):
        check_canary(buf, p["M"], p["N"], p["L"])
        assert_close_full(c, p)


@pytest.mark.parametrize("mode", ["auto", "sk"])
@pytest.mark.parametrize("M,N,K,L", [(256, 512, 2048, 1), (200, 136, 1024, 2), (129, 264, 512, 1),
                                     (128, 7168, 4096, 1), (384, 1024, 1024, 1)])
def test_parity_wide_tiles(mode, M, N, K, L, monkeypatch):
    """128 x 256 output tiles (two scale atoms per B k-tile, one accumulator)."""
    binding = require_gpu()
    monkeypatch.setenv("NVFP4_BN", "256")
    monkeypatch.setenv("NVFP4_SCHEDULE", mode)
    p = workloads.make_random_problem(M + 3 * N + K, M, N, K, L)
    d = to_device(p)
    buf, C = alloc_c(M, N, L)
    run_single(d, C)
    binding.nvfp4_gemm_check_device_status()
    assert_close_full(C, p)
    check_canary(buf, M, N, L)


@pytest.mark.parametrize("bn", ["128", "256"])
@pytest.mark.parametrize("M,N,K,L", [(256, 512, 1024, 1), (512, 1024, 2048, 1), (200, 264, 512, 2),
                                     (1024, 136, 768, 1)])
def test_parity_cluster_pairs(bn, M, N, K, L, monkeypatch):
    """Clusters of two CTAs sharing each B tile through multicast."""
    binding = require_gpu()
    monkeypatch.setenv("NVFP4_BN", bn)
    monkeypatch.setenv("NVFP4_SCHEDULE", "dp")
    monkeypatch.setenv("NVFP4_CLUSTER", "2")
    plan = binding.nvfp4_gemm_plan([M], [N], [K], [L], torch.cuda.get_device_properties(0).multi_processor_count)
    assert plan["cluster"] == 2
    p = workloads.make_random_problem(M + N + 5 * K + int(bn), M, N, K, L)
    d = to_device(p)
    buf, C = alloc_c(M, N, L)
    run_single(d, C)
    assert binding.nvfp4_gemm_last_launch()["variant"] in ("multicast", "pair")
    binding.nvfp4_gemm_check_device_status()
    assert_close_full(C, p)
    check_canary(buf, M, N, L)


@pytest.mark.parametrize("pair", ["1", "0"])
@pytest.mark.parametrize("M,N,K,L", [(256, 512, 1024, 1), (512, 1024, 2048, 1), (200, 264, 512, 2),
                                     (1024, 136, 768, 1), (256, 256, 256, 1), (768, 520, 1536, 1)])
def test_parity_pair_tiles(pair, M, N, K, L, monkeypatch):
    """256 x 256 tiles of two CTAs: 2-SM MMAs with half of B in each CTA
    (pair=1) or B shared by multicast (pair=0).  Ragged M leaves the odd
    CTA's rows partly or wholly past M; ragged N leaves the last tile's
    second scale block past the last row of B."""
    binding = require_gpu()
    monkeypatch.setenv("NVFP4_BN", "256")
    monkeypatch.setenv("NVFP4_SCHEDULE", "dp")
    monkeypatch.setenv("NVFP4_CLUSTER", "2")
    monkeypatch.setenv("NVFP4_PAIR", pair)
    plan = binding.nvfp4_gemm_plan([M], [N], [K], [L], torch.cuda.get_device_properties(0).multi_processor_count)
    assert plan["cluster"] == 2 and plan["pair"] == int(pair)
    p = workloads.make_random_problem(3 * M + N + K + L, M, N, K, L)
    d = to_device(p)
    buf, C = alloc_c(M, N, L)
    run_single(d, C)
    assert binding.nvfp4_gemm_last_launch()["variant"] == ("pair" if pair == "1" else "multicast")
    binding.nvfp4_gemm_check_device_status()
    assert_close_full(C, p)
    check_canary(buf, M, N, L)


def test_parity_pair_tiles_grouped(monkeypatch):
    """Grouped problem on 2-SM pair tiles, every group with an even number of
    m-tiles, against the oracle group by group."""
    binding = require_gpu()
    monkeypatch.setenv("NVFP4_BN", "256")
    monkeypatch.setenv("NVFP4_SCHEDULE", "dp")
    monkeypatch.setenv("NVFP4_CLUSTER", "2")
    monkeypatch.setenv("NVFP4_PAIR", "1")    # short K: the planner alone would pick multicast pairs
    Ms, Ns, Ks = [256, 512, 200], [512, 264, 1024], [1024, 512, 768]
    plan = binding.nvfp4_gemm_plan(Ms, Ns, Ks, [1] * 3, torch.cuda.get_device_properties(0).multi_processor_count)
    assert plan["pair"] == 1
    probs = [workloads.make_random_problem(900 + g, Ms[g], Ns[g], Ks[g], 1) for g in range(3)]
    ds = [to_device(p) for p in probs]
    Cs = [alloc_c(Ms[g], Ns[g], 1) for g in range(3)]
    binding.nvfp4_gemm_run_grouped(3, [d["A"] for d in ds], [d["B"] for d in ds], [d["SFA"] for d in ds],
                                   [d["SFB"] for d in ds], [c[1] for c in Cs], Ms, Ns, Ks, [1] * 3)
    assert binding.nvfp4_gemm_last_launch()["variant"] == "pair"
    binding.nvfp4_gemm_check_device_status()
    for g in range(3):
        assert_close_full(Cs[g][1], probs[g])
        check_canary(Cs[g][0], Ms[g], Ns[g], 1)


@pytest.mark.parametrize("config", ["multicast", "pair"])
def test_cluster_timeout_is_reported(config, monkeypatch):
    """A skipped k-tile in a cluster pair: both CTAs give up, the host sees it."""
    binding = require_gpu()
    monkeypatch.setenv("NVFP4_SCHEDULE", "dp")
    monkeypatch.setenv("NVFP4_CLUSTER", "2")
    if config == "pair":
        monkeypatch.setenv("NVFP4_BN", "256")
        monkeypatch.setenv("NVFP4_PAIR", "1")
    M, N, K = 256, 512, 1024
    p = workloads.make_random_problem(5, M, N, K)
    d = to_device(p)
    try:
        binding.nvfp4_gemm_set_wait_timeout_ns(50_000_000)
        binding.nvfp4_gemm_debug_inject_skip(1)
        _, C = alloc_c(M, N, 1)
        run_single(d, C)
        with pytest.raises(binding.Nvfp4Error) as e:
            binding.nvfp4_gemm_check_device_status()
        assert e.value.code == -4
    finally:
        binding.nvfp4_gemm_debug_inject_skip(-1)
        binding.nvfp4_gemm_set_wait_timeout_ns(2_000_000_000)
    _, C = alloc_c(M, N, 1)
    run_single(d, C)
    binding.nvfp4_gemm_check_device_status()
    assert_close_full(C, p)


@pytest.mark.parametrize("mode", ["dp", "sk"])
@pytest.mark.parametrize("M,N,K,L", [(128, 448, 2048, 1), (200, 136, 512, 2), (64, 264, 1024, 1),
                                     (256, 192, 768, 1)])
def test_parity_narrow_tiles(mode, M, N, K, L, monkeypatch):
    """128 x 64 output tiles: an odd n-tile reads the upper half of its
    128-row B scale atom."""
    binding = require_gpu()
    monkeypatch.setenv("NVFP4_BN", "64")
    monkeypatch.setenv("NVFP4_SCHEDULE", mode)
    p = workloads.make_random_problem(7 * M + N + K, M, N, K, L)
    d = to_device(p)
    buf, C = alloc_c(M, N, L)
    run_single(d, C)
    binding.nvfp4_gemm_check_device_status()
    assert_close_full(C, p)
    check_canary(buf, M, N, L)


PARTIAL_K_CONFIGS = {
    "auto": {},
    "dp": {"NVFP4_SCHEDULE": "dp"},
    "sk": {"NVFP4_SCHEDULE": "sk"},
    "wide": {"NVFP4_BN": "256", "NVFP4_SCHEDULE": "dp", "NVFP4_CLUSTER": "1"},
    "narrow": {"NVFP4_BN": "64"},
}


@pytest.mark.parametrize("config", sorted(PARTIAL_K_CONFIGS))
@pytest.mark.parametrize("M,N,K,L", [(128, 128, 64, 1), (256, 512, 320, 1), (200, 136, 192, 2),
                                     (512, 1024, 1088, 1), (64, 2048, 4160, 1), (1, 8, 128, 1)])
def test_parity_partial_k_tiles(config, M, N, K, L, monkeypatch):
    """K % 256 != 0: the last k-tile is partial (zero codes past the row end,
    zero-padded scales), under every schedule and tile width."""
    binding = require_gpu()
    for k, v in PARTIAL_K_CONFIGS[config].items():
        monkeypatch.setenv(k, v)
    p = workloads.make_random_problem(5 * M + N + 3 * K + L, M, N, K, L)
    d = to_device(p)
    buf, C = alloc_c(M, N, L)
    run_single(d, C)
    binding.nvfp4_gemm_check_device_status()
    assert_close_full(C, p)
    check_canary(buf, M, N, L)


@pytest.mark.parametrize("pair", ["1", "0"])
@pytest.mark.parametrize("M,N,K", [(256, 512, 320), (512, 264, 704)])
def test_parity_partial_k_tiles_pairs(pair, M, N, K, monkeypatch):
    """Partial last k-tile on 2-CTA tiles (2-SM MMAs or B multicast)."""
    binding = require_gpu()
    monkeypatch.setenv("NVFP4_BN", "256")
    monkeypatch.setenv("NVFP4_SCHEDULE", "dp")
    monkeypatch.setenv("NVFP4_CLUSTER", "2")
    monkeypatch.setenv("NVFP4_PAIR", pair)
    plan = binding.nvfp4_gemm_plan([M], [N], [K], [1], torch.cuda.get_device_properties(0).multi_processor_count)
    assert plan["cluster"] == 2 and plan["pair"] == int(pair)
    p = workloads.make_random_problem(M + 7 * N + K, M, N, K, 1)
    d = to_device(p)
    buf, C = alloc_c(M, N, 1)
    run_single(d, C)
    assert binding.nvfp4_gemm_last_launch()["variant"] == ("pair" if pair == "1" else "multicast")
    binding.nvfp4_gemm_check_device_status()
    assert_close_full(C, p)
    check_canary(buf, M, N, 1)


@pytest.mark.parametrize("M,N,K,L", [(128, 7168, 16384, 1), (128, 512, 4096, 1), (100, 1032, 2048, 1),
                                     (64, 2048, 4096, 1), (200, 264, 2048, 2), (128, 3072, 1984, 1)])
def test_cluster_reduction_matches_workspace_path(M, N, K, L, monkeypatch):
    """Stream-K segments summed in distributed shared memory (clusters of 2 or
    4 CTAs) give the same bits as the workspace path (same k-order sums),
    and both match the oracle."""
    binding = require_gpu()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    monkeypatch.delenv("NVFP4_SKRED", raising=False)
    plan = binding.nvfp4_gemm_plan([M], [N], [K], [L], sms)
    assert plan["cluster_reduce"] == 1, plan
    p = workloads.make_random_problem(M * 3 + N + K * 5 + L, M, N, K, L)
    d = to_device(p)
    buf, C = alloc_c(M, N, L)
    run_single(d, C)
    launched = binding.nvfp4_gemm_last_launch()
    assert launched["variant"] == "cluster_reduce" and launched["cluster"] == plan["cluster"]
    binding.nvfp4_gemm_check_device_status()
    check_canary(buf, M, N, L)
    monkeypatch.setenv("NVFP4_SKRED", "0")
    assert binding.nvfp4_gemm_plan([M], [N], [K], [L], sms)["cluster_reduce"] == 0
    buf2, C2 = alloc_c(M, N, L)
    run_single(d, C2)
    assert binding.nvfp4_gemm_last_launch()["variant"] == "single"
    binding.nvfp4_gemm_check_device_status()
    assert torch.equal(C.view(torch.int16), C2.view(torch.int16))
    if M * N * K <= 128 * 7168 * 4096:
        assert_close_full(C, p)
    else:
        ls, ms, ns = sample_points(M, N, L, 3000, seed=9)
        assert_close_points(C, p, ls, ms, ns)


def test_cluster_reduction_timeout_is_reported(monkeypatch):
    """A skipped k-tile in one segment of a reduction cluster: every CTA of the
    cluster gives up, the host sees the timeout, and the next call is right."""
    binding = require_gpu()
    monkeypatch.delenv("NVFP4_SKRED", raising=False)
    M, N, K = 128, 512, 4096
    assert binding.nvfp4_gemm_plan([M], [N], [K], [1], torch.cuda.get_device_properties(0).multi_processor_count)[
        "cluster_reduce"] == 1
    p = workloads.make_random_problem(17, M, N, K)
    d = to_device(p)
    try:
        binding.nvfp4_gemm_set_wait_timeout_ns(50_000_000)
        binding.nvfp4_gemm_debug_inject_skip(1)
        _, C = alloc_c(M, N, 1)
        run_single(d, C)
        with pytest.raises(binding.Nvfp4Error) as e:
            binding.nvfp4_gemm_check_device_status()
        assert e.value.code == -4
    finally:
        binding.nvfp4_gemm_debug_inject_skip(-1)
        binding.nvfp4_gemm_set_wait_timeout_ns(2_000_000_000)
    buf, C = alloc_c(M, N, 1)
    run_single(d, C)
    binding.nvfp4_gemm_check_device_status()
    assert_close_full(C, p)
    check_canary(buf, M, N, 1)


_PAIR_ENV = {"NVFP4_BN": "256", "NVFP4_SCHEDULE": "dp", "NVFP4_CLUSTER": "2", "NVFP4_PAIR": "1"}


@pytest.mark.parametrize("M,N,K,env,variant", [(128, 1024, 4096, {}, "cluster_reduce"),
                                               (512, 2048, 2048, {}, "cluster_reduce"),
                                               (384, 4096, 1024, {}, "single"),
                                               (512, 512, 1024, _PAIR_ENV, "pair")])
def test_optional_l2_prefetch_changes_no_result(M, N, K, env, variant, monkeypatch):
    """The optional L2 prefetch of each CTA's first k-tiles before the launch
    dependency (NVFP4_PREFETCH, off by default) leaves every result as it is,
    for cluster-reduced stream-K, plain stream-K and 2-SM pair plans alike."""
    binding = require_gpu()
    monkeypatch.setenv("NVFP4_PREFETCH", "6")
    for k, v in env.items():
        monkeypatch.setenv(k, v)
    p = workloads.make_random_problem(M + 3 * N + K, M, N, K, 1)
    d = to_device(p)
    buf, C = alloc_c(M, N, 1)
    run_single(d, C)
    assert binding.nvfp4_gemm_last_launch()["variant"] == variant
    binding.nvfp4_gemm_check_device_status()
    assert_close_full(C, p)
    check_canary(buf, M, N, 1)


# Planner overrides crossed with random shapes: every combination either runs
# as asked or the planner falls back to a valid plan; the results must match
# the oracle either way.
_SWEEP_ENVS = [
    {},
    {"NVFP4_BN": "64"},
    {"NVFP4_BN": "128", "NVFP4_SCHEDULE": "dp"},
    {"NVFP4_BN": "128", "NVFP4_SCHEDULE": "sk"},
    {"NVFP4_BN": "128", "NVFP4_SCHEDULE": "sk", "NVFP4_SKRED": "0"},
    {"NVFP4_BN": "256", "NVFP4_SCHEDULE": "dp", "NVFP4_CLUSTER": "1"},
    {"NVFP4_BN": "256", "NVFP4_SCHEDULE": "dp", "NVFP4_CLUSTER": "2", "NVFP4_PAIR": "0"},
    {"NVFP4_BN": "256", "NVFP4_SCHEDULE": "dp", "NVFP4_CLUSTER": "2", "NVFP4_PAIR": "1"},
    {"NVFP4_BN": "128", "NVFP4_SCHEDULE": "dp", "NVFP4_CLUSTER": "2"},
    {"NVFP4_BN": "256", "NVFP4_SCHEDULE": "sk"},
]
_SWEEP_KEYS = ("NVFP4_BN", "NVFP4_SCHEDULE", "NVFP4_CLUSTER", "NVFP4_PAIR", "NVFP4_SKRED")


def _sweep_shapes(case):
    """1-3 problems; N a multiple of 8 up to 520, K a multiple of 64, L 1-2.
    Cluster overrides get an even number of 128-row m-tiles (ragged inside
    the last one); stream-K ones get long K (up to 4096) and few tiles, so
    that 2- and 4-segment reductions occur."""
    env = _SWEEP_ENVS[case % len(_SWEEP_ENVS)]
    rng = np.random.default_rng(1000 + case)
    wants_cluster = env.get("NVFP4_CLUSTER") == "2"
    wants_sk = env.get("NVFP4_SCHEDULE") == "sk" or not env
    shapes = []
    for _ in range(int(rng.integers(1, 4))):
        if wants_cluster:
            M = 256 * int(rng.integers(1, 3)) - int(rng.integers(0, 128))
        elif wants_sk:
            M = int(rng.integers(1, 257))
        else:
            M = int(rng.choice([int(rng.integers(1, 385)), 128 * int(rng.integers(1, 4))]))
        N = 8 * int(rng.integers(1, 66))
        K = 64 * int(rng.integers(16, 65)) if wants_sk else 64 * int(rng.integers(1, 17))
        L = int(rng.integers(1, 3))
        shapes.append((M, N, K, L))
    return shapes


@pytest.mark.parametrize("case", range(20))
def test_random_shapes_and_plans(case, monkeypatch):
    """Seeded random groups under a rotating planner override (tile width,
    schedule, clusters, 2-SM pairs, cluster reduction), element by element
    against the oracle."""
    binding = require_gpu()
    shapes = _sweep_shapes(case)
    for k in _SWEEP_KEYS:
        monkeypatch.delenv(k, raising=False)
    for k, v in _SWEEP_ENVS[case % len(_SWEEP_ENVS)].items():
        monkeypatch.setenv(k, v)
    probs = [workloads.make_random_problem(5000 + 10 * case + i, *s) for i, s in enumerate(shapes)]
    devs = [to_device(p) for p in probs]
    Cs = [alloc_c(p["M"], p["N"], p["L"]) for p in probs]
    _grouped(binding, devs, probs, Cs)
    for p, (buf, c) in zip(probs, Cs):
        check_canary(buf, p["M"], p["N"], p["L"])
        assert_close_full(c, p)


@pytest.mark.parametrize("shapes", [[(384, 2048, 1024, 1), (64, 1024, 1024, 1)],
                                    [(200, 1536, 1024, 1), (100, 512, 1280, 2)],
                                    [(300, 768, 2048, 2)]])
def test_padded_pair_tiles(shapes, monkeypatch):
    """2-SM pairs over groups with an odd number of 128-row m-tiles, each such
    group padded by one m-tile: the padding rows load as zeros (including the
    next batch's scale block read past the last row block when L > 1) and are
    never stored; every real element matches the oracle."""
    binding = require_gpu()
    for k, v in {"NVFP4_PAD_PAIRS": "2", "NVFP4_BN": "256", "NVFP4_SCHEDULE": "dp"}.items():
        monkeypatch.setenv(k, v)
    for k in ("NVFP4_PAIR", "NVFP4_CLUSTER"):
        monkeypatch.delenv(k, raising=False)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    M, N, K, L = ([s[i] for s in shapes] for i in range(4))
    plan = binding.nvfp4_gemm_plan(M, N, K, L, sms)
    padded = sum(((m + 127) // 128 + 1) // 2 * 2 * ((n + 255) // 256) * l for m, n, _, l in shapes)
    assert plan["pair"] == 1 and plan["tiles"] == padded, plan
    probs = [workloads.make_random_problem(7000 + 13 * i + m, *s) for i, (m, s) in enumerate(zip(M, shapes))]
    devs = [to_device(p) for p in probs]
    Cs = [alloc_c(p["M"], p["N"], p["L"]) for p in probs]
    _grouped(binding, devs, probs, Cs)
    assert binding.nvfp4_gemm_last_launch()["variant"] == "pair"
    for p, (buf, c) in zip(probs, Cs):
        check_canary(buf, p["M"], p["N"], p["L"])
        assert_close_full(c, p)


@pytest.mark.parametrize("M,N,K,L", [
    (128, 256, 65536, 1),    # K = 2^16: 64 stream-K segments per tile, summed through the workspace
    (1, 8, 65536, 1),        # a single 1 x 8 output row over 64 segments
    (8, 65528, 256, 1),      # very wide, 8 rows: 256 tiles of 128 x 256, mostly padding rows
    (4096, 8, 512, 1),       # very tall, 8 columns: N smaller than every tile width
    (300, 200, 4096, 6),     # six batches, ragged everywhere, clusters of four reducing
])
def test_parity_extreme_shapes(M, N, K, L):
    """Extreme aspect ratios and depths under the default planner, element by
    element against the oracle."""
    binding = require_gpu()
    p = workloads.make_random_problem(M + N + K + L, M, N, K, L)
    d = to_device(p)
    buf, C = alloc_c(M, N, L)
    run_single(d, C)
    binding.nvfp4_gemm_check_device_status()
    assert_close_full(C, p)
    check_canary(buf, M, N, L)
