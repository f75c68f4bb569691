"""Stream-K tails of CTA-pair plans (opt-in: NVFP4_PAIR_SK), element by element
against the oracle.

Pair plans (2-SM MMAs, or B shared by multicast) run their trailing tiles as
stream-K: a split tile has two segments; the one holding the tile's last
k-tiles publishes an fp32 partial and a ready flag per epilogue warp, the one
holding its first k-tiles adds it and stores the tile.  The tests force such
tails on small problems (NVFP4_PAIR_SK=2), cover grouped and padded plans and
partial k-tiles, check that results do not change from run to run, and that a
wait that runs out is reported and leaves the next launch correct.
"""
import pytest
import torch

from block_scaled_fp4_nvfp4_gb300 import workloads
from gpu_util import alloc_c, assert_close_full, check_canary, require_gpu, to_device

pytestmark = pytest.mark.gpu

_KEYS = ("NVFP4_BN", "NVFP4_SCHEDULE", "NVFP4_CLUSTER", "NVFP4_PAIR", "NVFP4_SKRED", "NVFP4_PAD_PAIRS",
         "NVFP4_PAIR_SK")


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def _env(monkeypatch, pair, extra=None):
    for k in _KEYS:
        monkeypatch.delenv(k, raising=False)
    env = {"NVFP4_BN": "256", "NVFP4_SCHEDULE": "dp", "NVFP4_CLUSTER": "2", "NVFP4_PAIR": pair,
           "NVFP4_PAIR_SK": "2"}
    env.update(extra or {})
    for k, v in env.items():
        monkeypatch.setenv(k, v)


def _run_grouped(binding, probs):
    devs = [to_device(p) for p in probs]
    Cs = [alloc_c(p["M"], p["N"], p["L"]) for p in probs]
    binding.nvfp4_gemm_run_grouped(
        len(probs), [d["A"] for d in devs], [d["B"] for d in devs], [d["SFA"] for d in devs],
        [d["SFB"] for d in devs], [c for _, c in Cs], [p["M"] for p in probs], [p["N"] for p in probs],
        [p["K"] for p in probs], [p["L"] for p in probs])
    return devs, Cs


SHAPES = [
    [(2048, 2560, 2048, 1)],                         # 80 pair tiles: a partial second wave
    [(1024, 2048, 1536, 2)],                         # L = 2
    [(2048, 2048, 4096, 1), (2048, 1032, 2048, 1)],  # two groups of different K, ragged N
    [(256, 2048, 1088, 1)],                          # partial last k-tile
    [(1000, 3000, 2048, 1)],                         # ragged M and N
]


@pytest.mark.parametrize("pair", ["1", "0"])
@pytest.mark.parametrize("case", range(len(SHAPES)))
def test_pair_stream_k_tail_parity(case, pair, monkeypatch):
    binding = require_gpu()
    _env(monkeypatch, pair)
    shapes = SHAPES[case]
    M, N, K, L = ([s[i] for s in shapes] for i in range(4))
    plan = binding.nvfp4_gemm_plan(M, N, K, L, _sms())
    assert plan["cluster"] == 2 and plan["pair"] == int(pair)
    if plan["sk_tiles"] == 0:
        pytest.skip("no valid stream-K tail for this shape on %d SMs" % _sms())
    assert plan["sk_max_segs"] == 2
    probs = [workloads.make_random_problem(4000 + 17 * case + i, *s) for i, s in enumerate(shapes)]
    _, Cs = _run_grouped(binding, probs)
    assert binding.nvfp4_gemm_last_launch()["variant"] == ("pair" if pair == "1" else "multicast")
    binding.nvfp4_gemm_check_device_status()
    for p, (buf, c) in zip(probs, Cs):
        check_canary(buf, p["M"], p["N"], p["L"])
        assert_close_full(c, p)


@pytest.mark.parametrize("shapes", [[(384, 2048, 2048, 1), (64, 1024, 2048, 1)],
                                    [(640, 2560, 1024, 1), (192, 512, 1024, 2)]])
def test_padded_pairs_with_stream_k_tail(shapes, monkeypatch):
    """Groups with an odd number of m-tiles, padded to 2-SM pairs, with a
    stream-K tail: padding rows are computed from zero-filled loads and
    never stored, and their partials are exchanged like any other rows."""
    binding = require_gpu()
    for k in _KEYS:
        monkeypatch.delenv(k, raising=False)
    for k, v in {"NVFP4_BN": "256", "NVFP4_SCHEDULE": "dp", "NVFP4_PAD_PAIRS": "2", "NVFP4_PAIR_SK": "2"}.items():
        monkeypatch.setenv(k, v)
    M, N, K, L = ([s[i] for s in shapes] for i in range(4))
    plan = binding.nvfp4_gemm_plan(M, N, K, L, _sms())
    assert plan["pair"] == 1
    if plan["sk_tiles"] == 0:
        pytest.skip("no valid stream-K tail for this shape on %d SMs" % _sms())
    probs = [workloads.make_random_problem(4500 + i + M[i], *s) for i, s in enumerate(shapes)]
    _, Cs = _run_grouped(binding, probs)
    assert binding.nvfp4_gemm_last_launch()["variant"] == "pair"
    binding.nvfp4_gemm_check_device_status()
    for p, (buf, c) in zip(probs, Cs):
        check_canary(buf, p["M"], p["N"], p["L"])
        assert_close_full(c, p)


def test_pair_stream_k_is_deterministic(monkeypatch):
    binding = require_gpu()
    _env(monkeypatch, "1")
    p = workloads.make_random_problem(77, 2048, 2560, 2048)
    d = to_device(p)
    outs = []
    for _ in range(3):
        _, C = alloc_c(2048, 2560, 1)
        binding.nvfp4_gemm_run(d["A"], d["B"], d["SFA"], d["SFB"], C, 2048, 2560, 2048, 1)
        torch.cuda.synchronize()
        outs.append(C.clone())
    binding.nvfp4_gemm_check_device_status()
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    assert torch.equal(outs[0].view(torch.int16), outs[2].view(torch.int16))
    # and equal to the same tiles computed whole (two addends: order-free)
    monkeypatch.setenv("NVFP4_PAIR_SK", "0")
    assert binding.nvfp4_gemm_plan([2048], [2560], [2048], [1], _sms())["sk_tiles"] == 0
    _, C = alloc_c(2048, 2560, 1)
    binding.nvfp4_gemm_run(d["A"], d["B"], d["SFA"], d["SFB"], C, 2048, 2560, 2048, 1)
    binding.nvfp4_gemm_check_device_status()
    assert_close_full(outs[0], p)
    assert_close_full(C, p)


@pytest.mark.parametrize("pair", ["1", "0"])
def test_pair_stream_k_timeout_is_reported(pair, monkeypatch):
    """CTA 0 skips one k-tile's arrival (host-side injection, nothing in
    flight): its pair gives up, any segment waiting for its partial gives up
    at its bounded wait, the host sees the timeout, and the next launch --
    with the ready flags cleared by the status query -- is correct."""
    binding = require_gpu()
    _env(monkeypatch, pair)
    M, N, K = 2048, 2560, 2048
    p = workloads.make_random_problem(91, M, N, K)
    d = to_device(p)
    try:
        binding.nvfp4_gemm_set_wait_timeout_ns(50_000_000)
        binding.nvfp4_gemm_debug_inject_skip(1)
        _, C = alloc_c(M, N, 1)
        binding.nvfp4_gemm_run(d["A"], d["B"], d["SFA"], d["SFB"], C, M, N, K, 1)
        with pytest.raises(binding.Nvfp4Error) as e:
            binding.nvfp4_gemm_check_device_status()
        assert e.value.code == -4
    finally:
        binding.nvfp4_gemm_debug_inject_skip(-1)
        binding.nvfp4_gemm_set_wait_timeout_ns(2_000_000_000)
    buf, C = alloc_c(M, N, 1)
    binding.nvfp4_gemm_run(d["A"], d["B"], d["SFA"], d["SFB"], C, M, N, K, 1)
    binding.nvfp4_gemm_check_device_status()
    check_canary(buf, M, N, 1)
    assert_close_full(C, p)
