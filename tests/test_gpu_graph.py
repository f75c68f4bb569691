"""Launches captured in CUDA graphs and replayed, element by element against
the oracle: a replay computes what an eager launch computes, a graph captured
before the split-K workspace grew stays valid after it grew (the replaced
buffer is kept), and a launch that would grow the workspace during capture is
refused before anything is recorded.  The preparation kernels (quantize,
repack) are captured with the GEMM too."""
import pytest
import torch

from block_scaled_fp4_nvfp4_gb300 import workloads
from gpu_util import alloc_c, assert_close_full, check_canary, require_gpu, to_device

pytestmark = pytest.mark.gpu

_KEYS = ("NVFP4_BN", "NVFP4_SCHEDULE", "NVFP4_CLUSTER", "NVFP4_PAIR", "NVFP4_SKRED", "NVFP4_PAD_PAIRS",
         "NVFP4_PAIR_SK")


def _env(monkeypatch, **kv):
    for k in _KEYS:
        monkeypatch.delenv(k, raising=False)
    for k, v in kv.items():
        monkeypatch.setenv(k, str(v))


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def _workspace_plan(binding, M, N, K):
    plan = binding.nvfp4_gemm_plan([M], [N], [K], [1], _sms())
    assert plan["sk_max_segs"] > 1 and plan["cluster_reduce"] == 0, plan
    return plan


def _run(binding, d, C, stream):
    binding.nvfp4_gemm_run(d["A"], d["B"], d["SFA"], d["SFB"], C, d["M"], d["N"], d["K"], d["L"], stream=stream)


@pytest.mark.parametrize("shape,env", [
    ((2048, 2048, 2048, 1), {}),                                         # default plan
    ((1024, 2048, 1024, 1), {"NVFP4_BN": 256, "NVFP4_SCHEDULE": "dp", "NVFP4_CLUSTER": 2,
                             "NVFP4_PAIR": 1}),                          # 2-SM pairs
    ((128, 1024, 8192, 1), {"NVFP4_SCHEDULE": "sk", "NVFP4_BN": 128}),   # workspace stream-K
    ((128, 9728, 2048, 1), {}),                                          # cluster reduction (152 SMs)
])
def test_graph_replay_matches_oracle(shape, env, monkeypatch):
    binding = require_gpu()
    _env(monkeypatch, **env)
    p = workloads.make_random_problem(2100 + shape[0] + shape[2], *shape)
    d = to_device(p)
    stream = torch.cuda.Stream()
    buf, C = alloc_c(*shape[:2], shape[3])
    _run(binding, d, C, stream)          # eager first: creates any workspace outside the capture
    stream.synchronize()
    C.fill_(float("nan"))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        _run(binding, d, C, stream)
    for _ in range(2):
        C.fill_(float("nan"))
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        binding.nvfp4_gemm_check_device_status(stream)
        check_canary(buf, shape[0], shape[1], shape[3])
        assert_close_full(C, p)


def test_graph_survives_workspace_growth(monkeypatch):
    """Capture a stream-K launch with a small workspace, run a problem whose
    plan needs a larger one on the same stream (the workspace grows), then
    replay the first graph: it still names the first buffer, which must still
    be allocated, and its result must still be right."""
    binding = require_gpu()
    _env(monkeypatch, NVFP4_SCHEDULE="sk", NVFP4_BN=128)
    small = (128, 1024, 8192, 1)
    big = (256, 4096, 8192, 1)
    ws_small = _workspace_plan(binding, *small[:3])
    _env(monkeypatch, NVFP4_SCHEDULE="sk", NVFP4_BN=256)
    ws_big = _workspace_plan(binding, *big[:3])
    assert ws_big["sk_tiles"] * 256 * ws_big["sk_max_segs"] > ws_small["sk_tiles"] * 128 * ws_small["sk_max_segs"]
    stream = torch.cuda.Stream()
    p1 = workloads.make_random_problem(2201, *small)
    p2 = workloads.make_random_problem(2202, *big)
    d1, d2 = to_device(p1), to_device(p2)

    _env(monkeypatch, NVFP4_SCHEDULE="sk", NVFP4_BN=128)
    buf1, C1 = alloc_c(*small[:2], 1)
    _run(binding, d1, C1, stream)
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        _run(binding, d1, C1, stream)

    _env(monkeypatch, NVFP4_SCHEDULE="sk", NVFP4_BN=256)
    buf2, C2 = alloc_c(*big[:2], 1)
    _run(binding, d2, C2, stream)         # grows this stream's workspace
    stream.synchronize()
    binding.nvfp4_gemm_check_device_status(stream)
    assert_close_full(C2, p2)

    for _ in range(2):
        C1.fill_(float("nan"))
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        binding.nvfp4_gemm_check_device_status(stream)
        check_canary(buf1, small[0], small[1], 1)
        assert_close_full(C1, p1)


def test_workspace_growth_during_capture_is_refused(monkeypatch):
    """A fresh stream has no workspace: capturing a stream-K launch on it
    first is refused (INVALID_ARG, nothing recorded, nothing allocated); after
    one eager launch the same capture works."""
    binding = require_gpu()
    _env(monkeypatch, NVFP4_SCHEDULE="sk", NVFP4_BN=128)
    shape = (128, 1024, 8192, 1)
    _workspace_plan(binding, *shape[:3])
    p = workloads.make_random_problem(2301, *shape)
    d = to_device(p)
    stream = torch.cuda.Stream()
    _, C = alloc_c(*shape[:2], 1)
    g = torch.cuda.CUDAGraph()
    with pytest.raises(binding.Nvfp4Error) as e:
        with torch.cuda.graph(g, stream=stream):
            _run(binding, d, C, stream)
    assert e.value.code == -1 and "captured" in str(e.value)
    torch.cuda.synchronize()
    _run(binding, d, C, stream)
    stream.synchronize()
    g2 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g2, stream=stream):
        _run(binding, d, C, stream)
    C.fill_(float("nan"))
    torch.cuda.synchronize()
    g2.replay()
    torch.cuda.synchronize()
    binding.nvfp4_gemm_check_device_status(stream)
    assert_close_full(C, p)


def test_graph_of_quantize_repack_and_gemm():
    """The whole preparation and the GEMM in one graph: quantize A from bf16,
    repack B's row-major scales, multiply; three kernels launched as
    programmatic dependents of one another, replayed twice (outputs cleared
    in between), against the oracle's quantization and GEMM."""
    import oracle
    binding = require_gpu()
    M, N, K = 256, 512, 2048
    g = torch.Generator().manual_seed(77)
    xa = torch.randn((1, M, K), generator=g).to(torch.bfloat16)
    pb = workloads.make_random_problem(78, M, N, K)
    stream = torch.cuda.Stream()
    xa_d = xa.cuda()
    B = pb["B"].cuda()
    sfb_raw = pb["SFB"].cuda()
    codes_a = torch.empty((1, M, K // 2), dtype=torch.uint8, device="cuda")
    sfa = torch.empty(binding.nvfp4_gemm_repacked_scales_bytes(M, K, 1), dtype=torch.uint8, device="cuda")
    sfb = torch.empty(binding.nvfp4_gemm_repacked_scales_bytes(N, K, 1), dtype=torch.uint8, device="cuda")
    buf, C = alloc_c(M, N, 1)

    def step():
        binding.nvfp4_quantize(xa_d, binding.DTYPE_BF16, codes_a, sfa, M, K, 1, stream)
        binding.nvfp4_gemm_repack_scales(sfb_raw, sfb, N, K, 1, stream)
        binding.nvfp4_gemm_run(codes_a, B, sfa, sfb, C, M, N, K, 1, stream)

    with torch.cuda.stream(stream):
        step()
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step()
    ca, sa = oracle.quantize(xa, M, K)
    for _ in range(2):
        for t in (codes_a, sfa, sfb):
            t.zero_()
        C.fill_(float("nan"))
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        binding.nvfp4_gemm_check_device_status()
        assert_close_full(C, dict(A=ca, B=pb["B"], SFA=sa, SFB=pb["SFB"], M=M, N=N, K=K, L=1))
        check_canary(buf, M, N, 1)
