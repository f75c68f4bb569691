"""The C-ABI library on a host without a GPU: it loads, exports every function
the header declares, its descriptor encoders reproduce the pages' constants,
the launch planner behaves, and argument errors are reported before any CUDA
call."""
import ctypes
import json
import os

import pytest

import __graft_entry__
from block_scaled_fp4_nvfp4_gb300 import binding

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module")
def lib():
    __graft_entry__.build()
    return binding.load_library()


def test_exports_every_header_function(lib):
    names = binding.header_functions()
    assert len(names) == 15
    for n in names:
        assert hasattr(lib, n), n
        ctypes.cast(getattr(lib, n), ctypes.c_void_p)


def test_instruction_descriptor_matches_page_constant(lib):
    spec = json.load(open(os.path.join(GOLDEN, "instr_desc.json")))
    for c in spec["cases"]:
        assert binding.nvfp4_gemm_encode_idesc(c["M"], c["N"]) == c["idesc"]
    # N field is N >> 3 at bit 17, M field M >> 7 at bit 27
    assert binding.nvfp4_gemm_encode_idesc(128, 128) == c["idesc"] + ((16 - 8) << 17)
    assert binding.nvfp4_gemm_encode_idesc(128, 256) >> 17 & 0x3F == 32


def test_smem_descriptors_match_page_construction(lib):
    spec = json.load(open(os.path.join(GOLDEN, "smem_desc.json")))
    for c in spec["cases"]:
        got = binding.nvfp4_gemm_encode_smem_desc(c["addr"], c["kind"] == "ab_sw128")
        assert got == int(c["desc_hex"], 16), (c, hex(got))


def test_repacked_bytes(lib):
    assert binding.nvfp4_gemm_repacked_scales_bytes(128, 256, 1) == 2048
    assert binding.nvfp4_gemm_repacked_scales_bytes(7168, 16384, 1) == 7168 * 1024
    assert binding.nvfp4_gemm_repacked_scales_bytes(200, 512, 3) == 3 * 2 * 8 * 512
    assert binding.nvfp4_gemm_repacked_scales_bytes(1, 320, 1) == 1 * 8 * 512  # K padded to 512
    assert binding.nvfp4_gemm_repacked_scales_bytes(0, 256, 1) == 0
    assert binding.nvfp4_gemm_repacked_scales_bytes(128, 24, 1) == 0


def test_plan_single_tile_and_full_machine(lib):
    p = binding.nvfp4_gemm_plan([128], [128], [256], [1], 152)
    assert p["bn"] == 128 and p["tiles"] == 1 and p["grid"] == 1
    assert p["stages"] >= 4 and p["sk_max_segs"] == 1
    p = binding.nvfp4_gemm_plan([8192], [8192], [8192], [1], 152)
    # 128 x 256 tiles: 2048 of them as 2-SM pairs, the last wave and a half stream-K
    assert p["bn"] == 256 and p["tiles"] == 2048 and p["grid"] == 152
    assert p["dp_tiles"] + p["sk_tiles"] == 2048


def test_plan_stream_k_for_skinny_problem(lib):
    p = binding.nvfp4_gemm_plan([128], [7168], [16384], [1], 152)
    assert p["tiles"] == 56 and p["dp_tiles"] == 0 and p["sk_tiles"] == 56
    assert p["grid"] == 112 and p["sk_iters"] == 56 * 64    # two equal segments per tile
    assert p["sk_max_segs"] == 2
    p = binding.nvfp4_gemm_plan([128], [512], [4096], [1], 152)
    assert p["grid"] == 16 and p["sk_max_segs"] == 4         # capped: >= 4 k-tiles per CTA


def test_plan_data_parallel_from_one_wave(lib, monkeypatch):
    Ms = [384, 64, 1024, 256, 192, 512, 128, 768]
    p = binding.nvfp4_gemm_plan(Ms, [4096] * 8, [7168] * 8, [1] * 8, 152)
    tiles = sum(-(-m // 128) for m in Ms) * 16
    assert p["bn"] == 256 and p["tiles"] == tiles == 432 and p["dp_tiles"] == 432 and p["sk_tiles"] == 0
    # by the intake rule with a stream-K tail: padded to 2-SM pairs (30
    # m-tiles instead of 27), two whole waves, the rest stream-K
    monkeypatch.setenv("NVFP4_PAD_PAIRS", "1")
    monkeypatch.setenv("NVFP4_PAIR_SK", "1")
    p = binding.nvfp4_gemm_plan(Ms, [4096] * 8, [7168] * 8, [1] * 8, 152)
    padded = sum((-(-m // 128) + 1) // 2 * 2 for m in Ms) * 16
    assert p["bn"] == 256 and p["pair"] == 1 and p["tiles"] == padded == 480
    assert p["dp_tiles"] == 2 * 2 * 76 and p["sk_tiles"] == 480 - 304
    _check_pair_sk(Ms, [4096] * 8, [7168] * 8, [1] * 8, 152)
    monkeypatch.delenv("NVFP4_PAD_PAIRS")
    monkeypatch.delenv("NVFP4_PAIR_SK")
    p = binding.nvfp4_gemm_plan([1024, 2048], [4096, 7168], [7168, 2048], [1, 1], 152)
    assert p["bn"] == 256 and p["tiles"] == 8 * 16 + 16 * 28 == p["dp_tiles"] + p["sk_tiles"]


SCHED_CASES = [
    ([128], [7168], [16384], [1]),
    ([128], [128], [256], [1]),
    ([64], [2048], [4096], [1]),
    ([300], [264], [1024], [2]),
    ([384, 64, 1024, 256, 192, 512, 128, 768], [4096] * 8, [7168] * 8, [1] * 8),
    ([1024, 2048], [4096, 7168], [7168, 2048], [1, 1]),
    ([128, 256, 64], [1024, 512, 256], [4096, 1024, 8192], [1, 2, 1]),
]


def _tiles_m(M, N, L, plan):
    """m-tiles per group as planned: 2-SM pair plans over groups with an odd
    number of m-tiles pad each such group by one m-tile."""
    tm = [-(-m // 128) for m in M]
    plain = sum(t * -(-n // plan["bn"]) * l for t, n, l in zip(tm, N, L))
    if plan["tiles"] != plain:
        tm = [(t + 1) // 2 * 2 for t in tm]
        assert plan["pair"] == 1 and plan["tiles"] == sum(t * -(-n // plan["bn"]) * l for t, n, l in zip(tm, N, L))
    return tm


def _check_schedule(M, N, K, L, sms):
    plan = binding.nvfp4_gemm_plan(M, N, K, L, sms)
    tms = _tiles_m(M, N, L, plan)
    cover = {}
    segs = {}
    sk_lengths = []
    for cta in range(plan["grid"]):
        items = binding.nvfp4_gemm_debug_schedule(M, N, K, L, sms, cta)
        sk = 0
        for w in items:
            g = w["g"]
            tiles_m, tiles_n, kt = tms[g], -(-N[g] // plan["bn"]), K[g] // 256
            assert 0 <= w["tm"] < tiles_m and 0 <= w["tn"] < tiles_n and 0 <= w["l"] < L[g]
            assert 0 <= w["kt0"] < w["kt1"] <= kt
            key = (g, w["l"], w["tm"], w["tn"])
            for k in range(w["kt0"], w["kt1"]):
                assert (key, k) not in cover, "k-tile covered twice"
                cover[(key, k)] = cta
            segs.setdefault(w["tile"], []).append((w["seg"], w["nseg"], w["kt0"], w["kt1"], key))
            if w["tile"] >= plan["dp_tiles"]:
                sk += w["kt1"] - w["kt0"]
        sk_lengths.append(sk)
    # every k-tile of every tile exactly once
    total = sum(tms[g] * -(-N[g] // plan["bn"]) * L[g] * (K[g] // 256) for g in range(len(M)))
    assert len(cover) == total
    # segments of a tile: indices 0..n-1, consistent count, in k order, same coordinates
    assert len(segs) == plan["tiles"]
    for t, lst in segs.items():
        lst.sort()
        n = lst[0][1]
        assert [x[0] for x in lst] == list(range(n)) and all(x[1] == n for x in lst)
        assert n <= plan["sk_max_segs"] and len({x[4] for x in lst}) == 1
        assert lst[0][2] == 0 and all(lst[i][3] == lst[i + 1][2] for i in range(n - 1))
        if t < plan["dp_tiles"]:
            assert n == 1
    # stream-K ranges are equal to within one k-tile
    if plan["sk_tiles"]:
        assert max(sk_lengths) - min(sk_lengths) <= 1


@pytest.mark.parametrize("case", range(len(SCHED_CASES)))
def test_schedule_covers_every_k_tile_once(lib, case):
    _check_schedule(*SCHED_CASES[case], 152)


@pytest.mark.parametrize("mode", ["dp", "sk"])
def test_schedule_forced_modes(lib, mode, monkeypatch):
    monkeypatch.setenv("NVFP4_SCHEDULE", mode)
    for case in (SCHED_CASES[0], SCHED_CASES[3], SCHED_CASES[5]):
        _check_schedule(*case, 152)
        p = binding.nvfp4_gemm_plan(*case, 152)
        assert (p["sk_tiles"] == 0) if mode == "dp" else (p["dp_tiles"] == 0)


def test_partial_k_tiles_planned(lib):
    """K % 256 != 0: the last k-tile of each tile is partial, and the
    decomposition still covers every k-tile exactly once."""
    p = binding.nvfp4_gemm_plan([256], [512], [320], [1], 152)
    assert p["tiles"] == 2 * 4 and p["dp_tiles"] == 0 and p["sk_tiles"] == 8
    _check_schedule_k([256], [512], [320], [1], 152)
    _check_schedule_k([128], [7168], [16384 + 64], [1], 152)
    _check_schedule_k([300, 64], [264, 512], [1088, 192], [2, 1], 152)


def _check_schedule_k(M, N, K, L, sms):
    plan = binding.nvfp4_gemm_plan(M, N, K, L, sms)
    seen = set()
    for cta in range(plan["grid"]):
        for w in binding.nvfp4_gemm_debug_schedule(M, N, K, L, sms, cta):
            kt = -(-K[w["g"]] // 256)
            assert 0 <= w["kt0"] < w["kt1"] <= kt
            for k in range(w["kt0"], w["kt1"]):
                key = (w["g"], w["l"], w["tm"], w["tn"], k)
                assert key not in seen
                seen.add(key)
    total = sum(-(-M[g] // 128) * -(-N[g] // plan["bn"]) * L[g] * -(-K[g] // 256) for g in range(len(M)))
    assert len(seen) == total


def test_schedule_other_machine_sizes(lib):
    for sms in (1, 7, 148, 160):
        _check_schedule([128], [7168], [16384], [1], sms)
        _check_schedule([1024, 2048], [4096, 7168], [7168, 2048], [1, 1], sms)


@pytest.mark.parametrize("M,N,K,L,code", [
    (128, 128, 200, 1, -2),   # K % 64
    (128, 128, 96, 1, -2),    # K % 64
    (128, 100, 256, 1, -2),   # N % 8
    (0, 128, 256, 1, -1),
    (128, 128, 256, 0, -1),
])
def test_shape_errors_without_gpu(lib, M, N, K, L, code):
    with pytest.raises(binding.Nvfp4Error) as e:
        binding.nvfp4_gemm_run(16, 16, 16, 16, 16, M, N, K, L, stream=0)
    assert e.value.code == code
    assert binding.nvfp4_gemm_last_error_string()


def test_pointer_errors_without_gpu(lib):
    with pytest.raises(binding.Nvfp4Error) as e:
        binding.nvfp4_gemm_run(0, 16, 16, 16, 16, 128, 128, 256, 1, stream=0)
    assert e.value.code == -1
    with pytest.raises(binding.Nvfp4Error) as e:
        binding.nvfp4_gemm_run(24, 16, 16, 16, 16, 128, 128, 256, 1, stream=0)   # misaligned
    assert e.value.code == -1
    with pytest.raises(binding.Nvfp4Error) as e:
        binding.nvfp4_gemm_run_grouped(9, [16] * 9, [16] * 9, [16] * 9, [16] * 9, [16] * 9,
                                       [128] * 9, [128] * 9, [256] * 9, [1] * 9, stream=0)
    assert e.value.code == -1
    with pytest.raises(binding.Nvfp4Error) as e:
        binding.nvfp4_gemm_repack_scales(16, 8, 128, 256, 1, stream=0)
    assert e.value.code == -1


def test_last_launch_before_any_launch(lib):
    info = binding.nvfp4_gemm_last_launch()
    assert info["variant"] is None or info["variant"] in ("single", "multicast", "pair", "cluster_reduce")
    with pytest.raises(binding.Nvfp4Error):
        _check_rc = lib.nvfp4_gemm_last_launch(None, 5)
        binding._check(_check_rc, "nvfp4_gemm_last_launch")


def test_quantize_argument_errors_without_gpu(lib):
    for args in ((0, 0, 16, 16, 128, 256, 1),      # null x
                 (16, 0, 16, 24, 128, 256, 1),     # misaligned scales
                 (16, 2, 16, 16, 128, 256, 1),     # unknown dtype
                 (16, 0, 16, 16, 128, 200, 1),     # K % 16
                 (16, 1, 16, 16, 0, 256, 1)):      # rows
        with pytest.raises(binding.Nvfp4Error) as e:
            binding.nvfp4_quantize(*args, stream=0)
        assert e.value.code == -1


def test_timeout_setting_validated(lib):
    with pytest.raises(binding.Nvfp4Error):
        binding.nvfp4_gemm_set_wait_timeout_ns(10)
    binding.nvfp4_gemm_set_wait_timeout_ns(2_000_000_000)


def test_cluster_pairs_share_b_columns(lib, monkeypatch):
    """Clusters of two CTAs: rank 0 and rank 1 run tiles with the same group,
    batch and n-tile, adjacent m-tiles and identical k-ranges, in lockstep."""
    for case in ([8192], [8192], [8192], [1]), ([1024, 2048], [4096, 7168], [7168, 2048], [1, 1]):
        p = binding.nvfp4_gemm_plan(*case, 152)
        assert p["cluster"] == 2 and p["grid"] % 2 == 0
        _check_schedule(*case, 152)
        for c in range(0, min(p["grid"], 12), 2):
            w0 = binding.nvfp4_gemm_debug_schedule(*case, 152, c)
            w1 = binding.nvfp4_gemm_debug_schedule(*case, 152, c + 1)
            assert len(w0) == len(w1) > 0
            for a, b in zip(w0, w1):
                assert (a["g"], a["l"], a["tn"], a["kt0"], a["kt1"]) == (b["g"], b["l"], b["tn"], b["kt0"], b["kt1"])
                assert b["tm"] == a["tm"] + 1 and a["tm"] % 2 == 0
    # odd m-tile counts, stream-K plans and the override fall back to single CTAs
    assert binding.nvfp4_gemm_plan([384, 64], [4096, 4096], [7168, 7168], [1, 1], 152)["cluster"] == 1
    p = binding.nvfp4_gemm_plan([128], [7168], [16384], [1], 152)   # stream-K: clusters only for the reduction
    assert p["pair"] == 0 and (p["cluster"] == 1 or p["cluster_reduce"] == 1)
    monkeypatch.setenv("NVFP4_CLUSTER", "1")
    assert binding.nvfp4_gemm_plan([8192], [8192], [8192], [1], 152)["cluster"] == 1
    monkeypatch.setenv("NVFP4_CLUSTER", "2")
    p = binding.nvfp4_gemm_plan([256], [512], [1024], [1], 152)
    assert p["cluster"] == 1 or p["dp_tiles"] == p["tiles"]


def test_pair_tiles_planned_for_wide_clusters(lib, monkeypatch):
    """Clustered 256-wide plans run as 2-SM pair tiles (half of B per CTA, so
    one more stage fits); NVFP4_PAIR=0 keeps B multicast; 128-wide clusters
    and single CTAs never pair."""
    p = binding.nvfp4_gemm_plan([8192], [8192], [8192], [1], 152)
    assert p["cluster"] == 2 and p["pair"] == 1 and p["stages"] == 5
    monkeypatch.setenv("NVFP4_PAIR", "0")
    p = binding.nvfp4_gemm_plan([8192], [8192], [8192], [1], 152)
    assert p["cluster"] == 2 and p["pair"] == 0 and p["stages"] == 4
    monkeypatch.delenv("NVFP4_PAIR")
    monkeypatch.setenv("NVFP4_BN", "128")
    p = binding.nvfp4_gemm_plan([8192], [8192], [8192], [1], 152)
    assert p["cluster"] == 2 and p["pair"] == 0
    monkeypatch.delenv("NVFP4_BN")
    assert binding.nvfp4_gemm_plan([128], [7168], [16384], [1], 152)["pair"] == 0
    # the two-group workload (12.4 k-tiles per tile on average) runs as pairs too
    p = binding.nvfp4_gemm_plan([1024, 2048], [4096, 7168], [7168, 2048], [1, 1], 152)
    assert p["cluster"] == 2 and p["pair"] == 1
    assert binding.nvfp4_gemm_plan([2048], [8192], [4096], [1], 152)["pair"] == 1
    # tiles shorter than one ring (K = 512: 2 k-tiles) keep B multicast
    p = binding.nvfp4_gemm_plan([4096], [8192], [512], [1], 152)
    assert p["cluster"] == 2 and p["pair"] == 0


def test_cluster_reduction_planned_for_one_segment_per_cta(lib, monkeypatch):
    """Stream-K plans whose CTAs each run one of S = 2 or 4 equal segments
    launch each tile's segments as one cluster (rank = segment) and need no
    workspace; other plans keep the workspace path."""
    p = binding.nvfp4_gemm_plan([128], [7168], [16384], [1], 152)
    assert p["cluster_reduce"] == 1 and p["cluster"] == 2 and p["grid"] == 112
    p4 = binding.nvfp4_gemm_plan([128], [512], [4096], [1], 152)
    assert p4["cluster_reduce"] == 1 and p4["cluster"] == 4 and p4["grid"] == 16
    for M, N, K, L in (([128], [7168], [16384], [1]), ([128], [512], [4096], [1]), ([300], [264], [1024], [2])):
        p = binding.nvfp4_gemm_plan(M, N, K, L, 152)
        if not p["cluster_reduce"]:
            continue
        S = p["cluster"]
        for cta in range(p["grid"]):
            (w,) = binding.nvfp4_gemm_debug_schedule(M, N, K, L, 152, cta)
            assert w["nseg"] == S and w["seg"] == cta % S and w["tile"] == cta // S
        _check_schedule(M, N, K, L, 152)
    assert binding.nvfp4_gemm_plan([8192], [8192], [8192], [1], 152)["cluster_reduce"] == 0
    monkeypatch.setenv("NVFP4_SKRED", "0")
    p = binding.nvfp4_gemm_plan([128], [7168], [16384], [1], 152)
    assert p["cluster_reduce"] == 0 and p["cluster"] == 1 and p["grid"] == 112
    monkeypatch.setenv("NVFP4_SKRED", "1")
    monkeypatch.setenv("NVFP4_SCHEDULE", "sk")   # uneven ranges: workspace path
    assert binding.nvfp4_gemm_plan([128], [7168], [16384], [1], 152)["cluster_reduce"] == 0


# ------------------------------------------------------------------ stream-K tails of CTA-pair plans
def _check_pair_sk(M, N, K, L, sms):
    """A cluster plan with a stream-K tail: every k-tile once (checked by
    _check_schedule), at most two segments per tile, both CTAs of a cluster
    on the same k-range of tiles 2q and 2q+1, and the order the reduction
    relies on: segment 1 of a split tile is the first stream-K item of its
    cluster, segment 0 the last item of its cluster."""
    _check_schedule(M, N, K, L, sms)
    plan = binding.nvfp4_gemm_plan(M, N, K, L, sms)
    assert plan["cluster"] == 2 and plan["sk_max_segs"] <= 2
    items = [binding.nvfp4_gemm_debug_schedule(M, N, K, L, sms, c) for c in range(plan["grid"])]
    for c in range(0, plan["grid"], 2):
        a, b = items[c], items[c + 1]
        assert len(a) == len(b)
        for x, y in zip(a, b):
            assert (x["g"], x["l"], x["tn"], x["kt0"], x["kt1"], x["seg"], x["nseg"]) == \
                   (y["g"], y["l"], y["tn"], y["kt0"], y["kt1"], y["seg"], y["nseg"])
            assert y["tm"] == x["tm"] + 1 and x["tm"] % 2 == 0
    for cta, lst in enumerate(items):
        sk = [w for w in lst if w["tile"] >= plan["dp_tiles"]]
        for i, w in enumerate(sk):
            assert w["nseg"] in (1, 2)
            if w["nseg"] == 2:
                assert (w["seg"] == 1 and i == 0) or (w["seg"] == 0 and i == len(sk) - 1 and w is lst[-1]), (cta, w)
    return plan


def test_dense_pair_plan_gets_a_stream_k_tail(lib, monkeypatch):
    """8192^3 as 2-SM pairs on 152 SMs: 1024 pair tiles over 76 clusters leave a
    partial 14th wave; by the rule (NVFP4_PAIR_SK=1) one wave plus the
    remainder (112 pair tiles) run as stream-K, 47.2 k-tiles per cluster
    instead of whole 32-k-tile tiles."""
    monkeypatch.setenv("NVFP4_PAIR_SK", "1")
    plan = _check_pair_sk([8192], [8192], [8192], [1], 152)
    assert plan["pair"] == 1 and plan["sk_tiles"] == 2 * 112 and plan["dp_tiles"] == 2 * 912


def test_grouped_pair_plan_never_worse_than_whole_tiles(lib, monkeypatch):
    """Two groups whose tiles have 28 and 8 k-tiles: whole tiles dealt
    round-robin leave the busiest cluster 52 k-tiles (47.2 on average); a
    stream-K tail is taken only where its estimate (busiest cluster plus the
    reduction) is lower, so the busiest cluster never gets more."""
    monkeypatch.setenv("NVFP4_PAIR_SK", "1")
    M, N, K, L = [1024, 2048], [4096, 7168], [7168, 2048], [1, 1]
    plan = _check_pair_sk(M, N, K, L, 152)
    per = []
    for c in range(0, plan["grid"], 2):
        per.append(sum(w["kt1"] - w["kt0"] for w in binding.nvfp4_gemm_debug_schedule(M, N, K, L, 152, c)))
    assert max(per) <= 52 and sum(per) == 3584


@pytest.mark.parametrize("shape", [([512], [1024], [4096], [1]), ([256, 768], [512, 264], [2048, 1024], [1, 2]),
                                   ([1024], [2048], [1536], [2])])
@pytest.mark.parametrize("sms", [16, 36, 152])
def test_forced_pair_stream_k_tails(lib, shape, sms, monkeypatch):
    for k, v in {"NVFP4_BN": "256", "NVFP4_SCHEDULE": "dp", "NVFP4_CLUSTER": "2", "NVFP4_PAIR_SK": "2"}.items():
        monkeypatch.setenv(k, v)
    for pair in ("1", "0"):
        monkeypatch.setenv("NVFP4_PAIR", pair)
        plan = binding.nvfp4_gemm_plan(*shape, sms)
        if plan["cluster"] != 2:
            continue
        _check_pair_sk(*shape, sms)


def test_pair_stream_k_is_off_by_default(lib, monkeypatch):
    monkeypatch.delenv("NVFP4_PAIR_SK", raising=False)
    plan = binding.nvfp4_gemm_plan([8192], [8192], [8192], [1], 152)
    assert plan["pair"] == 1 and plan["sk_tiles"] == 0
    monkeypatch.setenv("NVFP4_PAIR_SK", "1")
    assert binding.nvfp4_gemm_plan([8192], [8192], [8192], [1], 152)["sk_tiles"] > 0
