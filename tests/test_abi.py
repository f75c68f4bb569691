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
    assert len(names) == 12
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
    assert p["bn"] == 128 and p["units"] == 1 and p["grid"] == 1 and p["splits"] == [1]
    assert p["stages"] >= 4
    p = binding.nvfp4_gemm_plan([8192], [8192], [8192], [1], 152)
    assert p["splits"] == [1] and p["units"] == 4096 and p["grid"] == 152


def test_plan_splits_skinny_problem(lib):
    p = binding.nvfp4_gemm_plan([128], [7168], [16384], [1], 152)
    s = p["splits"][0]
    assert s == 2 and p["units"] == 112 and p["grid"] == 112    # one wave of units
    p = binding.nvfp4_gemm_plan([128], [512], [4096], [1], 152)
    assert p["splits"] == [4]                                    # capped: >= 4 k-tiles per unit
    p = binding.nvfp4_gemm_plan([128], [128], [256], [1], 152)
    assert p["splits"] == [1]


def test_plan_grouped(lib):
    p = binding.nvfp4_gemm_plan([1024, 2048], [4096, 7168], [7168, 2048], [1, 1], 152)
    assert p["splits"] == [1, 1] and p["units"] == 8 * 32 + 16 * 56
    Ms = [384, 64, 1024, 256, 192, 512, 128, 768]
    p = binding.nvfp4_gemm_plan(Ms, [4096] * 8, [7168] * 8, [1] * 8, 152)
    assert p["units"] == sum(-(-m // 128) for m in Ms) * 32


@pytest.mark.parametrize("M,N,K,L,code", [
    (128, 128, 200, 1, -2),   # K % 256
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


def test_timeout_setting_validated(lib):
    with pytest.raises(binding.Nvfp4Error):
        binding.nvfp4_gemm_set_wait_timeout_ns(10)
    binding.nvfp4_gemm_set_wait_timeout_ns(2_000_000_000)
