"""The C ABI used from a plain C program (no Python in the call path): a
grouped GEMM with a closed-form result and the documented argument errors."""
import os
import shutil
import subprocess

import pytest

from gpu_util import require_gpu

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_c_client(tmp_path):
    require_gpu()
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    cc = shutil.which("gcc") or shutil.which("cc")
    assert cc, "no C compiler"
    lib_dir = os.path.join(ROOT, "block_scaled_fp4_nvfp4_gb300")
    exe = str(tmp_path / "c_abi_client")
    subprocess.run([cc, "-std=c99", "-O1", "-I" + os.path.join(ROOT, "include"), "-I" + os.path.join(cuda, "include"),
                    os.path.join(ROOT, "tests", "c_abi_client.c"), "-o", exe, "-L" + lib_dir, "-lnvfp4gemm",
                    "-Wl,-rpath," + lib_dir, "-L" + os.path.join(cuda, "lib64"), "-lcudart",
                    "-Wl,-rpath," + os.path.join(cuda, "lib64")], check=True)
    out = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, out.stderr
    assert "c abi ok" in out.stdout
