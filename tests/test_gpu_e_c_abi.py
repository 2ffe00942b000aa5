"""The C ABI used from plain C: compile tests/c_abi/c_abi_example.c with gcc
against include/mxg.h and libmxg.so, run it on the GPU."""
import os
import subprocess

import pytest

from gpu_util import require_gpu

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_c_program_through_the_abi(tmp_path):
    require_gpu()
    from moe_grouped_block_gb300 import mxg
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    exe = str(tmp_path / "c_abi_example")
    libdir = os.path.dirname(mxg.LIB_PATH)
    r = subprocess.run(["gcc", "-O1", "-std=c11", "-Wall", "-Werror", os.path.join(ROOT, "tests", "c_abi", "c_abi_example.c"),
                    "-I" + os.path.join(ROOT, "include"), "-I" + os.path.join(cuda, "include"),
                    "-L" + libdir, "-lmxg", "-L" + os.path.join(cuda, "lib64"), "-lcudart",
                    "-Wl,-rpath," + libdir + ":" + os.path.join(cuda, "lib64"), "-o", exe],
                   capture_output=True, text=True)
    assert r.returncode == 0, "gcc failed:\n" + r.stdout + r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "c_abi_example ok" in r.stdout
