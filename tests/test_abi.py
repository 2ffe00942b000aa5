"""The C-ABI library loads, exports every function include/mxg.h declares,
and rejects bad arguments synchronously -- all without a GPU.  Every call
below fails validation before any device work, so it is safe anywhere."""
import ctypes

import pytest
import torch

from moe_grouped_block_gb300 import build as mxg_build
from moe_grouped_block_gb300 import mxg


@pytest.fixture(scope="module")
def lib():
    mxg_build.build()
    return mxg.load()


def test_exports_every_declared_function(lib):
    names = mxg.declared_functions()
    assert len(names) >= 9
    for n in names:
        assert hasattr(lib, n), "libmxg.so does not export " + n


def test_scalar_queries(lib):
    assert mxg.mxg_offsets_workspace_bytes(8) == (2 * 8 + 1) * 8
    assert mxg.mxg_offsets_workspace_bytes(0) == 0
    assert mxg.mxg_grouped_gemm_workspace_bytes(1, 0, 8, 16384, 14336) == 0
    assert mxg.mxg_version() >= 100
    for code, name in mxg.STATUS_NAMES.items():
        assert mxg.mxg_status_string(code) == name
    assert mxg.mxg_status_string(99) == "MXG_ERR_UNKNOWN"


FAKE = 1 << 20  # a 16-byte-aligned non-null value; never dereferenced (validation fails first)

# The calls below pass fake device pointers that every one of them must
# reject before any device work.  They are run only where there is no CUDA
# device, so a validation gap can never turn into a launch.
no_device_only = pytest.mark.skipif(torch.cuda.is_available(),
                                    reason="fake-pointer validation tests run without a GPU")


@no_device_only
def test_offsets_argument_errors(lib):
    L = lib
    assert L.mxg_group_offsets(None, 0, 4, 1, 128, 512, FAKE, None, None) == 1
    assert L.mxg_group_offsets(FAKE, 0, 0, 1, 128, 512, FAKE, None, None) == 1
    assert L.mxg_group_offsets(FAKE, 0, 4, 0, 128, 512, FAKE, None, None) == 1
    assert L.mxg_group_offsets(FAKE, 0, 4, 1, 0, 512, FAKE, None, None) == 1
    assert L.mxg_group_offsets(FAKE, 0, 4, 1, 128, -1, None, None, None) == 1


@no_device_only
def test_offsets_bounds_keep_products_in_int64(lib):
    """Multiplier above 2^31, capacity above 2^62, capacity * last_dim past
    int64: refused, for both offsets entry points."""
    for f in (lib.mxg_group_offsets, lib.mxg_group_offsets_unaligned):
        assert f(FAKE, 1, 4, (1 << 31) + 1, 128, 512, FAKE, None, None) == 1
        assert f(FAKE, 1, 4, 1, 128, (1 << 62) + 128, FAKE, None, None) == 1
        assert f(FAKE, 1, 4, 1, 1 << 40, 1 << 24, FAKE, None, None) == 1


@no_device_only
def test_unaligned_quantize_rejects_padded_rows_past_int32(lib):
    q = lib.mxg_group_quantize_unaligned
    # 0x7FFFFF00 + 128 * 1024 padded rows do not fit the kernels' 32-bit row tables
    assert q(3, FAKE, 0x7FFFFF00, 128, FAKE, 1024, FAKE, FAKE, FAKE, FAKE, None, None) == 1


@no_device_only
def test_debug_entry_validates_its_overrides(lib):
    op = mxg.Operand(FAKE, FAKE, None)
    r = ctypes.byref
    d = lib.mxg_grouped_gemm_debug
    args = (1, 0, r(op), r(op), FAKE, 4, 512, 256, 256, None, None, None, FAKE, 0, None)
    assert d(*args, 64, 0, 0, 0, None) == 1     # tile width 64 does not exist
    assert d(*args, 0, 256, 0, 0, None) == 1    # only 128-byte stages can be forced
    assert d(*args, 0, 0, 2, 0, None) == 1      # unknown inject bit
    assert d(*args, 0, 0, 0, -1, None) == 1     # negative wait bound


@no_device_only
def test_quantize_argument_errors(lib):
    L = lib
    q = L.mxg_group_quantize
    # bad format / layout
    assert q(7, 1, FAKE, 128, 128, None, 1, FAKE, FAKE, None, None, None, None, None, None) == 1
    assert q(1, 4, FAKE, 128, 128, None, 1, FAKE, FAKE, None, None, None, None, None, None) == 1
    # missing outputs
    assert q(1, 3, FAKE, 128, 128, None, 1, FAKE, FAKE, None, None, None, None, None, None) == 1
    # NVFP4 colwise needs its [G, cols] outer-scale output
    assert q(2, 2, FAKE, 128, 128, None, 1, None, None, FAKE, FAKE, None, None, None, None) == 1
    # sizes not multiples of 128, misaligned pointer
    assert q(1, 1, FAKE, 100, 128, None, 1, FAKE, FAKE, None, None, None, None, None, None) == 2
    assert q(1, 1, FAKE, 128, 96, None, 1, FAKE, FAKE, None, None, None, None, None, None) == 2
    assert q(1, 1, FAKE + 8, 128, 128, None, 1, FAKE, FAKE, None, None, None, None, None, None) == 2


@no_device_only
def test_gemm_argument_errors(lib):
    L = lib
    op = mxg.Operand(FAKE, FAKE, None)
    opo = mxg.Operand(FAKE, FAKE, FAKE)
    r = ctypes.byref
    g = L.mxg_grouped_gemm
    assert g(1, 0, None, r(op), FAKE, 4, 512, 256, 256, None, None, None, FAKE, 0, None, 0, None, None) == 1
    assert g(1, 0, r(op), r(op), None, 4, 512, 256, 256, None, None, None, FAKE, 0, None, 0, None, None) == 1
    assert g(1, 0, r(op), r(op), FAKE, 0, 512, 256, 256, None, None, None, FAKE, 0, None, 0, None, None) == 1
    assert g(1, 0, r(op), r(op), FAKE, 1025, 512, 256, 256, None, None, None, FAKE, 0, None, 0, None, None) == 1
    assert g(1, 5, r(op), r(op), FAKE, 4, 512, 256, 256, None, None, None, FAKE, 0, None, 0, None, None) == 1
    # NVFP4: dgrad, beta and missing outer scales are rejected
    assert g(2, 2, r(opo), r(opo), FAKE, 4, 512, 256, 256, None, None, None, FAKE, 0, None, 0, None, None) == 1
    assert g(2, 0, r(opo), r(opo), FAKE, 4, 512, 256, 256, None, FAKE, None, FAKE, 0, None, 0, None, None) == 1
    assert g(2, 0, r(op), r(opo), FAKE, 4, 512, 256, 256, None, None, None, FAKE, 0, None, 0, None, None) == 1
    # bias has no meaning for wgrad
    assert g(1, 1, r(op), r(op), FAKE, 4, 512, 256, 256, None, None, FAKE, FAKE, 0, None, 0, None, None) == 1
    # alignment
    assert g(1, 0, r(op), r(op), FAKE, 4, 500, 256, 256, None, None, None, FAKE, 0, None, 0, None, None) == 2
    assert g(1, 0, r(op), r(op), FAKE, 4, 512, 200, 256, None, None, None, FAKE, 0, None, 0, None, None) == 2
    assert g(2, 0, r(opo), r(opo), FAKE, 4, 512, 256, 200, None, None, None, FAKE, 0, None, 0, None, None) == 2
    assert g(1, 0, r(op), r(op), FAKE, 4, 512, 256, 256, None, None, None, FAKE + 4, 0, None, 0, None, None) == 2


@no_device_only
def test_gemm_operand_descriptor_errors(lib):
    """rows / cols other than the mode's, a leading dimension below cols or
    not a multiple of 16 bytes: refused before any launch."""
    r = ctypes.byref
    g = lib.mxg_grouped_gemm
    ok = mxg.Operand(FAKE, FAKE, None, 0, 0, 0)

    def call(a, b, fmt=1, mode=0):
        return g(fmt, mode, r(a), r(b), FAKE, 4, 512, 256, 256, None, None, None, FAKE, 0, None, 0,
                 None, None)

    # fprop: A is M_cap x K = 512 x 256, B is G*N x K = 1024 x 256
    assert call(mxg.Operand(FAKE, FAKE, None, 256, 0, 0), ok) == 1      # A rows
    assert call(ok, mxg.Operand(FAKE, FAKE, None, 0, 512, 0)) == 1      # B cols
    assert call(mxg.Operand(FAKE, FAKE, None, 0, 0, 128), ok) == 1      # ld < cols
    assert call(mxg.Operand(FAKE, FAKE, None, 0, 0, 264), ok) == 2      # 264 bytes
    # wgrad: A is N x M_cap = 256 x 512
    assert call(mxg.Operand(FAKE, FAKE, None, 256, 256, 0), ok, mode=1) == 1
    # NVFP4 (outer scales present): ld counts elements, two per byte
    opo = mxg.Operand(FAKE, FAKE, FAKE, 0, 0, 0)
    assert call(mxg.Operand(FAKE, FAKE, FAKE, 0, 0, 257), opo, fmt=2) == 2   # odd
    assert call(mxg.Operand(FAKE, FAKE, FAKE, 0, 0, 272), opo, fmt=2) == 2   # 136 bytes


@no_device_only
def test_dequantize_argument_errors(lib):
    L = lib
    assert L.mxg_dequantize(1, 1, None, FAKE, None, 128, 128, FAKE, 0, None) == 1
    assert L.mxg_dequantize(2, 2, FAKE, FAKE, FAKE, 128, 128, FAKE, 0, None) == 6
    assert L.mxg_dequantize(1, 1, FAKE, FAKE, None, 120, 128, FAKE, 0, None) == 2


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU path")
def test_no_device_is_reported_not_launched(lib):
    # valid arguments but no usable device: refused before any launch
    assert lib.mxg_group_offsets(FAKE, 0, 4, 1, 128, 512, FAKE, None, None) == 3


def test_binding_refuses_host_tensors(lib):
    with pytest.raises(ValueError):
        mxg.mxg_group_offsets(torch.zeros(4, dtype=torch.int32), 1, 128, 512,
                              torch.zeros(9, dtype=torch.int64))


def test_c_program_compiles_against_the_header(lib, tmp_path):
    """The plain-C example (run on the GPU by test_gpu_e_c_abi) compiles and
    links against include/mxg.h and libmxg.so with -Wall -Werror."""
    import os
    import shutil
    import subprocess
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    if shutil.which("gcc") is None or not os.path.exists(os.path.join(cuda, "include")):
        pytest.skip("needs gcc and the CUDA headers")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run(["gcc", "-O1", "-std=c11", "-Wall", "-Werror",
                        os.path.join(root, "tests", "c_abi", "c_abi_example.c"),
                        "-I" + os.path.join(root, "include"), "-I" + os.path.join(cuda, "include"),
                        "-L" + os.path.dirname(mxg.LIB_PATH), "-lmxg",
                        "-L" + os.path.join(cuda, "lib64"), "-lcudart",
                        "-o", str(tmp_path / "c_abi_example")], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
