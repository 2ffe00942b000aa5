"""Python binding of libmxg.so (include/mxg.h): argument marshalling only.

Every function here has the name of the C entry point it calls and passes
device pointers and sizes straight through; all arithmetic runs in the
library's sm_103a kernels.  torch tensors are used as device buffers and the
current torch stream is the default stream.  There is no fallback: if the
library is missing or the call fails, an exception is raised.

The ``alloc_*`` helpers only size and allocate output buffers (torch.empty)
for the shapes include/mxg.h documents.
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmxg.so")
HEADER_PATH = os.path.join(os.path.dirname(_PKG), "include", "mxg.h")

# enums of include/mxg.h
MXG_OK = 0
MXG_MXFP8_E4M3, MXG_NVFP4_ROWSCALED = 1, 2
MXG_ROWWISE, MXG_COLWISE, MXG_BOTH = 1, 2, 3
MXG_FPROP_TN, MXG_WGRAD_NT, MXG_DGRAD_NN = 0, 1, 2
MXG_OUT_F32, MXG_OUT_BF16 = 0, 1
MXG_DEV_NEG_SIZE, MXG_DEV_MISALIGNED, MXG_DEV_SUM_OVER_CAPACITY = 1, 2, 4
MXG_DEV_BOUNDS, MXG_DEV_TIMEOUT = 8, 16
STATUS_NAMES = {0: "MXG_OK", 1: "MXG_ERR_INVALID_ARG", 2: "MXG_ERR_ALIGNMENT",
                3: "MXG_ERR_UNSUPPORTED_ARCH", 4: "MXG_ERR_LAUNCH",
                5: "MXG_ERR_WORKSPACE_TOO_SMALL", 6: "MXG_ERR_UNSUPPORTED"}


class MxgError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__("%s failed: %s (%d)" % (fn, STATUS_NAMES.get(code, "?"), code))
        self.code = code


class Operand(ctypes.Structure):
    """mxg_operand_t"""
    _fields_ = [("data", ctypes.c_void_p), ("scale", ctypes.c_void_p), ("outer", ctypes.c_void_p),
                ("rows", ctypes.c_int64), ("cols", ctypes.c_int64), ("ld", ctypes.c_int64)]


def _operand(T, elems_per_byte: int) -> Operand:
    """(data, scale[, outer]) -> mxg_operand_t.  A 2-D data tensor passes its
    leading dimension (row stride in elements), so a view of rows inside a
    wider buffer is described as such; rows and cols are left to the library
    (0: as the GEMM mode implies)."""
    data = T[0]
    ld = 0
    if isinstance(data, torch.Tensor) and data.dim() == 2:
        ld = data.stride(0) * elems_per_byte
    return Operand(_p(data), _p(T[1]), _p(T[2]) if len(T) > 2 else None, 0, 0, ld)


_lib = None


def load() -> ctypes.CDLL:
    """Load libmxg.so (built by moe_grouped_block_gb300.build)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libmxg.so is not built: run `python -m moe_grouped_block_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        vp, i64, i32, c_int, sz = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_int,
                                   ctypes.c_size_t)
        L.mxg_offsets_workspace_bytes.restype = sz
        L.mxg_offsets_workspace_bytes.argtypes = [c_int]
        L.mxg_group_offsets.restype = c_int
        L.mxg_group_offsets.argtypes = [vp, c_int, c_int, i64, i64, i64, vp, vp, vp]
        L.mxg_group_quantize.restype = c_int
        L.mxg_group_quantize.argtypes = [c_int, c_int, vp, i64, i64, vp, c_int, vp, vp, vp, vp, vp,
                                         vp, vp, vp]
        L.mxg_grouped_gemm.restype = c_int
        L.mxg_grouped_gemm.argtypes = [c_int, c_int, ctypes.POINTER(Operand), ctypes.POINTER(Operand),
                                       vp, c_int, i64, i64, i64, vp, vp, vp, vp, c_int, vp, sz, vp,
                                       vp]
        L.mxg_grouped_gemm_debug.restype = c_int
        L.mxg_grouped_gemm_debug.argtypes = [c_int, c_int, ctypes.POINTER(Operand),
                                             ctypes.POINTER(Operand), vp, c_int, i64, i64, i64, vp,
                                             vp, vp, vp, c_int, vp, c_int, c_int, c_int, i64, vp]
        L.mxg_grouped_gemm_workspace_bytes.restype = sz
        L.mxg_grouped_gemm_workspace_bytes.argtypes = [c_int, c_int, c_int, i64, i64]
        L.mxg_dequantize.restype = c_int
        L.mxg_dequantize.argtypes = [c_int, c_int, vp, vp, vp, i64, i64, vp, c_int, vp]
        L.mxg_status_string.restype = ctypes.c_char_p
        L.mxg_status_string.argtypes = [c_int]
        L.mxg_version.restype = c_int
        L.mxg_version.argtypes = []
        L.mxg_launch_count.restype = ctypes.c_uint64
        L.mxg_launch_count.argtypes = []
        L.mxg_unaligned_rows_capacity.restype = i64
        L.mxg_unaligned_rows_capacity.argtypes = [i64, c_int]
        L.mxg_group_offsets_unaligned.restype = c_int
        L.mxg_group_offsets_unaligned.argtypes = [vp, c_int, c_int, i64, i64, i64, vp, vp, vp]
        L.mxg_group_quantize_unaligned.restype = c_int
        L.mxg_group_quantize_unaligned.argtypes = [c_int, vp, i64, i64, vp, c_int, vp, vp, vp, vp,
                                                   vp, vp]
        L.mxg_grouped_gemm_unaligned.restype = c_int
        L.mxg_grouped_gemm_unaligned.argtypes = [c_int, ctypes.POINTER(Operand),
                                                 ctypes.POINTER(Operand), vp, c_int, i64, i64, i64,
                                                 vp, vp, vp, vp, c_int, vp, vp]
        _lib = L
    return _lib


def declared_functions() -> list:
    """Names of the functions include/mxg.h declares."""
    text = open(HEADER_PATH).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mxg_[a-z0-9_]+)\s*\(", text)))


def _p(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise ValueError("libmxg takes device tensors; got a %s tensor" % t.device)
    return t.data_ptr()


def _s(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check(fn: str, code: int) -> None:
    if code != MXG_OK:
        raise MxgError(fn, code)


# ----------------------------------------------------------------- entry points
def mxg_offsets_workspace_bytes(G: int) -> int:
    return load().mxg_offsets_workspace_bytes(G)


def mxg_group_offsets(sizes: torch.Tensor, multiplier: int, last_dim: int, rows_capacity: int,
                      ws: torch.Tensor, dev_status: torch.Tensor | None = None, stream=None) -> None:
    assert sizes.dtype in (torch.int32, torch.int64) and ws.dtype == torch.int64
    _check("mxg_group_offsets",
           load().mxg_group_offsets(_p(sizes), 1 if sizes.dtype == torch.int64 else 0, sizes.numel(),
                                    multiplier, last_dim, rows_capacity, _p(ws), _p(dev_status),
                                    _s(stream)))


def mxg_group_quantize(fmt: int, layout: int, x: torch.Tensor, rows_capacity: int, cols: int,
                       group_ws: torch.Tensor | None, G: int, q_row=None, sf_row=None, q_col=None,
                       sf_col=None, outer_row=None, dev_status=None, stream=None,
                       outer_col=None) -> None:
    assert x.dtype == torch.bfloat16 and x.is_contiguous()
    _check("mxg_group_quantize",
           load().mxg_group_quantize(fmt, layout, _p(x), rows_capacity, cols, _p(group_ws), G,
                                     _p(q_row), _p(sf_row), _p(q_col), _p(sf_col), _p(outer_row),
                                     _p(outer_col), _p(dev_status), _s(stream)))


def mxg_grouped_gemm(fmt: int, mode: int, A: tuple, B: tuple, group_ws: torch.Tensor, G: int,
                     M_cap: int, N: int, K: int, alpha=None, beta=None, C=None,
                     out_type: int = MXG_OUT_F32, workspace=None, workspace_bytes: int = 0,
                     dev_status=None, stream=None, bias=None) -> None:
    """A, B: (data, scale, outer-or-None) device tensors."""
    epb = 2 if fmt == MXG_NVFP4_ROWSCALED else 1
    a, b = _operand(A, epb), _operand(B, epb)
    _check("mxg_grouped_gemm",
           load().mxg_grouped_gemm(fmt, mode, ctypes.byref(a), ctypes.byref(b), _p(group_ws), G,
                                   M_cap, N, K, _p(alpha), _p(beta), _p(bias), _p(C), out_type,
                                   _p(workspace),
                                   workspace_bytes, _p(dev_status), _s(stream)))


def mxg_grouped_gemm_debug(fmt: int, mode: int, A: tuple, B: tuple, group_ws, G: int, M_cap: int,
                           N: int, K: int, alpha=None, beta=None, C=None,
                           out_type: int = MXG_OUT_F32, dev_status=None, tile_n: int = 0,
                           stage_bytes: int = 0, inject_flags: int = 0, wait_timeout_ns: int = 0,
                           stream=None, bias=None) -> None:
    epb = 2 if fmt == MXG_NVFP4_ROWSCALED else 1
    a, b = _operand(A, epb), _operand(B, epb)
    _check("mxg_grouped_gemm_debug",
           load().mxg_grouped_gemm_debug(fmt, mode, ctypes.byref(a), ctypes.byref(b), _p(group_ws),
                                         G, M_cap, N, K, _p(alpha), _p(beta), _p(bias), _p(C),
                                         out_type, _p(dev_status), tile_n, stage_bytes,
                                         inject_flags, wait_timeout_ns, _s(stream)))


def mxg_grouped_gemm_workspace_bytes(fmt: int, mode: int, G: int, M_cap: int, N: int) -> int:
    return load().mxg_grouped_gemm_workspace_bytes(fmt, mode, G, M_cap, N)


def mxg_dequantize(fmt: int, layout: int, q, sf, outer, rows: int, cols: int, out,
                   out_type: int = MXG_OUT_F32, stream=None) -> None:
    _check("mxg_dequantize",
           load().mxg_dequantize(fmt, layout, _p(q), _p(sf), _p(outer), rows, cols, _p(out),
                                 out_type, _s(stream)))


def mxg_unaligned_rows_capacity(rows_capacity: int, G: int) -> int:
    return load().mxg_unaligned_rows_capacity(rows_capacity, G)


def mxg_group_offsets_unaligned(sizes: torch.Tensor, multiplier: int, last_dim: int,
                                rows_capacity: int, ws: torch.Tensor,
                                dev_status: torch.Tensor | None = None, stream=None) -> None:
    assert sizes.dtype in (torch.int32, torch.int64) and ws.dtype == torch.int64
    _check("mxg_group_offsets_unaligned",
           load().mxg_group_offsets_unaligned(_p(sizes), 1 if sizes.dtype == torch.int64 else 0,
                                              sizes.numel(), multiplier, last_dim, rows_capacity,
                                              _p(ws), _p(dev_status), _s(stream)))


def mxg_group_quantize_unaligned(layout: int, x: torch.Tensor, rows_capacity: int, cols: int,
                                 group_ws: torch.Tensor, G: int, q_row=None, sf_row=None,
                                 q_col=None, sf_col=None, dev_status=None, stream=None) -> None:
    assert x.dtype == torch.bfloat16 and x.is_contiguous()
    _check("mxg_group_quantize_unaligned",
           load().mxg_group_quantize_unaligned(layout, _p(x), rows_capacity, cols, _p(group_ws), G,
                                               _p(q_row), _p(sf_row), _p(q_col), _p(sf_col),
                                               _p(dev_status), _s(stream)))


def mxg_grouped_gemm_unaligned(mode: int, A: tuple, B: tuple, group_ws: torch.Tensor, G: int,
                               M_cap: int, N: int, K: int, alpha=None, beta=None, C=None,
                               out_type: int = MXG_OUT_F32, dev_status=None, stream=None,
                               bias=None) -> None:
    """A, B: (data, scale) device tensors (MXFP8)."""
    a, b = _operand(A[:2], 1), _operand(B[:2], 1)
    _check("mxg_grouped_gemm_unaligned",
           load().mxg_grouped_gemm_unaligned(mode, ctypes.byref(a), ctypes.byref(b), _p(group_ws),
                                             G, M_cap, N, K, _p(alpha), _p(beta), _p(bias), _p(C),
                                             out_type, _p(dev_status), _s(stream)))


def mxg_status_string(code: int) -> str:
    return load().mxg_status_string(code).decode()


def mxg_version() -> int:
    return load().mxg_version()


def mxg_launch_count() -> int:
    return load().mxg_launch_count()


# ----------------------------------------------------------------- buffer helpers
def alloc_offsets(G: int, device="cuda") -> torch.Tensor:
    return torch.empty(2 * G + 1, dtype=torch.int64, device=device)


def alloc_mxfp8(rows: int, cols: int, rowwise=True, colwise=False, device="cuda") -> dict:
    out = {}
    if rowwise:
        out["q_row"] = torch.empty((rows, cols), dtype=torch.uint8, device=device)
        out["sf_row"] = torch.empty(rows * cols // 32, dtype=torch.uint8, device=device)
    if colwise:
        out["q_col"] = torch.empty((cols, rows), dtype=torch.uint8, device=device)
        out["sf_col"] = torch.empty(rows * cols // 32, dtype=torch.uint8, device=device)
    return out


def alloc_mxfp8_unaligned(rows: int, cols: int, G: int, rowwise=True, colwise=False,
                          device="cuda") -> dict:
    """Buffers for mxg_group_quantize_unaligned: dense rowwise data, scales and
    colwise copy over the padded row count rows + 128 G."""
    rp = rows + 128 * G
    out = {}
    if rowwise:
        out["q_row"] = torch.empty((rows, cols), dtype=torch.uint8, device=device)
        out["sf_row"] = torch.empty(rp * cols // 32, dtype=torch.uint8, device=device)
    if colwise:
        out["q_col"] = torch.empty((cols, rp), dtype=torch.uint8, device=device)
        out["sf_col"] = torch.empty(rp * cols // 32, dtype=torch.uint8, device=device)
    return out


def alloc_nvfp4(rows: int, cols: int, device="cuda", rowwise=True, colwise=False,
                G: int = 1) -> dict:
    out = {}
    if rowwise:
        out["q_row"] = torch.empty((rows, cols // 2), dtype=torch.uint8, device=device)
        out["sf_row"] = torch.empty(rows * cols // 16, dtype=torch.uint8, device=device)
        out["outer_row"] = torch.empty(rows, dtype=torch.float32, device=device)
    if colwise:
        out["q_col"] = torch.empty((cols, rows // 2), dtype=torch.uint8, device=device)
        out["sf_col"] = torch.empty(rows * cols // 16, dtype=torch.uint8, device=device)
        out["outer_col"] = torch.empty((G, cols), dtype=torch.float32, device=device)
    return out
