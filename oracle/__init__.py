"""Oracle for the grouped block-scaled quantize + grouped GEMM path.

TEST INFRASTRUCTURE ONLY.  This package is imported by ``tests/``, by
``__graft_entry__.smoke()`` and by the CPU-baseline / reference legs of
``bench.py``; the product library (``moe_grouped_block_gb300``) never imports,
links or executes anything here, and nothing here imports the product.  The two
share only the seeded input generators, which hold none of the method's
arithmetic.

Bit-level work (codecs, the MXFP8 and row-scaled NVFP4 quantizers, the scale
swizzle, the group offsets, dequantization) is plain C in ``mxg_oracle.c``,
built by :func:`build` with gcc.  The grouped GEMM is the per-expert dense
product over the dequantized operands in fp64, with a library matmul as the
one primitive step:

* fprop (TN, ragged rows), TransformerEngine gemm.py ``grouped_gemm`` with its
  default contracting dims: ``C[off_g+i, n] = alpha_g * sum_k dq(A)[off_g+i, k]
  * dq(B)[g, n, k] + beta_g * C_in``, alpha = 1 and beta = 0 by default
  (gemm.py ``grouped_gemm``: alpha ones, beta zeros).
* wgrad (NT, ragged contraction), gemm.py ``grouped_gemm`` wgrad branch:
  ``dW[g, n, k] = alpha_g * sum_{m in group g} dq(dY)[m, n] * dq(X)[m, k]``;
  an empty group gives ``beta_g * dW_in`` (zeros by default).
* row-scaled NVFP4 (PR #3661 description): the product runs on operands with
  neutral outer scales, then the per-row (activation) and per-column (weight)
  FP32 outer scales are applied to the fp64 result.

Every GEMM here is pinned by tests against brute-force loops on tiny inputs,
the per-expert-dense invariant, the G = 1 dense case and exact integer cases.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mxg_oracle.c")
_SO = os.path.join(_HERE, "libmxg_oracle.so")
_lock = threading.Lock()
_lib = None

ST_NEG_SIZE = 1
ST_MISALIGNED = 2
ST_SUM_OVER_CAPACITY = 4


def build(force: bool = False) -> str:
    """Compile mxg_oracle.c with gcc (no fused multiply-add, no fast-math)."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + ".tmp.%d" % os.getpid()
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
               "-fno-fast-math", "-Wall", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _SO)
    return _SO


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_SO)
            c_p = ctypes.c_void_p
            i64, i32 = ctypes.c_int64, ctypes.c_int32
            L.mxg_oracle_e4m3_decode.restype = ctypes.c_double
            L.mxg_oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
            L.mxg_oracle_e4m3_encode.restype = ctypes.c_uint8
            L.mxg_oracle_e4m3_encode.argtypes = [ctypes.c_double]
            L.mxg_oracle_e2m1_decode.restype = ctypes.c_double
            L.mxg_oracle_e2m1_decode.argtypes = [ctypes.c_uint8]
            L.mxg_oracle_e2m1_encode.restype = ctypes.c_uint8
            L.mxg_oracle_e2m1_encode.argtypes = [ctypes.c_double]
            L.mxg_oracle_e8m0_decode.restype = ctypes.c_double
            L.mxg_oracle_e8m0_decode.argtypes = [ctypes.c_uint8]
            L.mxg_oracle_mx_scale_exponent.restype = ctypes.c_int
            L.mxg_oracle_mx_scale_exponent.argtypes = [ctypes.c_float]
            L.mxg_oracle_swizzle_index.restype = i64
            L.mxg_oracle_swizzle_index.argtypes = [i64, i64, i64]
            L.mxg_oracle_unswizzle.argtypes = [c_p, i64, i64, c_p]
            L.mxg_oracle_swizzle.argtypes = [c_p, i64, i64, c_p]
            L.mxg_oracle_group_offsets.restype = i32
            L.mxg_oracle_group_offsets.argtypes = [c_p, ctypes.c_int, i64, i64, i64, c_p]
            L.mxg_oracle_group_offsets_unaligned.restype = i32
            L.mxg_oracle_group_offsets_unaligned.argtypes = [c_p, ctypes.c_int, i64, i64, i64, c_p]
            L.mxg_oracle_mxfp8_quantize_rowwise.argtypes = [c_p, i64, i64, c_p, c_p]
            L.mxg_oracle_mxfp8_quantize_colwise.argtypes = [c_p, i64, i64, i64, c_p, c_p]
            L.mxg_oracle_nvfp4_quantize_rowwise.argtypes = [c_p, i64, i64, c_p, c_p, c_p]
            L.mxg_oracle_nvfp4_quantize_colwise.argtypes = [c_p, c_p, ctypes.c_int, i64, i64, c_p,
                                                            c_p, c_p]
            L.mxg_oracle_mxfp8_dequantize_rows.argtypes = [c_p, c_p, i64, c_p, i64, c_p]
            L.mxg_oracle_nvfp4_dequantize_rows.argtypes = [c_p, c_p, c_p, ctypes.c_int, i64, c_p,
                                                           i64, c_p]
            L.mxg_oracle_e4m3_encode_array.argtypes = [c_p, i64, c_p]
            L.mxg_oracle_e2m1_encode_array.argtypes = [c_p, i64, c_p]
            L.mxg_oracle_mx_scale_exponent_array.argtypes = [c_p, i64, c_p]
            _lib = L
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"], "oracle buffers must be C-contiguous"
    return a.ctypes.data


def _u16(x) -> np.ndarray:
    """bf16 input as its uint16 bit pattern (numpy array or torch tensor)."""
    if hasattr(x, "view") and hasattr(x, "dtype") and str(x.dtype) == "torch.bfloat16":
        import torch  # only the input container; no arithmetic
        x = x.contiguous().view(torch.int16).numpy().view(np.uint16)
    x = np.ascontiguousarray(x)
    assert x.dtype == np.uint16, "bf16 inputs are passed as uint16 bit patterns"
    return x


# --------------------------------------------------------------------------
# codecs (scalar and array)
# --------------------------------------------------------------------------
def e4m3_decode(b: int) -> float:
    return lib().mxg_oracle_e4m3_decode(int(b))


def e4m3_encode(v: float) -> int:
    return lib().mxg_oracle_e4m3_encode(float(v))


def e2m1_decode(n: int) -> float:
    return lib().mxg_oracle_e2m1_decode(int(n))


def e2m1_encode(v: float) -> int:
    return lib().mxg_oracle_e2m1_encode(float(v))


def e8m0_decode(b: int) -> float:
    return lib().mxg_oracle_e8m0_decode(int(b))


def e4m3_encode_array(v: np.ndarray) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float64)
    out = np.empty(v.shape, np.uint8)
    lib().mxg_oracle_e4m3_encode_array(_ptr(v), v.size, _ptr(out))
    return out


def e2m1_encode_array(v: np.ndarray) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float64)
    out = np.empty(v.shape, np.uint8)
    lib().mxg_oracle_e2m1_encode_array(_ptr(v), v.size, _ptr(out))
    return out


def e4m3_decode_table() -> np.ndarray:
    return np.array([e4m3_decode(b) for b in range(256)], dtype=np.float64)


def e2m1_decode_table() -> np.ndarray:
    return np.array([e2m1_decode(n) for n in range(16)], dtype=np.float64)


def mx_scale_exponent(amax: float) -> int:
    return lib().mxg_oracle_mx_scale_exponent(float(amax))


def mx_scale_exponent_array(amax: np.ndarray) -> np.ndarray:
    amax = np.ascontiguousarray(amax, dtype=np.float32)
    out = np.empty(amax.shape, np.int32)
    lib().mxg_oracle_mx_scale_exponent_array(_ptr(amax), amax.size, _ptr(out))
    return out


# --------------------------------------------------------------------------
# swizzle
# --------------------------------------------------------------------------
def swizzle_index(r: int, c: int, C: int) -> int:
    return lib().mxg_oracle_swizzle_index(r, c, C)


def swizzle(plain: np.ndarray) -> np.ndarray:
    plain = np.ascontiguousarray(plain, dtype=np.uint8)
    R, C = plain.shape
    out = np.empty(R * C, np.uint8)
    lib().mxg_oracle_swizzle(_ptr(plain), R, C, _ptr(out))
    return out


def unswizzle(swz: np.ndarray, R: int, C: int) -> np.ndarray:
    swz = np.ascontiguousarray(swz, dtype=np.uint8).reshape(-1)
    assert swz.size == R * C
    out = np.empty((R, C), np.uint8)
    lib().mxg_oracle_unswizzle(_ptr(swz), R, C, _ptr(out))
    return out


# --------------------------------------------------------------------------
# offsets
# --------------------------------------------------------------------------
def group_offsets(sizes, multiplier: int, last_dim: int, rows_capacity: int):
    """Returns (workspace int64[2G+1] = [sizes | offsets], status bits)."""
    s = np.ascontiguousarray(np.asarray(sizes).astype(np.int64))
    G = s.size
    ws = np.zeros(2 * G + 1, np.int64)
    st = lib().mxg_oracle_group_offsets(_ptr(s), G, multiplier, last_dim, rows_capacity, _ptr(ws))
    return ws, int(st)


def live_rows(ws: np.ndarray, G: int) -> np.ndarray:
    """Row offsets [G+1] from a workspace (element offsets / last_dim is not
    needed: the sanitised sizes are stored in the first G slots)."""
    return np.concatenate([[0], np.cumsum(ws[:G])]).astype(np.int64)


# --------------------------------------------------------------------------
# quantizers
# --------------------------------------------------------------------------
def mxfp8_quantize(x, rows_live: int, rows_capacity: int, rowwise=True, colwise=False,
                   fill: int = 0):
    """MXFP8 (R1) quantize of bf16 x[rows_capacity, cols].  Buffers are
    pre-filled with ``fill``; rows >= rows_live are left untouched."""
    x = _u16(x)
    R, cols = x.shape
    assert R == rows_capacity and cols % 128 == 0 and R % 128 == 0 and rows_live % 32 == 0
    out = {}
    if rowwise:
        q = np.full((R, cols), fill, np.uint8)
        sf = np.full(R * cols // 32, fill, np.uint8)
        lib().mxg_oracle_mxfp8_quantize_rowwise(_ptr(x), rows_live, cols, _ptr(q), _ptr(sf))
        out["q_row"], out["sf_row"] = q, sf
    if colwise:
        qT = np.full((cols, R), fill, np.uint8)
        sfT = np.full(cols * R // 32, fill, np.uint8)
        lib().mxg_oracle_mxfp8_quantize_colwise(_ptr(x), rows_live, R, cols, _ptr(qT), _ptr(sfT))
        out["q_col"], out["sf_col"] = qT, sfT
    return out


def nvfp4_quantize(x, rows_live: int, rows_capacity: int, fill: int = 0):
    """Row-scaled NVFP4 (R2) quantize of bf16 x[rows_capacity, cols]."""
    x = _u16(x)
    R, cols = x.shape
    assert R == rows_capacity and cols % 128 == 0 and R % 128 == 0
    q = np.full((R, cols // 2), fill, np.uint8)
    sf = np.full(R * cols // 16, fill, np.uint8)
    outer = np.full(R, np.nan, np.float32)
    lib().mxg_oracle_nvfp4_quantize_rowwise(_ptr(x), rows_live, cols, _ptr(q), _ptr(sf),
                                            _ptr(outer))
    return {"q_row": q, "sf_row": sf, "outer_row": outer}


def nvfp4_quantize_colwise(x, group_rows, rows_capacity: int, fill: int = 0):
    """Row-scaled NVFP4 (R2) of the columns of each group, written transposed:
    q_col [cols, rows_cap/2], sf_col swizzled [cols, rows_cap/16], outer_col
    [G, cols] (per group and column)."""
    x = _u16(x)
    R, cols = x.shape
    offs = np.ascontiguousarray(np.asarray(group_rows, np.int64))
    G = offs.size - 1
    assert R == rows_capacity and cols % 128 == 0 and R % 128 == 0
    qT = np.full((cols, R // 2), fill, np.uint8)
    sfT = np.full(cols * R // 16, fill, np.uint8)
    outer = np.full((G, cols), np.nan, np.float32)
    lib().mxg_oracle_nvfp4_quantize_colwise(_ptr(x), _ptr(offs), G, R, cols, _ptr(qT), _ptr(sfT),
                                            _ptr(outer))
    return {"q_col": qT, "sf_col": sfT, "outer_col": outer}


# --------------------------------------------------------------------------
# dequantize
# --------------------------------------------------------------------------
def dequantize_rows(fmt: str, q: np.ndarray, sf: np.ndarray, cols: int, rows,
                    outer: np.ndarray | None = None, with_outer: bool = True) -> np.ndarray:
    """fp64 values of the given rows of a rowwise-quantized [*, cols] matrix."""
    idx = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1))
    out = np.empty((idx.size, cols), np.float64)
    q = np.ascontiguousarray(q)
    sf = np.ascontiguousarray(sf)
    if fmt == "mxfp8":
        lib().mxg_oracle_mxfp8_dequantize_rows(_ptr(q), _ptr(sf), cols, _ptr(idx), idx.size,
                                               _ptr(out))
    elif fmt == "nvfp4":
        o = np.ascontiguousarray(outer if outer is not None else np.ones(1, np.float32),
                                 dtype=np.float32)
        lib().mxg_oracle_nvfp4_dequantize_rows(_ptr(q), _ptr(sf), _ptr(o),
                                               1 if (with_outer and outer is not None) else 0,
                                               cols, _ptr(idx), idx.size, _ptr(out))
    else:
        raise ValueError(fmt)
    return out


def dequantize(fmt: str, q, sf, rows: int, cols: int, outer=None) -> np.ndarray:
    return dequantize_rows(fmt, q, sf, cols, np.arange(rows), outer)


# --------------------------------------------------------------------------
# grouped GEMM (fp64, per expert)
# --------------------------------------------------------------------------
def _per_group(alpha, G):
    return np.ones(G) if alpha is None else np.asarray(alpha, np.float64).reshape(G)


def grouped_gemm_fprop(fmt: str, a: dict, b: dict, group_rows, N: int, K: int,
                       alpha=None, beta=None, c_in=None, sample_rows=None, sample_cols=None,
                       bias=None):
    """fprop TN over ragged row groups.

    a: {"q", "sf"[, "outer"]} rowwise-quantized activations [M_cap, K].
    b: {"q", "sf"[, "outer"]} rowwise-quantized weights [G*N, K].
    group_rows: int64[G+1] row offsets.  Returns a dict row -> fp64 vector
    over ``sample_cols`` (default all N) for every live row in
    ``sample_rows`` (default all live rows), as an array [rows, cols] plus
    the row list.
    """
    offs = np.asarray(group_rows, np.int64)
    G = offs.size - 1
    al, be = _per_group(alpha, G), (np.zeros(G) if beta is None else
                                    np.asarray(beta, np.float64).reshape(G))
    cols = np.arange(N) if sample_cols is None else np.asarray(sample_cols, np.int64)
    rows = (np.arange(offs[-1]) if sample_rows is None else
            np.asarray(sample_rows, np.int64))
    out = np.zeros((rows.size, cols.size), np.float64)
    for g in range(G):
        sel = np.nonzero((rows >= offs[g]) & (rows < offs[g + 1]))[0]
        if sel.size == 0:
            continue
        ra = rows[sel]
        rb = g * N + cols
        if fmt == "mxfp8":
            A = dequantize_rows("mxfp8", a["q"], a["sf"], K, ra)
            B = dequantize_rows("mxfp8", b["q"], b["sf"], K, rb)
            acc = A @ B.T
        else:
            # neutral outer scales, product, then the row / column post-scale
            A = dequantize_rows("nvfp4", a["q"], a["sf"], K, ra, a["outer"], with_outer=False)
            B = dequantize_rows("nvfp4", b["q"], b["sf"], K, rb, b["outer"], with_outer=False)
            acc = A @ B.T
            acc = acc * np.asarray(a["outer"], np.float64)[ra][:, None]
            acc = acc * np.asarray(b["outer"], np.float64)[rb][None, :]
        res = al[g] * acc
        if bias is not None:
            res = res + np.asarray(bias, np.float64)[g][cols][None, :]
        if c_in is not None and be[g] != 0.0:
            res = res + be[g] * np.asarray(c_in, np.float64)[np.ix_(ra, cols)]
        out[sel] = res
    return rows, cols, out


def grouped_gemm_wgrad(a_t: dict, b_t: dict, group_rows, M_cap: int, N: int, K: int,
                       alpha=None, beta=None, c_in=None, sample_n=None, sample_k=None,
                       fmt: str = "mxfp8"):
    """wgrad NT over ragged contraction groups (MXFP8, or row-scaled NVFP4 with
    per-(group, column) outer scales "outer" [G, N] / [G, K] applied after
    the neutral-scale product, PR #3661's wgrad).

    a_t: colwise (transposed) copy of dY: {"q": [N, M_cap], "sf": [N, M_cap/32] swizzled}.
    b_t: colwise (transposed) copy of X:  {"q": [K, M_cap], "sf": [K, M_cap/32] swizzled}.
    Returns an array [G, len(sample_n), len(sample_k)] in fp64.
    """
    offs = np.asarray(group_rows, np.int64)
    G = offs.size - 1
    al = _per_group(alpha, G)
    be = np.zeros(G) if beta is None else np.asarray(beta, np.float64).reshape(G)
    ns = np.arange(N) if sample_n is None else np.asarray(sample_n, np.int64)
    ks = np.arange(K) if sample_k is None else np.asarray(sample_k, np.int64)
    if fmt == "mxfp8":
        dYT = dequantize_rows("mxfp8", a_t["q"], a_t["sf"], M_cap, ns)
        XT = dequantize_rows("mxfp8", b_t["q"], b_t["sf"], M_cap, ks)
    else:  # neutral outer scales; the per-(group, column) ones come after the product
        dYT = dequantize_rows("nvfp4", a_t["q"], a_t["sf"], M_cap, ns)
        XT = dequantize_rows("nvfp4", b_t["q"], b_t["sf"], M_cap, ks)
    out = np.zeros((G, ns.size, ks.size), np.float64)
    for g in range(G):
        lo, hi = offs[g], offs[g + 1]
        res = al[g] * (dYT[:, lo:hi] @ XT[:, lo:hi].T) if hi > lo else np.zeros((ns.size, ks.size))
        if fmt == "nvfp4":
            res = res * np.asarray(a_t["outer"], np.float64)[g][ns][:, None]
            res = res * np.asarray(b_t["outer"], np.float64)[g][ks][None, :]
        if c_in is not None and be[g] != 0.0:
            res = res + be[g] * np.asarray(c_in, np.float64)[g][np.ix_(ns, ks)]
        out[g] = res
    return ns, ks, out


def grouped_gemm_dgrad(a: dict, b_t: dict, group_rows, G: int, N: int, K: int, alpha=None,
                       beta=None, c_in=None, sample_rows=None, sample_cols=None, bias=None):
    """dgrad NN over ragged row groups (MXFP8), TransformerEngine gemm.py
    grouped_gemm with the weights not transposed (its _quantize_gemm_operands
    quantizes such an RHS colwise, i.e. in blocks along N).

    a:   rowwise dY {"q": [M_cap, N], "sf": swizzled [M_cap, N/32]}.
    b_t: colwise (transposed) copy of W viewed as [G*N, K]:
         {"q": [K, G*N], "sf": swizzled [K, G*N/32]}.
    dX[off_g+i, k] = alpha_g * sum_n dq(dY)[off_g+i, n] * dq(W)[g*N+n, k]
                     (+ beta_g * c_in).  Returns (rows, cols, [rows, cols]).
    """
    offs = np.asarray(group_rows, np.int64)
    al = _per_group(alpha, G)
    be = np.zeros(G) if beta is None else np.asarray(beta, np.float64).reshape(G)
    cols = np.arange(K) if sample_cols is None else np.asarray(sample_cols, np.int64)
    rows = np.arange(offs[-1]) if sample_rows is None else np.asarray(sample_rows, np.int64)
    WT = dequantize_rows("mxfp8", b_t["q"], b_t["sf"], G * N, cols)  # [len(cols), G*N]
    out = np.zeros((rows.size, cols.size), np.float64)
    for g in range(G):
        sel = np.nonzero((rows >= offs[g]) & (rows < offs[g + 1]))[0]
        if sel.size == 0:
            continue
        A = dequantize_rows("mxfp8", a["q"], a["sf"], N, rows[sel])
        res = al[g] * (A @ WT[:, g * N:(g + 1) * N].T)
        if bias is not None:
            res = res + np.asarray(bias, np.float64)[g][cols][None, :]
        if c_in is not None and be[g] != 0.0:
            res = res + be[g] * np.asarray(c_in, np.float64)[np.ix_(rows[sel], cols)]
        out[sel] = res
    return rows, cols, out


# --------------------------------------------------------------------------
# groups of any size (MXFP8): each group is its own tensor, zero-padded to a
# multiple of 128 rows.  TransformerEngine gemm.py grouped_gemm: padding is
# part of a group and filled with zeros so that it does not change the
# result; gemm.py apply_padding_to_scale_inv pads scale matrices of non-128
# dims; PR #2763 review thread: the 128-row rule comes from the offset
# arithmetic of the grouped quantize and GEMM setup.  Everything below is
# composed from the aligned (pinned) quantizer, dequantizer and swizzle.
# --------------------------------------------------------------------------
def group_offsets_unaligned(sizes, multiplier: int, last_dim: int, rows_capacity: int):
    """As group_offsets, with sizes kept as given (no rounding to 128)."""
    s = np.ascontiguousarray(np.asarray(sizes).astype(np.int64))
    G = s.size
    ws = np.zeros(2 * G + 1, np.int64)
    st = lib().mxg_oracle_group_offsets_unaligned(_ptr(s), G, multiplier, last_dim,
                                                  rows_capacity, _ptr(ws))
    return ws, int(st)


def padded_rows(ws: np.ndarray, G: int) -> np.ndarray:
    """Padded row offsets [G+1]: prefix sums of each group's rows rounded up to 128."""
    sizes = np.asarray(ws[:G], np.int64)
    return np.concatenate([[0], np.cumsum((sizes + 127) // 128 * 128)]).astype(np.int64)


def unaligned_rows_capacity(rows_capacity: int, G: int) -> int:
    return rows_capacity + 128 * G


def mxfp8_quantize_unaligned(x, ws: np.ndarray, G: int, rows_capacity: int, rowwise=True,
                             colwise=False, fill: int = 0):
    """MXFP8 quantize of each group of bf16 x[rows_capacity, cols] as its own
    tensor zero-padded to P_g = ceil128(M_g) rows.  Outputs (pre-filled with
    ``fill`` where nothing is written):
      q_row  [rows_capacity, cols] dense (group g at its data rows);
      sf_row swizzled [R_pad, cols/32], group g's scale rows at its padded offset;
      q_col  [cols, R_pad] and sf_col swizzled [cols, R_pad/32], group g's slab at
      its padded offset;   R_pad = rows_capacity + 128 G."""
    xu = _u16(x)
    R, cols = xu.shape
    assert R == rows_capacity and cols % 128 == 0 and R % 128 == 0
    offs = live_rows(ws, G)
    poffs = padded_rows(ws, G)
    Rp = unaligned_rows_capacity(R, G)
    C = cols // 32
    out = {}
    q_row = np.full((R, cols), fill, np.uint8)
    sfp_row = np.full((Rp, C), fill, np.uint8)
    q_col = np.full((cols, Rp), fill, np.uint8)
    sfp_col = np.full((cols, Rp // 32), fill, np.uint8)
    for g in range(G):
        m, lo, plo = int(ws[g]), int(offs[g]), int(poffs[g])
        if m == 0:
            continue
        P = (m + 127) // 128 * 128
        slab = np.zeros((P, cols), np.uint16)
        slab[:m] = xu[lo:lo + m]
        qs = mxfp8_quantize(slab, P, P, rowwise=rowwise, colwise=colwise)
        if rowwise:
            q_row[lo:lo + m] = qs["q_row"][:m]
            sfp_row[plo:plo + P] = unswizzle(qs["sf_row"], P, C)
        if colwise:
            q_col[:, plo:plo + P] = qs["q_col"]
            sfp_col[:, plo // 32:(plo + P) // 32] = unswizzle(qs["sf_col"], cols, P // 32)
    if rowwise:
        out["q_row"], out["sf_row"] = q_row, swizzle(sfp_row)
    if colwise:
        out["q_col"], out["sf_col"] = q_col, swizzle(sfp_col)
    return out


def _padded_rowwise(a: dict, ws: np.ndarray, G: int, cols: int) -> np.ndarray:
    """Dense rowwise data moved to the padded rows of its scales (zero rows
    in the padding), so that dequantize_rows reads data and scales alike."""
    offs, poffs = live_rows(ws, G), padded_rows(ws, G)
    q_pad = np.zeros((int(poffs[-1]) + 128, cols), np.uint8)
    for g in range(G):
        m = int(ws[g])
        q_pad[poffs[g]:poffs[g] + m] = a["q"][offs[g]:offs[g] + m]
    return q_pad


def grouped_gemm_fprop_unaligned(a: dict, b: dict, ws: np.ndarray, G: int, N: int, K: int,
                                 alpha=None, beta=None, c_in=None, bias=None, sample_rows=None,
                                 sample_cols=None):
    """fprop TN (MXFP8) for groups of any size: a = {"q": dense rowwise data
    [M_cap, K], "sf": padded swizzled scales}.  Returns (rows, [rows, cols])
    over the live data rows in ``sample_rows`` (default all) and the columns
    in ``sample_cols`` (default all N); the per-group product is as in
    grouped_gemm_fprop."""
    offs, poffs = live_rows(ws, G), padded_rows(ws, G)
    q_pad = _padded_rowwise(a, ws, G, K)
    al = _per_group(alpha, G)
    be = np.zeros(G) if beta is None else np.asarray(beta, np.float64).reshape(G)
    rows = np.arange(offs[-1]) if sample_rows is None else np.asarray(sample_rows, np.int64)
    cols = np.arange(N) if sample_cols is None else np.asarray(sample_cols, np.int64)
    out = np.zeros((rows.size, cols.size), np.float64)
    for g in range(G):
        sel = np.nonzero((rows >= offs[g]) & (rows < offs[g + 1]))[0]
        if sel.size == 0:
            continue
        r = rows[sel]
        A = dequantize_rows("mxfp8", q_pad, a["sf"], K, poffs[g] + (r - offs[g]))
        B = dequantize_rows("mxfp8", b["q"], b["sf"], K, g * N + cols)
        res = al[g] * (A @ B.T)
        if bias is not None:
            res = res + np.asarray(bias, np.float64)[g][cols][None, :]
        if c_in is not None and be[g] != 0.0:
            res = res + be[g] * np.asarray(c_in, np.float64)[np.ix_(r, cols)]
        out[sel] = res
    return rows, out


def grouped_gemm_wgrad_unaligned(a_t: dict, b_t: dict, ws: np.ndarray, G: int, M_cap: int,
                                 N: int, K: int, alpha=None, beta=None, c_in=None):
    """wgrad NT (MXFP8) for groups of any size: the colwise copies are padded
    per group, so each group contracts over its padded slab (zeros add
    nothing) -- grouped_gemm_wgrad over the padded offsets."""
    poffs = padded_rows(ws, G)
    return grouped_gemm_wgrad(a_t, b_t, poffs, unaligned_rows_capacity(M_cap, G), N, K,
                              alpha=alpha, beta=beta, c_in=c_in)


def grouped_gemm_dgrad_unaligned(a: dict, b_t: dict, ws: np.ndarray, G: int, N: int, K: int,
                                 alpha=None, beta=None, c_in=None, bias=None):
    """dgrad NN (MXFP8) for groups of any size: a = rowwise dY (dense data,
    padded scales); b_t = colwise copy of W as in grouped_gemm_dgrad."""
    offs, poffs = live_rows(ws, G), padded_rows(ws, G)
    q_pad = _padded_rowwise(a, ws, G, N)
    al = _per_group(alpha, G)
    be = np.zeros(G) if beta is None else np.asarray(beta, np.float64).reshape(G)
    WT = dequantize_rows("mxfp8", b_t["q"], b_t["sf"], G * N, np.arange(K))
    rows = np.arange(offs[-1])
    out = np.zeros((rows.size, K), np.float64)
    for g in range(G):
        m = int(ws[g])
        if m == 0:
            continue
        A = dequantize_rows("mxfp8", q_pad, a["sf"], N, poffs[g] + np.arange(m))
        res = al[g] * (A @ WT[:, g * N:(g + 1) * N].T)
        if bias is not None:
            res = res + np.asarray(bias, np.float64)[g][None, :]
        r = offs[g] + np.arange(m)
        if c_in is not None and be[g] != 0.0:
            res = res + be[g] * np.asarray(c_in, np.float64)[r]
        out[r] = res
    return rows, out
