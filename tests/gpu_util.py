"""Helpers for the GPU parity tests: run the CUDA path through the C ABI and
the oracle on the same seeded inputs.  Imported by tests only."""
from __future__ import annotations


import numpy as np
import pytest
import torch

import oracle
from moe_grouped_block_gb300 import mxg, workloads

DEV = "cuda"


def require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    major, minor = torch.cuda.get_device_capability()
    if (major, minor) != (10, 3):
        pytest.skip("needs sm_103 (GB300)")
    mxg.load()


def u8(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().numpy().reshape(-1)


def status_tensor():
    return torch.zeros(1, dtype=torch.int32, device=DEV)


def gpu_offsets(sizes: torch.Tensor, last_dim: int, cap: int, mult: int = 1):
    G = sizes.numel()
    ws = mxg.alloc_offsets(G, DEV)
    st = status_tensor()
    mxg.mxg_group_offsets(sizes.to(DEV), mult, last_dim, cap, ws, st)
    return ws, st


def gpu_mxfp8(x_dev: torch.Tensor, ws, G: int, layout: int, fill: int | None = None):
    R, C = x_dev.shape
    out = mxg.alloc_mxfp8(R, C, rowwise=bool(layout & 1), colwise=bool(layout & 2), device=DEV)
    if fill is not None:
        for t in out.values():
            t.fill_(fill)
    st = status_tensor()
    mxg.mxg_group_quantize(mxg.MXG_MXFP8_E4M3, layout, x_dev, R, C, ws, G, out.get("q_row"),
                           out.get("sf_row"), out.get("q_col"), out.get("sf_col"), None, st)
    return out, st


def gpu_nvfp4(x_dev: torch.Tensor, ws, G: int, fill: int | None = None):
    R, C = x_dev.shape
    out = mxg.alloc_nvfp4(R, C, device=DEV)
    if fill is not None:
        out["q_row"].fill_(fill)
        out["sf_row"].fill_(fill)
        out["outer_row"].fill_(float("nan"))
    st = status_tensor()
    mxg.mxg_group_quantize(mxg.MXG_NVFP4_ROWSCALED, mxg.MXG_ROWWISE, x_dev, R, C, ws, G,
                           out["q_row"], out["sf_row"], None, None, out["outer_row"], st)
    return out, st


def normwise_errors(got: np.ndarray, ref: np.ndarray, offs, rows=None):
    """max |got-ref| / max |ref| per expert (over the rows of each expert
    present in `rows`, default all rows)."""
    rows = np.arange(got.shape[0]) if rows is None else np.asarray(rows)
    errs = []
    for g in range(len(offs) - 1):
        sel = (rows >= offs[g]) & (rows < offs[g + 1])
        if not sel.any():
            continue
        r, gg = ref[sel], got[sel]
        den = np.max(np.abs(r))
        errs.append(np.max(np.abs(gg - r)) / den if den > 0 else np.max(np.abs(gg)))
    return np.array(errs)


# Elementwise relative error is taken over the elements with |ref| >= 1e-2 of
# their expert's max|ref| (near-cancelling elements have no meaningful
# relative error); it is reported beside the normwise gate, with a loose
# sanity bound.
ELEM_FLOOR = 1e-2
ELEM_BOUND = 1e-2


def elementwise_error(got: np.ndarray, ref: np.ndarray) -> float:
    """max |got-ref| / |ref| over the elements of one expert block with
    |ref| >= ELEM_FLOOR * max|ref|."""
    den = np.max(np.abs(ref)) if ref.size else 0.0
    if den == 0:
        return 0.0
    sel = np.abs(ref) >= ELEM_FLOOR * den
    return float(np.max(np.abs(got[sel] - ref[sel]) / np.abs(ref[sel])))


def elementwise_errors(got: np.ndarray, ref: np.ndarray, offs, rows=None):
    """elementwise_error per expert (rows grouped as in normwise_errors)."""
    rows = np.arange(got.shape[0]) if rows is None else np.asarray(rows)
    errs = []
    for g in range(len(offs) - 1):
        sel = (rows >= offs[g]) & (rows < offs[g + 1])
        if sel.any():
            errs.append(elementwise_error(got[sel], ref[sel]))
    return np.array(errs)


def report_errors(name: str, normwise, elementwise) -> None:
    """One line per full-size check (shown with pytest -rP)."""
    print("%s: normwise max %.3e, elementwise max over |R| >= %.0e max|R|: %.3e"
          % (name, float(np.max(normwise)), ELEM_FLOOR, float(np.max(elementwise))))


class gemm_override:
    """Context manager that routes mxg.mxg_grouped_gemm through the test entry
    point mxg_grouped_gemm_debug with a forced kernel choice: tile_n = 256 or
    128 selects the single-CTA kernel with that tile width, stage_bytes = 128
    forces 128-byte K stages.  With neither set, calls are left unchanged."""

    def __init__(self, tile_n=None, stage_bytes=None):
        self.tile_n = tile_n or 0
        self.stage_bytes = stage_bytes or 0

    def __enter__(self):
        self.orig = mxg.mxg_grouped_gemm
        if not self.tile_n and not self.stage_bytes:
            return self
        orig_debug = mxg.mxg_grouped_gemm_debug
        tn, sb = self.tile_n, self.stage_bytes

        def forced(fmt, mode, A, B, group_ws, G, M_cap, N, K, alpha=None, beta=None, C=None,
                   out_type=mxg.MXG_OUT_F32, workspace=None, workspace_bytes=0, dev_status=None,
                   stream=None, bias=None):
            orig_debug(fmt, mode, A, B, group_ws, G, M_cap, N, K, alpha=alpha, beta=beta, C=C,
                       out_type=out_type, dev_status=dev_status, tile_n=tn, stage_bytes=sb,
                       stream=stream, bias=bias)

        mxg.mxg_grouped_gemm = forced
        return self

    def __exit__(self, *a):
        mxg.mxg_grouped_gemm = self.orig


def tile_n(n):
    """gemm_override forcing the single-CTA kernel's tile width (None: default)."""
    return gemm_override(tile_n=n)


def fprop_case(wl: workloads.Workload, layout_x=mxg.MXG_ROWWISE, out_type=mxg.MXG_OUT_F32,
               alpha=None, beta=None, c_in=None, fill_c=0.0, bias=None, c_offset=0):
    """Quantize x and w and run the fprop GEMM on the GPU.  Returns a dict of
    host inputs, device outputs and the offsets.  With c_offset > 0, C starts
    c_offset elements into a larger buffer (returned as "C_buf")."""
    inp = workloads.make_inputs(wl)
    G, N, K, R = wl.G, wl.N, wl.K, wl.rows_capacity
    x = inp["x"].to(DEV)
    w = inp["w"].to(DEV).reshape(G * N, K)
    ws, st = gpu_offsets(inp["sizes"], K, R)
    fmt = mxg.MXG_MXFP8_E4M3 if wl.fmt == "mxfp8" else mxg.MXG_NVFP4_ROWSCALED
    if wl.fmt == "mxfp8":
        qx, _ = gpu_mxfp8(x, ws, G, layout_x)
        qw, _ = gpu_mxfp8(w, None, G, mxg.MXG_ROWWISE)
        A = (qx["q_row"], qx["sf_row"], None)
        B = (qw["q_row"], qw["sf_row"], None)
    else:
        qx, _ = gpu_nvfp4(x, ws, G)
        qw, _ = gpu_nvfp4(w, None, G)
        A = (qx["q_row"], qx["sf_row"], qx["outer_row"])
        B = (qw["q_row"], qw["sf_row"], qw["outer_row"])
    cdt = torch.float32 if out_type == mxg.MXG_OUT_F32 else torch.bfloat16
    C_buf = torch.full((c_offset + R * N,), fill_c, dtype=cdt, device=DEV)
    C = C_buf[c_offset:].view(R, N)
    if c_in is not None:
        C.copy_(c_in.to(DEV, cdt))
    al = None if alpha is None else torch.tensor(alpha, dtype=torch.float32, device=DEV)
    be = None if beta is None else torch.tensor(beta, dtype=torch.float32, device=DEV)
    bi = None if bias is None else torch.as_tensor(bias, dtype=torch.float32).to(DEV)
    mxg.mxg_grouped_gemm(fmt, mxg.MXG_FPROP_TN, A, B, ws, G, R, N, K, al, be, C, out_type,
                         dev_status=st, bias=bi)
    torch.cuda.synchronize()
    return {"inp": inp, "ws": ws, "status": st, "qx": qx, "qw": qw, "C": C, "C_buf": C_buf,
            "G": G, "N": N, "K": K, "R": R}


def oracle_quantized_operands(wl: workloads.Workload, inp: dict):
    """The oracle's own quantization of the seeded inputs (never the GPU's)."""
    G, N, K, R = wl.G, wl.N, wl.K, wl.rows_capacity
    ws, _ = oracle.group_offsets(inp["sizes"].numpy(), 1, K, R)
    offs = oracle.live_rows(ws, G)
    live = int(offs[-1])
    w2 = inp["w"].reshape(G * N, K)
    if wl.fmt == "mxfp8":
        ox = oracle.mxfp8_quantize(inp["x"], live, R, rowwise=True)
        ow = oracle.mxfp8_quantize(w2, G * N, G * N, rowwise=True)
        a = {"q": ox["q_row"], "sf": ox["sf_row"]}
        b = {"q": ow["q_row"], "sf": ow["sf_row"]}
    else:
        ox = oracle.nvfp4_quantize(inp["x"], live, R)
        ow = oracle.nvfp4_quantize(w2, G * N, G * N)
        a = {"q": ox["q_row"], "sf": ox["sf_row"], "outer": ox["outer_row"]}
        b = {"q": ow["q_row"], "sf": ow["sf_row"], "outer": ow["outer_row"]}
    return ws, offs, a, b


def oracle_fprop(wl: workloads.Workload, inp: dict, rows=None, cols=None, alpha=None, beta=None,
                 c_in=None, bias=None):
    ws, offs, a, b = oracle_quantized_operands(wl, inp)
    r, c, ref = oracle.grouped_gemm_fprop(wl.fmt, a, b, offs, wl.N, wl.K, alpha=alpha, beta=beta,
                                          c_in=c_in, sample_rows=rows, sample_cols=cols, bias=bias)
    return offs, r, c, ref, a, b
