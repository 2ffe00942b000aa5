"""GPU parity at the full workload sizes, in the launch configuration the
benchmark times (default tile choice, bf16 inputs resident on the device).

Quantized bytes, scales and offsets are compared in full, bit for bit.  GEMM
outputs are compared on samples the oracle computes one by one: for every
expert its first and last rows plus random rows, against a column sample that
covers the first and last output tiles (normwise error per expert <= 1e-3).
The fine-grained 64-expert workload is small enough to check in full."""
import numpy as np
import pytest
import torch

import oracle
from moe_grouped_block_gb300 import mxg, workloads

from gpu_util import DEV, fprop_case, gpu_mxfp8, gpu_offsets, normwise_errors, require_gpu, u8

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
TOL = 1e-3


@pytest.fixture(autouse=True)
def _gpu():
    require_gpu()


def _sample(offs, N, rng, per_group=6, n_cols=1024):
    rows = []
    for g in range(len(offs) - 1):
        lo, hi = int(offs[g]), int(offs[g + 1])
        if hi > lo:
            rows += [lo, hi - 1] + list(rng.integers(lo, hi, per_group))
    cols = np.unique(np.concatenate([np.arange(0, 256), np.arange(N - 256, N),
                                     rng.integers(0, N, n_cols)]))
    return np.unique(rows), cols


def _fprop_fullsize(name, check_all=False):
    wl = workloads.WORKLOADS[name]
    case = fprop_case(wl, out_type=mxg.MXG_OUT_F32,
                      layout_x=mxg.MXG_BOTH if wl.fmt == "mxfp8" else mxg.MXG_ROWWISE)
    assert int(case["status"].item()) == 0
    inp = case["inp"]
    G, N, K, R = wl.G, wl.N, wl.K, wl.rows_capacity
    ws, _ = oracle.group_offsets(inp["sizes"].numpy(), 1, K, R)
    assert np.array_equal(case["ws"].cpu().numpy(), ws)
    offs = oracle.live_rows(ws, G)
    w2 = inp["w"].reshape(G * N, K)
    if wl.fmt == "mxfp8":
        ox = oracle.mxfp8_quantize(inp["x"], R, R, rowwise=True, colwise=True)
        ow = oracle.mxfp8_quantize(w2, G * N, G * N)
        for k in ("q_row", "sf_row", "q_col", "sf_col"):
            assert np.array_equal(u8(case["qx"][k]), ox[k].reshape(-1)), k
        a = {"q": ox["q_row"], "sf": ox["sf_row"]}
        b = {"q": ow["q_row"], "sf": ow["sf_row"]}
    else:
        ox = oracle.nvfp4_quantize(inp["x"], R, R)
        ow = oracle.nvfp4_quantize(w2, G * N, G * N)
        for k in ("q_row", "sf_row", "outer_row"):
            assert np.array_equal(case["qx"][k].cpu().numpy().reshape(-1), ox[k].reshape(-1)), k
        a = {"q": ox["q_row"], "sf": ox["sf_row"], "outer": ox["outer_row"]}
        b = {"q": ow["q_row"], "sf": ow["sf_row"], "outer": ow["outer_row"]}
    for k in ("q_row", "sf_row"):
        assert np.array_equal(u8(case["qw"][k]), ow[k].reshape(-1)), "w " + k
    rng = np.random.default_rng(123)
    if check_all:
        rows, cols = np.arange(int(offs[-1])), np.arange(N)
    else:
        rows, cols = _sample(offs, N, rng)
    _, _, ref = oracle.grouped_gemm_fprop(wl.fmt, a, b, offs, N, K, sample_rows=rows,
                                          sample_cols=cols)
    got = case["C"].cpu().numpy()[np.ix_(rows, cols)].astype(np.float64)
    errs = normwise_errors(got, ref, offs, rows)
    assert errs.max() <= TOL, errs
    return errs


def test_mixtral_fprop_fullsize():
    _fprop_fullsize("mixtral_fprop_mxfp8")


def test_finegrained_fprop_fullsize_all_outputs():
    _fprop_fullsize("finegrained_fprop_mxfp8", check_all=True)


def test_rowscaled_nvfp4_fprop_fullsize():
    _fprop_fullsize("rowscaled_fprop_nvfp4")


def test_wgrad_fullsize():
    wl = workloads.WORKLOADS["wgrad_mxfp8"]
    inp = workloads.make_inputs(wl)
    G, N, K, M = wl.G, wl.N, wl.K, wl.M
    ws, st = gpu_offsets(inp["sizes"], K, M)
    qx, _ = gpu_mxfp8(inp["x"].to(DEV), ws, G, mxg.MXG_COLWISE)
    qd, _ = gpu_mxfp8(inp["dy"].to(DEV), ws, G, mxg.MXG_COLWISE)
    dW = torch.empty((G, N, K), dtype=torch.float32, device=DEV)
    mxg.mxg_grouped_gemm(mxg.MXG_MXFP8_E4M3, mxg.MXG_WGRAD_NT, (qd["q_col"], qd["sf_col"], None),
                         (qx["q_col"], qx["sf_col"], None), ws, G, M, N, K, C=dW, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    rws, _ = oracle.group_offsets(inp["sizes"].numpy(), 1, K, M)
    offs = oracle.live_rows(rws, G)
    ox = oracle.mxfp8_quantize(inp["x"], M, M, rowwise=False, colwise=True)
    od = oracle.mxfp8_quantize(inp["dy"], M, M, rowwise=False, colwise=True)
    for k in ("q_col", "sf_col"):
        assert np.array_equal(u8(qx[k]), ox[k].reshape(-1)), k
        assert np.array_equal(u8(qd[k]), od[k].reshape(-1)), k
    rng = np.random.default_rng(7)
    ns = np.unique(np.concatenate([[0, 127, 128, N - 1], rng.integers(0, N, 60)]))
    ks = np.unique(np.concatenate([np.arange(0, 256), np.arange(K - 256, K), rng.integers(0, K, 256)]))
    _, _, ref = oracle.grouped_gemm_wgrad({"q": od["q_col"], "sf": od["sf_col"]},
                                          {"q": ox["q_col"], "sf": ox["sf_col"]}, offs, M, N, K,
                                          sample_n=ns, sample_k=ks)
    got = dW.cpu().numpy()
    sizes = inp["sizes"].numpy()
    for g in range(G):
        gg = got[g][np.ix_(ns, ks)].astype(np.float64)
        if sizes[g] == 0:
            assert not got[g].any()
        else:
            assert np.abs(gg - ref[g]).max() / np.abs(ref[g]).max() <= TOL, g
