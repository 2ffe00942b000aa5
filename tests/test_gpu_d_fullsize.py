"""GPU parity at the full workload sizes, in the launch configuration the
benchmark times (default tile choice, bf16 inputs resident on the device).

Quantized bytes, scales and offsets are compared in full, bit for bit.  GEMM
outputs are compared on samples the oracle computes one by one: for every
expert its first and last rows plus random rows, against a column sample that
covers the first and last output tiles (normwise error per expert <= 1e-3).
The fine-grained 64-expert workload is small enough to check in full.  Beside
the normwise gate each check reports the elementwise relative error over the
elements with |R| >= 1e-2 max|R| of their expert (with a loose bound of 1e-2;
shown with pytest -rP)."""
import numpy as np
import pytest
import torch

import oracle
from moe_grouped_block_gb300 import mxg, workloads

from gpu_util import (DEV, ELEM_BOUND, elementwise_error, elementwise_errors, fprop_case,
                      gpu_mxfp8, gpu_offsets, normwise_errors, report_errors, require_gpu, u8)

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
    elem = elementwise_errors(got, ref, offs, rows)
    report_errors(name, errs, elem)
    assert errs.max() <= TOL, errs
    assert elem.max() <= ELEM_BOUND, elem
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
    nw, el = [], []
    for g in range(G):
        gg = got[g][np.ix_(ns, ks)].astype(np.float64)
        if sizes[g] == 0:
            assert not got[g].any()
        else:
            nw.append(np.abs(gg - ref[g]).max() / np.abs(ref[g]).max())
            el.append(elementwise_error(gg, ref[g]))
    report_errors("wgrad_mxfp8", nw, el)
    assert max(nw) <= TOL, nw
    assert max(el) <= ELEM_BOUND, el


def test_dgrad_fullsize():
    """dX = dY . W_g at the dgrad workload's full size: rowwise dY, colwise
    (transposed) copy of W, both bit-exact; dX sampled."""
    wl = workloads.WORKLOADS["dgrad_mxfp8"]
    inp = workloads.make_inputs(wl)
    G, N, K, M = wl.G, wl.N, wl.K, wl.M
    ws, st = gpu_offsets(inp["sizes"], N, M)
    qd, _ = gpu_mxfp8(inp["dy"].to(DEV), ws, G, mxg.MXG_ROWWISE)
    w2 = inp["w"].reshape(G * N, K)
    qwt, _ = gpu_mxfp8(w2.to(DEV), None, G, mxg.MXG_COLWISE)
    dX = torch.empty((M, K), dtype=torch.float32, device=DEV)
    mxg.mxg_grouped_gemm(mxg.MXG_MXFP8_E4M3, mxg.MXG_DGRAD_NN, (qd["q_row"], qd["sf_row"], None),
                         (qwt["q_col"], qwt["sf_col"], None), ws, G, M, N, K, C=dX, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    rws, _ = oracle.group_offsets(inp["sizes"].numpy(), 1, N, M)
    offs = oracle.live_rows(rws, G)
    od = oracle.mxfp8_quantize(inp["dy"], M, M, rowwise=True)
    ow = oracle.mxfp8_quantize(w2, G * N, G * N, rowwise=False, colwise=True)
    for k in ("q_row", "sf_row"):
        assert np.array_equal(u8(qd[k]), od[k].reshape(-1)), k
    for k in ("q_col", "sf_col"):
        assert np.array_equal(u8(qwt[k]), ow[k].reshape(-1)), k
    rows, cols = _sample(offs, K, np.random.default_rng(8))
    _, _, ref = oracle.grouped_gemm_dgrad({"q": od["q_row"], "sf": od["sf_row"]},
                                          {"q": ow["q_col"], "sf": ow["sf_col"]}, offs, G, N, K,
                                          sample_rows=rows, sample_cols=cols)
    got = dX.cpu().numpy()[np.ix_(rows, cols)].astype(np.float64)
    errs, elem = normwise_errors(got, ref, offs, rows), elementwise_errors(got, ref, offs, rows)
    report_errors("dgrad_mxfp8", errs, elem)
    assert errs.max() <= TOL
    assert elem.max() <= ELEM_BOUND


def test_nvfp4_wgrad_fullsize():
    """Row-scaled NVFP4 wgrad at the full wgrad size: colwise NVFP4 copies of
    X and dY with per-(group, column) outer scales, bit-exact; dW sampled."""
    wl = workloads.WORKLOADS["wgrad_nvfp4"]
    inp = workloads.make_inputs(wl)
    G, N, K, M = wl.G, wl.N, wl.K, wl.M
    sizes = inp["sizes"].numpy()
    ws, st = gpu_offsets(inp["sizes"], K, M)
    qx = mxg.alloc_nvfp4(M, K, device=DEV, rowwise=False, colwise=True, G=G)
    qd = mxg.alloc_nvfp4(M, N, device=DEV, rowwise=False, colwise=True, G=G)
    for q, t, C in ((qx, inp["x"], K), (qd, inp["dy"], N)):
        mxg.mxg_group_quantize(mxg.MXG_NVFP4_ROWSCALED, mxg.MXG_COLWISE, t.to(DEV), M, C, ws, G,
                               None, None, q["q_col"], q["sf_col"], None, st,
                               outer_col=q["outer_col"])
    dW = torch.empty((G, N, K), dtype=torch.float32, device=DEV)
    mxg.mxg_grouped_gemm(mxg.MXG_NVFP4_ROWSCALED, mxg.MXG_WGRAD_NT,
                         (qd["q_col"], qd["sf_col"], qd["outer_col"]),
                         (qx["q_col"], qx["sf_col"], qx["outer_col"]), ws, G, M, N, K, C=dW,
                         dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    offs = np.concatenate([[0], np.cumsum(sizes)])
    ox = oracle.nvfp4_quantize_colwise(inp["x"], offs, M)
    od = oracle.nvfp4_quantize_colwise(inp["dy"], offs, M)
    for k in ("q_col", "sf_col", "outer_col"):
        assert np.array_equal(qx[k].cpu().numpy().reshape(-1), ox[k].reshape(-1)), k
        assert np.array_equal(qd[k].cpu().numpy().reshape(-1), od[k].reshape(-1)), k
    rng = np.random.default_rng(9)
    ns = np.unique(np.concatenate([[0, 127, 128, N - 1], rng.integers(0, N, 60)]))
    ks = np.unique(np.concatenate([np.arange(0, 256), np.arange(K - 256, K), rng.integers(0, K, 256)]))
    _, _, ref = oracle.grouped_gemm_wgrad(
        {"q": od["q_col"], "sf": od["sf_col"], "outer": od["outer_col"]},
        {"q": ox["q_col"], "sf": ox["sf_col"], "outer": ox["outer_col"]}, offs, M, N, K,
        sample_n=ns, sample_k=ks, fmt="nvfp4")
    got = dW.cpu().numpy()
    nw, el = [], []
    for g in range(G):
        gg = got[g][np.ix_(ns, ks)].astype(np.float64)
        if sizes[g] == 0:
            assert not got[g].any()
        else:
            nw.append(np.abs(gg - ref[g]).max() / np.abs(ref[g]).max())
            el.append(elementwise_error(gg, ref[g]))
    report_errors("wgrad_nvfp4", nw, el)
    assert max(nw) <= TOL, nw
    assert max(el) <= ELEM_BOUND, el


def test_unaligned_fprop_fullsize():
    """Groups of any size at the Mixtral shape: unaligned offsets and padded
    quantize bit-exact in full, the GEMM sampled (first / last rows of every
    group, so each group boundary inside a 128-row tile is checked)."""
    wl = workloads.WORKLOADS["mixtral_fprop_mxfp8_unaligned"]
    inp = workloads.make_inputs(wl)
    G, N, K, R = wl.G, wl.N, wl.K, wl.rows_capacity
    sizes = inp["sizes"]
    assert (sizes.numpy() % 128 != 0).any()
    ws = mxg.alloc_offsets(G, DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    mxg.mxg_group_offsets_unaligned(sizes.to(DEV), 1, K, R, ws, st)
    qx = mxg.alloc_mxfp8_unaligned(R, K, G, rowwise=True, colwise=True, device=DEV)
    mxg.mxg_group_quantize_unaligned(mxg.MXG_BOTH, inp["x"].to(DEV), R, K, ws, G, qx["q_row"],
                                     qx["sf_row"], qx["q_col"], qx["sf_col"], st)
    w2 = inp["w"].reshape(G * N, K)
    qw, _ = gpu_mxfp8(w2.to(DEV), None, G, mxg.MXG_ROWWISE)
    C = torch.empty((R, N), dtype=torch.float32, device=DEV)
    mxg.mxg_grouped_gemm_unaligned(mxg.MXG_FPROP_TN, (qx["q_row"], qx["sf_row"]),
                                   (qw["q_row"], qw["sf_row"]), ws, G, R, N, K, C=C, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    wsn, _ = oracle.group_offsets_unaligned(sizes.numpy(), 1, K, R)
    assert np.array_equal(ws.cpu().numpy(), wsn)
    ox = oracle.mxfp8_quantize_unaligned(inp["x"], wsn, G, R, rowwise=True, colwise=True)
    for k in ("q_row", "sf_row", "q_col", "sf_col"):
        got_k = u8(qx[k])
        if k == "q_row":  # rows past the live count are untouched
            n = int(wsn[:G].sum()) * K
            assert np.array_equal(got_k[:n], ox[k].reshape(-1)[:n]), k
        else:
            Rp = oracle.unaligned_rows_capacity(R, G)
            used = int(oracle.padded_rows(wsn, G)[-1])
            if k == "sf_row":  # scale bands of the padded groups
                assert np.array_equal(got_k[:used * K // 32], ox[k][:used * K // 32]), k
            elif k == "q_col":
                assert np.array_equal(qx[k].cpu().numpy()[:, :used], ox[k][:, :used]), k
            else:
                gu = oracle.unswizzle(got_k, K, Rp // 32)[:, :used // 32]
                ou = oracle.unswizzle(ox[k], K, Rp // 32)[:, :used // 32]
                assert np.array_equal(gu, ou), k
    ow = oracle.mxfp8_quantize(w2, G * N, G * N)
    offs = oracle.live_rows(wsn, G)
    rows, cols = _sample(offs, N, np.random.default_rng(10))
    _, ref = oracle.grouped_gemm_fprop_unaligned({"q": ox["q_row"], "sf": ox["sf_row"]},
                                                 {"q": ow["q_row"], "sf": ow["sf_row"]}, wsn, G,
                                                 N, K, sample_rows=rows, sample_cols=cols)
    got = C.cpu().numpy()[np.ix_(rows, cols)].astype(np.float64)
    errs, elem = normwise_errors(got, ref, offs, rows), elementwise_errors(got, ref, offs, rows)
    report_errors("mixtral_fprop_mxfp8_unaligned", errs, elem)
    assert errs.max() <= TOL
    assert elem.max() <= ELEM_BOUND
