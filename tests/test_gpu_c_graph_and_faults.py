"""CUDA-graph safety and host-made failures.

* The whole path (offsets -> quantize -> GEMM) is captured once into a CUDA
  graph; new group sizes are written into the captured device buffer and the
  graph is replayed: results must follow the new routing with no host sync
  (the reason PR #2763 moves group sizes to device-side offsets).  Likewise
  for groups of any size, dgrad and row-scaled NVFP4 wgrad.
* Bad group sizes made on the host (negative, not a multiple of 128, summing
  past the capacity) set the sticky status bits and are clamped exactly as
  the oracle's sanitisation defines; nothing outside the buffers is touched.
"""
import numpy as np
import pytest
import torch

import oracle
from moe_grouped_block_gb300 import mxg, workloads

from gpu_util import DEV, gpu_offsets, normwise_errors, require_gpu, u8

pytestmark = pytest.mark.gpu
TOL = 1e-3


@pytest.fixture(autouse=True)
def _gpu():
    require_gpu()


def _oracle_fprop(x, w, sizes, G, N, K, R):
    ws, st = oracle.group_offsets(sizes, 1, K, R)
    offs = oracle.live_rows(ws, G)
    ox = oracle.mxfp8_quantize(x, int(offs[-1]), R)
    ow = oracle.mxfp8_quantize(w, G * N, G * N)
    _, _, ref = oracle.grouped_gemm_fprop("mxfp8", {"q": ox["q_row"], "sf": ox["sf_row"]},
                                          {"q": ow["q_row"], "sf": ow["sf_row"]}, offs, N, K)
    return ws, st, offs, ref


def test_graph_capture_replay_with_new_routing():
    G, N, K, R = 8, 256, 512, 2048
    x_h = workloads.random_bf16((R, K), seed=31)
    w_h = workloads.random_bf16((G * N, K), seed=32, scale=0.02)
    x, w = x_h.to(DEV), w_h.to(DEV)
    sizes = torch.zeros(G, dtype=torch.int32, device=DEV)
    ws = mxg.alloc_offsets(G, DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    qx = mxg.alloc_mxfp8(R, K, rowwise=True, colwise=True, device=DEV)
    qw = mxg.alloc_mxfp8(G * N, K, device=DEV)
    C = torch.zeros((R, N), dtype=torch.float32, device=DEV)

    def path():
        mxg.mxg_group_offsets(sizes, 1, K, R, ws, st)
        mxg.mxg_group_quantize(mxg.MXG_MXFP8_E4M3, mxg.MXG_BOTH, x, R, K, ws, G, qx["q_row"],
                               qx["sf_row"], qx["q_col"], qx["sf_col"], None, st)
        mxg.mxg_group_quantize(mxg.MXG_MXFP8_E4M3, mxg.MXG_ROWWISE, w, G * N, K, None, G,
                               qw["q_row"], qw["sf_row"], None, None, None, st)
        mxg.mxg_grouped_gemm(mxg.MXG_MXFP8_E4M3, mxg.MXG_FPROP_TN, (qx["q_row"], qx["sf_row"], None),
                             (qw["q_row"], qw["sf_row"], None), ws, G, R, N, K, C=C, dev_status=st)

    sizes.copy_(torch.tensor([256] * 8, dtype=torch.int32))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        path()  # eager warm-up on the capture stream
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        path()
    for routing in ([256] * 8, [0, 512, 128, 0, 896, 128, 256, 128], [2048, 0, 0, 0, 0, 0, 0, 0],
                    [128, 128, 0, 0, 0, 0, 0, 0]):
        C.fill_(-1.0)
        sizes.copy_(torch.tensor(routing, dtype=torch.int32))
        g.replay()
        torch.cuda.synchronize()
        rws, rst, offs, ref = _oracle_fprop(x_h, w_h, np.array(routing), G, N, K, R)
        assert np.array_equal(ws.cpu().numpy(), rws)
        live = int(offs[-1])
        got = C.cpu().numpy().astype(np.float64)
        errs = normwise_errors(got[:live], ref, offs)
        assert errs.max() <= TOL, (routing, errs)
        assert np.all(got[live:] == -1.0), "rows past the live count were written"
    assert int(st.item()) == 0


def _capture(path):
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        path()  # eager warm-up on the capture stream
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        path()
    return g


def test_graph_replay_unaligned_groups():
    """Groups of any size: offsets, the per-group padded quantize and the
    GEMM captured once, replayed under new routings of any sizes."""
    G, N, K, R = 4, 256, 256, 1024
    x_h = workloads.random_bf16((R, K), seed=33)
    w_h = workloads.random_bf16((G * N, K), seed=34, scale=0.02)
    x, w = x_h.to(DEV), w_h.to(DEV)
    sizes = torch.zeros(G, dtype=torch.int32, device=DEV)
    ws = mxg.alloc_offsets(G, DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    qx = mxg.alloc_mxfp8_unaligned(R, K, G, device=DEV)
    qw = mxg.alloc_mxfp8(G * N, K, device=DEV)
    mxg.mxg_group_quantize(mxg.MXG_MXFP8_E4M3, mxg.MXG_ROWWISE, w, G * N, K, None, G, qw["q_row"],
                           qw["sf_row"], None, None, None, st)
    C = torch.zeros((R, N), dtype=torch.float32, device=DEV)

    def path():
        mxg.mxg_group_offsets_unaligned(sizes, 1, K, R, ws, st)
        mxg.mxg_group_quantize_unaligned(mxg.MXG_ROWWISE, x, R, K, ws, G, qx["q_row"],
                                         qx["sf_row"], None, None, st)
        mxg.mxg_grouped_gemm_unaligned(mxg.MXG_FPROP_TN, (qx["q_row"], qx["sf_row"]),
                                       (qw["q_row"], qw["sf_row"]), ws, G, R, N, K, C=C,
                                       dev_status=st)

    sizes.copy_(torch.tensor([100, 200, 300, 400], dtype=torch.int32))
    g = _capture(path)
    ow = oracle.mxfp8_quantize(w_h, G * N, G * N)
    for routing in ([100, 200, 300, 400], [1, 0, 1000, 23], [0, 0, 0, 1024], [129, 127, 5, 0]):
        C.fill_(-1.0)
        sizes.copy_(torch.tensor(routing, dtype=torch.int32))
        g.replay()
        torch.cuda.synchronize()
        wsn, _ = oracle.group_offsets_unaligned(np.array(routing), 1, K, R)
        assert np.array_equal(ws.cpu().numpy(), wsn)
        ox = oracle.mxfp8_quantize_unaligned(x_h, wsn, G, R, rowwise=True)
        rows, ref = oracle.grouped_gemm_fprop_unaligned({"q": ox["q_row"], "sf": ox["sf_row"]},
                                                        {"q": ow["q_row"], "sf": ow["sf_row"]},
                                                        wsn, G, N, K)
        got = C.cpu().numpy().astype(np.float64)
        live = rows.size
        assert normwise_errors(got[:live], ref, oracle.live_rows(wsn, G)).max() <= TOL, routing
        assert np.all(got[live:] == -1.0)
    assert int(st.item()) == 0


def test_graph_replay_backward_paths():
    """dgrad (rowwise dY, colwise W) and row-scaled NVFP4 wgrad (colwise
    copies with per-(group, column) outer scales) captured once and replayed
    under a new routing."""
    G, N, K, R = 4, 256, 256, 1024
    dy_h = workloads.random_bf16((R, N), seed=35, scale=1e-3)
    x_h = workloads.random_bf16((R, K), seed=36)
    w_h = workloads.random_bf16((G * N, K), seed=37, scale=0.02)
    dy, x, w = dy_h.to(DEV), x_h.to(DEV), w_h.to(DEV)
    sizes = torch.zeros(G, dtype=torch.int32, device=DEV)
    ws_n, ws_k = mxg.alloc_offsets(G, DEV), mxg.alloc_offsets(G, DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    qd = mxg.alloc_mxfp8(R, N, device=DEV)
    qwt = mxg.alloc_mxfp8(G * N, K, rowwise=False, colwise=True, device=DEV)
    nx = mxg.alloc_nvfp4(R, K, device=DEV, rowwise=False, colwise=True, G=G)
    nd = mxg.alloc_nvfp4(R, N, device=DEV, rowwise=False, colwise=True, G=G)
    dX = torch.zeros((R, K), dtype=torch.float32, device=DEV)
    dW = torch.zeros((G, N, K), dtype=torch.float32, device=DEV)

    def path():
        mxg.mxg_group_offsets(sizes, 1, N, R, ws_n, st)
        mxg.mxg_group_quantize(mxg.MXG_MXFP8_E4M3, mxg.MXG_ROWWISE, dy, R, N, ws_n, G, qd["q_row"],
                               qd["sf_row"], None, None, None, st)
        mxg.mxg_group_quantize(mxg.MXG_MXFP8_E4M3, mxg.MXG_COLWISE, w, G * N, K, None, G, None,
                               None, qwt["q_col"], qwt["sf_col"], None, st)
        mxg.mxg_grouped_gemm(mxg.MXG_MXFP8_E4M3, mxg.MXG_DGRAD_NN, (qd["q_row"], qd["sf_row"], None),
                             (qwt["q_col"], qwt["sf_col"], None), ws_n, G, R, N, K, C=dX,
                             dev_status=st)
        mxg.mxg_group_offsets(sizes, 1, K, R, ws_k, st)
        for q, t, C_ in ((nx, x, K), (nd, dy, N)):
            mxg.mxg_group_quantize(mxg.MXG_NVFP4_ROWSCALED, mxg.MXG_COLWISE, t, R, C_, ws_k, G,
                                   None, None, q["q_col"], q["sf_col"], None, st,
                                   outer_col=q["outer_col"])
        mxg.mxg_grouped_gemm(mxg.MXG_NVFP4_ROWSCALED, mxg.MXG_WGRAD_NT,
                             (nd["q_col"], nd["sf_col"], nd["outer_col"]),
                             (nx["q_col"], nx["sf_col"], nx["outer_col"]), ws_k, G, R, N, K, C=dW,
                             dev_status=st)

    sizes.copy_(torch.tensor([256, 256, 256, 256], dtype=torch.int32))
    g = _capture(path)
    ow = oracle.mxfp8_quantize(w_h, G * N, G * N, rowwise=False, colwise=True)
    for routing in ([256, 256, 256, 256], [128, 0, 640, 256]):
        dX.fill_(-1.0)
        sizes.copy_(torch.tensor(routing, dtype=torch.int32))
        g.replay()
        torch.cuda.synchronize()
        rws, _ = oracle.group_offsets(np.array(routing), 1, N, R)
        offs = oracle.live_rows(rws, G)
        live = int(offs[-1])
        od = oracle.mxfp8_quantize(dy_h, live, R, rowwise=True)
        _, _, ref = oracle.grouped_gemm_dgrad({"q": od["q_row"], "sf": od["sf_row"]},
                                              {"q": ow["q_col"], "sf": ow["sf_col"]}, offs, G, N, K)
        got = dX.cpu().numpy().astype(np.float64)
        assert normwise_errors(got[:live], ref, offs).max() <= TOL, routing
        assert np.all(got[live:] == -1.0)
        ox = oracle.nvfp4_quantize_colwise(x_h, offs, R)
        odc = oracle.nvfp4_quantize_colwise(dy_h, offs, R)
        _, _, refw = oracle.grouped_gemm_wgrad(
            {"q": odc["q_col"], "sf": odc["sf_col"], "outer": odc["outer_col"]},
            {"q": ox["q_col"], "sf": ox["sf_col"], "outer": ox["outer_col"]}, offs, R, N, K,
            fmt="nvfp4")
        gw = dW.cpu().numpy().astype(np.float64)
        for gi in range(G):
            if routing[gi] == 0:
                assert not gw[gi].any()
            else:
                assert np.abs(gw[gi] - refw[gi]).max() / np.abs(refw[gi]).max() <= TOL, (routing, gi)
    assert int(st.item()) == 0


@pytest.mark.parametrize("routing,bits", [
    ([256, -128, 384, 256], mxg.MXG_DEV_NEG_SIZE),
    ([256, 100, 384, 256], mxg.MXG_DEV_MISALIGNED),
    ([512, 512, 512, 512], mxg.MXG_DEV_SUM_OVER_CAPACITY),
    ([-5, 1000, 1024, 64], mxg.MXG_DEV_NEG_SIZE | mxg.MXG_DEV_MISALIGNED |
     mxg.MXG_DEV_SUM_OVER_CAPACITY),
])
def test_bad_group_sizes_are_flagged_and_clamped(routing, bits):
    G, N, K, R = 4, 256, 256, 1024
    x_h = workloads.random_bf16((R, K), seed=41)
    w_h = workloads.random_bf16((G * N, K), seed=42, scale=0.02)
    sizes = torch.tensor(routing, dtype=torch.int32)
    ws, st = gpu_offsets(sizes, K, R)
    qx = mxg.alloc_mxfp8(R, K, rowwise=True, colwise=True, device=DEV)
    for t in qx.values():
        t.fill_(0x77)
    qw = mxg.alloc_mxfp8(G * N, K, device=DEV)
    guard = torch.full((R + 128, N), 5.0, device=DEV)  # one extra band of guard rows
    C = guard[:R]
    mxg.mxg_group_quantize(mxg.MXG_MXFP8_E4M3, mxg.MXG_BOTH, x_h.to(DEV), R, K, ws, G, qx["q_row"],
                           qx["sf_row"], qx["q_col"], qx["sf_col"], None, st)
    mxg.mxg_group_quantize(mxg.MXG_MXFP8_E4M3, mxg.MXG_ROWWISE, w_h.to(DEV), G * N, K, None, G,
                           qw["q_row"], qw["sf_row"], None, None, None, st)
    mxg.mxg_grouped_gemm(mxg.MXG_MXFP8_E4M3, mxg.MXG_FPROP_TN, (qx["q_row"], qx["sf_row"], None),
                         (qw["q_row"], qw["sf_row"], None), ws, G, R, N, K, C=C, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == bits
    rws, rst, offs, ref = _oracle_fprop(x_h, w_h, np.array(routing), G, N, K, R)
    assert rst == bits and np.array_equal(ws.cpu().numpy(), rws)
    live = int(offs[-1])
    got = guard.cpu().numpy().astype(np.float64)
    errs = normwise_errors(got[:live], ref, offs)
    assert errs.max() <= TOL
    assert np.all(got[live:] == 5.0)
    assert np.all(qx["q_row"][live:].cpu().numpy() == 0x77)


@pytest.mark.parametrize("tn", [None, 256, 128])
def test_bounded_wait_runs_out_and_the_device_stays_usable(tn):
    """A flag that nothing sets: CTA 0 withholds its first accumulator-ready
    arrival, so its epilogue's wait runs out after 20 ms.  The launch must
    report MXG_DEV_TIMEOUT, drain, free tensor memory and return; the next
    normal launch on the same context must be correct."""
    import time
    G, N, K, R = 4, 256, 256, 1024
    x_h = workloads.random_bf16((R, K), seed=51)
    w_h = workloads.random_bf16((G * N, K), seed=52, scale=0.02)
    sizes = torch.tensor([256, 256, 256, 256], dtype=torch.int32)
    ws, st = gpu_offsets(sizes, K, R)
    qx = mxg.alloc_mxfp8(R, K, device=DEV)
    qw = mxg.alloc_mxfp8(G * N, K, device=DEV)
    mxg.mxg_group_quantize(mxg.MXG_MXFP8_E4M3, mxg.MXG_ROWWISE, x_h.to(DEV), R, K, ws, G,
                           qx["q_row"], qx["sf_row"], None, None, None, st)
    mxg.mxg_group_quantize(mxg.MXG_MXFP8_E4M3, mxg.MXG_ROWWISE, w_h.to(DEV), G * N, K, None, G,
                           qw["q_row"], qw["sf_row"], None, None, None, st)
    A = (qx["q_row"], qx["sf_row"], None)
    B = (qw["q_row"], qw["sf_row"], None)
    C = torch.zeros((R, N), dtype=torch.float32, device=DEV)
    bad = torch.zeros(1, dtype=torch.int32, device=DEV)
    t0 = time.time()
    mxg.mxg_grouped_gemm_debug(mxg.MXG_MXFP8_E4M3, mxg.MXG_FPROP_TN, A, B, ws, G, R, N, K, C=C,
                               dev_status=bad, tile_n=tn or 0, inject_flags=1,
                               wait_timeout_ns=20_000_000)
    torch.cuda.synchronize()
    assert time.time() - t0 < 10.0
    assert int(bad.item()) & mxg.MXG_DEV_TIMEOUT
    # the context is intact: a normal launch is correct
    mxg.mxg_grouped_gemm_debug(mxg.MXG_MXFP8_E4M3, mxg.MXG_FPROP_TN, A, B, ws, G, R, N, K, C=C,
                               dev_status=st, tile_n=tn or 0)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    _, _, offs, ref = _oracle_fprop(x_h, w_h, sizes.numpy(), G, N, K, R)
    errs = normwise_errors(C.cpu().numpy().astype(np.float64), ref, offs)
    assert errs.max() <= TOL
