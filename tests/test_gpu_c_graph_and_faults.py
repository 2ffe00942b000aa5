"""CUDA-graph safety and host-made failures.

* The whole path (offsets -> quantize -> GEMM) is captured once into a CUDA
  graph; new group sizes are written into the captured device buffer and the
  graph is replayed: results must follow the new routing with no host sync
  (the reason PR #2763 moves group sizes to device-side offsets).
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
    from gpu_util import tile_n
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
    with tile_n(tn):
        t0 = time.time()
        mxg.mxg_grouped_gemm_debug(mxg.MXG_MXFP8_E4M3, mxg.MXG_FPROP_TN, A, B, ws, G, R, N, K, C=C,
                                   dev_status=bad, inject_flags=1, wait_timeout_ns=20_000_000)
        torch.cuda.synchronize()
        assert time.time() - t0 < 10.0
        assert int(bad.item()) & mxg.MXG_DEV_TIMEOUT
        # the context is intact: a normal launch is correct
        mxg.mxg_grouped_gemm(mxg.MXG_MXFP8_E4M3, mxg.MXG_FPROP_TN, A, B, ws, G, R, N, K, C=C,
                             dev_status=st)
        torch.cuda.synchronize()
    assert int(st.item()) == 0
    _, _, offs, ref = _oracle_fprop(x_h, w_h, sizes.numpy(), G, N, K, R)
    errs = normwise_errors(C.cpu().numpy().astype(np.float64), ref, offs)
    assert errs.max() <= TOL
