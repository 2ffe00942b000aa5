"""GPU parity at the largest expert count the C ABI accepts (G = 1024): the
per-CTA group tables of the quantize and GEMM kernels are at their largest,
and almost every group is empty.  Aligned fprop on both K-stage widths of the
CTA-pair kernel, wgrad (every dW_g written: zeros for the empty groups), and
the unaligned quantize + fprop with 1024 groups of a few rows each."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import (DEV, fprop_case, normwise_errors, oracle_fprop, require_gpu, status_tensor,
                      u8)
from moe_grouped_block_gb300 import mxg, workloads

pytestmark = pytest.mark.gpu
TOL = 1e-3
G = 1024


@pytest.fixture(autouse=True)
def _gpu():
    require_gpu()


def _aligned_sizes(rows, live_groups, seed):
    """rows (a multiple of 128) over live_groups random experts, >= 128 each."""
    rng = np.random.default_rng(seed)
    units = rows // 128
    s = np.zeros(G, np.int64)
    live = rng.choice(G, size=live_groups, replace=False)
    s[live] = 128 * (1 + rng.multinomial(units - live_groups, np.full(live_groups, 1 / live_groups)))
    assert s.sum() == rows
    return tuple(int(v) for v in s)


@pytest.mark.parametrize("K", [256, 384])
def test_fprop_max_groups(K):
    # K = 256: 256-byte K stages; K = 384: 128-byte stages.  N = 128 also makes
    # every column unit half wide.
    wl = workloads.WORKLOADS["mixtral_fprop_mxfp8"].scaled(
        G=G, M=4096, K=K, N=128, sizes="fixed", fixed_sizes=_aligned_sizes(4096, 20, 91))
    case = fprop_case(wl, fill_c=7.0)
    assert int(case["status"].item()) == 0
    offs, rows, cols, ref, a, b = oracle_fprop(wl, case["inp"])
    got = case["C"].cpu().numpy().astype(np.float64)
    errs = normwise_errors(got[:wl.M], ref, offs)
    assert errs.max() <= TOL, errs


@pytest.mark.parametrize("fmt,K", [("mxfp8", 256), ("mxfp8", 384), ("nvfp4", 256),
                                   ("nvfp4", 384)])
def test_fprop_max_groups_bias(fmt, K):
    # The CTA-pair kernel's largest shared-memory layouts: 1024 groups' tables
    # beside every epilogue warp's staged bias (and, NVFP4, column outer
    # scales), on each stage variant (MXFP8 3 x 256 / 6 x 128 bytes of K,
    # NVFP4 5 x 128 / 10 x 64).
    base = "mixtral_fprop_mxfp8" if fmt == "mxfp8" else "rowscaled_fprop_nvfp4"
    wl = workloads.WORKLOADS[base].scaled(
        G=G, M=4096, K=K, N=256, sizes="fixed", fixed_sizes=_aligned_sizes(4096, 20, 93))
    rng = np.random.default_rng(94)
    bias = rng.standard_normal((G, wl.N)).astype(np.float32)
    alpha = (0.5 + rng.random(G)).astype(np.float32).tolist()
    case = fprop_case(wl, fill_c=7.0, bias=bias, alpha=alpha)
    assert int(case["status"].item()) == 0
    offs, rows, cols, ref, a, b = oracle_fprop(wl, case["inp"], alpha=alpha, bias=bias)
    got = case["C"].cpu().numpy().astype(np.float64)
    errs = normwise_errors(got[:wl.M], ref, offs)
    assert errs.max() <= TOL, errs


def test_wgrad_max_groups():
    wl = workloads.WORKLOADS["wgrad_mxfp8"].scaled(
        G=G, M=4096, K=256, N=128, sizes="fixed", fixed_sizes=_aligned_sizes(4096, 24, 92))
    inp = workloads.make_inputs(wl)
    N, K, M = wl.N, wl.K, wl.M
    from gpu_util import gpu_mxfp8, gpu_offsets
    ws, st = gpu_offsets(inp["sizes"], K, M)
    qx, _ = gpu_mxfp8(inp["x"].to(DEV), ws, G, mxg.MXG_COLWISE)
    qd, _ = gpu_mxfp8(inp["dy"].to(DEV), ws, G, mxg.MXG_COLWISE)
    dW = torch.full((G, N, K), 3.0, dtype=torch.float32, device=DEV)
    mxg.mxg_grouped_gemm(mxg.MXG_MXFP8_E4M3, mxg.MXG_WGRAD_NT, (qd["q_col"], qd["sf_col"], None),
                         (qx["q_col"], qx["sf_col"], None), ws, G, M, N, K, None, None, dW,
                         dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    rws, _ = oracle.group_offsets(inp["sizes"].numpy(), 1, K, M)
    offs = oracle.live_rows(rws, G)
    ox = oracle.mxfp8_quantize(inp["x"], M, M, rowwise=False, colwise=True)
    od = oracle.mxfp8_quantize(inp["dy"], M, M, rowwise=False, colwise=True)
    assert np.array_equal(qx["q_col"].cpu().numpy(), ox["q_col"])
    assert np.array_equal(qd["q_col"].cpu().numpy(), od["q_col"])
    _, _, ref = oracle.grouped_gemm_wgrad({"q": od["q_col"], "sf": od["sf_col"]},
                                          {"q": ox["q_col"], "sf": ox["sf_col"]}, offs, M, N, K)
    got = dW.cpu().numpy().astype(np.float64)
    sizes = np.asarray(wl.fixed_sizes)
    assert np.all(got[sizes == 0] == 0.0), "empty groups get dW_g = 0"
    for g in np.flatnonzero(sizes):
        den = max(np.abs(ref[g]).max(), 1e-30)
        assert np.abs(got[g] - ref[g]).max() / den <= TOL, g


def test_unaligned_max_groups():
    rng = np.random.default_rng(93)
    sizes = rng.integers(0, 13, G)
    sizes[rng.choice(G, 300, replace=False)] = 0
    N, K = 256, 256
    R = int(-(-sizes.sum() // 128) * 128)
    x = workloads.random_bf16((R, K), seed=94)
    w = workloads.random_bf16((G * N, K), seed=95, scale=0.02)
    t = torch.tensor(sizes, dtype=torch.int32)
    ws = mxg.alloc_offsets(G, DEV)
    st = status_tensor()
    mxg.mxg_group_offsets_unaligned(t.to(DEV), 1, K, R, ws, st)
    qa = mxg.alloc_mxfp8_unaligned(R, K, G, rowwise=True, colwise=True, device=DEV)
    for v in qa.values():
        v.fill_(0x5A)
    mxg.mxg_group_quantize_unaligned(mxg.MXG_BOTH, x.to(DEV), R, K, ws, G, qa["q_row"],
                                     qa["sf_row"], qa["q_col"], qa["sf_col"], st)
    qw = mxg.alloc_mxfp8(G * N, K, device=DEV)
    mxg.mxg_group_quantize(mxg.MXG_MXFP8_E4M3, mxg.MXG_ROWWISE, w.to(DEV), G * N, K, None, G,
                           qw["q_row"], qw["sf_row"])
    C = torch.full((R, N), 7.0, dtype=torch.float32, device=DEV)
    mxg.mxg_grouped_gemm_unaligned(mxg.MXG_FPROP_TN, (qa["q_row"], qa["sf_row"]),
                                   (qw["q_row"], qw["sf_row"]), ws, G, R, N, K, C=C,
                                   out_type=mxg.MXG_OUT_F32, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    wsn = ws.cpu().numpy()
    ref_q = oracle.mxfp8_quantize_unaligned(x, wsn, G, R, rowwise=True, colwise=True, fill=0x5A)
    for name in qa:
        assert np.array_equal(u8(qa[name]), ref_q[name].reshape(-1)), name
    a = {"q": qa["q_row"].cpu().numpy(), "sf": u8(qa["sf_row"])}
    b = {"q": qw["q_row"].cpu().numpy(), "sf": u8(qw["sf_row"])}
    rows, ref = oracle.grouped_gemm_fprop_unaligned(a, b, wsn, G, N, K)
    live = rows.size
    got = C.cpu().numpy().astype(np.float64)
    assert normwise_errors(got[:live], ref, oracle.live_rows(wsn, G)).max() <= TOL
    assert np.all(got[live:] == 7.0)
