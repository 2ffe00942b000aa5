"""GPU parity of the epilogue's accumulate-into-bf16 branch: bf16 output C
with a nonzero per-group beta and a nonzero bf16 C on input, for fprop,
dgrad and wgrad (TransformerEngine gemm.py grouped_gemm: per-group alpha /
beta; PR #3661: the FP32 result is copied or accumulated into the output).

The oracle computes alpha_g * (A . B^T) + beta_g * C_in in fp64 from its own
quantization of the inputs and C_in's bf16 values; the kernel's bf16 output
must equal that result rounded to bf16 within one bf16 ulp (the kernel rounds
its fp32 value once, which may land on the neighbouring bf16 value).  C
starts either 32-byte aligned (whole-sector stores) or 16 bytes into its
buffer (16-byte stores); nothing outside the written rows changes.
"""
import numpy as np
import pytest
import torch

import oracle
from moe_grouped_block_gb300 import mxg, workloads

from gpu_util import (DEV, fprop_case, gpu_mxfp8, gpu_offsets, oracle_fprop, require_gpu,
                      tile_n)

pytestmark = pytest.mark.gpu

BETAS = (0.0, 1.0, -1.0, 2.0)


@pytest.fixture(autouse=True)
def _gpu():
    require_gpu()


def _betas(G):
    return [BETAS[g % len(BETAS)] for g in range(G)]


def _bf16_close(got: np.ndarray, ref: np.ndarray, scale: float):
    """|got - bf16(ref)| within one bf16 ulp of bf16(ref), plus fp32
    accumulation slack relative to the magnitudes involved."""
    refb = torch.from_numpy(ref).to(torch.bfloat16).double().numpy()
    bound = np.abs(refb) * 2.0 ** -7 + 1e-5 * scale
    bad = np.abs(got - refb) > bound
    assert not bad.any(), "%d of %d outside one bf16 ulp; worst %.3g" % (
        bad.sum(), bad.size, np.max(np.abs(got - refb) - bound))


def _c_buffer(shape, c_in_bf16, c_offset):
    """A bf16 buffer holding c_in at element offset c_offset, with a
    sentinel in front; returns (buffer, view)."""
    n = int(np.prod(shape))
    buf = torch.full((c_offset + n,), 7.0, dtype=torch.bfloat16, device=DEV)
    view = buf[c_offset:].view(*shape)
    view.copy_(c_in_bf16.to(DEV))
    return buf, view


@pytest.mark.parametrize("tn", [None, 128])
@pytest.mark.parametrize("c_offset_bytes", [0, 16])
def test_fprop_beta_bf16_output(tn, c_offset_bytes):
    wl = workloads.WORKLOADS["mixtral_fprop_mxfp8"].scaled(M=1024, K=256, N=512, M_cap=1152)
    G, N, R = wl.G, wl.N, wl.rows_capacity
    c_in = workloads.random_bf16((R, N), seed=91)
    alpha = [0.5 + 0.25 * g for g in range(G)]
    beta = _betas(G)
    with tile_n(tn):
        case = fprop_case(wl, out_type=mxg.MXG_OUT_BF16, alpha=alpha, beta=beta, c_in=c_in,
                          fill_c=7.0, c_offset=c_offset_bytes // 2)
    assert int(case["status"].item()) == 0
    offs, rows, cols, ref, _, _ = oracle_fprop(wl, case["inp"], alpha=alpha, beta=beta,
                                               c_in=c_in.double().numpy())
    live = int(offs[-1])
    got = case["C"].cpu().double().numpy()
    scale = np.abs(ref).max() + np.abs(c_in.double().numpy()).max() * 2.0
    _bf16_close(got[:live], ref, scale)
    # capacity rows keep C_in; the prefix before C keeps the sentinel
    assert np.array_equal(got[live:], c_in.double().numpy()[live:])
    pre = case["C_buf"][:c_offset_bytes // 2].cpu().double().numpy()
    assert np.all(pre == 7.0)


@pytest.mark.parametrize("c_offset_bytes", [0, 16])
def test_dgrad_beta_bf16_output(c_offset_bytes):
    wl = workloads.WORKLOADS["finegrained_fprop_mxfp8"].scaled(M=2048, K=512, N=256, G=8)
    inp = workloads.make_inputs(wl)
    G, N, K, M = wl.G, wl.N, wl.K, wl.M
    dy_h = workloads.random_bf16((M, N), seed=92, scale=1e-3)
    ws, st = gpu_offsets(inp["sizes"], N, M)
    qd, _ = gpu_mxfp8(dy_h.to(DEV), ws, G, mxg.MXG_ROWWISE)
    w2 = inp["w"].reshape(G * N, K)
    qwt, _ = gpu_mxfp8(w2.to(DEV), None, G, mxg.MXG_COLWISE)
    c_in = workloads.random_bf16((M, K), seed=93, scale=1e-3)
    buf, dX = _c_buffer((M, K), c_in, c_offset_bytes // 2)
    alpha = [1.0, 0.5, 2.0, -1.0, 1.0, 1.0, 4.0, 0.25]
    beta = _betas(G)
    al = torch.tensor(alpha, dtype=torch.float32, device=DEV)
    be = torch.tensor(beta, dtype=torch.float32, device=DEV)
    mxg.mxg_grouped_gemm(mxg.MXG_MXFP8_E4M3, mxg.MXG_DGRAD_NN, (qd["q_row"], qd["sf_row"], None),
                         (qwt["q_col"], qwt["sf_col"], None), ws, G, M, N, K, al, be, dX,
                         out_type=mxg.MXG_OUT_BF16, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    rws, _ = oracle.group_offsets(inp["sizes"].numpy(), 1, N, M)
    offs = oracle.live_rows(rws, G)
    live = int(offs[-1])
    od = oracle.mxfp8_quantize(dy_h, M, M, rowwise=True)
    ow = oracle.mxfp8_quantize(w2, G * N, G * N, rowwise=False, colwise=True)
    _, _, ref = oracle.grouped_gemm_dgrad({"q": od["q_row"], "sf": od["sf_row"]},
                                          {"q": ow["q_col"], "sf": ow["sf_col"]}, offs, G, N, K,
                                          alpha=alpha, beta=beta, c_in=c_in.double().numpy())
    got = dX.cpu().double().numpy()
    scale = np.abs(ref).max() + np.abs(c_in.double().numpy()).max() * 2.0
    _bf16_close(got[:live], ref, scale)
    assert np.array_equal(got[live:], c_in.double().numpy()[live:])
    assert np.all(buf[:c_offset_bytes // 2].cpu().double().numpy() == 7.0)


@pytest.mark.parametrize("tn", [None, 128])
@pytest.mark.parametrize("c_offset_bytes", [0, 16])
def test_wgrad_beta_bf16_output(tn, c_offset_bytes):
    # one empty group: its dW is beta * C_in rounded to bf16
    wl = workloads.WORKLOADS["wgrad_mxfp8"].scaled(M=1024, K=256, N=384, sizes="fixed",
                                                     fixed_sizes=(256, 0, 384, 128, 0, 128, 128, 0))
    inp = workloads.make_inputs(wl)
    G, N, K, M = wl.G, wl.N, wl.K, wl.rows_capacity
    ws, st = gpu_offsets(inp["sizes"], K, M)
    qx, _ = gpu_mxfp8(inp["x"].to(DEV), ws, G, mxg.MXG_COLWISE)
    qd, _ = gpu_mxfp8(inp["dy"].to(DEV), ws, G, mxg.MXG_COLWISE)
    c_in = workloads.random_bf16((G, N, K), seed=94, scale=1e-3)
    buf, dW = _c_buffer((G, N, K), c_in, c_offset_bytes // 2)
    beta = _betas(G)
    alpha = [2.0 - 0.25 * g for g in range(G)]
    al = torch.tensor(alpha, dtype=torch.float32, device=DEV)
    be = torch.tensor(beta, dtype=torch.float32, device=DEV)
    with tile_n(tn):
        mxg.mxg_grouped_gemm(mxg.MXG_MXFP8_E4M3, mxg.MXG_WGRAD_NT,
                             (qd["q_col"], qd["sf_col"], None), (qx["q_col"], qx["sf_col"], None),
                             ws, G, M, N, K, al, be, dW, out_type=mxg.MXG_OUT_BF16,
                             dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    rws, _ = oracle.group_offsets(inp["sizes"].numpy(), 1, K, M)
    offs = oracle.live_rows(rws, G)
    live = int(offs[-1])
    ox = oracle.mxfp8_quantize(inp["x"], live, M, rowwise=False, colwise=True)
    od = oracle.mxfp8_quantize(inp["dy"], live, M, rowwise=False, colwise=True)
    _, _, ref = oracle.grouped_gemm_wgrad({"q": od["q_col"], "sf": od["sf_col"]},
                                          {"q": ox["q_col"], "sf": ox["sf_col"]}, offs, M, N, K,
                                          alpha=alpha, beta=beta, c_in=c_in.double().numpy())
    got = dW.cpu().double().numpy()
    for g in range(G):
        scale = np.abs(ref[g]).max() + np.abs(c_in[g].double().numpy()).max() * 2.0
        _bf16_close(got[g], ref[g], scale)
    assert np.all(buf[:c_offset_bytes // 2].cpu().double().numpy() == 7.0)
