"""GPU parity: the grouped block-scaled GEMM through the C ABI against the
oracle's fp64 per-expert GEMM over the oracle's own quantized operands.

Tolerance: max |C - R| / max |R| <= 1e-3 per expert (the normwise reading of
"max relative error 1e-3"); FP32 accumulation over K <= 4096 products of
exactly-representable values sits near 1e-6, so 1e-3 leaves the margin the
statement allows.  bf16 output is compared with the oracle rounded to bf16,
within one bf16 ulp.  The quantized operands are also checked bit-exact
against the oracle here, so a GEMM failure is never a quantize failure."""
import numpy as np
import pytest
import torch

import oracle
from moe_grouped_block_gb300 import mxg, workloads

from gpu_util import (DEV, fprop_case, gpu_mxfp8, gpu_offsets, normwise_errors, oracle_fprop,
                      oracle_quantized_operands, require_gpu, status_tensor, tile_n, u8,
                      gemm_override)

pytestmark = pytest.mark.gpu
TOL = 1e-3


@pytest.fixture(autouse=True)
def _gpu():
    require_gpu()


def _assert_operands_match(case, a, b, live):
    assert np.array_equal(case["qx"]["q_row"][:live].cpu().numpy(), a["q"][:live])
    assert np.array_equal(case["qw"]["q_row"].cpu().numpy(), b["q"])
    assert np.array_equal(u8(case["qw"]["sf_row"]), b["sf"])


def _run_fprop(wl, tn=None, **kw):
    with tile_n(tn):
        case = fprop_case(wl, **kw)
    offs, rows, cols, ref, a, b = oracle_fprop(wl, case["inp"], alpha=kw.get("alpha"),
                                               beta=kw.get("beta"), bias=kw.get("bias"),
                                               c_in=None if kw.get("c_in") is None else
                                               kw["c_in"].double().numpy())
    _assert_operands_match(case, a, b, int(offs[-1]))
    assert int(case["status"].item()) == 0
    return case, offs, rows, ref


def test_single_tile_one_hot():
    # one expert, one 128x128 tile, one K block: C[m, n] = W[n, m] exactly
    G, N, K, M = 1, 128, 128, 128
    xf = torch.zeros((M, K))
    xf[torch.arange(M), torch.arange(M)] = 1.0
    wl = workloads.Workload("one_hot", "fprop", "mxfp8", G, K, N, M, 0, "fixed", (M,))
    w = torch.randint(-8, 9, (G, N, K)).float()
    inp = {"x": xf.to(torch.bfloat16), "w": w.to(torch.bfloat16),
           "sizes": torch.tensor([M], dtype=torch.int32)}
    x = inp["x"].to(DEV)
    ws, st = gpu_offsets(inp["sizes"], K, M)
    qx, _ = gpu_mxfp8(x, ws, G, mxg.MXG_ROWWISE)
    qw, _ = gpu_mxfp8(inp["w"].to(DEV).reshape(N, K), None, 1, mxg.MXG_ROWWISE)
    C = torch.full((M, N), 7.0, device=DEV)
    mxg.mxg_grouped_gemm(mxg.MXG_MXFP8_E4M3, mxg.MXG_FPROP_TN, (qx["q_row"], qx["sf_row"], None),
                         (qw["q_row"], qw["sf_row"], None), ws, G, M, N, K, C=C, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(C.cpu(), w[0].t().contiguous())


def test_pair_unit_upper_half_past_end():
    # one expert of 128 rows, N = 256: the CTA-pair kernel's odd CTA reads rows
    # 128..255, past the end of A (zero fill), and must store nothing
    G, N, K, M = 1, 256, 256, 128
    xf = torch.zeros((M, K))
    xf[torch.arange(M), torch.arange(M) + 64] = 1.0
    w = torch.randint(-8, 9, (G, N, K)).float()
    sizes = torch.tensor([M], dtype=torch.int32)
    ws, st = gpu_offsets(sizes, K, M)
    qx, _ = gpu_mxfp8(xf.to(torch.bfloat16).to(DEV), ws, G, mxg.MXG_ROWWISE)
    qw, _ = gpu_mxfp8(w.to(torch.bfloat16).to(DEV).reshape(N, K), None, 1, mxg.MXG_ROWWISE)
    C = torch.full((M, N), 7.0, device=DEV)
    mxg.mxg_grouped_gemm(mxg.MXG_MXFP8_E4M3, mxg.MXG_FPROP_TN, (qx["q_row"], qx["sf_row"], None),
                         (qw["q_row"], qw["sf_row"], None), ws, G, M, N, K, C=C, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(C.cpu(), w[0][:, 64:64 + M].t().contiguous())


@pytest.mark.parametrize("tn", [None, 256, 128])
def test_fprop_tiny_workload(tn):
    wl = workloads.WORKLOADS["tiny_fprop_mxfp8"]
    case, offs, rows, ref = _run_fprop(wl, tn)
    got = case["C"].cpu().numpy().astype(np.float64)
    errs = normwise_errors(got[:wl.M], ref, offs)
    assert errs.max() <= TOL, errs


@pytest.mark.parametrize("tn", [None, 256, 128])
def test_fprop_mixtral_shape_scaled(tn):
    wl = workloads.WORKLOADS["mixtral_fprop_mxfp8"].scaled(M=2048, K=512, N=512)
    case, offs, rows, ref = _run_fprop(wl, tn)
    errs = normwise_errors(case["C"].cpu().numpy().astype(np.float64)[:wl.M], ref, offs)
    assert errs.max() <= TOL, errs


def test_fprop_finegrained_empty_groups():
    wl = workloads.WORKLOADS["finegrained_fprop_mxfp8"].scaled(M=4096, K=256)
    inp_sizes = workloads.group_sizes(wl)
    assert (inp_sizes == 0).any()
    case, offs, rows, ref = _run_fprop(wl)
    errs = normwise_errors(case["C"].cpu().numpy().astype(np.float64)[:wl.M], ref, offs)
    assert errs.max() <= TOL, errs


def test_fprop_alpha_beta_and_capacity_padding():
    wl = workloads.WORKLOADS["tiny_fprop_mxfp8"].scaled(M_cap=768)
    G, N = wl.G, wl.N
    c_in = torch.linspace(-1, 1, 768 * N).reshape(768, N).float()
    alpha = [1.0, 3.0, -0.5, 0.125]
    beta = [0.0, 1.0, 2.0, -1.0]
    case, offs, rows, ref = _run_fprop(wl, alpha=alpha, beta=beta, c_in=c_in)
    got = case["C"].cpu().numpy().astype(np.float64)
    errs = normwise_errors(got[:wl.M], ref, offs)
    assert errs.max() <= TOL, errs
    # rows beyond the live count keep their previous contents
    assert np.array_equal(got[wl.M:], c_in.numpy()[wl.M:].astype(np.float64))


@pytest.mark.parametrize("tn", [None, 256, 128])
def test_fprop_per_group_bias(tn):
    wl = workloads.WORKLOADS["mixtral_fprop_mxfp8"].scaled(M=1024, K=256, N=512)
    bias = np.random.default_rng(3).standard_normal((wl.G, wl.N)).astype(np.float32)
    case, offs, rows, ref = _run_fprop(wl, tn, bias=bias, alpha=[0.5] * wl.G)
    errs = normwise_errors(case["C"].cpu().numpy().astype(np.float64)[:wl.M], ref, offs)
    assert errs.max() <= TOL, errs


@pytest.mark.parametrize("tn", [None, 256, 128])
def test_fprop_bf16_output(tn):
    wl = workloads.WORKLOADS["mixtral_fprop_mxfp8"].scaled(M=1024, K=256, N=512)
    case, offs, rows, ref = _run_fprop(wl, tn, out_type=mxg.MXG_OUT_BF16)
    got = case["C"].cpu().float().numpy().astype(np.float64)[:wl.M]
    refb = torch.from_numpy(ref).to(torch.bfloat16).double().numpy()
    ulp = np.abs(refb) * 2.0 ** -7 + 1e-30
    assert np.all(np.abs(got - refb) <= ulp + 1e-6 * np.abs(ref).max())


@pytest.mark.parametrize("out_type", [mxg.MXG_OUT_F32, mxg.MXG_OUT_BF16])
@pytest.mark.parametrize("c_offset_bytes", [0, 16])
def test_fprop_stores_stay_in_bounds(out_type, c_offset_bytes):
    # C starts 16 (not 32) bytes into its buffer in one case (16-byte stores
    # instead of whole-sector ones), the buffer has 256 spare capacity rows,
    # and the Dirichlet sizes put group ends inside the CTA-pair units: every
    # row < M matches the oracle and nothing else in the buffer (the prefix,
    # the capacity rows) changes from the sentinel.
    wl = workloads.WORKLOADS["mixtral_fprop_mxfp8"].scaled(M=2048, K=256, N=512, M_cap=2304)
    esize = 4 if out_type == mxg.MXG_OUT_F32 else 2
    sentinel = 7.0
    case, offs, rows, ref = _run_fprop(wl, out_type=out_type, fill_c=sentinel,
                                       c_offset=c_offset_bytes // esize)
    buf = case["C_buf"].cpu().float().numpy().astype(np.float64)
    assert np.all(buf[:c_offset_bytes // esize] == sentinel)
    got = case["C"].cpu().float().numpy().astype(np.float64)
    assert np.all(got[wl.M:] == sentinel)
    if out_type == mxg.MXG_OUT_BF16:
        refb = torch.from_numpy(ref).to(torch.bfloat16).double().numpy()
        assert np.all(np.abs(got[:wl.M] - refb) <= np.abs(refb) * 2.0 ** -7 + 1e-6 * np.abs(ref).max())
    else:
        errs = normwise_errors(got[:wl.M], ref, offs)
        assert errs.max() <= TOL, errs


@pytest.mark.parametrize("out_type", [mxg.MXG_OUT_F32, mxg.MXG_OUT_BF16])
def test_fprop_half_wide_last_column_unit(out_type):
    # N = 384: the CTA-pair kernel's last 256-wide column unit is half wide; its
    # upper 128 columns (the next expert's weight rows, or the zero fill past
    # the end) are computed but never stored
    wl = workloads.WORKLOADS["mixtral_fprop_mxfp8"].scaled(M=1024, K=256, N=384)
    bias = np.random.default_rng(5).standard_normal((wl.G, wl.N)).astype(np.float32)
    case, offs, rows, ref = _run_fprop(wl, bias=bias, out_type=out_type)
    got = case["C"].cpu().float().numpy().astype(np.float64)[:wl.M]
    if out_type == mxg.MXG_OUT_BF16:
        refb = torch.from_numpy(ref).to(torch.bfloat16).double().numpy()
        assert np.all(np.abs(got - refb) <= np.abs(refb) * 2.0 ** -7 + 1e-6 * np.abs(ref).max())
    else:
        errs = normwise_errors(got, ref, offs)
        assert errs.max() <= TOL, errs


def test_nvfp4_fprop_k_not_multiple_of_256():
    # K = 384: 128-byte stages would overrun K, so the pair kernel runs with
    # 64-byte stages (64-byte swizzle, two MMAs and two scale tiles per band)
    wl = workloads.WORKLOADS["rowscaled_fprop_nvfp4"].scaled(M=1024, K=384, N=512, G=4)
    case, offs, rows, ref = _run_fprop(wl)
    errs = normwise_errors(case["C"].cpu().numpy().astype(np.float64)[:wl.M], ref, offs)
    assert errs.max() <= TOL, errs


def test_nvfp4_fprop_half_wide_last_column_unit():
    wl = workloads.WORKLOADS["rowscaled_fprop_nvfp4"].scaled(M=1024, K=256, N=384, G=4)
    case, offs, rows, ref = _run_fprop(wl)
    errs = normwise_errors(case["C"].cpu().numpy().astype(np.float64)[:wl.M], ref, offs)
    assert errs.max() <= TOL, errs


# --------------------------------------------------------------------------- wgrad
def _wgrad_case(wl, tn=None, beta=None):
    inp = workloads.make_inputs(wl)
    G, N, K, M = wl.G, wl.N, wl.K, wl.rows_capacity
    ws, st = gpu_offsets(inp["sizes"], K, M)
    qx, _ = gpu_mxfp8(inp["x"].to(DEV), ws, G, mxg.MXG_COLWISE)
    qd, _ = gpu_mxfp8(inp["dy"].to(DEV), ws, G, mxg.MXG_COLWISE)
    c0 = torch.linspace(-2, 2, G * N * K).reshape(G, N, K).float()
    dW = c0.to(DEV).clone()
    be = None if beta is None else torch.tensor(beta, dtype=torch.float32, device=DEV)
    with tile_n(tn):
        mxg.mxg_grouped_gemm(mxg.MXG_MXFP8_E4M3, mxg.MXG_WGRAD_NT, (qd["q_col"], qd["sf_col"], None),
                             (qx["q_col"], qx["sf_col"], None), ws, G, M, N, K, None, be, dW,
                             dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    # oracle on its own colwise quantization
    rws, _ = oracle.group_offsets(inp["sizes"].numpy(), 1, K, M)
    offs = oracle.live_rows(rws, G)
    live = int(offs[-1])
    ox = oracle.mxfp8_quantize(inp["x"], live, M, rowwise=False, colwise=True)
    od = oracle.mxfp8_quantize(inp["dy"], live, M, rowwise=False, colwise=True)
    assert np.array_equal(qx["q_col"][:, :live].cpu().numpy(), ox["q_col"][:, :live])
    assert np.array_equal(qd["q_col"][:, :live].cpu().numpy(), od["q_col"][:, :live])
    _, _, ref = oracle.grouped_gemm_wgrad({"q": od["q_col"], "sf": od["sf_col"]},
                                          {"q": ox["q_col"], "sf": ox["sf_col"]}, offs, M, N, K,
                                          beta=beta, c_in=c0.double().numpy())
    return dW.cpu().numpy().astype(np.float64), ref, offs


@pytest.mark.parametrize("tn,K,N", [(None, 512, 256), (None, 512, 384), (None, 384, 256),
                                    (256, 512, 256), (128, 512, 256)])
def test_wgrad_scaled(tn, K, N):
    wl = workloads.WORKLOADS["wgrad_mxfp8"].scaled(M=2048, K=K, N=N)
    sizes = workloads.group_sizes(wl)
    got, ref, offs = _wgrad_case(wl, tn)
    for g in range(wl.G):
        den = np.abs(ref[g]).max()
        if sizes[g] == 0:
            assert not got[g].any(), "empty group must be zero-filled"
        else:
            assert np.abs(got[g] - ref[g]).max() / den <= TOL


def test_wgrad_empty_group_beta():
    wl = workloads.WORKLOADS["wgrad_mxfp8"].scaled(M=1024, K=256, N=256, sizes="fixed",
                                                     fixed_sizes=(256, 0, 512, 0, 128, 128, 0, 0))
    beta = [0.0, 1.0, 0.5, -1.0, 2.0, 0.0, 0.0, 3.0]
    got, ref, offs = _wgrad_case(wl, beta=beta)
    for g in range(wl.G):
        den = max(np.abs(ref[g]).max(), 1e-30)
        assert np.abs(got[g] - ref[g]).max() / den <= TOL, g


# --------------------------------------------------------------------------- NVFP4
@pytest.mark.parametrize("tn", [None, 256, 128])
def test_nvfp4_fprop_scaled(tn):
    wl = workloads.WORKLOADS["rowscaled_fprop_nvfp4"].scaled(M=4096, K=512, N=512)
    case, offs, rows, ref = _run_fprop(wl, tn)
    errs = normwise_errors(case["C"].cpu().numpy().astype(np.float64)[:wl.M], ref, offs)
    assert errs.max() <= TOL, errs


def test_nvfp4_fprop_alpha():
    wl = workloads.WORKLOADS["rowscaled_fprop_nvfp4"].scaled(M=1024, K=256, N=256, G=4)
    alpha = [1.0, -2.0, 0.5, 4.0]
    case, offs, rows, ref = _run_fprop(wl, alpha=alpha)
    errs = normwise_errors(case["C"].cpu().numpy().astype(np.float64)[:wl.M], ref, offs)
    assert errs.max() <= TOL, errs


# --------------------------------------------------------------------------- dgrad
@pytest.mark.parametrize("tn,K", [(None, 512), (None, 384), (256, 512), (128, 256)])
def test_dgrad_scaled(tn, K):
    """dX = dY . W_g: rowwise dY, colwise (transposed) copy of W."""
    _dgrad_check(tn, K, 256)


@pytest.mark.parametrize("N", [384, 512, 768])
@pytest.mark.parametrize("bk", [None, 128])
def test_stage_width_fprop_and_dgrad(N, bk):
    """The MXFP8 CTA-pair kernel takes 256 bytes of K per fprop stage when K
    is a multiple of 256 and 128 otherwise (or when the test entry point
    forces 128); dgrad keeps 128.  Both widths, with one and several stages,
    and dgrad over the same contraction lengths, match the oracle."""
    wl = workloads.WORKLOADS["mixtral_fprop_mxfp8"].scaled(M=1024, K=N, N=512)
    with gemm_override(stage_bytes=bk):
        case, offs, rows, ref = _run_fprop(wl)
    errs = normwise_errors(case["C"].cpu().numpy().astype(np.float64)[:wl.M], ref, offs)
    assert errs.max() <= TOL, errs
    _dgrad_check(None, 512, N)


@pytest.mark.parametrize("tn", [None, 128])
def test_fprop_one_k_block(tn):
    # K = 128: every unit is one 128-byte K stage (the 256-byte stages need
    # K % 256 == 0), so the first K block is also the last
    wl = workloads.WORKLOADS["mixtral_fprop_mxfp8"].scaled(M=1024, K=128, N=512)
    case, offs, rows, ref = _run_fprop(wl, tn)
    errs = normwise_errors(case["C"].cpu().numpy().astype(np.float64)[:wl.M], ref, offs)
    assert errs.max() <= TOL, errs


def test_nvfp4_fprop_one_k_block():
    # K = 128: one 64-byte stage (two MMAs) per unit
    wl = workloads.WORKLOADS["rowscaled_fprop_nvfp4"].scaled(M=1024, K=128, N=512, G=4)
    case, offs, rows, ref = _run_fprop(wl)
    errs = normwise_errors(case["C"].cpu().numpy().astype(np.float64)[:wl.M], ref, offs)
    assert errs.max() <= TOL, errs


@pytest.mark.parametrize("tn", [None, 128])
def test_dgrad_one_k_block(tn):
    """dgrad contracting over N = 128: one 128-byte K block per unit."""
    _dgrad_check(tn, 256, 128)


def _dgrad_check(tn, K, N):
    wl = workloads.WORKLOADS["finegrained_fprop_mxfp8"].scaled(M=2048, K=K, N=N, G=8)
    inp = workloads.make_inputs(wl)
    G, N, M = wl.G, wl.N, wl.M
    dy_h = workloads.random_bf16((M, N), seed=71, scale=1e-3)
    ws, st = gpu_offsets(inp["sizes"], N, M)
    qd, _ = gpu_mxfp8(dy_h.to(DEV), ws, G, mxg.MXG_ROWWISE)
    w2 = inp["w"].reshape(G * N, K)
    qwt, _ = gpu_mxfp8(w2.to(DEV), None, G, mxg.MXG_COLWISE)
    c0 = torch.linspace(-1, 1, M * K).reshape(M, K).float()
    dX = c0.to(DEV).clone()
    alpha = [1.0, 0.5, 2.0, -1.0, 1.0, 1.0, 4.0, 0.25]
    beta = [0.0, 1.0, 0.0, 0.5, 0.0, 2.0, 0.0, 0.0]
    al = torch.tensor(alpha, dtype=torch.float32, device=DEV)
    be = torch.tensor(beta, dtype=torch.float32, device=DEV)
    with tile_n(tn):
        mxg.mxg_grouped_gemm(mxg.MXG_MXFP8_E4M3, mxg.MXG_DGRAD_NN, (qd["q_row"], qd["sf_row"], None),
                             (qwt["q_col"], qwt["sf_col"], None), ws, G, M, N, K, al, be, dX,
                             dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    rws, _ = oracle.group_offsets(inp["sizes"].numpy(), 1, N, M)
    offs = oracle.live_rows(rws, G)
    od = oracle.mxfp8_quantize(dy_h, M, M, rowwise=True)
    ow = oracle.mxfp8_quantize(w2, G * N, G * N, rowwise=False, colwise=True)
    assert np.array_equal(qwt["q_col"].cpu().numpy(), ow["q_col"])
    _, _, ref = oracle.grouped_gemm_dgrad({"q": od["q_row"], "sf": od["sf_row"]},
                                          {"q": ow["q_col"], "sf": ow["sf_col"]}, offs, G, N, K,
                                          alpha=alpha, beta=beta, c_in=c0.double().numpy())
    errs = normwise_errors(dX.cpu().numpy().astype(np.float64), ref, offs)
    assert errs.max() <= TOL, errs


# --------------------------------------------------------------------------- NVFP4 wgrad
@pytest.mark.parametrize("K,sizes", [(512, None), (384, None),
                                     (256, (128, 384, 0, 128, 640, 256, 128, 384))])
def test_nvfp4_wgrad_scaled(K, sizes):
    """Row-scaled NVFP4 wgrad: colwise copies with per-(group, column) outer
    scales (PR #3661's wgrad direction).  The fixed sizes end groups inside a
    256-element K stage (128 and 384 rows) and leave one group empty."""
    wl = workloads.WORKLOADS["wgrad_mxfp8"].scaled(M=2048, K=K, N=256)
    if sizes is not None:
        wl = wl.scaled(sizes="fixed", fixed_sizes=sizes)
    inp = workloads.make_inputs(wl)
    G, N, M = wl.G, wl.N, wl.M
    sizes = inp["sizes"].numpy()
    ws, st = gpu_offsets(inp["sizes"], K, M)
    qx = mxg.alloc_nvfp4(M, K, device=DEV, rowwise=False, colwise=True, G=G)
    qd = mxg.alloc_nvfp4(M, N, device=DEV, rowwise=False, colwise=True, G=G)
    for q, t, C in ((qx, inp["x"], K), (qd, inp["dy"], N)):
        mxg.mxg_group_quantize(mxg.MXG_NVFP4_ROWSCALED, mxg.MXG_COLWISE, t.to(DEV), M, C, ws, G,
                               None, None, q["q_col"], q["sf_col"], None, st,
                               outer_col=q["outer_col"])
    dW = torch.full((G, N, K), 3.0, dtype=torch.float32, device=DEV)
    mxg.mxg_grouped_gemm(mxg.MXG_NVFP4_ROWSCALED, mxg.MXG_WGRAD_NT,
                         (qd["q_col"], qd["sf_col"], qd["outer_col"]),
                         (qx["q_col"], qx["sf_col"], qx["outer_col"]), ws, G, M, N, K, C=dW,
                         dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    offs = np.concatenate([[0], np.cumsum(sizes)])
    ox = oracle.nvfp4_quantize_colwise(inp["x"], offs, M)
    od = oracle.nvfp4_quantize_colwise(inp["dy"], offs, M)
    assert np.array_equal(qx["q_col"].cpu().numpy(), ox["q_col"])
    assert np.array_equal(qd["outer_col"].cpu().numpy(), od["outer_col"])
    _, _, ref = oracle.grouped_gemm_wgrad(
        {"q": od["q_col"], "sf": od["sf_col"], "outer": od["outer_col"]},
        {"q": ox["q_col"], "sf": ox["sf_col"], "outer": ox["outer_col"]}, offs, M, N, K,
        fmt="nvfp4")
    got = dW.cpu().numpy().astype(np.float64)
    for g in range(G):
        if sizes[g] == 0:
            assert not got[g].any()
        else:
            assert np.abs(got[g] - ref[g]).max() / np.abs(ref[g]).max() <= TOL, g


@pytest.mark.parametrize("entry", ["aligned", "unaligned", "nvfp4"])
@pytest.mark.parametrize("out_type", [mxg.MXG_OUT_F32, mxg.MXG_OUT_BF16])
def test_wgrad_without_rows(entry, out_type):
    """M_cap = 0: every group is empty, so each dW_g is beta_g * dW_g, or 0
    where there is no beta or beta_g is 0 (the oracle's empty group); the
    operands have no columns and are not read.  fprop and dgrad with
    M_cap = 0 write nothing."""
    G, N, K = 4, 256, 384
    zero = torch.zeros(G, dtype=torch.int32)
    ws = mxg.alloc_offsets(G, DEV)
    st = status_tensor()
    if entry == "unaligned":
        mxg.mxg_group_offsets_unaligned(zero.to(DEV), 1, K, 0, ws, st)
    else:
        mxg.mxg_group_offsets(zero.to(DEV), 1, K, 0, ws, st)
    dummy = torch.zeros(64, dtype=torch.uint8, device=DEV)  # valid pointers, never read
    outer = torch.zeros(64, dtype=torch.float32, device=DEV)
    cdt = torch.float32 if out_type == mxg.MXG_OUT_F32 else torch.bfloat16
    old = workloads.random_bf16((G, N, K), seed=44).float().to(cdt)
    for beta in ([0.5, 0.0, -2.0, 1.0], None):
        if entry == "nvfp4" and beta is not None:
            continue  # beta is rejected with NVFP4
        dW = old.to(DEV).clone()
        be = None if beta is None else torch.tensor(beta, dtype=torch.float32, device=DEV)
        if entry == "unaligned":
            mxg.mxg_grouped_gemm_unaligned(mxg.MXG_WGRAD_NT, (dummy, dummy), (dummy, dummy), ws, G,
                                           0, N, K, None, be, dW, out_type, dev_status=st)
        elif entry == "nvfp4":
            mxg.mxg_grouped_gemm(mxg.MXG_NVFP4_ROWSCALED, mxg.MXG_WGRAD_NT, (dummy, dummy, outer),
                                 (dummy, dummy, outer), ws, G, 0, N, K, None, None, dW, out_type,
                                 dev_status=st)
        else:
            mxg.mxg_grouped_gemm(mxg.MXG_MXFP8_E4M3, mxg.MXG_WGRAD_NT, (dummy, dummy, None),
                                 (dummy, dummy, None), ws, G, 0, N, K, None, be, dW, out_type,
                                 dev_status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        b = torch.zeros(G) if beta is None else torch.tensor(beta)
        want = (old.float() * b.view(G, 1, 1)).to(cdt)  # one rounding, as the epilogue's
        want[b == 0] = 0
        assert torch.equal(dW.cpu(), want), beta
    if entry == "aligned":
        C = torch.full((128, N), 5.0, dtype=torch.float32, device=DEV)
        for mode, n_ in ((mxg.MXG_FPROP_TN, N), (mxg.MXG_DGRAD_NN, N)):
            mxg.mxg_grouped_gemm(mxg.MXG_MXFP8_E4M3, mode, (dummy, dummy, None),
                                 (dummy, dummy, None), ws, G, 0, n_, K, C=C, dev_status=st)
        torch.cuda.synchronize()
        assert torch.all(C == 5.0)


@pytest.mark.parametrize("tn", [None, 128])
def test_empty_routing_fprop_is_a_noop_and_wgrad_zero_fills(tn):
    """Every group empty (M = 0 live rows): fprop writes nothing, wgrad writes
    dW_g = 0 for every group (no beta), and no status bit is set."""
    G, N, K, R = 4, 256, 512, 1024
    zero = torch.zeros(G, dtype=torch.int32)
    x = workloads.random_bf16((R, K), seed=41).to(DEV)
    w = workloads.random_bf16((G * N, K), seed=42, scale=0.02).to(DEV)
    dy = workloads.random_bf16((R, N), seed=43, scale=1e-3).to(DEV)
    # fprop
    ws, st = gpu_offsets(zero, K, R)
    qx, _ = gpu_mxfp8(x, ws, G, mxg.MXG_ROWWISE)
    qw, _ = gpu_mxfp8(w, None, G, mxg.MXG_ROWWISE)
    C = torch.full((R, N), 5.0, dtype=torch.float32, device=DEV)
    with tile_n(tn):
        mxg.mxg_grouped_gemm(mxg.MXG_MXFP8_E4M3, mxg.MXG_FPROP_TN, (qx["q_row"], qx["sf_row"], None),
                             (qw["q_row"], qw["sf_row"], None), ws, G, R, N, K, C=C, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.all(C == 5.0), "fprop wrote rows with no live group"
    # wgrad
    ws2, st2 = gpu_offsets(zero, K, R)
    qxc, _ = gpu_mxfp8(x, ws2, G, mxg.MXG_COLWISE)
    qdc, _ = gpu_mxfp8(dy, ws2, G, mxg.MXG_COLWISE)
    dW = torch.full((G, N, K), 3.0, dtype=torch.float32, device=DEV)
    with tile_n(tn):
        mxg.mxg_grouped_gemm(mxg.MXG_MXFP8_E4M3, mxg.MXG_WGRAD_NT, (qdc["q_col"], qdc["sf_col"], None),
                             (qxc["q_col"], qxc["sf_col"], None), ws2, G, R, N, K, None, None, dW,
                             dev_status=st2)
    torch.cuda.synchronize()
    assert int(st2.item()) == 0
    assert torch.all(dW == 0.0), "wgrad must zero-fill every dW_g of an empty group"
