"""GPU: GEMM operands given as views inside wider buffers (the
operand descriptor's leading dimension; TransformerEngine PR #2763's GEMM
setup derives per-group operand pointers from offsets and leading
dimensions).  The data is copied into a buffer with extra columns and the
GEMM reads it through the descriptor's ld; the output must be bit-identical
to the dense call (same kernel, same operand values, same accumulation
order).  Column operands of the epilogue (bias, NVFP4 column outer scales)
given 4 bytes off a 16-byte boundary take the 4-byte copy path and must give
the same result as aligned ones.  Shapes that disagree with the mode are
refused on the host (tests/test_abi.py)."""
import pytest
import torch

from moe_grouped_block_gb300 import mxg, workloads

from gpu_util import DEV, gpu_mxfp8, gpu_nvfp4, gpu_offsets, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _gpu():
    require_gpu()


def _widen(q: torch.Tensor, extra_bytes: int) -> torch.Tensor:
    """The same rows as a view into a buffer extra_bytes wider (filled with
    0xFF so that a read past the row shows up in the result)."""
    rows, width = q.shape
    buf = torch.full((rows, width + extra_bytes), 0xFF, dtype=torch.uint8, device=q.device)
    buf[:, :width].copy_(q)
    return buf[:, :width]


def _same(fmt, mode, A, B, A_wide, B_wide, ws, G, M, N, K, out_shape):
    dense = torch.zeros(out_shape, dtype=torch.float32, device=DEV)
    strided = torch.zeros(out_shape, dtype=torch.float32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    mxg.mxg_grouped_gemm(fmt, mode, A, B, ws, G, M, N, K, C=dense, dev_status=st)
    mxg.mxg_grouped_gemm(fmt, mode, A_wide, B_wide, ws, G, M, N, K, C=strided, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(dense, strided)


@pytest.mark.parametrize("extra", [16, 384])
def test_fprop_mxfp8_strided(extra):
    wl = workloads.WORKLOADS["mixtral_fprop_mxfp8"].scaled(M=1024, K=512, N=384)
    inp = workloads.make_inputs(wl)
    G, N, K, M = wl.G, wl.N, wl.K, wl.M
    ws, _ = gpu_offsets(inp["sizes"], K, M)
    qx, _ = gpu_mxfp8(inp["x"].to(DEV), ws, G, mxg.MXG_ROWWISE)
    qw, _ = gpu_mxfp8(inp["w"].to(DEV).reshape(G * N, K), None, G, mxg.MXG_ROWWISE)
    A = (qx["q_row"], qx["sf_row"], None)
    B = (qw["q_row"], qw["sf_row"], None)
    Aw = (_widen(qx["q_row"], extra), qx["sf_row"], None)
    Bw = (_widen(qw["q_row"], extra + 128), qw["sf_row"], None)
    _same(mxg.MXG_MXFP8_E4M3, mxg.MXG_FPROP_TN, A, B, Aw, Bw, ws, G, M, N, K, (M, N))


def test_fprop_nvfp4_strided():
    wl = workloads.WORKLOADS["rowscaled_fprop_nvfp4"].scaled(M=1024, K=512, N=256, G=4)
    inp = workloads.make_inputs(wl)
    G, N, K, M = wl.G, wl.N, wl.K, wl.M
    ws, _ = gpu_offsets(inp["sizes"], K, M)
    qx, _ = gpu_nvfp4(inp["x"].to(DEV), ws, G)
    qw, _ = gpu_nvfp4(inp["w"].to(DEV).reshape(G * N, K), None, G)
    A = (qx["q_row"], qx["sf_row"], qx["outer_row"])
    B = (qw["q_row"], qw["sf_row"], qw["outer_row"])
    Aw = (_widen(qx["q_row"], 48), qx["sf_row"], qx["outer_row"])
    Bw = (_widen(qw["q_row"], 256), qw["sf_row"], qw["outer_row"])
    _same(mxg.MXG_NVFP4_ROWSCALED, mxg.MXG_FPROP_TN, A, B, Aw, Bw, ws, G, M, N, K, (M, N))


def test_wgrad_mxfp8_strided():
    wl = workloads.WORKLOADS["wgrad_mxfp8"].scaled(M=1024, K=256, N=512)
    inp = workloads.make_inputs(wl)
    G, N, K, M = wl.G, wl.N, wl.K, wl.M
    ws, _ = gpu_offsets(inp["sizes"], K, M)
    qx, _ = gpu_mxfp8(inp["x"].to(DEV), ws, G, mxg.MXG_COLWISE)
    qd, _ = gpu_mxfp8(inp["dy"].to(DEV), ws, G, mxg.MXG_COLWISE)
    A = (qd["q_col"], qd["sf_col"], None)
    B = (qx["q_col"], qx["sf_col"], None)
    Aw = (_widen(qd["q_col"], 32), qd["sf_col"], None)
    Bw = (_widen(qx["q_col"], 1024), qx["sf_col"], None)
    _same(mxg.MXG_MXFP8_E4M3, mxg.MXG_WGRAD_NT, A, B, Aw, Bw, ws, G, M, N, K, (G, N, K))


def test_dgrad_mxfp8_strided():
    wl = workloads.WORKLOADS["dgrad_mxfp8"].scaled(M=1024, K=512, N=256)
    inp = workloads.make_inputs(wl)
    G, N, K, M = wl.G, wl.N, wl.K, wl.M
    ws, _ = gpu_offsets(inp["sizes"], N, M)
    qd, _ = gpu_mxfp8(inp["dy"].to(DEV), ws, G, mxg.MXG_ROWWISE)
    qwt, _ = gpu_mxfp8(inp["w"].to(DEV).reshape(G * N, K), None, G, mxg.MXG_COLWISE)
    A = (qd["q_row"], qd["sf_row"], None)
    B = (qwt["q_col"], qwt["sf_col"], None)
    Aw = (_widen(qd["q_row"], 64), qd["sf_row"], None)
    Bw = (_widen(qwt["q_col"], 512), qwt["sf_col"], None)
    _same(mxg.MXG_MXFP8_E4M3, mxg.MXG_DGRAD_NN, A, B, Aw, Bw, ws, G, M, N, K, (M, K))


def _shifted(t: torch.Tensor) -> torch.Tensor:
    """The same fp32 values in a buffer one element further on: 4-byte but not
    16-byte aligned, so the epilogue copies them 4 bytes at a time."""
    buf = torch.empty(t.numel() + 1, dtype=torch.float32, device=t.device)
    view = buf[1:].view(t.shape)
    view.copy_(t)
    assert view.data_ptr() % 16 != 0
    return view


def test_fprop_mxfp8_bias_not_16_byte_aligned():
    wl = workloads.WORKLOADS["mixtral_fprop_mxfp8"].scaled(M=1024, K=256, N=512)
    inp = workloads.make_inputs(wl)
    G, N, K, M = wl.G, wl.N, wl.K, wl.M
    ws, _ = gpu_offsets(inp["sizes"], K, M)
    qx, _ = gpu_mxfp8(inp["x"].to(DEV), ws, G, mxg.MXG_ROWWISE)
    qw, _ = gpu_mxfp8(inp["w"].to(DEV).reshape(G * N, K), None, G, mxg.MXG_ROWWISE)
    A = (qx["q_row"], qx["sf_row"], None)
    B = (qw["q_row"], qw["sf_row"], None)
    bias = torch.randn(G, N, dtype=torch.float32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    outs = []
    for bi in (bias, _shifted(bias)):
        C = torch.zeros((M, N), dtype=torch.float32, device=DEV)
        mxg.mxg_grouped_gemm(mxg.MXG_MXFP8_E4M3, mxg.MXG_FPROP_TN, A, B, ws, G, M, N, K, C=C,
                             dev_status=st, bias=bi)
        outs.append(C)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(outs[0], outs[1])


def test_nvfp4_outer_and_bias_not_16_byte_aligned():
    wl = workloads.WORKLOADS["rowscaled_fprop_nvfp4"].scaled(M=1024, K=512, N=256, G=4)
    inp = workloads.make_inputs(wl)
    G, N, K, M = wl.G, wl.N, wl.K, wl.M
    ws, _ = gpu_offsets(inp["sizes"], K, M)
    qx, _ = gpu_nvfp4(inp["x"].to(DEV), ws, G)
    qw, _ = gpu_nvfp4(inp["w"].to(DEV).reshape(G * N, K), None, G)
    A = (qx["q_row"], qx["sf_row"], qx["outer_row"])
    bias = torch.randn(G, N, dtype=torch.float32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    outs = []
    for outer, bi in ((qw["outer_row"], bias), (_shifted(qw["outer_row"]), _shifted(bias))):
        C = torch.zeros((M, N), dtype=torch.float32, device=DEV)
        mxg.mxg_grouped_gemm(mxg.MXG_NVFP4_ROWSCALED, mxg.MXG_FPROP_TN, A,
                             (qw["q_row"], qw["sf_row"], outer), ws, G, M, N, K, C=C,
                             dev_status=st, bias=bi)
        outs.append(C)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(outs[0], outs[1])
