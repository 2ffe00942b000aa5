"""GPU parity for group sizes that are not multiples of 128 (MXFP8):
offsets, the per-group padded quantize and the fprop / wgrad / dgrad GEMMs,
all through the C ABI, against the oracle on the same seeded inputs.  The
quantize is bit-exact, sentinel bytes included (nothing outside the padded
groups is written); the GEMMs are within 1e-3 normwise per group."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import DEV, normwise_errors, require_gpu, status_tensor, u8
from moe_grouped_block_gb300 import mxg, workloads

pytestmark = pytest.mark.gpu
TOL = 1e-3
FILL = 0x5A


@pytest.fixture(autouse=True)
def _gpu():
    require_gpu()


def _offsets(sizes, last_dim, cap):
    t = torch.tensor(sizes, dtype=torch.int32)
    ws = mxg.alloc_offsets(t.numel(), DEV)
    st = status_tensor()
    mxg.mxg_group_offsets_unaligned(t.to(DEV), 1, last_dim, cap, ws, st)
    return ws, st


def _quantize(x, ws, G, layout):
    R, C = x.shape
    out = mxg.alloc_mxfp8_unaligned(R, C, G, rowwise=bool(layout & 1), colwise=bool(layout & 2),
                                    device=DEV)
    for t in out.values():
        t.fill_(FILL)
    st = status_tensor()
    mxg.mxg_group_quantize_unaligned(layout, x.to(DEV), R, C, ws, G, out.get("q_row"),
                                     out.get("sf_row"), out.get("q_col"), out.get("sf_col"), st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return out


@pytest.mark.parametrize("sizes,cap,bits", [
    ((5, 0, 300, 7), 512, 0),
    ((-3, 200, 400, 9), 512, oracle.ST_NEG_SIZE | oracle.ST_SUM_OVER_CAPACITY),
    ((128, 256, 1), 1024, 0),
])
def test_offsets_unaligned(sizes, cap, bits):
    ws, st = _offsets(sizes, 96, cap)
    torch.cuda.synchronize()
    ref, rst = oracle.group_offsets_unaligned(np.array(sizes), 1, 96, cap)
    assert np.array_equal(ws.cpu().numpy(), ref)
    assert int(st.item()) == rst == bits


SIZE_SETS = [(37, 0, 129, 200), (1, 127, 128, 255), (300,), (128, 0, 256, 128)]


@pytest.mark.parametrize("sizes", SIZE_SETS)
@pytest.mark.parametrize("layout", [mxg.MXG_ROWWISE, mxg.MXG_COLWISE, mxg.MXG_BOTH])
def test_quantize_unaligned_bit_exact(sizes, layout):
    R, K = 640, 256
    G = len(sizes)
    x = workloads.random_bf16((R, K), seed=81)
    ws, _ = _offsets(sizes, K, R)
    out = _quantize(x, ws, G, layout)
    ref = oracle.mxfp8_quantize_unaligned(x, ws.cpu().numpy(), G, R, rowwise=bool(layout & 1),
                                          colwise=bool(layout & 2), fill=FILL)
    for name in out:
        assert np.array_equal(u8(out[name]), ref[name].reshape(-1)), name


def test_quantize_unaligned_many_groups():
    # 64 groups of random sizes (some empty) over a 4096-row buffer
    rng = np.random.default_rng(82)
    sizes = rng.integers(0, 120, 64)
    sizes[[3, 17, 40]] = 0
    R, K = 4096, 512
    x = workloads.random_bf16((R, K), seed=83)
    ws, _ = _offsets(tuple(int(s) for s in sizes), K, R)
    out = _quantize(x, ws, 64, mxg.MXG_BOTH)
    ref = oracle.mxfp8_quantize_unaligned(x, ws.cpu().numpy(), 64, R, rowwise=True, colwise=True,
                                          fill=FILL)
    for name in out:
        assert np.array_equal(u8(out[name]), ref[name].reshape(-1)), name


def _per_group_err(got, ref, offs):
    return normwise_errors(got, ref, offs)


@pytest.mark.parametrize("sizes", [(37, 0, 129, 200), (1, 127, 128, 255), (300, 5)])
@pytest.mark.parametrize("out_type", [mxg.MXG_OUT_F32, mxg.MXG_OUT_BF16])
def test_fprop_unaligned(sizes, out_type):
    G, N, K, R = len(sizes), 256, 512, 640
    x = workloads.random_bf16((R, K), seed=84)
    w = workloads.random_bf16((G * N, K), seed=85, scale=0.02)
    ws, _ = _offsets(sizes, K, R)
    qa = _quantize(x, ws, G, mxg.MXG_ROWWISE)
    qw = mxg.alloc_mxfp8(G * N, K, device=DEV)
    mxg.mxg_group_quantize(mxg.MXG_MXFP8_E4M3, mxg.MXG_ROWWISE, w.to(DEV), G * N, K, None, G,
                           qw["q_row"], qw["sf_row"])
    bias = torch.from_numpy(np.random.default_rng(86).standard_normal((G, N)).astype(np.float32))
    alpha = torch.tensor([0.5 + g for g in range(G)], dtype=torch.float32)
    dt = torch.float32 if out_type == mxg.MXG_OUT_F32 else torch.bfloat16
    C = torch.full((R, N), 7.0, dtype=dt, device=DEV)
    st = status_tensor()
    mxg.mxg_grouped_gemm_unaligned(mxg.MXG_FPROP_TN, (qa["q_row"], qa["sf_row"]),
                                   (qw["q_row"], qw["sf_row"]), ws, G, R, N, K,
                                   alpha=alpha.to(DEV), C=C, out_type=out_type, dev_status=st,
                                   bias=bias.to(DEV))
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    wsn = ws.cpu().numpy()
    a = {"q": qa["q_row"].cpu().numpy(), "sf": u8(qa["sf_row"])}
    b = {"q": qw["q_row"].cpu().numpy(), "sf": u8(qw["sf_row"])}
    rows, ref = oracle.grouped_gemm_fprop_unaligned(a, b, wsn, G, N, K, alpha=alpha.numpy(),
                                                    bias=bias.numpy())
    live = rows.size
    got = C.float().cpu().numpy().astype(np.float64)
    offs = oracle.live_rows(wsn, G)
    if out_type == mxg.MXG_OUT_F32:
        assert _per_group_err(got[:live], ref, offs).max() <= TOL
    else:
        refb = torch.from_numpy(ref).to(torch.bfloat16).double().numpy()
        assert np.all(np.abs(got[:live] - refb) <= np.abs(refb) * 2.0 ** -7 + 1e-6 * np.abs(ref).max())
    assert np.all(got[live:] == 7.0), "rows past the live groups must stay untouched"


@pytest.mark.parametrize("sizes", [(37, 0, 129, 200), (1, 127, 128, 255)])
def test_wgrad_unaligned(sizes):
    G, N, K, R = len(sizes), 256, 384, 640
    x = workloads.random_bf16((R, K), seed=87)
    dy = workloads.random_bf16((R, N), seed=88, scale=1e-3)
    ws, _ = _offsets(sizes, K, R)
    qx = _quantize(x, ws, G, mxg.MXG_COLWISE)
    qd = _quantize(dy, ws, G, mxg.MXG_COLWISE)
    beta = torch.tensor([0.0, 1.0, 0.5, -1.0][:G], dtype=torch.float32)
    c0 = torch.linspace(-1, 1, G * N * K).reshape(G, N, K).float()
    dW = c0.to(DEV).clone()
    st = status_tensor()
    mxg.mxg_grouped_gemm_unaligned(mxg.MXG_WGRAD_NT, (qd["q_col"], qd["sf_col"]),
                                   (qx["q_col"], qx["sf_col"]), ws, G, R, N, K,
                                   beta=beta.to(DEV), C=dW, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    wsn = ws.cpu().numpy()
    _, _, ref = oracle.grouped_gemm_wgrad_unaligned(
        {"q": qd["q_col"].cpu().numpy(), "sf": u8(qd["sf_col"])},
        {"q": qx["q_col"].cpu().numpy(), "sf": u8(qx["sf_col"])}, wsn, G, R, N, K,
        beta=beta.numpy(), c_in=c0.double().numpy())
    got = dW.cpu().numpy().astype(np.float64)
    for g in range(G):
        den = max(np.abs(ref[g]).max(), 1e-30)
        assert np.abs(got[g] - ref[g]).max() / den <= TOL, g


def test_dgrad_unaligned():
    sizes = (37, 0, 129, 200)
    G, N, K, R = 4, 256, 512, 640
    dy = workloads.random_bf16((R, N), seed=89, scale=1e-3)
    w = workloads.random_bf16((G * N, K), seed=90, scale=0.02)
    ws, _ = _offsets(sizes, N, R)
    qd = _quantize(dy, ws, G, mxg.MXG_ROWWISE)
    qwt = mxg.alloc_mxfp8(G * N, K, rowwise=False, colwise=True, device=DEV)
    mxg.mxg_group_quantize(mxg.MXG_MXFP8_E4M3, mxg.MXG_COLWISE, w.to(DEV), G * N, K, None, G,
                           None, None, qwt["q_col"], qwt["sf_col"])
    dX = torch.zeros((R, K), dtype=torch.float32, device=DEV)
    st = status_tensor()
    mxg.mxg_grouped_gemm_unaligned(mxg.MXG_DGRAD_NN, (qd["q_row"], qd["sf_row"]),
                                   (qwt["q_col"], qwt["sf_col"]), ws, G, R, N, K, C=dX,
                                   dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    wsn = ws.cpu().numpy()
    rows, ref = oracle.grouped_gemm_dgrad_unaligned(
        {"q": qd["q_row"].cpu().numpy(), "sf": u8(qd["sf_row"])},
        {"q": qwt["q_col"].cpu().numpy(), "sf": u8(qwt["sf_col"])}, wsn, G, N, K)
    offs = oracle.live_rows(wsn, G)
    got = dX.cpu().numpy().astype(np.float64)
    assert _per_group_err(got[:rows.size], ref, offs).max() <= TOL


def test_unaligned_gemm_rejects_small_b():
    # the unaligned GEMM runs on the CTA-pair kernel only: B needs >= 256 rows
    ws, _ = _offsets((5,), 128, 128)
    q = torch.zeros((128, 128), dtype=torch.uint8, device=DEV)
    sf = torch.zeros(256 * 4, dtype=torch.uint8, device=DEV)
    C = torch.zeros((128, 128), dtype=torch.float32, device=DEV)
    with pytest.raises(mxg.MxgError):
        mxg.mxg_grouped_gemm_unaligned(mxg.MXG_FPROP_TN, (q, sf), (q, sf), ws, 1, 128, 128, 128,
                                       C=C)
