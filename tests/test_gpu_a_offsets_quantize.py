"""GPU parity: group offsets, MXFP8 / row-scaled NVFP4 grouped quantize and
dequantize, through the C ABI, against the oracle on the same seeded inputs.
Quantized bytes, swizzled scales, outer scales and offsets are compared
bit for bit."""
import numpy as np
import pytest
import torch

import oracle
from moe_grouped_block_gb300 import mxg, workloads

from gpu_util import DEV, gpu_mxfp8, gpu_nvfp4, gpu_offsets, require_gpu, u8

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _gpu():
    require_gpu()


# --------------------------------------------------------------------------- offsets
@pytest.mark.parametrize("G", [1, 4, 8, 33, 64, 1024])
@pytest.mark.parametrize("dtype", [torch.int32, torch.int64])
def test_offsets_parity(G, dtype):
    rng = np.random.default_rng(G)
    sizes = torch.from_numpy(rng.integers(0, 40, G) * 128).to(dtype)
    cap = int(sizes.sum()) + 256
    ws, st = gpu_offsets(sizes, 4096, cap)
    ref, rst = oracle.group_offsets(sizes.numpy(), 1, 4096, cap)
    assert np.array_equal(ws.cpu().numpy(), ref)
    assert int(st.item()) == rst == 0


def _offsets_by_definition(sizes, mult, last_dim, cap, round128=True):
    """The sanitised workspace from its definition in exact (Python) integer
    arithmetic: rows = size * multiplier, negative -> 0, rounded down to 128,
    the running sum kept within the capacity."""
    bits, kept, p = 0, [], 0
    for s in sizes:
        v = int(s) * mult
        if v < 0:
            bits |= mxg.MXG_DEV_NEG_SIZE
            v = 0
        if round128 and v % 128:
            bits |= mxg.MXG_DEV_MISALIGNED
            v -= v % 128
        v = min(v, cap)
        before, p = min(p, cap), p + v
        if p > cap and v > 0:
            bits |= mxg.MXG_DEV_SUM_OVER_CAPACITY
        kept.append(min(p, cap) - before)
    offs = np.concatenate([[0], np.cumsum(kept)]) * last_dim
    return np.concatenate([np.array(kept, np.int64), offs.astype(np.int64)]), bits


def test_offsets_definition_matches_the_oracle():
    """The exact-integer definition above agrees with the oracle wherever the
    oracle's 64-bit products do not overflow (so it can stand for the oracle
    on the overflow cases below)."""
    rng = np.random.default_rng(5)
    for mult in (1, 3, 128):
        sizes = rng.integers(-300, 3000, 40)
        ref, rst = oracle.group_offsets(sizes, mult, 4096, 1 << 18)
        mine, bits = _offsets_by_definition(sizes, mult, 4096, 1 << 18)
        assert np.array_equal(ref, mine) and rst == bits


@pytest.mark.parametrize("mult", [1, 4, 1 << 31])
def test_offsets_huge_sizes_do_not_overflow(mult):
    """Sizes whose product with the multiplier overflows int64 are clamped
    to the capacity like any other oversize group, with the status bits of
    the exact product."""
    sizes = torch.tensor([(1 << 62) + 5, -5, 384, 1000, (1 << 40) + 1, 1 << 61],
                         dtype=torch.int64)
    cap = 1 << 20
    ws, st = gpu_offsets(sizes, 4096, cap, mult=mult)
    ref, bits = _offsets_by_definition(sizes.tolist(), mult, 4096, cap)
    assert np.array_equal(ws.cpu().numpy(), ref)
    assert int(st.item()) == bits


def test_offsets_multiplier():
    sizes = torch.tensor([1, 0, 3, 2, 7], dtype=torch.int32)
    ws, st = gpu_offsets(sizes, 7168, 1 << 20, mult=128)
    ref, rst = oracle.group_offsets(sizes.numpy(), 128, 7168, 1 << 20)
    assert np.array_equal(ws.cpu().numpy(), ref) and int(st.item()) == rst == 0


@pytest.mark.parametrize("sizes,cap", [
    ([-128, 200, 256, 512], 512),            # negative, misaligned, over capacity
    ([128, 128, 128], 256),                  # over capacity at the end
    ([0, 0, 0, 0], 0),                       # all empty, zero capacity
    ([1000, -5, 129, 384] * 20, 4096),       # many groups, mixed faults
])
def test_offsets_sanitisation(sizes, cap):
    s = torch.tensor(sizes, dtype=torch.int32)
    ws, st = gpu_offsets(s, 10, cap)
    ref, rst = oracle.group_offsets(s.numpy(), 1, 10, cap)
    assert np.array_equal(ws.cpu().numpy(), ref)
    assert int(st.item()) == rst


# --------------------------------------------------------------------------- MXFP8
def _check_mxfp8(x_host, ws_dev, G, layout, live, fill=None):
    R, C = x_host.shape
    got, st = gpu_mxfp8(x_host.to(DEV), ws_dev, G, layout, fill=fill)
    ref = oracle.mxfp8_quantize(x_host, live, R, rowwise=bool(layout & 1),
                                colwise=bool(layout & 2), fill=0 if fill is None else fill)
    if fill is None:  # only the live part is defined
        if layout & 1:
            assert np.array_equal(got["q_row"][:live].cpu().numpy(), ref["q_row"][:live])
            n = live * C // 32
            assert np.array_equal(u8(got["sf_row"])[:n], ref["sf_row"][:n])
        if layout & 2:
            assert np.array_equal(got["q_col"][:, :live].cpu().numpy(), ref["q_col"][:, :live])
            sfc_g = oracle.unswizzle(u8(got["sf_col"]), C, R // 32)
            sfc_r = oracle.unswizzle(ref["sf_col"], C, R // 32)
            assert np.array_equal(sfc_g[:, :live // 32], sfc_r[:, :live // 32])
    else:  # everything, including the untouched fill beyond the live rows
        for k in ref:
            assert np.array_equal(u8(got[k]), ref[k].reshape(-1)), k
    return st


@pytest.mark.parametrize("layout", [mxg.MXG_ROWWISE, mxg.MXG_COLWISE, mxg.MXG_BOTH])
def test_mxfp8_tiny_workload(layout):
    wl = workloads.WORKLOADS["tiny_fprop_mxfp8"]
    inp = workloads.make_inputs(wl)
    ws, _ = gpu_offsets(inp["sizes"], wl.K, wl.M)
    st = _check_mxfp8(inp["x"], ws, wl.G, layout, wl.M, fill=0x5A)
    assert int(st.item()) == 0


@pytest.mark.parametrize("name,M,K", [("mixtral_fprop_mxfp8", 2048, 1024),
                                      ("finegrained_fprop_mxfp8", 4096, 512),
                                      ("wgrad_mxfp8", 1024, 384)])
def test_mxfp8_scaled_workloads_both(name, M, K):
    wl = workloads.WORKLOADS[name].scaled(M=M, K=K)
    inp = workloads.make_inputs(wl)
    ws, _ = gpu_offsets(inp["sizes"], K, M)
    _check_mxfp8(inp["x"], ws, wl.G, mxg.MXG_BOTH, M, fill=0xA5)
    if wl.mode == "wgrad":
        _check_mxfp8(inp["dy"], gpu_offsets(inp["sizes"], wl.N, M)[0], wl.G, mxg.MXG_BOTH, M,
                     fill=0xA5)


def test_mxfp8_special_values():
    R, C = 256, 256
    x = workloads.random_bf16((R, C), seed=77, scale=2.0).to(torch.float32)
    x[0, :32] = 0.0                       # zero block
    x[1, :] = -0.0                        # negative zeros
    x[2, 32:64] = 2.0 ** -130             # subnormal block
    x[3, 64:96] = 3.0e38                  # near bf16 max
    x[4, 96:128] = torch.linspace(-448, 448, 32)
    x[5, :] = 1e-30
    x[6, :] = torch.arange(C, dtype=torch.float32) * 2.0 ** -20
    x[7, 5] = 1e30                        # one huge element beside normal ones
    x[:, 200] = 0.0                       # zero column (colwise zero blocks)
    xb = x.to(torch.bfloat16)
    _check_mxfp8(xb, None, 1, mxg.MXG_BOTH, R, fill=0x33)


def test_mxfp8_live_rows_below_capacity_leave_the_rest_untouched():
    R, C, G = 1024, 256, 5
    sizes = torch.tensor([128, 0, 256, 128, 0], dtype=torch.int32)  # 512 live rows of 1024
    x = workloads.random_bf16((R, C), seed=5)
    ws, _ = gpu_offsets(sizes, C, R)
    st = _check_mxfp8(x, ws, G, mxg.MXG_BOTH, 512, fill=0xEE)
    assert int(st.item()) == 0


def test_mxfp8_empty_routing_writes_nothing():
    R, C, G = 512, 128, 3
    ws, _ = gpu_offsets(torch.zeros(G, dtype=torch.int32), C, R)
    _check_mxfp8(workloads.random_bf16((R, C), seed=6), ws, G, mxg.MXG_BOTH, 0, fill=0x11)


def test_mxfp8_weights_uniform_groups():
    G, N, K = 4, 384, 512
    w = workloads.random_bf16((G * N, K), seed=8, scale=0.02)
    _check_mxfp8(w, None, G, mxg.MXG_ROWWISE, G * N, fill=0)


# --------------------------------------------------------------------------- NVFP4
def _check_nvfp4(x_host, ws_dev, G, live, fill=0x3C):
    R, C = x_host.shape
    got, st = gpu_nvfp4(x_host.to(DEV), ws_dev, G, fill=fill)
    ref = oracle.nvfp4_quantize(x_host, live, R, fill=fill)
    assert np.array_equal(got["q_row"].cpu().numpy(), ref["q_row"])
    assert np.array_equal(u8(got["sf_row"]), ref["sf_row"])
    o = got["outer_row"].cpu().numpy()
    assert np.array_equal(o[:live], ref["outer_row"][:live])
    assert np.all(np.isnan(o[live:]))
    return st


def test_nvfp4_scaled_workload():
    wl = workloads.WORKLOADS["rowscaled_fprop_nvfp4"].scaled(M=2048, K=1024)
    inp = workloads.make_inputs(wl)
    ws, _ = gpu_offsets(inp["sizes"], wl.K, wl.M)
    st = _check_nvfp4(inp["x"], ws, wl.G, wl.M)
    assert int(st.item()) == 0
    _check_nvfp4(inp["w"].reshape(-1, wl.K)[:512], None, 1, 512)


@pytest.mark.parametrize("cols", [7168, 7296])
def test_nvfp4_row_width_either_side_of_staging_limit(cols):
    # rows up to 7168 columns are staged whole in shared memory; wider rows
    # take the kernel that reads them twice from global memory
    R = 256
    x = workloads.random_bf16((R, cols), seed=12, dist="uniform", scale=3.0)
    _check_nvfp4(x, None, 1, R)


def test_nvfp4_special_rows():
    R, C = 256, 384
    x = workloads.random_bf16((R, C), seed=9, dist="student_t3").to(torch.float32)
    x[0] = 0.0
    x[1] = -0.0
    x[2] = 0.0
    x[2, 17] = -3.5                       # single nonzero: scale 448, code -6
    x[3, 32:48] = 1e-8                    # block far below the row amax
    x[4] = torch.linspace(-1e30, 1e30, C)
    x[5] = 2.0 ** -133
    x[6, ::2] = 6.0
    x[6, 1::2] = -0.25
    _check_nvfp4(x.to(torch.bfloat16), None, 1, R)


def test_nvfp4_live_rows_below_capacity():
    R, C, G = 512, 256, 3
    sizes = torch.tensor([128, 0, 128], dtype=torch.int32)
    ws, _ = gpu_offsets(sizes, C, R)
    st = _check_nvfp4(workloads.random_bf16((R, C), seed=10), ws, G, 256)
    assert int(st.item()) == 0


# --------------------------------------------------------------------------- dequantize
def test_dequantize_mxfp8_row_and_col():
    R, C = 256, 384
    x = workloads.random_bf16((R, C), seed=11, scale=5.0)
    q, _ = gpu_mxfp8(x.to(DEV), None, 1, mxg.MXG_BOTH)
    ref = oracle.mxfp8_quantize(x, R, R, rowwise=True, colwise=True)
    want = oracle.dequantize("mxfp8", ref["q_row"], ref["sf_row"], R, C)
    for layout, qk, sk in [(mxg.MXG_ROWWISE, "q_row", "sf_row"), (mxg.MXG_COLWISE, "q_col", "sf_col")]:
        out = torch.empty((R, C), dtype=torch.float32, device=DEV)
        mxg.mxg_dequantize(mxg.MXG_MXFP8_E4M3, layout, q[qk], q[sk], None, R, C, out)
        got = out.cpu().numpy().astype(np.float64)
        if layout == mxg.MXG_ROWWISE:
            assert np.array_equal(got, want)
        else:
            wantc = oracle.dequantize("mxfp8", ref["q_col"], ref["sf_col"], C, R).T
            assert np.array_equal(got, wantc)
        outb = torch.empty((R, C), dtype=torch.bfloat16, device=DEV)
        mxg.mxg_dequantize(mxg.MXG_MXFP8_E4M3, layout, q[qk], q[sk], None, R, C, outb,
                           mxg.MXG_OUT_BF16)
        assert torch.equal(outb.cpu(), out.cpu().to(torch.bfloat16))


def test_dequantize_nvfp4():
    R, C = 256, 512
    x = workloads.random_bf16((R, C), seed=12, dist="student_t3")
    q, _ = gpu_nvfp4(x.to(DEV), None, 1)
    ref = oracle.nvfp4_quantize(x, R, R)
    want = oracle.dequantize("nvfp4", ref["q_row"], ref["sf_row"], R, C, ref["outer_row"])
    out = torch.empty((R, C), dtype=torch.float32, device=DEV)
    mxg.mxg_dequantize(mxg.MXG_NVFP4_ROWSCALED, mxg.MXG_ROWWISE, q["q_row"], q["sf_row"],
                       q["outer_row"], R, C, out)
    got = out.cpu().numpy().astype(np.float64)
    # fp32 product e2m1 * scale * outer: one rounding of the exact fp64 value
    assert np.max(np.abs(got - want) / np.maximum(np.abs(want), 1e-38)) <= 2.0 ** -23


# --------------------------------------------------------------------------- NVFP4 colwise
@pytest.mark.parametrize("sizes", [(256, 0, 384, 128, 256), (1024,), (128,) * 8])
def test_nvfp4_colwise_parity(sizes):
    G, K = len(sizes), 384
    live = sum(sizes)
    R = live + 128  # capacity beyond the live rows
    x = workloads.random_bf16((R, K), seed=90 + G, dist="student_t3").to(torch.float32)
    x[:, 7] = 0.0
    x[:, 9] = -0.0
    xb = x.to(torch.bfloat16)
    ws, st = gpu_offsets(torch.tensor(sizes, dtype=torch.int32), K, R)
    out = mxg.alloc_nvfp4(R, K, device=DEV, rowwise=True, colwise=True, G=G)
    for k in ("q_col", "sf_col"):
        out[k].fill_(0x3C)
    mxg.mxg_group_quantize(mxg.MXG_NVFP4_ROWSCALED, mxg.MXG_BOTH, xb.to(DEV), R, K, ws, G,
                           out["q_row"], out["sf_row"], out["q_col"], out["sf_col"],
                           out["outer_row"], st, outer_col=out["outer_col"])
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    offs = np.concatenate([[0], np.cumsum(sizes)])
    ref = oracle.nvfp4_quantize_colwise(xb, offs, R, fill=0x3C)
    assert np.array_equal(out["q_col"].cpu().numpy(), ref["q_col"])
    assert np.array_equal(u8(out["sf_col"]), ref["sf_col"])
    assert np.array_equal(out["outer_col"].cpu().numpy(), ref["outer_col"])
    refr = oracle.nvfp4_quantize(xb, live, R)
    assert np.array_equal(out["q_row"][:live].cpu().numpy(), refr["q_row"][:live])
    assert np.array_equal(out["outer_row"][:live].cpu().numpy(), refr["outer_row"][:live])


def test_quantize_without_rows():
    """rows_capacity = 0: no rows are read or written; the NVFP4 colwise outer
    scales, one per (group, column), are those of empty groups: 0."""
    G, cols = 3, 256
    zero = torch.zeros(G, dtype=torch.int32)
    ws, st = gpu_offsets(zero, cols, 0)
    x = torch.zeros(64, dtype=torch.bfloat16, device=DEV)  # valid pointers, never touched
    dummy = torch.zeros(64, dtype=torch.uint8, device=DEV)
    outer = torch.full((G, cols), 7.0, dtype=torch.float32, device=DEV)
    mxg.mxg_group_quantize(mxg.MXG_NVFP4_ROWSCALED, mxg.MXG_COLWISE, x, 0, cols, ws, G, None,
                           None, dummy, dummy, None, st, outer_col=outer)
    mxg.mxg_group_quantize(mxg.MXG_MXFP8_E4M3, mxg.MXG_BOTH, x, 0, cols, ws, G, dummy, dummy,
                           dummy, dummy, None, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.all(outer == 0.0)
    assert torch.all(dummy == 0)


def test_nvfp4_colwise_special_columns():
    """Columns at the edges of the scale arithmetic, bit-exact against the
    oracle: zero and signed-zero columns, a single nonzero, a block far below
    its column's amax, magnitudes near the bf16 limits (the per-block ratio
    S / sb then leaves the normal fp32 range and the kernel falls back to the
    division), and columns scaled by powers of two across the exponent
    range."""
    sizes = (256, 128)
    G, K = len(sizes), 128
    live = sum(sizes)
    R = live + 128
    x = workloads.random_bf16((R, K), seed=95, dist="student_t3").to(torch.float32)
    x[:, 0] = 0.0
    x[:, 1] = -0.0
    x[:, 2] = 0.0
    x[17, 2] = -3.5                                   # single nonzero: scale 448, code -6
    x[32:48, 3] = 1e-8                                # a block far below the column amax
    x[:, 4] = torch.linspace(-1e30, 1e30, R)
    x[:, 5] = 2.0 ** -133                             # S = 2688 / A overflows to inf
    x[::2, 6] = 6.0
    x[1::2, 6] = -0.25
    x[:, 7] = 3.0e38 * torch.sign(x[:, 7])            # amax near the bf16 maximum
    x[:, 8] = x[:, 8] * 1e-37                         # tiny, partly subnormal bf16
    x[300:310, 9] = 3.0e38                            # one huge block in a group of small values
    x[310:, 9] = x[310:, 9] * 1e-30
    for c in range(10, K):
        x[:, c] = x[:, c] * 2.0 ** ((c * 37) % 201 - 100)
    xb = x.to(torch.bfloat16)
    assert torch.isfinite(xb).all()
    ws, st = gpu_offsets(torch.tensor(sizes, dtype=torch.int32), K, R)
    out = mxg.alloc_nvfp4(R, K, device=DEV, rowwise=False, colwise=True, G=G)
    for k in ("q_col", "sf_col"):
        out[k].fill_(0x3C)
    mxg.mxg_group_quantize(mxg.MXG_NVFP4_ROWSCALED, mxg.MXG_COLWISE, xb.to(DEV), R, K, ws, G,
                           None, None, out["q_col"], out["sf_col"], None, st,
                           outer_col=out["outer_col"])
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    offs = np.concatenate([[0], np.cumsum(sizes)])
    ref = oracle.nvfp4_quantize_colwise(xb, offs, R, fill=0x3C)
    assert np.array_equal(out["q_col"].cpu().numpy(), ref["q_col"])
    assert np.array_equal(u8(out["sf_col"]), ref["sf_col"])
    assert np.array_equal(out["outer_col"].cpu().numpy(), ref["outer_col"])
