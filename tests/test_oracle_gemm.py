"""Pins for the oracle's grouped GEMM (fprop TN, wgrad NT, row-scaled NVFP4).

* brute-force triple loops over tiny inputs, with operands decoded through
  torch's fp8 dtype and the page's reshape form of the swizzle (no oracle
  decode on that side);
* grouped result = per-expert dense GEMM on byte-identical operands (the
  parity invariant PR #3661's tests state);
* G = 1 reduces to one dense matmul;
* one-hot activations give exact weight entries;
* wgrad per group = dY_g^T X_g on the decoded colwise copies;
* NVFP4: unit outer scales reduce to the plain block-scaled product, and the
  row/column post-scale equals diag(s_row) C diag(s_col).
"""
import numpy as np
import pytest
import torch

import oracle
from moe_grouped_block_gb300 import workloads

E4M3 = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).to(
    torch.float64).numpy()


def page_unswizzle(swz, R, C):
    return np.asarray(swz).reshape(R // 128, C // 4, 32, 4, 4).transpose(0, 3, 2, 1, 4).reshape(R, C)


def decode_mxfp8(q, sf, R, K):
    """Independent decode: torch fp8 table x 2^(byte-127), page-form unswizzle."""
    s = page_unswizzle(sf, R, K // 32).astype(np.float64)
    return E4M3[q] * np.repeat(np.exp2(s - 127.0), 32, axis=1)


def quant_fprop(x, w, G, N, K, M_cap, live):
    qa = oracle.mxfp8_quantize(x, live, M_cap, rowwise=True)
    qb = oracle.mxfp8_quantize(w.reshape(G * N, K), G * N, G * N, rowwise=True)
    return {"q": qa["q_row"], "sf": qa["sf_row"]}, {"q": qb["q_row"], "sf": qb["sf_row"]}


def test_fprop_brute_force_tiny():
    wl = workloads.WORKLOADS["tiny_fprop_mxfp8"].scaled(K=128, N=128)
    inp = workloads.make_inputs(wl)
    G, N, K, M = wl.G, wl.N, wl.K, wl.M
    a, b = quant_fprop(inp["x"], inp["w"], G, N, K, M, M)
    offs = np.concatenate([[0], np.cumsum(inp["sizes"].numpy())])
    alpha = np.array([1.0, 2.0, -0.5, 0.25])
    rows, cols, C = oracle.grouped_gemm_fprop("mxfp8", a, b, offs, N, K, alpha=alpha)
    A = decode_mxfp8(a["q"], a["sf"], M, K)
    B = decode_mxfp8(b["q"], b["sf"], G * N, K)
    rng = np.random.default_rng(0)
    for m in rng.choice(M, 24, replace=False):
        g = int(np.searchsorted(offs, m, side="right") - 1)
        for n in rng.choice(N, 6, replace=False):
            acc = 0.0
            for k in range(K):
                acc += A[m, k] * B[g * N + n, k]
            assert abs(C[m, n] - alpha[g] * acc) <= 1e-12 * max(1.0, abs(acc))


def test_fprop_grouped_equals_per_expert_dense():
    wl = workloads.WORKLOADS["finegrained_fprop_mxfp8"].scaled(K=256, N=128, M=4096, G=16)
    inp = workloads.make_inputs(wl)
    G, N, K, M = wl.G, wl.N, wl.K, wl.M
    sizes = inp["sizes"].numpy()
    a, b = quant_fprop(inp["x"], inp["w"], G, N, K, M, M)
    offs = np.concatenate([[0], np.cumsum(sizes)])
    _, _, C = oracle.grouped_gemm_fprop("mxfp8", a, b, offs, N, K)
    C_sf = page_unswizzle(a["sf"], M, K // 32)
    B_sf = page_unswizzle(b["sf"], G * N, K // 32)
    for g in range(G):
        lo, hi = offs[g], offs[g + 1]
        if hi == lo:
            continue
        # byte-identical per-expert operands, G = 1 call
        ag = {"q": a["q"][lo:hi], "sf": oracle.swizzle(C_sf[lo:hi])}
        bg = {"q": b["q"][g * N:(g + 1) * N], "sf": oracle.swizzle(B_sf[g * N:(g + 1) * N])}
        _, _, Cg = oracle.grouped_gemm_fprop("mxfp8", ag, bg, [0, hi - lo], N, K)
        assert np.array_equal(C[lo:hi], Cg)


def test_fprop_single_group_is_dense_matmul():
    x = workloads.random_bf16((256, 256), seed=21)
    w = workloads.random_bf16((1, 128, 256), seed=22, scale=0.02)
    a, b = quant_fprop(x, w, 1, 128, 256, 256, 256)
    _, _, C = oracle.grouped_gemm_fprop("mxfp8", a, b, [0, 256], 128, 256)
    A = decode_mxfp8(a["q"], a["sf"], 256, 256)
    B = decode_mxfp8(b["q"], b["sf"], 128, 256)
    np.testing.assert_allclose(C, A @ B.T, rtol=1e-13, atol=1e-13)


def test_fprop_one_hot_exact():
    G, N, K = 2, 128, 256
    M = 256
    cols = (np.arange(M) * 37) % K
    xf = np.zeros((M, K), np.float32)
    xf[np.arange(M), cols] = 1.0
    rng = np.random.default_rng(1)
    wf = rng.integers(-8, 9, (G, N, K)).astype(np.float32)
    x = torch.from_numpy(xf).to(torch.bfloat16)
    w = torch.from_numpy(wf).to(torch.bfloat16)
    a, b = quant_fprop(x, w, G, N, K, M, M)
    offs = [0, 128, 256]
    _, _, C = oracle.grouped_gemm_fprop("mxfp8", a, b, offs, N, K)
    for m in range(M):
        g = 0 if m < 128 else 1
        assert np.array_equal(C[m], wf[g, :, cols[m]].astype(np.float64))


def test_fprop_beta_and_sampling():
    wl = workloads.WORKLOADS["tiny_fprop_mxfp8"]
    inp = workloads.make_inputs(wl)
    G, N, K, M = wl.G, wl.N, wl.K, wl.M
    a, b = quant_fprop(inp["x"], inp["w"], G, N, K, M, M)
    offs = np.concatenate([[0], np.cumsum(inp["sizes"].numpy())])
    c_in = np.arange(M * N, dtype=np.float64).reshape(M, N) / (M * N)
    beta = np.array([0.0, 1.0, 2.0, -1.0])
    _, _, C0 = oracle.grouped_gemm_fprop("mxfp8", a, b, offs, N, K)
    _, _, C1 = oracle.grouped_gemm_fprop("mxfp8", a, b, offs, N, K, beta=beta, c_in=c_in)
    g_of_row = np.searchsorted(offs, np.arange(M), side="right") - 1
    np.testing.assert_allclose(C1, C0 + beta[g_of_row][:, None] * c_in, rtol=0, atol=1e-15)
    bias = np.arange(G * N, dtype=np.float64).reshape(G, N) * 0.01
    _, _, Cb = oracle.grouped_gemm_fprop("mxfp8", a, b, offs, N, K, bias=bias)
    np.testing.assert_allclose(Cb, C0 + bias[g_of_row], rtol=0, atol=1e-15)
    rows, cols, Cs = oracle.grouped_gemm_fprop("mxfp8", a, b, offs, N, K, sample_rows=[5, 300, 511],
                                               sample_cols=[0, 7, 255])
    assert np.array_equal(Cs, C0[np.ix_([5, 300, 511], [0, 7, 255])])


def test_wgrad_equals_per_group_transpose_product():
    wl = workloads.WORKLOADS["wgrad_mxfp8"].scaled(K=128, N=256, M=1024, G=4, fixed_sizes=(256, 0, 640, 128),
                                                   sizes="fixed")
    inp = workloads.make_inputs(wl)
    G, N, K, M = wl.G, wl.N, wl.K, wl.M
    qx = oracle.mxfp8_quantize(inp["x"], M, M, rowwise=False, colwise=True)
    qd = oracle.mxfp8_quantize(inp["dy"], M, M, rowwise=False, colwise=True)
    offs = np.concatenate([[0], np.cumsum(inp["sizes"].numpy())])
    ns, ks, dW = oracle.grouped_gemm_wgrad({"q": qd["q_col"], "sf": qd["sf_col"]},
                                           {"q": qx["q_col"], "sf": qx["sf_col"]}, offs, M, N, K)
    dYT = decode_mxfp8(qd["q_col"], qd["sf_col"], N, M)
    XT = decode_mxfp8(qx["q_col"], qx["sf_col"], K, M)
    for g in range(G):
        lo, hi = offs[g], offs[g + 1]
        ref = dYT[:, lo:hi] @ XT[:, lo:hi].T if hi > lo else np.zeros((N, K))
        np.testing.assert_allclose(dW[g], ref, rtol=1e-13, atol=1e-18)
    assert not dW[1].any()  # the empty group
    # brute force on a few entries
    for (g, n, k) in [(0, 3, 5), (2, 255, 127), (3, 100, 0)]:
        lo, hi = offs[g], offs[g + 1]
        acc = sum(dYT[n, m] * XT[k, m] for m in range(lo, hi))
        assert abs(dW[g, n, k] - acc) <= 1e-12 * max(abs(acc), 1e-12)


def _nvfp4_operands(seed, G, N, K, M):
    x = workloads.random_bf16((M, K), seed=seed, dist="student_t3")
    w = workloads.random_bf16((G * N, K), seed=seed + 1, scale=0.02)
    qa = oracle.nvfp4_quantize(x, M, M)
    qb = oracle.nvfp4_quantize(w, G * N, G * N)
    a = {"q": qa["q_row"], "sf": qa["sf_row"], "outer": qa["outer_row"]}
    b = {"q": qb["q_row"], "sf": qb["sf_row"], "outer": qb["outer_row"]}
    return a, b


def _decode_nvfp4_neutral(q, sf, R, K):
    E2M1 = np.array([0, .5, 1, 1.5, 2, 3, 4, 6, -0., -.5, -1, -1.5, -2, -3, -4, -6])
    codes = np.empty((R, K), np.uint8)
    codes[:, 0::2] = q & 0xF
    codes[:, 1::2] = q >> 4
    s = page_unswizzle(sf, R, K // 16)
    return E2M1[codes] * np.repeat(E4M3[s], 16, axis=1)


def test_nvfp4_post_scale_definition():
    G, N, K, M = 2, 128, 256, 384
    a, b = _nvfp4_operands(30, G, N, K, M)
    offs = [0, 256, 384]
    _, _, C = oracle.grouped_gemm_fprop("nvfp4", a, b, offs, N, K)
    A = _decode_nvfp4_neutral(a["q"], a["sf"], M, K)
    B = _decode_nvfp4_neutral(b["q"], b["sf"], G * N, K)
    for g in range(G):
        lo, hi = offs[g], offs[g + 1]
        ref = A[lo:hi] @ B[g * N:(g + 1) * N].T
        ref = ref * a["outer"][lo:hi, None].astype(np.float64) * b["outer"][None, g * N:(g + 1) * N].astype(np.float64)
        np.testing.assert_allclose(C[lo:hi], ref, rtol=1e-12, atol=1e-300)
    # unit outer scales reduce to the plain block-scaled product
    a1 = dict(a, outer=np.ones_like(a["outer"]))
    b1 = dict(b, outer=np.ones_like(b["outer"]))
    _, _, C1 = oracle.grouped_gemm_fprop("nvfp4", a1, b1, offs, N, K)
    np.testing.assert_allclose(C1[:256], A[:256] @ B[:N].T, rtol=1e-13, atol=1e-300)
    # full dequantization (with outer scales) then product gives the same result
    Af = oracle.dequantize("nvfp4", a["q"], a["sf"], M, K, a["outer"])
    Bf = oracle.dequantize("nvfp4", b["q"], b["sf"], G * N, K, b["outer"])
    ref = Af[256:] @ Bf[N:].T  # summation order differs: compare normwise
    assert np.max(np.abs(C[256:] - ref)) <= 1e-12 * np.max(np.abs(ref))


def test_dgrad_brute_force_and_per_expert():
    G, N, K, M = 3, 128, 256, 512
    sizes = [128, 0, 384]
    offs = np.concatenate([[0], np.cumsum(sizes)])
    dy = workloads.random_bf16((M, N), seed=61)
    w = workloads.random_bf16((G * N, K), seed=62, scale=0.02)
    qd = oracle.mxfp8_quantize(dy, M, M, rowwise=True)
    qwt = oracle.mxfp8_quantize(w, G * N, G * N, rowwise=False, colwise=True)
    alpha = [2.0, 1.0, -0.5]
    rows, cols, dX = oracle.grouped_gemm_dgrad({"q": qd["q_row"], "sf": qd["sf_row"]},
                                               {"q": qwt["q_col"], "sf": qwt["sf_col"]}, offs,
                                               G, N, K, alpha=alpha)
    A = decode_mxfp8(qd["q_row"], qd["sf_row"], M, N)           # [M, N]
    WT = decode_mxfp8(qwt["q_col"], qwt["sf_col"], K, G * N)     # [K, G*N]
    for g in range(G):
        lo, hi = offs[g], offs[g + 1]
        if hi > lo:
            ref = alpha[g] * (A[lo:hi] @ WT[:, g * N:(g + 1) * N].T)
            assert np.max(np.abs(dX[lo:hi] - ref)) <= 1e-13 * np.max(np.abs(ref))
    for (m, k) in [(0, 0), (127, 255), (200, 17), (511, 100)]:
        g = int(np.searchsorted(offs, m, side="right") - 1)
        acc = sum(A[m, n] * WT[k, g * N + n] for n in range(N))
        assert abs(dX[m, k] - alpha[g] * acc) <= 1e-12 * max(1.0, abs(acc))
    # the colwise weight blocks run along N: each 32-block of a column of W_g
    # shares one scale, so quantizing W_g^T rowwise gives the same bytes
    wt = torch.from_numpy(w.float().numpy()[:N].T.copy()).to(torch.bfloat16)
    qr = oracle.mxfp8_quantize(wt, K, K, rowwise=True)
    assert np.array_equal(qr["q_row"], qwt["q_col"][:, :N])


def test_nvfp4_wgrad_brute_force():
    G, N, K, M = 3, 128, 128, 512
    offs = np.array([0, 256, 256, 512])
    x = workloads.random_bf16((M, K), seed=81, dist="student_t3")
    dy = workloads.random_bf16((M, N), seed=82, scale=1e-3)
    qx = oracle.nvfp4_quantize_colwise(x, offs, M)
    qd = oracle.nvfp4_quantize_colwise(dy, offs, M)
    a = {"q": qd["q_col"], "sf": qd["sf_col"], "outer": qd["outer_col"]}
    b = {"q": qx["q_col"], "sf": qx["sf_col"], "outer": qx["outer_col"]}
    ns, ks, dW = oracle.grouped_gemm_wgrad(a, b, offs, M, N, K, fmt="nvfp4")
    DT = _decode_nvfp4_neutral(qd["q_col"], qd["sf_col"], N, M)   # [N, M]
    XT = _decode_nvfp4_neutral(qx["q_col"], qx["sf_col"], K, M)   # [K, M]
    assert not dW[1].any()
    for (g, n, k) in [(0, 0, 0), (0, 127, 5), (2, 64, 127), (2, 3, 99)]:
        lo, hi = offs[g], offs[g + 1]
        acc = sum(DT[n, m] * XT[k, m] for m in range(lo, hi))
        ref = acc * float(qd["outer_col"][g, n]) * float(qx["outer_col"][g, k])
        assert abs(dW[g, n, k] - ref) <= 1e-12 * max(abs(ref), 1e-30)
    # against the full dequantization (outer scale per group and column)
    for g in (0, 2):
        lo, hi = offs[g], offs[g + 1]
        Df = DT[:, lo:hi] * qd["outer_col"][g][:, None].astype(np.float64)
        Xf = XT[:, lo:hi] * qx["outer_col"][g][:, None].astype(np.float64)
        ref = Df @ Xf.T
        assert np.max(np.abs(dW[g] - ref)) <= 1e-12 * np.max(np.abs(ref))
