"""Pins for the oracle of groups of any size (MXFP8).

Each check ties the unaligned oracle to something other than itself: the
aligned (already pinned) oracle where the two must agree, the grouping-
independence of rowwise quantization, the R1 rule written as a closed form
for an isolated row, and exact-integer inputs whose whole quantize + GEMM
pipeline must equal a plain fp64 product over each group's original rows --
so a wrong offset, a leaked padding row or a block spanning two groups fails.
"""
import numpy as np
import pytest
import torch

import oracle


def _bf16(a):
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16)

def _ws(sizes, cap, last_dim=1):
    ws, st = oracle.group_offsets_unaligned(np.asarray(sizes), 1, last_dim, cap)
    return ws, st

def test_offsets_brute_force():
    ws, st = _ws([5, 0, 300, 7], 512, last_dim=3)
    G = 4
    assert st == 0
    assert list(ws[:G]) == [5, 0, 300, 7]
    assert list(ws[G:]) == [0, 15, 15, 915, 936]
    # negative -> 0, running sum capped at the capacity
    ws, st = _ws([-3, 200, 400, 9], 512)
    assert st == oracle.ST_NEG_SIZE | oracle.ST_SUM_OVER_CAPACITY
    assert list(ws[:4]) == [0, 200, 312, 0]
    # no MISALIGNED bit and no rounding, unlike the aligned rule
    ws_a, st_a = oracle.group_offsets(np.array([5, 300]), 1, 1, 512)
    assert st_a & oracle.ST_MISALIGNED and list(ws_a[:2]) == [0, 256]

def test_offsets_equal_aligned_rule_on_multiples_of_128():
    sizes = np.array([128, 0, 384, 256, 128])
    for cap in (1024, 768):
        a = oracle.group_offsets(sizes, 1, 64, cap)
        u = oracle.group_offsets_unaligned(sizes, 1, 64, cap)
        assert np.array_equal(a[0], u[0]) and a[1] == u[1]

def test_padded_rows():
    ws, _ = _ws([5, 0, 300, 128, 1], 1024)
    assert list(oracle.padded_rows(ws, 5)) == [0, 128, 128, 512, 640, 768]

def _x(rows, cols, seed):
    return _bf16(np.random.default_rng(seed).standard_normal((rows, cols)))

def test_quantize_reduces_to_aligned_on_multiples_of_128():
    R, K = 768, 256
    x = _x(R, K, 1)
    sizes = np.array([128, 0, 384, 128])
    ws, _ = _ws(sizes, R)
    u = oracle.mxfp8_quantize_unaligned(x, ws, 4, R, rowwise=True, colwise=True, fill=0x5A)
    a = oracle.mxfp8_quantize(x, 640, R, rowwise=True, colwise=True, fill=0x5A)
    Rp = oracle.unaligned_rows_capacity(R, 4)
    assert np.array_equal(u["q_row"], a["q_row"])
    # the padded buffers are longer; their first R rows equal the aligned ones
    C = K // 32
    assert np.array_equal(oracle.unswizzle(u["sf_row"], Rp, C)[:R],
                          oracle.unswizzle(a["sf_row"], R, C))
    assert np.array_equal(u["q_col"][:, :R], a["q_col"])
    assert np.array_equal(oracle.unswizzle(u["sf_col"], K, Rp // 32)[:, :R // 32],
                          oracle.unswizzle(a["sf_col"], K, R // 32))

def test_rowwise_data_and_scales_do_not_depend_on_grouping():
    R, K = 512, 128
    x = _x(R, K, 2)
    sizes = np.array([37, 0, 129, 200])
    ws, _ = _ws(sizes, R)
    live = int(sizes.sum())
    u = oracle.mxfp8_quantize_unaligned(x, ws, 4, R, rowwise=True, fill=0x11)
    d = oracle.mxfp8_quantize(x, R, R, rowwise=True)
    assert np.array_equal(u["q_row"][:live], d["q_row"][:live])
    assert (u["q_row"][live:] == 0x11).all()
    Rp = oracle.unaligned_rows_capacity(R, 4)
    C = K // 32
    su, sd = oracle.unswizzle(u["sf_row"], Rp, C), oracle.unswizzle(d["sf_row"], R, C)
    offs, poffs = oracle.live_rows(ws, 4), oracle.padded_rows(ws, 4)
    for g in range(4):
        m = int(sizes[g])
        assert np.array_equal(su[poffs[g]:poffs[g] + m], sd[offs[g]:offs[g] + m])
        P = (m + 127) // 128 * 128
        assert (su[poffs[g] + m:poffs[g] + P] == 0).all()  # padding rows: byte 0

def test_colwise_blocks_start_at_each_group():
    # group 0 = 33 rows of small values, group 1 = 31 rows of large ones: a
    # dense colwise quantize would mix row 32 with group 1 in one 32-row
    # block; per-group blocks give row 32 a block (and a scale) of its own
    R, K = 128, 128
    rng = np.random.default_rng(3)
    xs = np.concatenate([rng.uniform(-1, 1, (33, K)), rng.uniform(-1000, 1000, (31, K)),
                         np.zeros((64, K))])
    x = _bf16(xs)
    ws, _ = _ws([33, 31], R)
    u = oracle.mxfp8_quantize_unaligned(x, ws, 2, R, colwise=True, rowwise=False)
    Rp = oracle.unaligned_rows_capacity(R, 2)
    sf = oracle.unswizzle(u["sf_col"], K, Rp // 32)
    xb = x.float().numpy()
    for k in range(K):
        # closed form of R1 for the one-row block: e = ceil(log2(|x| / 448))
        a = abs(float(xb[32, k]))
        e = -127 if a == 0 else max(-127, int(np.ceil(np.log2(a / 448.0) - 1e-12)))
        assert sf[k, 1] == e + 127
        assert (sf[k, 2:4] == 0).all()           # group 0's padding blocks
        assert sf[k, 4] == oracle.mx_scale_exponent(float(np.abs(xb[33:64, k]).max())) + 127
    assert (u["q_col"][:, 33:128] == 0).all()    # padding columns of group 0
    assert (u["q_col"][:, 128 + 31:256] == 0).all()

def _int_inputs(rows, cols, seed):
    # entries in {-2, ..., 2}: every 1x32 / 32x1 block quantizes exactly
    # (amax 1 or 2 -> scaled values 128 or 256, both E4M3 values)
    return np.random.default_rng(seed).integers(-2, 3, (rows, cols)).astype(np.float32)

@pytest.mark.parametrize("sizes", [(37, 0, 129, 200), (1, 127, 128, 255), (300,)])
def test_fprop_exact_integers(sizes):
    G, N, K = len(sizes), 128, 256
    R = 640
    xs = _int_inputs(R, K, 4)
    ws_ = _int_inputs(G * N, K, 5)
    ws, _ = _ws(sizes, R)
    qa = oracle.mxfp8_quantize_unaligned(_bf16(xs), ws, G, R, rowwise=True)
    qb = oracle.mxfp8_quantize(_bf16(ws_), G * N, G * N, rowwise=True)
    rows, C = oracle.grouped_gemm_fprop_unaligned({"q": qa["q_row"], "sf": qa["sf_row"]},
                                                  {"q": qb["q_row"], "sf": qb["sf_row"]},
                                                  ws, G, N, K)
    offs = oracle.live_rows(ws, G)
    for g in range(G):
        lo, hi = offs[g], offs[g + 1]
        ref = xs[lo:hi].astype(np.float64) @ ws_[g * N:(g + 1) * N].astype(np.float64).T
        assert np.array_equal(C[lo:hi], ref)

@pytest.mark.parametrize("sizes", [(37, 0, 129, 200), (1, 127, 128, 255)])
def test_wgrad_exact_integers(sizes):
    G, N, K = len(sizes), 128, 256
    R = 640
    xs = _int_inputs(R, K, 6)
    dys = _int_inputs(R, N, 7)
    ws, _ = _ws(sizes, R)
    qx = oracle.mxfp8_quantize_unaligned(_bf16(xs), ws, G, R, rowwise=False, colwise=True)
    qd = oracle.mxfp8_quantize_unaligned(_bf16(dys), ws, G, R, rowwise=False, colwise=True)
    _, _, dW = oracle.grouped_gemm_wgrad_unaligned({"q": qd["q_col"], "sf": qd["sf_col"]},
                                                   {"q": qx["q_col"], "sf": qx["sf_col"]},
                                                   ws, G, R, N, K)
    offs = oracle.live_rows(ws, G)
    for g in range(G):
        lo, hi = offs[g], offs[g + 1]
        ref = dys[lo:hi].astype(np.float64).T @ xs[lo:hi].astype(np.float64)
        assert np.array_equal(dW[g], ref)

def test_dgrad_exact_integers():
    sizes = (37, 0, 129, 200)
    G, N, K = 4, 128, 256
    R = 512
    dys = _int_inputs(R, N, 8)
    w = _int_inputs(G * N, K, 9)
    ws, _ = _ws(sizes, R)
    qd = oracle.mxfp8_quantize_unaligned(_bf16(dys), ws, G, R, rowwise=True)
    qwt = oracle.mxfp8_quantize(_bf16(w), G * N, G * N, rowwise=False, colwise=True)
    rows, dX = oracle.grouped_gemm_dgrad_unaligned({"q": qd["q_row"], "sf": qd["sf_row"]},
                                                   {"q": qwt["q_col"], "sf": qwt["sf_col"]},
                                                   ws, G, N, K)
    offs = oracle.live_rows(ws, G)
    for g in range(G):
        lo, hi = offs[g], offs[g + 1]
        ref = dys[lo:hi].astype(np.float64) @ w[g * N:(g + 1) * N].astype(np.float64)
        assert np.array_equal(dX[lo:hi], ref)

def test_fprop_matches_dense_rowwise_product():
    # layout independence: the unaligned fprop equals the product of the
    # dense rowwise quantization (scales are per row, whatever the groups)
    sizes = (37, 0, 129, 200)
    G, N, K, R = 4, 128, 256, 512
    x, w = _x(R, K, 10), _x(G * N, K, 11)
    ws, _ = _ws(sizes, R)
    qa = oracle.mxfp8_quantize_unaligned(x, ws, G, R, rowwise=True)
    qd = oracle.mxfp8_quantize(x, R, R, rowwise=True)
    qb = oracle.mxfp8_quantize(w, G * N, G * N, rowwise=True)
    _, C = oracle.grouped_gemm_fprop_unaligned({"q": qa["q_row"], "sf": qa["sf_row"]},
                                               {"q": qb["q_row"], "sf": qb["sf_row"]}, ws, G, N, K)
    offs = oracle.live_rows(ws, G)
    Bd = oracle.dequantize("mxfp8", qb["q_row"], qb["sf_row"], G * N, K)
    Ad = oracle.dequantize("mxfp8", qd["q_row"], qd["sf_row"], R, K)
    for g in range(G):
        lo, hi = offs[g], offs[g + 1]
        ref = Ad[lo:hi] @ Bd[g * N:(g + 1) * N].T
        assert np.allclose(C[lo:hi], ref, rtol=1e-12, atol=1e-12)
