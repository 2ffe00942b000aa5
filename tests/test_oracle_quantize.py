"""Pins for the oracle's MXFP8 (R1) and row-scaled NVFP4 (R2) quantizers and
its dequantizer.

Independent checks: a brute-force quantizer on tiny inputs (literal scale
definition + exhaustive nearest-code search, values decoded through torch's
fp8 dtype and the page's reshape form of the swizzle), the colwise = rowwise
of the transpose invariant, value idempotence, the E4M3 error bound, the
NVFP4 outer-scale closed form from gemm.py ``_get_nvfp4_tensor_scale_inv``
(amax / (6 * 448)) and its single-element special case.
"""
import numpy as np
import pytest
import torch

import oracle
from moe_grouped_block_gb300 import workloads

E4M3_POS = torch.arange(0x7F, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).to(
    torch.float64).numpy()
E2M1_POS = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def _nearest(a: float, grid: np.ndarray) -> int:
    d = np.abs(grid - a)
    best = np.nonzero(d == d.min())[0]
    if best.size > 1:
        best = best[(best & 1) == 0]
    return int(best[0])


def _f32(x_bf16: torch.Tensor) -> np.ndarray:
    return x_bf16.to(torch.float32).numpy()


def page_unswizzle(swz: np.ndarray, R: int, C: int) -> np.ndarray:
    """Inverse of gemm.py swizzled_scale's reshape/transpose, with numpy."""
    return swz.reshape(R // 128, C // 4, 32, 4, 4).transpose(0, 3, 2, 1, 4).reshape(R, C)


def brute_mxfp8_rowwise(x: np.ndarray):
    R, K = x.shape
    q = np.zeros((R, K), np.uint8)
    sf = np.zeros((R, K // 32), np.uint8)
    for r in range(R):
        for b in range(K // 32):
            blk = x[r, b * 32:(b + 1) * 32].astype(np.float64)
            amax = np.abs(blk).max()
            e = next(e for e in range(-127, 128) if amax <= 448.0 * 2.0 ** e)
            sf[r, b] = e + 127
            for i, v in enumerate(blk):
                code = _nearest(min(abs(v) * 2.0 ** -e, 448.0), E4M3_POS)
                q[r, b * 32 + i] = code | (0x80 if np.signbit(v) else 0)
    return q, sf


def test_mxfp8_rowwise_brute_force_tiny():
    x = workloads.random_bf16((128, 128), seed=1, scale=3.0)
    xf = _f32(x)
    xf[5, :32] = 0.0          # an all-zero block
    xf[6, 40] = -0.0
    xf[7, 64:96] = 2.0 ** -130  # subnormal block
    xf[8, 96:128] *= 1e30     # huge block
    x = torch.from_numpy(xf).to(torch.bfloat16)
    xf = _f32(x)
    got = oracle.mxfp8_quantize(x, 128, 128, rowwise=True)
    q_b, sf_b = brute_mxfp8_rowwise(xf)
    assert np.array_equal(got["q_row"], q_b)
    assert np.array_equal(page_unswizzle(got["sf_row"], 128, 4), sf_b)


def test_mxfp8_colwise_is_rowwise_of_transpose():
    x = workloads.random_bf16((256, 384), seed=2)
    both = oracle.mxfp8_quantize(x, 256, 256, rowwise=True, colwise=True)
    xt = x.t().contiguous()
    rowT = oracle.mxfp8_quantize(xt, 384, 384, rowwise=True)
    assert np.array_equal(both["q_col"], rowT["q_row"])
    assert np.array_equal(both["sf_col"], rowT["sf_row"])


def test_mxfp8_live_rows_only_and_rows_beyond_untouched():
    x = workloads.random_bf16((256, 128), seed=3)
    full = oracle.mxfp8_quantize(x, 256, 256, rowwise=True, colwise=True)
    part = oracle.mxfp8_quantize(x, 128, 256, rowwise=True, colwise=True, fill=0xAB)
    assert np.array_equal(part["q_row"][:128], full["q_row"][:128])
    assert np.all(part["q_row"][128:] == 0xAB)
    C = 128 // 32
    assert np.array_equal(part["sf_row"][:128 * C], full["sf_row"][:128 * C])
    assert np.all(part["sf_row"][128 * C:] == 0xAB)
    assert np.array_equal(part["q_col"][:, :128], full["q_col"][:, :128])
    assert np.all(part["q_col"][:, 128:] == 0xAB)
    sfc = page_unswizzle(part["sf_col"], 128, 256 // 32)
    sfc_full = page_unswizzle(full["sf_col"], 128, 256 // 32)
    assert np.array_equal(sfc[:, :4], sfc_full[:, :4]) and np.all(sfc[:, 4:] == 0xAB)


def test_mxfp8_dequant_value_idempotent_and_error_bound():
    x = workloads.random_bf16((256, 256), seed=4, scale=10.0, dist="student_t3")
    xf = _f32(x).astype(np.float64)
    q = oracle.mxfp8_quantize(x, 256, 256, rowwise=True)
    dq = oracle.dequantize("mxfp8", q["q_row"], q["sf_row"], 256, 256)
    # the dequantized values are bf16-representable here (<= 4 significant bits)
    x2 = torch.from_numpy(dq.astype(np.float32)).to(torch.bfloat16)
    assert np.array_equal(_f32(x2).astype(np.float64), dq)
    q2 = oracle.mxfp8_quantize(x2, 256, 256, rowwise=True)
    dq2 = oracle.dequantize("mxfp8", q2["q_row"], q2["sf_row"], 256, 256)
    assert np.array_equal(dq, dq2)
    sf = page_unswizzle(q["sf_row"], 256, 8).astype(np.float64)
    scale = np.repeat(np.exp2(sf - 127), 32, axis=1)
    normal = np.abs(xf) / scale >= 2.0 ** -6
    err = np.abs(dq - xf)
    assert np.all(err[normal] <= 2.0 ** -4 * np.abs(xf[normal]))
    assert np.all(err[~normal] <= 2.0 ** -10 * scale[~normal])


def test_mxfp8_exactly_representable_round_trip():
    # integers times powers of two with <= 4 significant bits and a block
    # range inside E4M3's are reproduced exactly
    rng = np.random.default_rng(9)
    m = rng.integers(-15, 16, (128, 128)).astype(np.float32)
    x = torch.from_numpy(m * 2.0 ** -3).to(torch.bfloat16)
    q = oracle.mxfp8_quantize(x, 128, 128, rowwise=True)
    dq = oracle.dequantize("mxfp8", q["q_row"], q["sf_row"], 128, 128)
    assert np.array_equal(dq, (m * 2.0 ** -3).astype(np.float64))


# --------------------------------------------------------------------------- NVFP4
def brute_nvfp4_rowwise(xf: np.ndarray):
    R, K = xf.shape
    f32 = np.float32
    q = np.zeros((R, K), np.uint8)  # one code per element before packing
    sf = np.zeros((R, K // 16), np.uint8)
    outer = np.zeros(R, np.float32)
    for r in range(R):
        A = f32(np.abs(xf[r]).max())
        if A == 0:
            q[r] = np.where(np.signbit(xf[r]), 8, 0)
            continue
        outer[r] = f32(A / f32(2688.0))
        S = f32(f32(2688.0) / A)
        for b in range(K // 16):
            blk = xf[r, b * 16:(b + 1) * 16]
            t = f32(f32(f32(np.abs(blk).max()) / f32(6.0)) * S)
            code = _nearest(min(float(t), 448.0), E4M3_POS)
            sf[r, b] = code
            sbv = f32(E4M3_POS[code])
            for i, v in enumerate(blk):
                sign = 8 if np.signbit(v) else 0
                if sbv == 0:
                    q[r, b * 16 + i] = sign
                else:
                    vv = f32(f32(v) * f32(S / sbv))
                    q[r, b * 16 + i] = _nearest(min(abs(float(vv)), 6.0), E2M1_POS) | sign
    packed = (q[:, 0::2] | (q[:, 1::2] << 4)).astype(np.uint8)
    return packed, sf, outer


def test_nvfp4_brute_force_tiny():
    x = workloads.random_bf16((128, 256), seed=5, dist="student_t3")
    xf = _f32(x)
    xf[3] = 0.0
    xf[4, 17] = -0.0
    xf[9, 32:48] = 1e-8  # a block far below the row amax (its scale rounds to 0)
    x = torch.from_numpy(xf).to(torch.bfloat16)
    xf = _f32(x)
    got = oracle.nvfp4_quantize(x, 128, 128)
    qb, sfb, ob = brute_nvfp4_rowwise(xf)
    assert np.array_equal(got["q_row"], qb)
    assert np.array_equal(page_unswizzle(got["sf_row"], 128, 16), sfb)
    assert np.array_equal(got["outer_row"], ob)


def test_nvfp4_outer_scale_closed_form_and_scale_range():
    x = workloads.random_bf16((256, 512), seed=6, dist="student_t3")
    xf = _f32(x)
    got = oracle.nvfp4_quantize(x, 256, 256)
    amax = np.abs(xf).max(axis=1)
    assert np.array_equal(got["outer_row"], (amax / np.float32(6.0 * 448.0)).astype(np.float32))
    assert np.all(got["sf_row"] <= 0x7E)  # UE4M3: sign clear, finite


def test_nvfp4_single_nonzero_row():
    xf = np.zeros((128, 128), np.float32)
    for r in range(128):
        xf[r, (r * 7) % 128] = (r + 1) * (-1.0 if r % 2 else 1.0) * 0.37
    x = torch.from_numpy(xf).to(torch.bfloat16)
    xf = _f32(x)
    got = oracle.nvfp4_quantize(x, 128, 128)
    sf = page_unswizzle(got["sf_row"], 128, 8)
    for r in range(128):
        c = (r * 7) % 128
        assert sf[r, c // 16] == 0x7E  # 448
        assert np.count_nonzero(sf[r]) == 1
        byte = got["q_row"][r, c // 2]
        nib = (byte >> 4) if c % 2 else (byte & 0xF)
        assert nib == (0xF if xf[r, c] < 0 else 0x7)  # +-6


def test_nvfp4_error_bound_and_nibble_order():
    x = workloads.random_bf16((128, 256), seed=7, dist="student_t3")
    xf = _f32(x).astype(np.float64)
    got = oracle.nvfp4_quantize(x, 128, 128)
    dq = oracle.dequantize("nvfp4", got["q_row"], got["sf_row"], 128, 256, got["outer_row"])
    blk_amax = np.repeat(np.abs(xf).reshape(128, 16, 16).max(axis=2), 16, axis=1)
    assert np.all(np.abs(dq - xf) <= blk_amax / 6.0 * 1.1 + 1e-30)
    # relative error is small on average for heavy-tailed rows
    assert np.mean(np.abs(dq - xf)) < 0.2 * np.mean(np.abs(xf))


# --------------------------------------------------------------------------- NVFP4 colwise
def test_nvfp4_colwise_single_group_is_rowwise_of_transpose():
    x = workloads.random_bf16((256, 384), seed=13, dist="student_t3")
    col = oracle.nvfp4_quantize_colwise(x, [0, 256], 256)
    xt = x.t().contiguous()
    row = oracle.nvfp4_quantize(xt, 384, 384)
    assert np.array_equal(col["q_col"], row["q_row"])
    assert np.array_equal(col["sf_col"], row["sf_row"])
    assert np.array_equal(col["outer_col"][0], row["outer_row"])


def test_nvfp4_colwise_groups_brute_force():
    R, K = 512, 128
    x = workloads.random_bf16((R, K), seed=14, dist="student_t3").to(torch.float32)
    x[:, 5] = 0.0          # a zero column in every group
    x[128:256, 7] = -0.0
    xb = x.to(torch.bfloat16)
    offs = [0, 128, 128, 384, 512]  # includes an empty group
    col = oracle.nvfp4_quantize_colwise(xb, offs, R)
    sf = page_unswizzle(col["sf_col"], K, R // 16)
    for g in range(4):
        lo, hi = offs[g], offs[g + 1]
        if hi == lo:
            assert np.all(col["outer_col"][g] == 0.0)
            continue
        slab = _f32(xb)[lo:hi].T.copy()  # [K, rows of g]
        qb, sfb, ob = brute_nvfp4_rowwise(slab)
        assert np.array_equal(col["q_col"][:, lo // 2:hi // 2], qb)
        assert np.array_equal(sf[:, lo // 16:hi // 16], sfb)
        assert np.array_equal(col["outer_col"][g], ob)
