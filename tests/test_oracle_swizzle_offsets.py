"""Pins for the oracle's scale swizzle and group offsets.

Swizzle: TransformerEngine gemm.py ``swizzled_scale`` defines the layout as a
reshape to (R/128, 4, 32, C/4, 4), an axis permutation (0, 3, 2, 1, 4) and a
flatten, with the colwise scale matrix transposed first.  The oracle writes
that as a flat index formula; here the page's reshape/transpose form is run
with numpy and must agree, plus structural invariants.

Offsets: PR #2763's offsets kernel review thread defines an exclusive prefix
sum of size * last_dim with G + 1 outputs; the workspace review thread lays
out [G sizes | G+1 offsets].  Checked against numpy cumsum, plus the
sanitisation rules of this library for invalid sizes.
"""
import numpy as np
import pytest

import oracle


def page_swizzle(scale: np.ndarray, is_colwise: bool) -> np.ndarray:
    """gemm.py swizzled_scale on a 2-D scale matrix, written with numpy."""
    if is_colwise:
        scale = scale.T
    rows, cols = scale.shape
    return scale.reshape(rows // 128, 4, 32, cols // 4, 4).transpose(0, 3, 2, 1, 4).reshape(-1)


@pytest.mark.parametrize("R,C", [(128, 4), (256, 8), (384, 12), (128, 128), (512, 4)])
def test_swizzle_matches_page_reshape(R, C):
    rng = np.random.default_rng(R * 1000 + C)
    plain = rng.integers(0, 256, (R, C), dtype=np.uint8)
    assert np.array_equal(oracle.swizzle(plain), page_swizzle(plain, False))


@pytest.mark.parametrize("Mb,K", [(4, 128), (8, 256), (12, 384)])
def test_colwise_swizzle_matches_page_reshape(Mb, K):
    # natural colwise scale matrix is [M/32, K]; the page transposes it first
    rng = np.random.default_rng(Mb + K)
    nat = rng.integers(0, 256, (Mb, K), dtype=np.uint8)
    assert np.array_equal(oracle.swizzle(np.ascontiguousarray(nat.T)), page_swizzle(nat, True))


def test_swizzle_is_a_bijection_and_unswizzle_inverts_it():
    R, C = 384, 16
    idx = np.array([[oracle.swizzle_index(r, c, C) for c in range(C)] for r in range(R)])
    assert np.array_equal(np.sort(idx.reshape(-1)), np.arange(R * C))
    rng = np.random.default_rng(2)
    plain = rng.integers(0, 256, (R, C), dtype=np.uint8)
    assert np.array_equal(oracle.unswizzle(oracle.swizzle(plain), R, C), plain)


def test_swizzle_tiles_are_512_contiguous_bytes():
    R, C = 256, 8
    for r0 in range(0, R, 128):
        for c0 in range(0, C, 4):
            idx = [oracle.swizzle_index(r, c, C) for r in range(r0, r0 + 128) for c in range(c0, c0 + 4)]
            base = min(idx)
            assert base % 512 == 0 and sorted(idx) == list(range(base, base + 512))
            assert base == ((r0 // 128) * (C // 4) + c0 // 4) * 512


def test_group_slices_of_global_swizzle_equal_per_group_swizzle():
    # groups aligned to 128 rows: group g's scales are the global swizzled buffer
    # from byte off_g * C on (PR #2763: per-group scale pointer = data offset / 32)
    rng = np.random.default_rng(4)
    sizes = [128, 0, 256, 128, 384]
    C = 8
    R = sum(sizes)
    plain = rng.integers(0, 256, (R, C), dtype=np.uint8)
    glob = oracle.swizzle(plain)
    off = 0
    for s in sizes:
        if s:
            assert np.array_equal(glob[off * C:(off + s) * C], oracle.swizzle(plain[off:off + s]))
        off += s


# --------------------------------------------------------------------------- offsets
@pytest.mark.parametrize("G", [1, 4, 8, 33, 64, 1024])
def test_offsets_closed_form(G):
    rng = np.random.default_rng(G)
    sizes = rng.integers(0, 20, G) * 128
    last_dim = 4096
    ws, st = oracle.group_offsets(sizes.astype(np.int32), 1, last_dim, int(sizes.sum()) + 128)
    assert st == 0
    assert np.array_equal(ws[:G], sizes)
    assert ws[G] == 0
    assert np.array_equal(ws[G + 1:], np.cumsum(sizes) * last_dim)


def test_offsets_multiplier_and_int64_range():
    sizes = np.array([1, 0, 3, 2], np.int64)
    ws, st = oracle.group_offsets(sizes, 128, 7168, 1 << 40)
    assert st == 0
    assert list(ws[:4]) == [128, 0, 384, 256]
    assert list(ws[4:]) == [0, 128 * 7168, 128 * 7168, 512 * 7168, 768 * 7168]
    big = np.array([2 ** 31 - 128, 2 ** 31 - 128], np.int64)
    ws, st = oracle.group_offsets(big, 1, 4096, 1 << 40)
    assert st == 0 and ws[-1] == 2 * (2 ** 31 - 128) * 4096  # needs int64


def test_offsets_sanitisation():
    # negative -> 0, misaligned -> rounded down, over capacity -> cut
    ws, st = oracle.group_offsets(np.array([-128, 200, 256, 512], np.int32), 1, 10, 512)
    assert st == oracle.ST_NEG_SIZE | oracle.ST_MISALIGNED | oracle.ST_SUM_OVER_CAPACITY
    assert list(ws[:4]) == [0, 128, 256, 128]
    assert list(ws[4:]) == [0, 0, 1280, 3840, 5120]
    ws, st = oracle.group_offsets(np.array([0, 0, 0], np.int32), 1, 10, 0)
    assert st == 0 and not ws.any()
