"""Pins for the oracle's element codecs and the MXFP8 scale rule (R1).

Each codec is checked against something other than itself: torch's own fp8 /
e8m0 dtypes, ml_dtypes' fp4 dtype (where installed) and brute-force
nearest-value search over the full code book with ties to the even code.
"""
import numpy as np
import pytest
import torch

import oracle


def _all_bf16_finite() -> np.ndarray:
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint32) << 16
    v = bits.view(np.float32)
    return v[np.isfinite(v)].astype(np.float64)


def _brute_round(values: np.ndarray, grid_vals: np.ndarray, grid_codes: np.ndarray,
                 even: np.ndarray, sat: float) -> np.ndarray:
    """Nearest code by exhaustive search; a tie goes to the code with an even
    mantissa; magnitudes above the largest value saturate."""
    out = np.empty(values.size, np.int64)
    for i, v in enumerate(values):
        a = min(abs(v), sat)
        d = np.abs(grid_vals - a)
        best = np.nonzero(d == d.min())[0]
        if best.size > 1:
            best = best[even[best]]
        c = int(grid_codes[best[0]])
        out[i] = c
    return out


# --------------------------------------------------------------------------- E4M3
def test_e4m3_decode_matches_torch():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    mine = oracle.e4m3_decode_table()
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(mine))
    assert nan.sum() == 2  # 0x7F and 0xFF
    assert np.array_equal(ref[~nan], mine[~nan])
    assert mine[0x7E] == 448.0 and mine[0x01] == 2.0 ** -9 and mine[0x08] == 2.0 ** -6


def test_e4m3_encode_brute_force():
    # magnitude grid of the positive codes 0x00..0x7E
    vals = np.array([oracle.e4m3_decode(c) for c in range(0x7F)])
    codes = np.arange(0x7F)
    even = (codes & 1) == 0
    rng = np.random.default_rng(11)
    mids = (vals[1:] + vals[:-1]) / 2
    probe = np.concatenate([
        vals, mids, np.nextafter(mids, 0), np.nextafter(mids, 1e9),
        rng.uniform(0, 500, 4000), np.exp2(rng.uniform(-14, 9, 4000)), [447.9, 448, 460, 464, 470, 1e6],
    ])
    probe = np.concatenate([probe, -probe])
    brute = _brute_round(probe, vals, codes, even, 448.0)
    brute = brute | np.where(np.signbit(probe), 0x80, 0)
    mine = oracle.e4m3_encode_array(probe)
    bad = np.nonzero(mine != brute)[0]
    assert bad.size == 0, [(probe[i], mine[i], brute[i]) for i in bad[:5]]


def test_e4m3_encode_matches_torch_on_all_bf16_in_range():
    v = _all_bf16_finite()
    v = v[np.abs(v) <= 448.0]
    ref = torch.from_numpy(v.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    mine = oracle.e4m3_encode_array(v)
    assert np.array_equal(mine, ref)


def test_e4m3_encode_signed_zero_and_saturation():
    assert oracle.e4m3_encode(-0.0) == 0x80
    assert oracle.e4m3_encode(-1e-30) == 0x80
    assert oracle.e4m3_encode(1e30) == 0x7E
    assert oracle.e4m3_encode(-1e30) == 0xFE
    assert oracle.e4m3_encode(2.0 ** -10) == 0x00      # tie 0 / 2^-9 -> even (0)
    assert oracle.e4m3_encode(3 * 2.0 ** -10) == 0x02  # tie 1 / 2 (x 2^-9) -> even (2)


# --------------------------------------------------------------------------- E2M1
E2M1_VALUES = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_e2m1_decode_table():
    t = oracle.e2m1_decode_table()
    assert list(t[:8]) == E2M1_VALUES
    assert list(-t[8:]) == E2M1_VALUES
    assert np.signbit(t[8])


def test_e2m1_encode_brute_force_and_ties():
    vals = np.array(E2M1_VALUES)
    codes = np.arange(8)
    even = (codes & 1) == 0
    rng = np.random.default_rng(5)
    mids = (vals[1:] + vals[:-1]) / 2
    probe = np.concatenate([vals, mids, np.nextafter(mids, 0), np.nextafter(mids, 10),
                            rng.uniform(0, 8, 5000), [6.5, 7.0, 100.0]])
    probe = np.concatenate([probe, -probe])
    brute = _brute_round(probe, vals, codes, even, 6.0) | np.where(np.signbit(probe), 8, 0)
    mine = oracle.e2m1_encode_array(probe)
    assert np.array_equal(mine, brute)
    # the tie table of the rule: 0.25->0, 0.75->1, 1.25->1, 1.75->2, 2.5->2, 3.5->4, 5->4
    for v, want in [(0.25, 0.0), (0.75, 1.0), (1.25, 1.0), (1.75, 2.0), (2.5, 2.0), (3.5, 4.0),
                    (5.0, 4.0), (7.0, 6.0)]:
        assert oracle.e2m1_decode(oracle.e2m1_encode(v)) == want


def test_e2m1_matches_ml_dtypes():
    ml = pytest.importorskip("ml_dtypes")
    rng = np.random.default_rng(3)
    v = np.concatenate([rng.uniform(-6, 6, 20000), np.linspace(-6, 6, 4801)])
    ref = v.astype(ml.float4_e2m1fn).astype(np.float64)
    mine = np.array([oracle.e2m1_decode(c) for c in oracle.e2m1_encode_array(v)])
    assert np.array_equal(ref, mine)


# --------------------------------------------------------------------------- E8M0
def test_e8m0_decode_matches_torch():
    codes = torch.arange(255, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    mine = np.array([oracle.e8m0_decode(b) for b in range(255)])
    assert np.array_equal(ref, mine)
    assert np.isnan(oracle.e8m0_decode(0xFF))


# --------------------------------------------------------------------------- R1
def _r1_literal(amax: float) -> int:
    """The R1 definition read literally: the smallest e in [-127, 127] with
    amax <= 448 * 2^e (e = -127 for an all-zero block)."""
    for e in range(-127, 128):
        if amax <= 448.0 * 2.0 ** e:
            return e
    return 127


def test_r1_scale_rule_literal_definition():
    rng = np.random.default_rng(0)
    am = np.concatenate([
        np.abs(_all_bf16_finite())[::7],
        [0.0, 448.0, np.nextafter(np.float32(448), np.float32(0)), np.nextafter(np.float32(448), np.float32(1e9)),
         1.75, 1.7500001, 2.0 ** -126, 2.0 ** -133, 3.3895e38],
        np.exp2(rng.uniform(-140, 127, 2000)),
    ]).astype(np.float32)
    mine = oracle.mx_scale_exponent_array(am)
    want = np.array([_r1_literal(float(a)) for a in am])
    assert np.array_equal(mine, want)


def test_r1_invariants():
    rng = np.random.default_rng(1)
    am = np.exp2(rng.uniform(-120, 120, 50000)).astype(np.float32)
    e = oracle.mx_scale_exponent_array(am).astype(np.float64)
    a = am.astype(np.float64)
    assert np.all(a <= 448.0 * np.exp2(e))
    assert np.all((e == -127) | (a > 448.0 * np.exp2(e - 1)))
    assert oracle.mx_scale_exponent(0.0) == -127
    assert oracle.mx_scale_exponent(448.0) == 0
    assert oracle.mx_scale_exponent(448.0 * 1.0000001) == 1
    assert oracle.mx_scale_exponent(1.0) == -8  # 1 <= 448 * 2^-8 = 1.75
