"""Pins for the oracle's uniform quantiser, fp32 FMA emulation and code packing."""

import json
import os
from fractions import Fraction

import numpy as np
import pytest

from oracle import quant

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "hand_cases.json")))


def exact_round_f32(v: Fraction) -> np.float32:
    """Correct RNE rounding of an exact rational to fp32 (independent of the oracle)."""
    r0 = np.float32(float(v))
    cands = {float(r0), float(np.nextafter(r0, np.float32(np.inf))),
             float(np.nextafter(r0, np.float32(-np.inf)))}
    best = None
    for c in sorted(cands):
        dist = abs(Fraction(c) - v)
        if best is None or dist < best[0]:
            best = (dist, c)
        elif dist == best[0]:
            # tie: choose the even significand
            m_c = np.float32(c).view(np.uint32) & 1
            if m_c == 0:
                best = (dist, c)
    return np.float32(best[1])


@pytest.mark.parametrize("case", GOLD["uniform_quant"])
def test_hand_cases(case):
    x = np.array(case["x"], np.float32)
    codes, s, z = quant.quantize_groups(x, case["bits"])
    assert codes.tolist() == case["codes"]
    assert float(s) == case["s"]
    assert float(z) == case["z"]
    if case["z"] == 0.0:
        assert not np.signbit(z)
    xh = quant.dequantize(codes, s, z)
    assert xh.tolist() == case["xhat"]


def test_fma32_matches_exact_rounding_random():
    rng = np.random.default_rng(0)
    n = 4000
    a = rng.integers(0, 16, n).astype(np.float32)
    b = (rng.standard_normal(n) * np.exp(rng.uniform(-20, 20, n))).astype(np.float32)
    c = (rng.standard_normal(n) * np.exp(rng.uniform(-20, 20, n))).astype(np.float32)
    got = quant.fma32(a, b, c)
    for i in range(n):
        want = exact_round_f32(Fraction(float(a[i])) * Fraction(float(b[i])) + Fraction(float(c[i])))
        assert got[i] == want, (a[i], b[i], c[i], got[i], want)


def test_fma32_double_rounding_cases():
    # a*b lands exactly on an fp32 midpoint and c is far below fp64 precision of
    # the product: fp64-then-fp32 would round to even, the true FMA must not.
    b = np.float32(1.0 + 2.0 ** -23)           # odd significand
    a = np.float32(3.0)                          # 3*b = 3 + 3*2^-23 -> needs 25 bits
    for c in (np.float32(2.0 ** -80), np.float32(-(2.0 ** -80))):
        got = quant.fma32(a, b, c)
        want = exact_round_f32(Fraction(3) * Fraction(float(b)) + Fraction(float(c)))
        assert got == want
    # and the plain fp64 route really does differ on one of them
    naive = [np.float32(np.float64(a) * np.float64(b) + np.float64(c))
             for c in (np.float32(2.0 ** -80), np.float32(-(2.0 ** -80)))]
    wants = [exact_round_f32(Fraction(3) * Fraction(float(b)) + Fraction(float(c)))
             for c in (np.float32(2.0 ** -80), np.float32(-(2.0 ** -80)))]
    assert naive != wants


def test_codes_are_nearest_grid_point():
    """Away from exact half-way points, codes equal the exact nearest level of m + k s."""
    rng = np.random.default_rng(1)
    for bits in (2, 4):
        x = (rng.standard_normal((300, 32)) * np.exp(rng.uniform(-3, 3, (300, 1)))).astype(np.float32)
        codes, s, z = quant.quantize_groups(x, bits)
        qmax = 2 ** bits - 1
        for g in range(x.shape[0]):
            if s[g] == 0:
                continue
            for i in range(32):
                t = (Fraction(float(x[g, i])) - Fraction(float(z[g]))) / Fraction(float(s[g]))
                frac = t - int(t)
                if abs(frac - Fraction(1, 2)) < Fraction(1, 10 ** 4):
                    continue                          # fp32 t may round across the tie
                k = min(qmax, max(0, int(t + Fraction(1, 2))))
                assert codes[g, i] == k


def test_error_bound_and_range():
    rng = np.random.default_rng(2)
    for bits in (2, 4):
        x = (rng.standard_normal((500, 32)) * 5).astype(np.float32)
        codes, s, z = quant.quantize_groups(x, bits)
        assert codes.max() <= 2 ** bits - 1
        xh = quant.dequantize(codes, s[:, None], z[:, None])
        err = np.abs(xh.astype(np.float64) - x)
        bound = s[:, None].astype(np.float64) / 2 * (1 + 1e-5) + np.spacing(np.abs(x)) * 2
        assert (err <= bound).all()
        # extremes are reproduced: the min exactly, the max within one step rounding
        assert (xh.min(axis=1) == x.min(axis=1)).all()


def test_padding_excluded():
    x = np.array([1.0, 2.0, 3.0, 100.0], np.float32)
    codes, s, z = quant.quantize_groups(x, 2, n_valid=3)
    assert codes.tolist() == [0, 2, 3, 0]
    assert float(z) == 1.0 and float(s) == np.float32(2.0) / np.float32(3.0)


def test_pack_bit_positions():
    codes = np.zeros(16, np.uint8)
    codes[0], codes[1], codes[2], codes[15] = 1, 2, 3, 3
    w = quant.pack_codes(codes, 2)
    assert w.tolist() == [1 | (2 << 2) | (3 << 4) | (3 << 30)]
    c4 = np.array([1, 15, 0, 0, 0, 0, 0, 9], np.uint8)
    assert quant.pack_codes(c4, 4).tolist() == [1 | (15 << 4) | (9 << 28)]
    rng = np.random.default_rng(3)
    for bits in (2, 4):
        c = rng.integers(0, 2 ** bits, (7, 128)).astype(np.uint8)
        assert (quant.unpack_codes(quant.pack_codes(c, bits), bits, 128) == c).all()


def test_round_to_dtype():
    x = np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1.0 + 2 ** -11, 1.0 + 3 * 2 ** -11], np.float32)
    bf = quant.round_to(x, "bf16")
    assert bf.tolist() == [1.0, 1.0 + 2 ** -6, 1.0, 1.0]  # RNE at 2^-7 spacing, ties to even
    f16 = quant.round_to(x, "f16")
    assert f16.tolist() == [1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1.0, 1.0 + 2 ** -9]
