"""Pins for the fp16-metadata cache variant of the oracle (quantiser and block format).

The WindowQuant note (主な結果: a 1.05 GB cache held in 0.19 GB) and the QuantWM card (Key
Results: up to 6.20x smaller) report caches far smaller than fp32 step / zero metadata allows;
the variant stores each (s, z) as two fp16 values and takes the codes against that stored
grid.  The hand cases are derived in tests/golden/hand_cases.json; the other pins use exact
rational arithmetic, exhaustive search over the codes and the byte format read by hand."""

import json
import os
from fractions import Fraction

import numpy as np
import pytest

from oracle import quant, layout
from bit_kv_cache_28_b300 import synth

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "hand_cases.json")))


@pytest.mark.parametrize("case", GOLD["meta16_quant"])
def test_hand_cases(case):
    x = np.array(case["x"], np.float32)
    codes, s, z = quant.quantize_groups(x, case["bits"], meta16=True)
    assert codes.tolist() == case["codes"], case["why"]
    assert float(s) == case["s"] and float(z) == case["z"]
    assert quant.dequantize(codes, s, z, meta16=True).tolist() == case["xhat"]
    if "codes_f32_meta" in case:
        assert quant.quantize_groups(x, case["bits"])[0].tolist() == case["codes_f32_meta"]


def _all_f16_nonneg():
    """Every finite non-negative fp16 value, from its bit patterns."""
    return np.arange(0, 0x7C00, dtype=np.uint16).view(np.float16).astype(np.float64)


def test_f16_round_against_every_fp16_value():
    """Exhaustive: each rounded value is an fp16 value, no fp16 value lies closer, ties go to
    the even significand; the library's fp64 -> fp16 conversion agrees."""
    grid = _all_f16_nonneg()
    rng = np.random.default_rng(21)
    mids = (grid[1:] + grid[:-1]) / 2                       # exact ties
    x = np.concatenate([grid, mids, rng.uniform(0, 65504, 3000), np.exp(rng.uniform(-20, 11, 3000)),
                        rng.uniform(0, 2 ** -14, 500), [65503.9, 65519.99, 65520.0, 1e6]])
    x = np.concatenate([x, -x])
    y = quant.f16_round(x)
    with np.errstate(over="ignore"):
        assert np.array_equal(y, x.astype(np.float16).astype(np.float64))
    fin = np.isfinite(y)
    assert (np.abs(x[~fin]) >= 65520).all() and (np.abs(x[fin]) < 65520).all()
    idx = np.searchsorted(grid, np.abs(x[fin]))
    lo = grid[np.maximum(idx - 1, 0)]
    hi = grid[np.minimum(idx, grid.size - 1)]
    ay, ax = np.abs(y[fin]), np.abs(x[fin])
    assert (np.minimum(np.abs(lo - ax), np.abs(hi - ax)) == np.abs(ay - ax)).all()
    tie = np.abs(lo - ax) == np.abs(hi - ax)
    bits = ay[tie & (lo != hi)].astype(np.float16).view(np.uint16)
    assert (bits & 1 == 0).all()


def test_fp16_dequantisation_is_one_rounding():
    """fp16 dequantisation: the fp16 value nearest to the exact code s + z (Fraction), where the
    fp32 FMA followed by an fp16 rounding may round twice."""
    rng = np.random.default_rng(22)
    s = quant.f16_rne(np.exp(rng.uniform(-8, 5, 4000)).astype(np.float32))
    z = quant.f16_rne((rng.standard_normal(4000) * 50).astype(np.float32))
    k = rng.integers(0, 16, 4000)
    got = quant.dequantize(k, s, z, meta16=True)
    grid = _all_f16_nonneg()
    for i in range(0, 4000, 7):
        ex = Fraction(int(k[i])) * Fraction(float(s[i])) + Fraction(float(z[i]))
        a = abs(ex)
        j = int(np.searchsorted(grid, float(a)))
        cands = [grid[max(j - 1, 0)], grid[min(j, grid.size - 1)], grid[min(j + 1, grid.size - 1)]]
        best = min(abs(Fraction(c) - a) for c in cands)
        assert abs(Fraction(abs(float(got[i]))) - a) == best


def _fp16_neighbours(v):
    h = np.float16(v)
    return [float(np.nextafter(h, np.float16(-np.inf))), float(h), float(np.nextafter(h, np.float16(np.inf)))]


def test_metadata_is_the_nearest_fp16():
    """s16 and z16 are fp16 values, and no fp16 value lies closer to the fp32 step (minimum)."""
    rng = np.random.default_rng(11)
    x = (rng.standard_normal((400, 32)) * np.exp(rng.uniform(-6, 6, (400, 1)))).astype(np.float32)
    for bits in (2, 4):
        _, s16, z16 = quant.quantize_groups(x, bits, meta16=True)
        _, s32, z32 = quant.quantize_groups(x, bits)
        for g in range(x.shape[0]):
            for v16, v32 in ((s16[g], s32[g]), (z16[g], z32[g])):
                assert float(np.float16(v16)) == float(v16)          # representable
                best = min(abs(Fraction(c) - Fraction(float(v32))) for c in _fp16_neighbours(v32))
                assert abs(Fraction(float(v16)) - Fraction(float(v32))) == best


def test_codes_are_nearest_level_of_the_stored_grid():
    """Exhaustive search: each code minimises |x - fmaf(k, s16, z16)| over k in [0, 2^b - 1],
    in exact arithmetic, away from exact half-way points."""
    rng = np.random.default_rng(12)
    for bits in (2, 4):
        qmax = 2 ** bits - 1
        x = (rng.standard_normal((120, 32)) * np.exp(rng.uniform(-4, 4, (120, 1)))).astype(np.float32)
        codes, s, z = quant.quantize_groups(x, bits, meta16=True)
        for g in range(x.shape[0]):
            if s[g] == 0:
                assert (codes[g] == 0).all()
                continue
            levels = [Fraction(k) * Fraction(float(s[g])) + Fraction(float(z[g])) for k in range(qmax + 1)]
            for i in range(32):
                dist = [abs(Fraction(float(x[g, i])) - lv) for lv in levels]
                order = sorted(range(qmax + 1), key=lambda k: dist[k])
                if dist[order[1]] - dist[order[0]] < Fraction(float(s[g])) * Fraction(1, 10 ** 4):
                    continue                                   # fp32 t may round across the tie
                assert codes[g, i] == order[0], (g, i)


def test_block_bytes_by_hand():
    """INT2, d 128: codes 1024 + 1024, key pairs 128 x 4, value pairs 4 x 32 x 4 -> 3072 (fp32: 4096)."""
    assert layout.block_bytes(layout.INT2, 128, meta16=True) == 3072
    assert layout.block_bytes(layout.INT4, 128, meta16=True) == 2048 * 2 + 512 + 512
    assert layout.block_bytes(layout.INT2, 64, meta16=True) == 1536
    assert layout.block_bytes(layout.INT4, 64, meta16=True) == 2560
    assert layout.block_bytes(layout.RAW16, 64, meta16=True) == layout.block_bytes(layout.RAW16, 64)
    # cache bytes per token and head at d 128, INT2, full blocks: 3072 / 32 = 96 B (fp16 raw: 256 B
    # per K or V row, 512 B both)
    assert layout.block_bytes(layout.INT2, 128, meta16=True) / 32 == 96


def test_stored_bytes_read_by_hand():
    """Decode one packed block byte by byte: Kc | Km half2[d] | Vc | Vm half2[d/32][32]."""
    rng = np.random.default_rng(13)
    d, bits, nv = 64, 2, 27
    Kb = (rng.standard_normal((1, 32, d)) * 3).astype(np.float32)
    Vb = rng.standard_normal((1, 32, d)).astype(np.float32)
    enc = layout.encode_int_blocks(Kb, Vb, bits, nv, meta16=True)
    raw = enc["bytes"][0]
    assert raw.size == 1536
    kc_bytes = 32 * d * bits // 8
    km = raw[kc_bytes:kc_bytes + 4 * d].view(np.float16).reshape(d, 2)
    vc0 = kc_bytes + 4 * d
    vm = raw[vc0 + kc_bytes:].view(np.float16).reshape(d // 32, 32, 2)
    # key metadata: channel c's (s, z) from the channel's valid tokens
    for c in (0, 17, 63):
        col = Kb[0, :nv, c]
        assert float(km[c, 1]) == float(np.float16(col.min()))
        assert float(km[c, 0]) == float(np.float16(np.float32(np.float32(col.max() - col.min()) / np.float32(3))))
    # value metadata: (group g, token t); pad tokens zero
    for g, t in ((0, 0), (1, 26)):
        row = Vb[0, t, 32 * g:32 * g + 32]
        assert float(vm[g, t, 1]) == float(np.float16(row.min()))
    assert (vm[:, nv:] == 0).all()
    # code words: channel 5 of token 3 sits at word 3*(d*b/32) + 5/16, bits 2*(5 mod 16)
    kw = raw[:kc_bytes].view(np.uint32)
    word = kw[3 * (d * bits // 32) + 5 // 16]
    assert (word >> (2 * 5)) & 3 == enc["kcode"][0, 3, 5]
    # the same values with fp32 metadata: identical code bytes wherever the codes agree
    enc32 = layout.encode_int_blocks(Kb, Vb, bits, nv)
    assert enc32["bytes"].shape[1] == 2048


def test_dequantised_error_bound():
    """|x_hat - x| <= s16 / 2 inside the stored grid's span, up to fp32 rounding; the grid's
    ends sit within half an fp16 step of the group's min and max."""
    rng = np.random.default_rng(14)
    for bits in (2, 4):
        qmax = 2 ** bits - 1
        x = (rng.standard_normal((300, 32)) * np.exp(rng.uniform(-3, 3, (300, 1)))).astype(np.float32)
        codes, s, z = quant.quantize_groups(x, bits, meta16=True)
        xh = quant.dequantize(codes, s[:, None], z[:, None], meta16=True).astype(np.float64)
        assert np.array_equal(xh, xh.astype(np.float16).astype(np.float64))     # fp16 values
        lo = z.astype(np.float64)
        hi = lo + qmax * s.astype(np.float64)
        xc = np.clip(x.astype(np.float64), lo[:, None], hi[:, None])
        err = np.abs(xh - xc)
        half_f16 = np.abs(np.spacing(np.abs(xh).astype(np.float16)).astype(np.float64)) / 2
        assert (err <= s[:, None] / 2 * (1 + 1e-5) + half_f16 + np.spacing(np.abs(x)) * 2).all()
        # the spans: |z - m| <= half an fp16 ulp of m, and the top level misses M by at most
        # qmax half-ulps of s plus half an ulp of m
        m, M = x.min(1).astype(np.float64), x.max(1).astype(np.float64)
        ulp = lambda v: np.abs(np.spacing(np.float16(v)).astype(np.float64))
        assert (np.abs(lo - m) <= ulp(m) / 2 + 1e-30).all()
        _, s32, _ = quant.quantize_groups(x, bits)
        slack = qmax * ulp(s32) / 2 + ulp(m) / 2 + np.abs(M) * 2 ** -22
        assert (np.abs(hi - M) <= slack).all()


def test_builders_keep_raw_windows_and_shrink_int_blocks():
    case = synth.decode_case(seed=15, B=1, Hq=2, Hkv=1, d=64, n_cache=200, dtype="f16")
    bits = np.array([[16, 4, 2, 2, 4, 16, 2]])
    caps = [2, 2, 3]
    c32 = layout.build_mixed(case["K_cache"], case["V_cache"], bits, caps, "f16")
    c16 = layout.build_mixed(case["K_cache"], case["V_cache"], bits, caps, "f16", meta16=True)
    rb = 2 * layout.block_bytes(layout.RAW16, 64)
    assert np.array_equal(c16.data[..., :rb], c32.data[..., :rb])
    assert c16.stream_bytes == rb + 2 * 2560 + 3 * 1536
    for r16, r32 in zip(c16.blocks[0][0], c32.blocks[0][0]):
        assert r16["pos"] == r32["pos"] and r16["len"] == r32["len"]
        if r16["quantised"]:
            # the key step sizes the Jensen term reads are the stored fp16 ones
            assert np.array_equal(r16["ks"], np.asarray(quant.f16_rne(r16["ks"])))
            assert np.abs(r16["khat"] - r32["khat"]).max() <= np.abs(r32["ks"]).max()
    u = layout.build_uniform(case["K_cache"][:, :, :100], case["V_cache"][:, :, :100], 2, [60, 40], 4, meta16=True)
    assert u.stream_bytes == 4 * 1536 and u.n_blocks == [4]
