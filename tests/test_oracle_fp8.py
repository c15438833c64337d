"""Pins of the oracle's FP8 E4M3 codec (CPU only).

Definition followed: FP8 E4M3 with dynamic range scaling from max|x|
("DeepSeek-R1 inference latency ... hardware-aware scheduling",
jsqmd.com/news/887038, section 2.2) as the KV-cache format ("DeepSeek R1
performance tips", ddd.cn, section 1), on the same (sequence, head, 64-token)
blocks as quantize_block: scale = max|x| / 448, code = E4M3(RN32(x / scale)),
round to nearest, ties to the even fraction, saturating.

The pins: values of particular codes derived by hand from the format's fields,
the structure of the code table (monotone, eight codes per binade, constant
spacing inside a binade), the nearest-value rule checked by exhaustive search in
exact rationals, a hand-worked block, every binary16 magnitude for the scale
and the absmax element, and the page's error bound of half a unit in the last
place of the 3-bit fraction.
"""
import os
from fractions import Fraction

import numpy as np
import pytest

from oracle import oracle as orc
from tests.exact import half_value, rn32

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
F = Fraction


def _f16(vals):
    return np.asarray(vals, dtype=np.float16).view(np.uint16)


def test_e4m3_code_values_by_hand():
    """Codes whose values follow from the fields alone (bias 7, 3 fraction bits)."""
    want = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x0F: 1.875 * 2.0 ** -6,
            0x38: 1.0, 0x3F: 1.875, 0x40: 2.0, 0x58: 16.0, 0x59: 18.0, 0x77: 240.0, 0x78: 256.0,
            0x7E: 448.0, 0xB8: -1.0, 0xC2: -2.5, 0xFE: -448.0}
    for c, v in want.items():
        assert orc.e4m3_to_float(c) == v, hex(c)
    nz = orc.e4m3_to_float(0x80)
    assert nz == 0.0 and np.signbit(nz)
    assert np.isnan(orc.e4m3_to_float(0x7F)) and np.isnan(orc.e4m3_to_float(0xFF))


def test_e4m3_code_table_structure():
    """0x00..0x7e strictly increasing; the subnormals step by 2^-9; each normal
    binade holds 8 codes spaced 2^(e-10); the sign bit negates."""
    v = [F(orc.e4m3_to_float(c)) for c in range(127)]
    assert all(v[i] < v[i + 1] for i in range(126))
    for c in range(8):
        assert v[c] == c * F(1, 512)
    for e in range(1, 16):
        codes = [c for c in range(127) if (c >> 3) == e]
        assert len(codes) == (8 if e < 15 else 7)
        assert v[codes[0]] == F(2) ** (e - 7)
        for c in codes[:-1]:
            assert v[c + 1] - v[c] == F(2) ** (e - 10)
    for c in range(127):
        assert orc.e4m3_to_float(c | 0x80) == -orc.e4m3_to_float(c)


def _nearest_e4m3(y):
    """Brute force: the nearest of the 127 finite non-negative values, the even
    code on a tie, saturating, then the sign bit."""
    table = [F(orc.e4m3_to_float(c)) for c in range(127)]
    ay = abs(F(float(y)))
    best = min(range(127), key=lambda c: (abs(table[c] - ay), c & 1))
    return best | (0x80 if np.signbit(y) else 0)


def test_e4m3_encode_is_nearest_ties_even():
    vals = [F(orc.e4m3_to_float(c)) for c in range(127)]
    ys = []
    for i in range(126):  # every code, every midpoint, and one binary32 ulp on either side
        mid = (vals[i] + vals[i + 1]) / 2
        for t in (vals[i], mid):
            f = np.float32(float(t))
            ys += [f, np.nextafter(f, np.float32(np.inf)), np.nextafter(f, np.float32(-np.inf))]
    rng = np.random.default_rng(7)
    ys += list((rng.standard_normal(2000) * 10.0 ** rng.uniform(-4, 2.7, 2000)).astype(np.float32))
    ys += [np.float32(v) for v in (448.0, 460.0, 463.99, 464.0, 500.0, 1e30, 1e-30, -1e-30, 0.0, -0.0)]
    for y in ys:
        for s in (y, -y):
            assert orc.float_to_e4m3(s) == _nearest_e4m3(s), (float(s),)


def test_fp8_worked_example():
    g = {}
    with open(os.path.join(GOLDEN, "fp8_e4m3_worked_example.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                k, v = line.split(":", 1)
                g[k] = v.split()
    xs = [float(v) for v in g["x"]]
    x = np.zeros((64, 1, 128), dtype=np.uint16)
    x[0, 0, :len(xs)] = _f16(xs)
    codes, scales = orc.quantize(orc.FP8, x)
    assert scales[0, 0] == np.float32(float(g["scale"][0]))
    want = np.zeros_like(codes[0, 0])
    rb = [int(v, 16) for v in g["row0_bytes"]]
    want[0, :len(rb)] = rb
    assert np.array_equal(codes[0, 0], want)


def test_fp8_scale_and_absmax_codes_exhaustive():
    """For every binary16 magnitude a: scale == RN32(a / 448); +a -> 0x7e and
    -a -> 0xfe (the quotient is 448 within binary32 rounding, far from the
    next E4M3 midpoint)."""
    mags = np.arange(1, 0x7C00, dtype=np.uint16)
    n = mags.size
    x = np.zeros((64 * n, 1, 2), dtype=np.uint16)
    x[0::64, 0, 0] = mags
    x[0::64, 0, 1] = mags | 0x8000
    codes, scales = orc.quantize(orc.FP8, x)
    for i, m in enumerate(mags.tolist()):
        assert F(float(scales[i, 0])) == rn32(half_value(m) / 448), hex(m)
    assert np.all(codes[:, 0, 0, 0] == 0x7E) and np.all(codes[:, 0, 0, 1] == 0xFE)


def _random_kv(T, H, D, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    v = rng.standard_normal((T, H, D)) * scale
    v[rng.random((T, H, D)) < 0.01] *= 10
    v[rng.random((T, H, D)) < 0.01] *= 1e-4
    return v.astype(np.float16).view(np.uint16)


def test_fp8_codes_follow_definition_exactly_small():
    """Every code == the nearest E4M3 (ties even) of RN32(x / scale) in exact
    rationals; rows past a tail block's end stay 0x00."""
    x = _random_kv(70, 2, 16, 3)
    codes, scales = orc.quantize(orc.FP8, x)
    table = [F(orc.e4m3_to_float(c)) for c in range(127)]
    for j in range(2):
        for h in range(2):
            rows = min(64, 70 - 64 * j)
            vals = [[half_value(int(x[64 * j + r, h, d])) for d in range(16)] for r in range(rows)]
            s = rn32(max(abs(v) for row in vals for v in row) / 448)
            assert F(float(scales[j, h])) == s
            for r in range(64):
                for d in range(16):
                    if r >= rows:
                        assert codes[j, h, r, d] == 0
                        continue
                    y = rn32(vals[r][d] / s)
                    best = min(range(127), key=lambda c: (abs(table[c] - abs(y)), c & 1))
                    neg = vals[r][d] < 0 or (vals[r][d] == 0 and int(x[64 * j + r, h, d]) & 0x8000)
                    assert codes[j, h, r, d] == best | (0x80 if neg else 0), (j, h, r, d)


def test_fp8_error_bound():
    """|x - deq| <= 1/2 ulp_E4M3(y) * scale (1 + 2^-19): half a unit in the last
    place of the 3-bit fraction at the quotient's binade (2^-9 below 2^-6), the
    bound of section 2.2, plus the binary32 rounding of the quotient y = x / scale
    (at most 2^-24 |y| < 2^-19 of that half unit); the bound is reached within 1%."""
    x = _random_kv(640, 4, 128, 11, scale=1.5)
    codes, scales = orc.quantize(orc.FP8, x)
    xf = x.view(np.float16).astype(np.float64).reshape(10, 64, 4, 128).transpose(0, 2, 1, 3)
    dq = np.vectorize(orc.e4m3_to_float)(np.arange(256)).astype(np.float64)[codes]
    s = scales.astype(np.float64)[:, :, None, None]
    y = np.abs(xf) / np.where(s > 0, s, 1.0)
    e = np.floor(np.log2(np.maximum(y, 2.0 ** -6)))
    half_ulp = 0.5 * 2.0 ** (e - 3)
    err = np.abs(xf - dq * s)
    bound = half_ulp * s * (1 + 2.0 ** -19)
    assert np.all(err <= bound)
    assert np.any(err >= 0.99 * bound)
    assert np.all(codes[..., :] != 0x7F) and np.all(codes != 0xFF)


def test_fp8_zero_block_and_negative_zero():
    """An all-zero block (even of -0.0) has scale 0 and codes 0x00; in a
    non-zero block -0.0 keeps its sign (0x80)."""
    x = np.zeros((128, 1, 4), dtype=np.uint16)
    x[:64, 0, :] = _f16([-0.0, 0.0, -0.0, 0.0])
    x[64, 0, :] = _f16([1.0, -0.0, 0.0, -1.0])
    codes, scales = orc.quantize(orc.FP8, x)
    assert scales[0, 0] == 0.0 and not codes[0, 0].any()
    assert codes[1, 0, 0, :4].tolist() == [0x7E, 0x80, 0x00, 0xFE]
