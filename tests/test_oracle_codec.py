"""Pins of the oracle's codec (CPU only) against what the pages and the
mathematics fix: the hand-worked examples, exact rational arithmetic with the
IEEE rounding rule, exhaustive sweeps over every binary16 magnitude, and the
error bounds of round-to-nearest.

Definition followed: quantize_block in "DeepSeek-R1 inference latency ...
hardware-aware scheduling" (jsqmd.com/news/887038) section 2.1, and the
per-chunk INT8 variant in "DeepSeek R1 performance overview"
(aicoding.csdn.net) section 2.2.
"""
import os
from fractions import Fraction

import numpy as np
import pytest

from oracle import oracle as orc
from tests.exact import half_value, rn32, round_half_even

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, v = line.split(":", 1)
            vals[k] = v.split()
    return vals


def _f16(vals):
    return np.asarray(vals, dtype=np.float16).view(np.uint16)


def _unpack_int4(codes):
    lo = (codes & 0xF).astype(np.int16)
    hi = (codes >> 4).astype(np.int16)
    lo = np.where(lo >= 8, lo - 16, lo)
    hi = np.where(hi >= 8, hi - 16, hi)
    out = np.empty(codes.shape[:-1] + (codes.shape[-1] * 2,), dtype=np.int16)
    out[..., 0::2] = lo
    out[..., 1::2] = hi
    return out


def test_half_decode_matches_numpy_all_finite():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float32)
    got = np.array([orc.half_to_float(int(b)) for b in bits[::7]], dtype=np.float32)
    r = ref[::7]
    fin = np.isfinite(r)
    assert np.array_equal(got[fin].view(np.uint32), r[fin].view(np.uint32))
    assert np.all(np.isnan(got[np.isnan(r)]))


@pytest.mark.parametrize("name,fmt", [("int4_worked_example.txt", orc.INT4),
                                      ("int8_worked_example.txt", orc.INT8)])
def test_worked_example(name, fmt):
    g = _load_golden(name)
    xs = [float(v) for v in g["x"]]
    D = 128
    x = np.zeros((64, 1, D), dtype=np.uint16)
    x[0, 0, :len(xs)] = _f16(xs)
    codes, scales = orc.quantize(fmt, x)
    assert scales[0, 0] == np.float32(float(g["scale"][0]))
    want = np.zeros_like(codes[0, 0])
    rb = [int(v, 16) for v in g["row0_bytes"]]
    want[0, :len(rb)] = rb
    assert np.array_equal(codes[0, 0], want)


def test_negative_zero_is_code_zero():
    x = np.zeros((1, 1, 4), dtype=np.uint16)
    x[0, 0, :] = _f16([1.0, -0.0, -1e-4, 1e-4])
    codes, _ = orc.quantize(orc.INT4, x)
    assert _unpack_int4(codes)[0, 0, 0, :4].tolist() == [7, 0, 0, 0]


@pytest.mark.parametrize("fmt", [orc.INT4, orc.INT8])
def test_zero_block_exact(fmt):
    x = np.zeros((130, 3, 8), dtype=np.uint16)
    x[64:128, 1, :] = _f16(np.linspace(-2, 2, 8))  # only block 1, head 1 is non-zero
    codes, scales = orc.quantize(fmt, x)
    assert scales.shape == (3, 3)
    for j in range(3):
        for h in range(3):
            if (j, h) == (1, 1):
                assert scales[j, h] > 0
            else:
                assert scales[j, h] == 0.0
                assert not codes[j, h].any()


def _absmax_sweep_blocks():
    """every positive finite binary16 magnitude a, one block per a: row 0 = (a, -a)"""
    mags = np.arange(1, 0x7C00, dtype=np.uint16)       # 31743 positive finite values
    n = mags.size
    x = np.zeros((64 * n, 1, 2), dtype=np.uint16)
    x[0::64, 0, 0] = mags
    x[0::64, 0, 1] = mags | 0x8000
    return mags, x


def test_int4_scale_and_absmax_codes_exhaustive():
    """For every binary16 a: scale == RN32(a / 7.5); the +a element maps to 7;
    the -a element maps to -8 exactly when RN32(a / scale) >= 7.5, else -7."""
    mags, x = _absmax_sweep_blocks()
    codes, scales = orc.quantize(orc.INT4, x)
    c = _unpack_int4(codes[:, 0, 0, :1])              # [n][2]
    neg_minus8 = 0
    for i, m in enumerate(mags.tolist()):
        a = half_value(m)
        s = rn32(a / Fraction(15, 2))
        assert Fraction(float(scales[i, 0])) == s, (hex(m),)
        y = rn32(a / s)
        assert c[i, 0] == 7
        want = -8 if y >= Fraction(15, 2) else -7
        neg_minus8 += want == -8
        assert c[i, 1] == want, (hex(m), float(y))
    # both outcomes occur: the fp32 quotient is not always exactly 7.5
    assert 0 < neg_minus8 < mags.size


def test_int8_scale_and_absmax_codes_exhaustive():
    mags, x = _absmax_sweep_blocks()
    codes, scales = orc.quantize(orc.INT8, x)
    c = codes[:, 0, 0, :2].view(np.int8)
    for i, m in enumerate(mags.tolist()):
        a = half_value(m)
        s = rn32(a / 127)
        assert Fraction(float(scales[i, 0])) == s
    assert np.all(c[:, 0] == 127) and np.all(c[:, 1] == -127)


def _random_kv(T, H, D, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    v = rng.standard_normal((T, H, D)) * scale
    v[rng.random((T, H, D)) < 0.01] *= 10
    return v.astype(np.float16).view(np.uint16)


@pytest.mark.parametrize("fmt", [orc.INT4, orc.INT8])
def test_codes_follow_definition_exactly_small(fmt):
    """Every code of a small random tensor equals clamp(round_half_even(RN32(x / scale)))
    evaluated in exact rational arithmetic."""
    x = _random_kv(70, 2, 16, 3)
    codes, scales = orc.quantize(fmt, x)
    lo, hi, div = (-8, 7, Fraction(15, 2)) if fmt == orc.INT4 else (-127, 127, Fraction(127))
    for j in range(2):
        for h in range(2):
            rows = min(64, 70 - 64 * j)
            vals = [[half_value(int(x[64 * j + r, h, d])) for d in range(16)] for r in range(rows)]
            a = max(abs(v) for row in vals for v in row)
            s = rn32(a / div)
            assert Fraction(float(scales[j, h])) == s
            got = _unpack_int4(codes[j, h]) if fmt == orc.INT4 else codes[j, h].view(np.int8)
            for r in range(64):
                for d in range(16):
                    if r >= rows:
                        assert got[r, d] == 0
                        continue
                    q = round_half_even(rn32(vals[r][d] / s))
                    assert got[r, d] == min(max(q, lo), hi)


@pytest.mark.parametrize("fmt", [orc.INT4, orc.INT8])
def test_rounding_error_bounds(fmt):
    """For unclamped elements |y - q| <= 1/2 + half an ulp of the binary32
    quotient y: |x - q*scale| <= scale/2 * (1 + 2^-21) for int4 (|y| < 8) and
    scale/2 * (1 + 2^-17) for int8 (|y| < 128); codes stay in the clamp range."""
    x = _random_kv(640, 4, 128, 11, scale=1.5)
    codes, scales = orc.quantize(fmt, x)
    xf = x.view(np.float16).astype(np.float64).reshape(10, 64, 4, 128).transpose(0, 2, 1, 3)
    q = (_unpack_int4(codes) if fmt == orc.INT4 else codes.view(np.int8)).astype(np.float64)
    s = scales.astype(np.float64)[:, :, None, None]
    lo, hi = (-8, 7) if fmt == orc.INT4 else (-127, 127)
    assert q.min() >= lo and q.max() <= hi
    unclamped = (q > lo) & (q < hi)
    err = np.abs(xf - q * s)
    rel = 2.0 ** -21 if fmt == orc.INT4 else 2.0 ** -17
    assert np.all(err[unclamped] <= (s / 2 * (1 + rel) * np.ones_like(err))[unclamped])
    # and the bound is not vacuous: some element comes within 1% of it
    assert np.any(err[unclamped] >= (0.99 * s / 2 * np.ones_like(err))[unclamped])
    # the absmax element of every block maps to the top of the range (or -8/-7 for int4)
    amax = np.abs(xf).max(axis=(2, 3))
    assert np.all(np.abs(q).max(axis=(2, 3)) >= (7 if fmt == orc.INT4 else 127))
    assert np.array_equal(s[:, :, 0, 0] > 0, amax > 0)


def test_tail_block_uses_valid_rows_only():
    x = _random_kv(65, 1, 8, 5)
    x[64, 0, :] = _f16([0.5, -0.25, 0, 0, 0, 0, 0, 0.125])
    codes, scales = orc.quantize(orc.INT4, x)
    assert scales[1, 0] == np.float32(0.5) / np.float32(7.5)
    got = _unpack_int4(codes[1, 0])
    assert got[0].tolist() == [7, -4, 0, 0, 0, 0, 0, 2]
    assert not got[1:].any()
