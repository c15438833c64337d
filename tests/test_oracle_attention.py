"""Pins of the oracle's decode attention (CPU only): closed forms worked out by
hand, special cases that reduce to a mean or to one value row, invariances of
the definition (page placement, token order within the softmax, splitting
and merging), and per-(sequence, head) independence.

The operation: one query per (sequence, head) attends over the dequantized
keys and values k^ = code * scale of its sequence, read through a block table
("DeepSeek R1 performance tips", ddd.cn, section 4, PagedAttention; decode
reading a quantized KV cache, "DeepSeek R1 performance overview" section 3.1).
"""
import math

import numpy as np
import pytest

from oracle import oracle as orc

D = 128
SM = 1.0 / math.sqrt(D)


def _f16(vals):
    return np.asarray(vals, dtype=np.float16).view(np.uint16)


def _empty_cache(fmt, num_pages, H, D=D):
    rb = orc.row_bytes(fmt, D)
    return (np.zeros((num_pages, H, 64, rb), np.uint8), np.zeros((num_pages, H, 64, rb), np.uint8),
            np.zeros((num_pages, H), np.float32), np.zeros((num_pages, H), np.float32))


def _set_code(fmt, codes, page, h, row, d, c):
    if fmt == orc.INT4:
        b = int(codes[page, h, row, d // 2])
        nib = c & 0xF
        b = (b & 0xF0) | nib if d % 2 == 0 else (b & 0x0F) | (nib << 4)
        codes[page, h, row, d // 2] = b
    elif fmt == orc.FP8:   # small integers are exact E4M3 values
        codes[page, h, row, d] = orc.float_to_e4m3(c)
        assert orc.e4m3_to_float(int(codes[page, h, row, d])) == c
    else:
        codes[page, h, row, d] = np.uint8(c & 0xFF)


@pytest.mark.parametrize("fmt", [orc.INT4, orc.INT8, orc.FP8])
def test_two_token_closed_form(fmt):
    """q = e_0.  Token 0: key code 7 at dim 0 (dim 1 code -3 is ignored by q),
    key scale 0.5 -> score 3.5/sqrt(128); token 1: key codes 0 -> score 0.
    Values: token 0 all codes 2, token 1 all codes -4, value scale 0.25.
    o = (0.5 e^s0 - 1) / (e^s0 + 1) in every dimension."""
    kc, vc, ks, vs = _empty_cache(fmt, 1, 1)
    _set_code(fmt, kc, 0, 0, 0, 0, 7)
    _set_code(fmt, kc, 0, 0, 0, 1, -3)
    for d in range(D):
        _set_code(fmt, vc, 0, 0, 0, d, 2)
        _set_code(fmt, vc, 0, 0, 1, d, -4)
    ks[0, 0] = 0.5
    vs[0, 0] = 0.25
    q = np.zeros((1, 1, D), np.uint16)
    q[0, 0, 0] = _f16([1.0])[0]
    out = orc.decode_attention(fmt, kc, vc, ks, vs, np.array([[0]]), np.array([2]), q, SM)
    s0 = 3.5 * SM
    want = (0.5 * math.exp(s0) - 1.0) / (math.exp(s0) + 1.0)
    np.testing.assert_allclose(out[0, 0], want, rtol=0, atol=1e-15)


def test_query_sign_and_dimension():
    """q = -2 e_5: only dim 5 of the keys matters and its sign flips the score."""
    fmt = orc.INT4
    kc, vc, ks, vs = _empty_cache(fmt, 1, 1)
    _set_code(fmt, kc, 0, 0, 0, 5, 3)        # token 0: k^_5 = 3 * 0.1
    _set_code(fmt, kc, 0, 0, 1, 4, 7)        # token 1: only dim 4 set -> score 0
    _set_code(fmt, vc, 0, 0, 0, 0, 1)
    _set_code(fmt, vc, 0, 0, 1, 0, -1)
    ks[0, 0] = np.float32(0.1)
    vs[0, 0] = 1.0
    q = np.zeros((1, 1, D), np.uint16)
    q[0, 0, 5] = _f16([-2.0])[0]
    out = orc.decode_attention(fmt, kc, vc, ks, vs, np.array([[0]]), np.array([2]), q, SM)
    s0 = -2.0 * 3 * float(np.float32(0.1)) * SM
    w0 = math.exp(s0) / (math.exp(s0) + 1.0)
    assert abs(out[0, 0, 0] - (w0 * 1 + (1 - w0) * -1)) < 1e-15
    assert np.all(out[0, 0, 1:] == 0)


def _random_cache(fmt, num_pages, H, seed):
    rng = np.random.default_rng(seed)
    rb = orc.row_bytes(fmt, D)
    kc = rng.integers(0, 256, (num_pages, H, 64, rb), dtype=np.uint8)
    vc = rng.integers(0, 256, (num_pages, H, 64, rb), dtype=np.uint8)
    if fmt == orc.INT8:   # -128 is outside the code range
        kc[kc == 0x80] = 0x81
        vc[vc == 0x80] = 0x81
    if fmt == orc.FP8:    # 0x7f / 0xff are NaN, never written by the codec
        kc[(kc & 0x7F) == 0x7F] &= 0xFE
        vc[(vc & 0x7F) == 0x7F] &= 0xFE
    ks = rng.uniform(0.05, 0.6, (num_pages, H)).astype(np.float32)
    vs = rng.uniform(0.05, 0.6, (num_pages, H)).astype(np.float32)
    return kc, vc, ks, vs


def _dequant(fmt, codes, scales, bt_row, L, h):
    rows = []
    for t in range(L):
        pg = bt_row[t // 64]
        r = codes[pg, h, t % 64]
        if fmt == orc.INT4:
            lo = (r & 0xF).astype(np.int64)
            hi = (r >> 4).astype(np.int64)
            c = np.empty(D, np.int64)
            c[0::2] = np.where(lo >= 8, lo - 16, lo)
            c[1::2] = np.where(hi >= 8, hi - 16, hi)
        elif fmt == orc.FP8:
            c = np.array([orc.e4m3_to_float(int(v)) for v in r])
        else:
            c = r.view(np.int8).astype(np.int64)
        rows.append(c * float(scales[pg, h]))
    return np.array(rows)


@pytest.mark.parametrize("fmt", [orc.INT4, orc.INT8, orc.FP8])
def test_single_token_returns_its_value_row(fmt):
    kc, vc, ks, vs = _random_cache(fmt, 3, 2, 1)
    q = np.random.default_rng(2).standard_normal((1, 2, D)).astype(np.float16).view(np.uint16)
    bt = np.array([[2, 0]], np.int32)
    out = orc.decode_attention(fmt, kc, vc, ks, vs, bt, np.array([1]), q, SM)
    for h in range(2):
        assert np.array_equal(out[0, h], _dequant(fmt, vc, vs, bt[0], 1, h)[0])


@pytest.mark.parametrize("fmt", [orc.INT4, orc.INT8, orc.FP8])
def test_zero_query_is_mean_of_values(fmt):
    kc, vc, ks, vs = _random_cache(fmt, 4, 2, 3)
    q = np.zeros((1, 2, D), np.uint16)
    bt = np.array([[3, 1, 0]], np.int32)
    L = 150
    out = orc.decode_attention(fmt, kc, vc, ks, vs, bt, np.array([L]), q, SM)
    for h in range(2):
        np.testing.assert_allclose(out[0, h], _dequant(fmt, vc, vs, bt[0], L, h).mean(axis=0),
                                   rtol=0, atol=1e-13)


def test_one_dominant_key_selects_its_value():
    fmt = orc.INT8
    kc, vc, ks, vs = _random_cache(fmt, 2, 1, 4)
    ks[:] = 1e-3                        # every score tiny ...
    kc[1, 0, 10, :] = 127               # ... except token 64 + 10
    ks[1, 0] = 1.0
    q = np.full((1, 1, D), _f16([1.0])[0], np.uint16)
    bt = np.array([[0, 1]], np.int32)
    out = orc.decode_attention(fmt, kc, vc, ks, vs, bt, np.array([128]), q, SM)
    np.testing.assert_allclose(out[0, 0], _dequant(fmt, vc, vs, bt[0], 128, 0)[74], rtol=0, atol=1e-12)


@pytest.mark.parametrize("fmt", [orc.INT4, orc.INT8, orc.FP8])
def test_page_placement_invariance_and_tail_rows_ignored(fmt):
    """Moving pages (and their scales) to other slots with the block table
    following them changes nothing; codes in rows past the sequence end, and
    pages not referenced, are never read."""
    kc, vc, ks, vs = _random_cache(fmt, 5, 3, 5)
    q = np.random.default_rng(6).standard_normal((2, 3, D)).astype(np.float16).view(np.uint16)
    bt = np.array([[0, 1, 2], [3, 4, 0]], np.int32)
    lens = np.array([129, 100], np.int32)
    ref = orc.decode_attention(fmt, kc, vc, ks, vs, bt, lens, q, SM)
    perm = np.array([4, 2, 0, 1, 3])            # new slot of old page i
    kc2, vc2, ks2, vs2 = [np.empty_like(a) for a in (kc, vc, ks, vs)]
    for i, p in enumerate(perm):
        kc2[p], vc2[p], ks2[p], vs2[p] = kc[i], vc[i], ks[i], vs[i]
    bt2 = perm[bt]
    # garbage beyond the ends: sequence 0 ends at row 0 of its 3rd page
    kc2[perm[2], :, 1:] = 0x77
    vc2[perm[2], :, 1:] = 0x77
    out = orc.decode_attention(fmt, kc2, vc2, ks2, vs2, bt2, lens, q, SM)
    assert np.array_equal(out[0], ref[0])
    # sequence 1 (100 tokens) reads pages 3 and 4 only; rows 36.. of page 4 unused
    assert np.array_equal(out[1], ref[1])


@pytest.mark.parametrize("fmt", [orc.INT4, orc.INT8, orc.FP8])
def test_split_merge_equals_direct(fmt):
    kc, vc, ks, vs = _random_cache(fmt, 6, 2, 7)
    q = np.random.default_rng(8).standard_normal((2, 2, D)).astype(np.float16).view(np.uint16)
    bt = np.array([[0, 1, 2], [3, 4, 5]], np.int32)
    lens = np.array([190, 65], np.int32)
    ref = orc.decode_attention(fmt, kc, vc, ks, vs, bt, lens, q, SM, num_splits=1)
    for s in (2, 3, 7, 64):
        out = orc.decode_attention(fmt, kc, vc, ks, vs, bt, lens, q, SM, num_splits=s)
        np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)


def test_each_sequence_and_head_is_independent():
    """The (b, h) output equals the output of a call holding only that (b, h)."""
    fmt = orc.INT4
    kc, vc, ks, vs = _random_cache(fmt, 4, 3, 9)
    q = np.random.default_rng(10).standard_normal((2, 3, D)).astype(np.float16).view(np.uint16)
    bt = np.array([[0, 1], [2, 3]], np.int32)
    lens = np.array([70, 128], np.int32)
    full = orc.decode_attention(fmt, kc, vc, ks, vs, bt, lens, q, SM)
    for b in range(2):
        for h in range(3):
            one = orc.decode_attention(fmt, np.ascontiguousarray(kc[:, h:h + 1]),
                                       np.ascontiguousarray(vc[:, h:h + 1]),
                                       np.ascontiguousarray(ks[:, h:h + 1]),
                                       np.ascontiguousarray(vs[:, h:h + 1]),
                                       bt[b:b + 1], lens[b:b + 1], q[b:b + 1, h:h + 1], SM)
            assert np.array_equal(one[0, 0], full[b, h])


def test_empty_sequence_gives_zero_and_bad_table_rejected():
    fmt = orc.INT4
    kc, vc, ks, vs = _random_cache(fmt, 2, 1, 11)
    q = np.random.default_rng(12).standard_normal((2, 1, D)).astype(np.float16).view(np.uint16)
    out = orc.decode_attention(fmt, kc, vc, ks, vs, np.array([[0], [1]]), np.array([0, 5]), q, SM)
    assert np.all(out[0] == 0) and np.any(out[1] != 0)
    with pytest.raises(ValueError):
        orc.decode_attention(fmt, kc, vc, ks, vs, np.array([[2]]), np.array([5]), q[:1], SM)
    with pytest.raises(ValueError):
        orc.decode_attention(fmt, kc, vc, ks, vs, np.array([[0]]), np.array([65]), q[:1], SM)


def test_matches_independent_numpy_softmax():
    """A cross-check (not a pin) against a vectorised numpy evaluation."""
    fmt = orc.INT4
    kc, vc, ks, vs = _random_cache(fmt, 4, 2, 13)
    q = np.random.default_rng(14).standard_normal((1, 2, D)).astype(np.float16)
    bt = np.array([[1, 3, 0]], np.int32)
    L = 131
    out = orc.decode_attention(fmt, kc, vc, ks, vs, bt, np.array([L]), q.view(np.uint16), SM)
    for h in range(2):
        K = _dequant(fmt, kc, ks, bt[0], L, h)
        V = _dequant(fmt, vc, vs, bt[0], L, h)
        s = K @ q[0, h].astype(np.float64) * SM
        p = np.exp(s - s.max())
        np.testing.assert_allclose(out[0, h], p @ V / p.sum(), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("fmt", [orc.INT4, orc.INT8, orc.FP8])
@pytest.mark.parametrize("g", [2, 3, 4, 8, 32])
def test_grouped_heads_equal_multi_head_over_repeated_heads(fmt, g):
    """Grouped query heads (Hq = g * Hkv, query head i reads cache head i // g)
    give exactly the multi-head result over a cache whose head i is a copy of
    cache head i // g: a wrong head mapping (i % Hkv, or the first head of the
    group for all) fails this."""
    Hkv = 3
    kc, vc, ks, vs = _random_cache(fmt, 5, Hkv, 21)
    rep = np.repeat(np.arange(Hkv), g)
    kc2, vc2, ks2, vs2 = kc[:, rep], vc[:, rep], ks[:, rep], vs[:, rep]
    bt = np.array([[4, 0, 2], [1, 3, 0]], np.int32)
    lens = np.array([150, 77], np.int32)
    q = np.random.default_rng(22).standard_normal((2, Hkv * g, D)).astype(np.float16).view(np.uint16)
    gqa = orc.decode_attention(fmt, kc, vc, ks, vs, bt, lens, q, SM)
    mha = orc.decode_attention(fmt, kc2, vc2, ks2, vs2, bt, lens, q, SM)
    assert gqa.shape == (2, Hkv * g, D)
    assert np.array_equal(gqa, mha)
    # the heads of one group differ (their queries differ) and follow their own cache head
    assert not np.array_equal(gqa[:, 0], gqa[:, 1])
    K = _dequant(fmt, kc, ks, bt[0], 150, 1)
    V = _dequant(fmt, vc, vs, bt[0], 150, 1)
    s = K @ q[0, g].view(np.float16).astype(np.float64) * SM  # query head g reads cache head 1
    p = np.exp(s - s.max())
    np.testing.assert_allclose(gqa[0, g], p @ V / p.sum(), rtol=1e-12, atol=1e-12)


def test_grouped_heads_reject_a_non_multiple():
    kc, vc, ks, vs = _random_cache(orc.INT4, 2, 2, 23)
    q = np.zeros((1, 3, D), np.uint16)
    with pytest.raises(ValueError):
        orc.decode_attention(orc.INT4, kc, vc, ks, vs, np.array([[0]], np.int32), np.array([10], np.int32), q, SM)
