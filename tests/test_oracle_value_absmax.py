"""Pin of the oracle's attention error normaliser, orc_value_absmax (CPU only).

The target states the attention error as a max-abs difference normalised by
max|v^| ("hardware-aware scheduling" page, jsqmd.com/news/887038, section 2.1,
and the error measure of the decode-attention target): for every (sequence,
head), the largest |code * value scale| over the sequence's valid tokens and
every head element, read through the block table.  Every attention parity test
divides by this value, so a mistake in it would loosen each of them silently.

The cache below is built by hand so that the answer for each (sequence, head)
is known by construction, and each plausible mistake gives a different one:
  * the block table is permuted, and the largest value of a sequence sits in
    its second or third page (a version that reads pages in order, or only the
    first page, misses it);
  * pages hold larger values in rows past the sequence's end (a version that
    ignores seq_lens returns those);
  * the value scale of a page applies to its own rows only (a version that
    pairs a row with a neighbouring page's scale returns another number);
  * the largest magnitude is a negative extreme code: int4 -8, int8 -127,
    FP8 0xfe = -448 (a version that drops the sign bit, or takes max instead of
    max |.|, returns something else);
  * heads and sequences have different answers (index mix-ups), and an empty
    sequence gives 0.
"""
import numpy as np
import pytest

from oracle import oracle as orc

D = 128
H = 3
# the most negative code of each format and its value, and the largest positive one
NEG = {orc.INT4: (-8, 8.0), orc.INT8: (-127, 127.0), orc.FP8: (-448, 448.0)}
POS = {orc.INT4: 7, orc.INT8: 127, orc.FP8: 448}


def _put(fmt, codes, page, h, row, d, c):
    if fmt == orc.INT4:
        b = int(codes[page, h, row, d // 2])
        nib = c & 0xF
        codes[page, h, row, d // 2] = (b & 0xF0) | nib if d % 2 == 0 else (b & 0x0F) | (nib << 4)
    elif fmt == orc.FP8:
        code = orc.float_to_e4m3(float(c))
        assert orc.e4m3_to_float(code) == c
        codes[page, h, row, d] = code
    else:
        codes[page, h, row, d] = np.uint8(c & 0xFF)


def _fill(fmt, codes, page, h, rows, c):
    for r in rows:
        for d in range(D):
            _put(fmt, codes, page, h, r, d, c)


def _cache(fmt):
    rb = orc.row_bytes(fmt, D)
    vc = np.zeros((5, H, 64, rb), np.uint8)
    vs = np.zeros((5, H), np.float32)
    neg, mag = NEG[fmt]
    pos = POS[fmt]
    # sequence 0: 150 tokens in pages 3, 0, 4 (page 4 holds tokens 128..149 in rows 0..21)
    # sequence 1: 70 tokens in pages 1, 2 (page 2 holds tokens 64..69 in rows 0..5)
    # sequence 2: empty
    table = np.array([[3, 0, 4], [1, 2, 0], [4, 4, 4]], np.int32)
    lens = np.array([150, 70, 0], np.int32)
    want = np.zeros((3, H))

    # (0, head 0): the negative extreme in the second page; page 4's valid rows
    # are 0 and its rows past the end hold the largest positive code at scale 10
    vs[3, 0], vs[0, 0], vs[4, 0] = 0.25, 0.5, 10.0
    _fill(fmt, vc, 3, 0, range(64), 1)
    _fill(fmt, vc, 0, 0, range(64), 2)
    _put(fmt, vc, 0, 0, 10, 5, neg)
    _fill(fmt, vc, 4, 0, range(22, 64), pos)
    want[0, 0] = mag * 0.5
    # (0, head 1): the negative extreme on the last valid token (row 21 of the
    # third page); rows 22.. of that page (past the end) hold the largest
    # positive code at the same scale, which must not count
    vs[3, 1], vs[0, 1], vs[4, 1] = 0.0625, 0.0625, 0.125
    _fill(fmt, vc, 3, 1, range(64), 1)
    _fill(fmt, vc, 0, 1, range(64), -1)
    _put(fmt, vc, 4, 1, 21, 127, neg)
    _fill(fmt, vc, 4, 1, range(22, 64), pos)
    want[0, 1] = mag * 0.125
    # (0, head 2): the largest positive code in the first page, last element
    vs[3, 2], vs[0, 2], vs[4, 2] = 1.0, 0.5, 0.5
    _put(fmt, vc, 3, 2, 0, 127, pos)
    _fill(fmt, vc, 0, 2, range(64), 3)
    want[0, 2] = max(float(pos) * 1.0, 3 * 0.5)

    # (1, head 0): the negative extreme on the last valid token (row 5 of page 2);
    # row 6 of page 2 (token 70, past the end) holds the largest positive code
    # at a larger scale on the same page -- scales are per (page, head), so the
    # row, not the scale, must exclude it
    vs[1, 0], vs[2, 0] = 0.75, 0.75
    _fill(fmt, vc, 1, 0, range(64), -1)
    _put(fmt, vc, 2, 0, 5, 64, neg)
    _fill(fmt, vc, 2, 0, range(6, 64), pos)
    want[1, 0] = mag * 0.75
    # (1, head 1): all values zero (codes zero, non-zero scales)
    vs[1, 1], vs[2, 1] = 3.0, 3.0
    want[1, 1] = 0.0
    # (1, head 2): code 3 at scale 2 in the first page; page 2 holds code 7 at
    # scale 4 only in rows past the end
    vs[1, 2], vs[2, 2] = 2.0, 4.0
    _put(fmt, vc, 1, 2, 63, 0, 3)
    _fill(fmt, vc, 2, 2, range(6, 64), 7)
    want[1, 2] = 6.0
    return vc, vs, table, lens, want


@pytest.mark.parametrize("fmt", [orc.INT4, orc.INT8, orc.FP8])
def test_value_absmax_known_by_construction(fmt):
    vc, vs, table, lens, want = _cache(fmt)
    got = orc.value_absmax(fmt, vc, vs, table, lens, H, D)
    assert got.shape == (3, H)
    assert np.array_equal(got, want), (got, want)


@pytest.mark.parametrize("fmt", [orc.INT4, orc.INT8, orc.FP8])
def test_value_absmax_scales_linearly(fmt):
    """Doubling every value scale doubles the normaliser (exact in binary64):
    it is |code| times the scale of the token's own page, not a function of
    the scales alone."""
    vc, vs, table, lens, want = _cache(fmt)
    got2 = orc.value_absmax(fmt, vc, (vs * 2).astype(np.float32), table, lens, H, D)
    assert np.array_equal(got2, 2 * want)


@pytest.mark.parametrize("fmt", [orc.INT4, orc.INT8, orc.FP8])
def test_value_absmax_matches_dequantized_brute_force(fmt):
    """Against max |v^| taken over an explicitly dequantized history built
    from the oracle's own codec on random data (the codes and scales of each
    sequence placed in permuted pages): the same number, exactly."""
    rng = np.random.default_rng(7)
    lens = np.array([1, 63, 64, 65, 130, 0], np.int32)
    B = len(lens)
    nb = 3
    table = rng.permutation(B * nb).astype(np.int32).reshape(B, nb)
    rb = orc.row_bytes(fmt, D)
    vc = np.zeros((B * nb, H, 64, rb), np.uint8)
    vs = np.zeros((B * nb, H), np.float32)
    want = np.zeros((B, H))
    for b, L in enumerate(lens):
        if L == 0:
            continue
        x = (rng.standard_normal((int(L), H, D)) * (1 + 3 * rng.random((1, H, 1)))).astype(np.float16)
        orc.quantize_into_pages(fmt, x.view(np.uint16), table[b], vc, vs)
        for h in range(H):
            for t in range(int(L)):
                pg = table[b, t // 64]
                row = [_decode(fmt, vc[pg, h, t % 64], d) for d in range(D)]
                want[b, h] = max(want[b, h], max(abs(c) for c in row) * float(vs[pg, h]))
    got = orc.value_absmax(fmt, vc, vs, table, lens, H, D)
    assert np.array_equal(got, want)


def _decode(fmt, row, d):
    """The signed value of element d of one stored code row (written from the
    storage layout: int4 low nibble = even element, two's complement)."""
    if fmt == orc.INT4:
        nib = (int(row[d // 2]) >> (4 * (d % 2))) & 0xF
        return nib - 16 if nib >= 8 else nib
    if fmt == orc.FP8:
        return orc.e4m3_to_float(int(row[d]))
    v = int(row[d])
    return v - 256 if v >= 128 else v


def test_normalized_error_known_by_construction():
    """The parity measure itself: for each (sequence, head) the largest
    |test - ref| over the head elements, divided by that (sequence, head)'s own
    max|v^|, then the maximum over all of them.  The numbers are chosen so that
    each plausible mistake gives another answer: the largest absolute error
    (0.006, head (0, 2)) is not the largest ratio (0.004, head (1, 2), where the
    test value is below the reference); one global max|v^| instead of the
    per-head one gives 0.0015; dropping the absolute value gives 0.0015; a
    zero-valued head with a zero error counts as 0 and one with
    any error as infinite."""
    ref = np.zeros((2, 3, 4))
    test = ref.copy()
    vmax = np.array([[2.0, 0.0, 4.0], [1.0, 0.0, 0.5]])
    test[0, 0, 3] = 0.002        # 0.001
    test[0, 2, 1] = 0.006        # 0.0015
    test[1, 0, 0] = 0.0015       # 0.0015
    ref[1, 2, 2] = 0.75
    test[1, 2, 2] = 0.748        # 0.004
    assert orc.normalized_error(test, ref, vmax) == pytest.approx(0.004, rel=1e-12)
    # a zero-valued head must match exactly
    test[0, 1, 0] = 1e-300
    assert orc.normalized_error(test, ref, vmax) == np.inf
    # shapes with no elements have no error
    assert orc.normalized_error(np.zeros((0, 3, 4)), np.zeros((0, 3, 4)), np.zeros((0, 3))) == 0.0
