"""Pins of the oracle's chunked-prefill attention (CPU only): a chunk of n
new tokens of a sequence of length L (the cache already holds them) -- query i
at position L - n + i attends causally to positions 0 .. L - n + i of the
dequantized cache.  Chunked prefill over the cache: "R1 performance overview"
(aicoding.csdn.net), dynamic chunked attention; paging: ddd.cn section 4.

Pinned by an independent numpy evaluation of the causal softmax over values
dequantized in the test, the first query of a chunk at position 0 (its own
value row), the chunk's last query against full-length decode attention, and
the causal mask (a change to a later token's value reaches only the queries
at or after it)."""
import math

import numpy as np
import pytest

from oracle import oracle as orc

D = 128
SM = 1.0 / math.sqrt(D)


def _cache(fmt, B, H, L, seed):
    rng = np.random.default_rng(seed)
    x_k = (rng.standard_normal((B, L, H, D)) * 1.5).astype(np.float16).view(np.uint16)
    x_v = rng.standard_normal((B, L, H, D)).astype(np.float16).view(np.uint16)
    nb = (L + 63) // 64
    rb = orc.row_bytes(fmt, D)
    kc = np.zeros((B * nb, H, 64, rb), np.uint8)
    vc = np.zeros_like(kc)
    ks = np.zeros((B * nb, H), np.float32)
    vs = np.zeros_like(ks)
    bt = rng.permutation(B * nb).astype(np.int32).reshape(B, nb)
    for b in range(B):
        orc.quantize_into_pages(fmt, x_k[b], bt[b], kc, ks)
        orc.quantize_into_pages(fmt, x_v[b], bt[b], vc, vs)
    return kc, vc, ks, vs, bt


def _dequant(fmt, codes, scales, bt_row, L, h):
    out = np.zeros((L, D))
    for t in range(L):
        pg = bt_row[t // 64]
        r = codes[pg, h, t % 64]
        if fmt == orc.INT4:
            lo = (r & 0xF).astype(np.int64)
            hi = (r >> 4).astype(np.int64)
            c = np.empty(D)
            c[0::2] = np.where(lo >= 8, lo - 16, lo)
            c[1::2] = np.where(hi >= 8, hi - 16, hi)
        elif fmt == orc.FP8:
            c = np.array([orc.e4m3_to_float(int(v)) for v in r])
        else:
            c = r.view(np.int8).astype(np.float64)
        out[t] = c * float(scales[pg, h])
    return out


@pytest.mark.parametrize("fmt", [orc.INT4, orc.INT8, orc.FP8])
@pytest.mark.parametrize("g", [1, 2, 3])
def test_matches_numpy_causal_softmax(fmt, g):
    B, H = 3, 2
    L = [70, 131, 64]
    n = [70, 5, 0]   # a whole sequence as one chunk, a short chunk after history, no new tokens
    kc, vc, ks, vs, bt = _cache(fmt, B, H, max(L), 3)
    cu = np.concatenate([[0], np.cumsum(n)])
    rng = np.random.default_rng(4)
    q = rng.standard_normal((cu[-1], H * g, D)).astype(np.float16)
    got = orc.prefill_attention(fmt, kc, vc, ks, vs, bt, L, cu, q.view(np.uint16), SM)
    for b in range(B):
        for hq in range(H * g):
            h = hq // g
            kh = _dequant(fmt, kc, ks, bt[b], L[b], h)
            vh = _dequant(fmt, vc, vs, bt[b], L[b], h)
            for i in range(n[b]):
                p = L[b] - n[b] + i
                s = kh[:p + 1] @ q[cu[b] + i, hq].astype(np.float64) * SM
                w = np.exp(s - s.max())
                want = (w / w.sum()) @ vh[:p + 1]
                np.testing.assert_allclose(got[cu[b] + i, hq], want, rtol=0, atol=1e-12)


def test_first_query_at_position_zero_is_its_value():
    kc, vc, ks, vs, bt = _cache(orc.INT4, 1, 1, 64, 5)
    q = np.random.default_rng(6).standard_normal((3, 1, D)).astype(np.float16).view(np.uint16)
    out = orc.prefill_attention(orc.INT4, kc, vc, ks, vs, bt, [3], [0, 3], q, SM)
    assert np.array_equal(out[0, 0], _dequant(orc.INT4, vc, vs, bt[0], 1, 0)[0])


def test_last_query_is_full_decode():
    kc, vc, ks, vs, bt = _cache(orc.INT8, 1, 2, 200, 7)
    q = np.random.default_rng(8).standard_normal((37, 2, D)).astype(np.float16).view(np.uint16)
    out = orc.prefill_attention(orc.INT8, kc, vc, ks, vs, bt, [200], [0, 37], q, SM)
    dec = orc.decode_attention(orc.INT8, kc, vc, ks, vs, bt, [200], q[-1:], SM)
    assert np.array_equal(out[-1], dec[0])


def test_causal_mask_reaches_only_later_queries():
    """Changing the value codes of token 150 changes queries at positions >=
    150 and no earlier one."""
    kc, vc, ks, vs, bt = _cache(orc.INT4, 1, 1, 180, 9)
    q = np.random.default_rng(10).standard_normal((80, 1, D)).astype(np.float16).view(np.uint16)
    a = orc.prefill_attention(orc.INT4, kc, vc, ks, vs, bt, [180], [0, 80], q, SM)
    vc2 = vc.copy()
    vc2[bt[0, 150 // 64], 0, 150 % 64] ^= 0x77
    b = orc.prefill_attention(orc.INT4, kc, vc2, ks, vs, bt, [180], [0, 80], q, SM)
    pos = 180 - 80 + np.arange(80)
    changed = np.any(a[:, 0] != b[:, 0], axis=1)
    assert not changed[pos < 150].any() and changed[pos >= 150].all()


def test_empty_and_oversized_chunks():
    """No new tokens anywhere gives an empty result; a chunk longer than its
    sequence (queries before position 0) is rejected."""
    kc, vc, ks, vs, bt = _cache(orc.INT4, 2, 1, 64, 11)
    q = np.zeros((0, 1, D), np.uint16)
    out = orc.prefill_attention(orc.INT4, kc, vc, ks, vs, bt, [10, 20], [0, 0, 0], q, SM)
    assert out.shape == (0, 1, D)
    q = np.zeros((11, 1, D), np.uint16)
    with pytest.raises(ValueError):
        orc.prefill_attention(orc.INT4, kc, vc, ks, vs, bt, [10, 20], [0, 11, 11], q, SM)
