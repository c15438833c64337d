"""ctypes binding of the CPU oracle (kvq_oracle.c).

Test infrastructure only: tests, the smoke check and the benchmark's CPU
baseline use it; the product path never does.  numpy arrays in, numpy arrays
out.  Every entry releases the GIL while the C code runs, so several Python
threads can run independent (sequence) samples side by side.
"""
import ctypes
import os

import numpy as np

from . import build as _build

INT4 = 0
INT8 = 1
FP8 = 2
BLOCK = 64

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        vp = ctypes.c_void_p
        L.orc_half_to_float.argtypes = [ctypes.c_uint16]
        L.orc_half_to_float.restype = ctypes.c_float
        L.orc_e4m3_to_double.argtypes = [ctypes.c_uint8]
        L.orc_e4m3_to_double.restype = ctypes.c_double
        L.orc_float_to_e4m3.argtypes = [ctypes.c_float]
        L.orc_float_to_e4m3.restype = ctypes.c_uint8
        L.orc_quantize.argtypes = [ctypes.c_int, vp, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, vp, vp]
        L.orc_quantize.restype = ctypes.c_int
        L.orc_decode_attention.argtypes = [ctypes.c_int, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                           vp, vp, vp, vp, vp, ctypes.c_int32, vp, ctypes.c_int32, vp,
                                           ctypes.c_double, ctypes.c_int32, vp]
        L.orc_decode_attention.restype = ctypes.c_int
        L.orc_decode_attention_gqa.argtypes = [ctypes.c_int, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                               ctypes.c_int32, vp, vp, vp, vp, vp, ctypes.c_int32, vp,
                                               ctypes.c_int32, vp, ctypes.c_double, ctypes.c_int32, vp]
        L.orc_decode_attention_gqa.restype = ctypes.c_int
        L.orc_value_absmax.argtypes = [ctypes.c_int, ctypes.c_int32, ctypes.c_int32, vp, vp, vp,
                                       ctypes.c_int32, vp, ctypes.c_int32, vp]
        L.orc_value_absmax.restype = ctypes.c_int
        _lib = L
    return _lib


def _p(a):
    return ctypes.c_void_p(a.ctypes.data)


def row_bytes(fmt, D):
    return D // 2 if fmt == INT4 else D


def half_to_float(bits):
    return lib().orc_half_to_float(int(bits))


def e4m3_to_float(code):
    """The value of one FP8 E4M3 code (binary64, exact; NaN for 0x7f / 0xff)."""
    return lib().orc_e4m3_to_double(int(code))


def float_to_e4m3(y):
    """E4M3 code of a binary32 value: nearest, ties to even, saturating at 448."""
    return int(lib().orc_float_to_e4m3(float(y)))


def quantize(fmt, x_bits):
    """Quantize x[T][H][D] (uint16 fp16 bits).  Returns (codes, scales):
    codes uint8 [ceil(T/64)][H][64][row_bytes], scales float32 [ceil(T/64)][H]."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    T, H, D = x.shape
    nb = (T + BLOCK - 1) // BLOCK
    codes = np.zeros((nb, H, BLOCK, row_bytes(fmt, D)), dtype=np.uint8)
    scales = np.zeros((nb, H), dtype=np.float32)
    rc = lib().orc_quantize(fmt, _p(x), T, H, D, _p(codes), _p(scales))
    if rc != 0:
        raise ValueError("orc_quantize rejected its arguments")
    return codes, scales


def decode_attention(fmt, k_codes, v_codes, k_scales, v_scales, block_table, seq_lens, q_bits,
                     softmax_scale, num_splits=1):
    """Binary64 decode attention over a paged cache.  Returns float64 [B][Hq][D].
    q may hold Hq = g * Hkv heads for a cache of Hkv heads (query head i reads
    cache head i // g); Hq == Hkv is multi-head attention."""
    k_codes = np.ascontiguousarray(k_codes, dtype=np.uint8)
    v_codes = np.ascontiguousarray(v_codes, dtype=np.uint8)
    k_scales = np.ascontiguousarray(k_scales, dtype=np.float32)
    v_scales = np.ascontiguousarray(v_scales, dtype=np.float32)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    q = np.ascontiguousarray(q_bits, dtype=np.uint16)
    B, Hq, D = q.shape
    num_pages, Hkv = k_codes.shape[0], k_codes.shape[1]
    out = np.zeros((B, Hq, D), dtype=np.float64)
    if Hq == Hkv:
        rc = lib().orc_decode_attention(fmt, Hq, D, num_pages, _p(k_codes), _p(v_codes), _p(k_scales),
                                        _p(v_scales), _p(bt), bt.shape[1], _p(sl), B, _p(q),
                                        float(softmax_scale), int(num_splits), _p(out))
    else:
        rc = lib().orc_decode_attention_gqa(fmt, Hkv, Hq, D, num_pages, _p(k_codes), _p(v_codes), _p(k_scales),
                                            _p(v_scales), _p(bt), bt.shape[1], _p(sl), B, _p(q),
                                            float(softmax_scale), int(num_splits), _p(out))
    if rc != 0:
        raise ValueError("orc_decode_attention rejected its arguments")
    return out


def prefill_attention(fmt, k_codes, v_codes, k_scales, v_scales, block_table, seq_lens, cu_seqlens_q, q_bits,
                      softmax_scale):
    """Binary64 causal attention of a chunk of new tokens over the paged cache
    that already holds them.  Sequence b's chunk is its last
    n_b = cu_seqlens_q[b+1] - cu_seqlens_q[b] tokens: query i (row
    cu_seqlens_q[b] + i of q [total][Hq][D]) sits at position
    p = seq_lens[b] - n_b + i and attends to the keys at positions 0 .. p.
    That is, by definition, decode attention of each query over the first
    p + 1 tokens of its sequence -- evaluated here with decode_attention, one
    query per row.  Returns float64 [total][Hq][D]."""
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    sl = np.asarray(seq_lens, dtype=np.int64)
    cu = np.asarray(cu_seqlens_q, dtype=np.int64)
    q = np.ascontiguousarray(q_bits, dtype=np.uint16)
    total = int(cu[-1])
    if total == 0:
        return np.zeros((0,) + q.shape[1:], dtype=np.float64)
    rows = np.zeros(total, dtype=np.int64)
    lens = np.zeros(total, dtype=np.int32)
    for b in range(len(sl)):
        n = int(cu[b + 1] - cu[b])
        if n > sl[b]:
            raise ValueError("a chunk longer than its sequence")
        rows[cu[b]:cu[b + 1]] = b
        lens[cu[b]:cu[b + 1]] = sl[b] - n + 1 + np.arange(n)
    return decode_attention(fmt, k_codes, v_codes, k_scales, v_scales, bt[rows], lens, q, softmax_scale)


def value_absmax(fmt, v_codes, v_scales, block_table, seq_lens, H, D):
    """max |v^| per (sequence, head), float64 [B][H]."""
    v_codes = np.ascontiguousarray(v_codes, dtype=np.uint8)
    v_scales = np.ascontiguousarray(v_scales, dtype=np.float32)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    B = sl.shape[0]
    out = np.zeros((B, H), dtype=np.float64)
    lib().orc_value_absmax(fmt, H, D, _p(v_codes), _p(v_scales), _p(bt), bt.shape[1], _p(sl), B, _p(out))
    return out


def quantize_into_pages(fmt, x_bits, block_table_row, k_codes_pages, k_scales_pages):
    """Quantize one sequence x[L][H][D] and place block j into page
    block_table_row[j] of a paged code array [num_pages][H][64][row_bytes] and
    scale array [num_pages][H] (placement is plain indexing)."""
    codes, scales = quantize(fmt, x_bits)
    for j in range(codes.shape[0]):
        pg = int(block_table_row[j])
        k_codes_pages[pg] = codes[j]
        k_scales_pages[pg] = scales[j]


def normalized_error(out_test, out_ref, vmax):
    """max over (b, h, d) of |test - ref| / max|v^|_(b,h); a (b, h) whose values
    are all zero must match exactly (0/0 reads as 0 only when the error is 0)."""
    err = np.abs(np.asarray(out_test, dtype=np.float64) - out_ref)
    per = err.max(axis=-1)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.where(vmax > 0, per / np.where(vmax > 0, vmax, 1.0), np.where(per > 0, np.inf, 0.0))
    return float(r.max()) if r.size else 0.0


__all__ = ["INT4", "INT8", "FP8", "BLOCK", "e4m3_to_float", "float_to_e4m3", "lib", "quantize", "decode_attention",
           "prefill_attention", "value_absmax",
           "quantize_into_pages", "normalized_error", "half_to_float", "row_bytes"]

if os.environ.get("KVQ_ORACLE_EAGER"):
    lib()
