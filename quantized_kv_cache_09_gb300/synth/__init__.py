"""Seeded synthetic inputs for the KV-cache workloads.

A module of its own: it generates inputs (fp16 keys, values and queries,
outlier channels, block tables, sequence lengths) and holds none of the
quantization or attention arithmetic.  The host build (numpy arrays) and the
device build (torch CUDA tensors) produce identical bits for every element;
a test checks that.

Element (t, h, d) of the key (or value) history of sequence b has global index
(t * H + h) * D + d in the stream of (tensor, b), so any token range of a
sequence -- the whole history, one appended token, one decode step -- can be
regenerated on its own and always agrees with the rest.
"""
import ctypes
import os

import numpy as np

from .. import build as _build

# stream ids (tensor kind in the high 32 bits, sequence / step in the low 32)
K_HIST = 1
V_HIST = 2
QUERY = 3
CHUNK_QUERY = 4  # queries of a prefill chunk, one stream per sequence
K_OUTLIER = 16
V_OUTLIER = 17
BLOCK_TABLE = 32
LENGTHS = 48
SAMPLE = 64

_host = None
_dev = None


def _host_lib():
    global _host
    if _host is None:
        if not os.path.exists(_build.LIB_SYNTH):
            _build.build()
        L = ctypes.CDLL(_build.LIB_SYNTH)
        vp, i64, u64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64, ctypes.c_int32
        L.kvq_synth_fill_f16.argtypes = [vp, i64, u64, u64, i64, ctypes.c_float, vp, i64, ctypes.c_float]
        L.kvq_synth_fill_f16.restype = None
        L.kvq_synth_outliers_per_head.argtypes = [vp, i32, i32, i32, u64, u64]
        L.kvq_synth_outliers_bernoulli.argtypes = [vp, i32, i32, ctypes.c_uint32, u64, u64]
        L.kvq_synth_permutation.argtypes = [vp, i64, u64, u64]
        L.kvq_synth_uniform_int.argtypes = [vp, i64, i32, i32, u64, u64]
        L.kvq_synth_f32_to_f16_export.argtypes = [ctypes.c_float]
        L.kvq_synth_f32_to_f16_export.restype = ctypes.c_uint16
        _host = L
    return _host


def _dev_lib():
    global _dev
    if _dev is None:
        if not os.path.exists(_build.LIB_SYNTH_CUDA):
            _build.build()
        L = ctypes.CDLL(_build.LIB_SYNTH_CUDA)
        vp, i64, u64 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64
        L.kvq_synth_fill_f16_cuda.argtypes = [vp, i64, u64, u64, i64, ctypes.c_float, vp, i64,
                                              ctypes.c_float, vp]
        L.kvq_synth_fill_f16_cuda.restype = ctypes.c_int
        _dev = L
    return _dev


def stream_id(kind, idx=0):
    return (int(kind) << 32) | (int(idx) & 0xFFFFFFFF)


def _ptr(a):
    return ctypes.c_void_p(a.ctypes.data) if a is not None else None


def f32_to_f16_bits(x):
    """The generator's binary32 -> binary16 rounding, one value."""
    return int(_host_lib().kvq_synth_f32_to_f16_export(float(np.float32(x))))


def fill_f16_host(n, seed, stream, index0=0, sigma=1.0, mask=None, outlier_mult=1.0):
    out = np.empty(int(n), dtype=np.uint16)
    m = None if mask is None else np.ascontiguousarray(mask, dtype=np.uint8)
    _host_lib().kvq_synth_fill_f16(_ptr(out), int(n), int(seed), int(stream), int(index0),
                                   float(sigma), _ptr(m), 0 if m is None else m.size, float(outlier_mult))
    return out


def fill_f16_device(out, seed, stream, index0=0, sigma=1.0, mask_dev=None, outlier_mult=1.0,
                    cuda_stream=None):
    """Fill a contiguous CUDA tensor (int16/uint16/float16, any shape) in place."""
    import torch
    assert out.is_cuda and out.is_contiguous() and out.element_size() == 2
    s = torch.cuda.current_stream(out.device).cuda_stream if cuda_stream is None else cuda_stream
    mp = None if mask_dev is None else ctypes.c_void_p(mask_dev.data_ptr())
    rc = _dev_lib().kvq_synth_fill_f16_cuda(ctypes.c_void_p(out.data_ptr()), out.numel(), int(seed),
                                            int(stream), int(index0), float(sigma), mp,
                                            0 if mask_dev is None else mask_dev.numel(),
                                            float(outlier_mult), ctypes.c_void_p(s))
    if rc != 0:
        raise RuntimeError(f"device generator failed (code {rc})")
    return out


def outliers_per_head(H, D, count, seed, stream):
    m = np.zeros((H, D), dtype=np.uint8)
    _host_lib().kvq_synth_outliers_per_head(_ptr(m), H, D, count, int(seed), int(stream))
    return m


def outliers_bernoulli(H, D, p, seed, stream):
    m = np.zeros((H, D), dtype=np.uint8)
    thr = min(int(round(p * 2 ** 32)), 2 ** 32 - 1)
    _host_lib().kvq_synth_outliers_bernoulli(_ptr(m), H, D, thr, int(seed), int(stream))
    return m


def permutation(n, seed, stream):
    out = np.empty(int(n), dtype=np.int32)
    _host_lib().kvq_synth_permutation(_ptr(out), int(n), int(seed), int(stream))
    return out


def uniform_int(n, lo, hi, seed, stream):
    out = np.empty(int(n), dtype=np.int32)
    _host_lib().kvq_synth_uniform_int(_ptr(out), int(n), int(lo), int(hi), int(seed), int(stream))
    return out


def synth_sample_heads(B, H, n, seed):
    """n seeded (sequence, head) pairs, for sampled full-size parity checks."""
    bs = uniform_int(n, 0, B - 1, seed, stream_id(SAMPLE, 0))
    hs = uniform_int(n, 0, H - 1, seed, stream_id(SAMPLE, 1))
    return [(int(b), int(h)) for b, h in zip(bs, hs)]


from .workloads import Workload, make_workload, RECIPES  # noqa: E402

__all__ = ["fill_f16_host", "fill_f16_device", "outliers_per_head", "outliers_bernoulli", "permutation",
           "uniform_int", "stream_id", "synth_sample_heads", "Workload", "make_workload", "RECIPES", "f32_to_f16_bits"]
