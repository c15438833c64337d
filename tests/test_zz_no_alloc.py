"""The allocation-free decode entry point, kvq_decode_attention_noalloc.

Some callers cannot allocate device memory at the moment they run decode
attention -- an inference-engine plugin whose execute step must not allocate,
a process whose device memory is reserved up front by another allocator, a
serving loop that cannot afford the synchronisation cudaMalloc / cudaFree may
cause.  The no-alloc entry point serves them from a fixed scratch array inside
the library instead of a caller workspace.

Through the C ABI, several calls in a row (different problems and formats, so
each finds the previous call's leftovers in the shared array) must give the
outputs of kvq_decode_attention with a caller workspace, and both must be
within the attention tolerance of the binary64 oracle (2e-3 of max|v^| per
sequence and head).  A call cut short by a bounded wait that ran out leaves
the shared array's counters non-zero; the caller cannot clear library memory,
so the next call must recover by itself.  This file is collected last so that
a run stopping at the first failure has already run every other test; it also
passes on its own in a fresh process.
"""
import math

import numpy as np
import pytest
import torch

from oracle import oracle as orc
from quantized_kv_cache_09_gb300 import kvq
from quantized_kv_cache_09_gb300.runner import DeviceWorkload
from quantized_kv_cache_09_gb300.synth import workloads as W

pytestmark = pytest.mark.gpu
TOL = 2e-3
D = 128


def _problem(fmt, lens, seed):
    wl = W.Workload(len(lens), 8, D, lens, fmt, 1.0, ("per_head", 4, 10.0), "permuted", seed=seed)
    dw = DeviceWorkload(wl)
    dw.prefill()
    q = torch.empty((wl.B, wl.H, wl.D), dtype=torch.float16, device="cuda")
    wl.q_device(q, seed)
    ref = torch.empty_like(q)
    kvq.kvq_decode_attention(dw.cache, q, dw.block_table, dw.lens, dw.softmax_scale, ref, dw.workspace)
    torch.cuda.synchronize()
    # the oracle's own cache of the same histories, and its attention over it
    rb = orc.row_bytes(fmt, D)
    kc = np.zeros((wl.num_pages, wl.H, 64, rb), np.uint8)
    vc = np.zeros_like(kc)
    ks = np.zeros((wl.num_pages, wl.H), np.float32)
    vs = np.zeros_like(ks)
    for b in range(wl.B):
        if wl.lens[b]:
            orc.quantize_into_pages(fmt, wl.kv_host("k", b, 0, int(wl.lens[b])), wl.block_table[b], kc, ks)
            orc.quantize_into_pages(fmt, wl.kv_host("v", b, 0, int(wl.lens[b])), wl.block_table[b], vc, vs)
    oref = orc.decode_attention(fmt, kc, vc, ks, vs, wl.block_table, wl.lens, wl.q_host(seed),
                                np.float32(1 / math.sqrt(D)))
    vmax = orc.value_absmax(fmt, vc, vs, wl.block_table, wl.lens, wl.H, wl.D)
    return dw, q, ref, oref, vmax


def _err(out, ref, vmax):
    return orc.normalized_error(out.float().cpu().numpy().astype(np.float64), np.asarray(ref, np.float64), vmax)


def _noalloc(dw, q):
    out = torch.full_like(q, float("nan"))
    kvq.kvq_decode_attention_noalloc(dw.cache, q, dw.block_table, dw.lens, dw.softmax_scale, out)
    torch.cuda.synchronize()
    return out


def test_noalloc_matches_workspace_entry_point_and_oracle(cuda_ok):
    problems = [_problem(kvq.KVQ_INT4_B64, [5000, 1, 777, 64, 0, 3000], 1),
                _problem(kvq.KVQ_INT8_PAGE, [129, 4096, 2000], 2),
                _problem(kvq.KVQ_FP8_E4M3, [3333, 65, 1000], 3)]
    for dw, q, ref, oref, vmax in problems + problems[:1]:
        assert _err(ref, oref, vmax) <= TOL
        out = _noalloc(dw, q)
        assert _err(out, ref.float().cpu().numpy(), vmax) <= TOL
        assert _err(out, oref, vmax) <= TOL
        assert kvq.kvq_get_device_status(dw.cache) == (0, 0)


def test_noalloc_recovers_after_a_call_cut_short(cuda_ok):
    """The test hook makes one call's bounded wait run out (1 ms, with no copy
    in flight); that call reports KVQ_ERR_TIMEOUT and leaves the shared
    array's counters non-zero.  The next two calls still match the oracle."""
    dw, q, ref, oref, vmax = _problem(kvq.KVQ_INT4_B64, [16384, 12000, 16385, 10000], 4)
    try:
        kvq.kvq_testing_set_decode_fault(1000, 1)
        _noalloc(dw, q)
    finally:
        kvq.kvq_testing_set_decode_fault(0, -1)
    rc, flags = kvq.kvq_get_device_status(dw.cache)
    assert rc == 5 and flags & kvq.KVQ_FLAG_TIMEOUT, (rc, flags)
    for _ in range(2):
        out = _noalloc(dw, q)
        assert kvq.kvq_get_device_status(dw.cache) == (0, 0)
        assert _err(out, oref, vmax) <= TOL
