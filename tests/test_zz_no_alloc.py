"""The allocation-free decode entry point, kvq_decode_attention_noalloc.

Some callers cannot allocate device memory at the moment they run decode
attention -- an inference-engine plugin whose execute step must not allocate,
a process whose device memory is reserved up front by another allocator, a
serving loop that cannot afford the synchronisation cudaMalloc / cudaFree may
cause.  The no-alloc entry point serves them from a fixed scratch array inside
the library instead of a caller workspace.

Through the C ABI, several calls in a row (different problems, so each finds
the previous call's leftovers in the shared array) must give the outputs of
kvq_decode_attention with a caller workspace, within the attention tolerance
the other tests use (2e-3 of max|v^| per sequence and head).  This file is
collected last so that a run stopping at the first failure has already run
every other test; it also passes on its own in a fresh process.
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


def _problem(fmt, lens, seed):
    wl = W.Workload(len(lens), 8, 128, lens, fmt, 1.0, ("per_head", 4, 10.0), "permuted", seed=seed)
    dw = DeviceWorkload(wl)
    dw.prefill()
    q = torch.empty((wl.B, wl.H, wl.D), dtype=torch.float16, device="cuda")
    wl.q_device(q, seed)
    ref = torch.empty_like(q)
    kvq.kvq_decode_attention(dw.cache, q, dw.block_table, dw.lens, dw.softmax_scale, ref, dw.workspace)
    torch.cuda.synchronize()
    vmax = orc.value_absmax(fmt, dw.cache.v_codes.cpu().numpy(), dw.cache.v_scales.cpu().numpy(),
                            wl.block_table, wl.lens, wl.H, wl.D)
    return dw, q, ref, vmax


def test_noalloc_matches_workspace_entry_point(cuda_ok):
    problems = [_problem(kvq.KVQ_INT4_B64, [5000, 1, 777, 64, 0, 3000], 1),
                _problem(kvq.KVQ_INT8_PAGE, [129, 4096, 2000], 2)]
    for dw, q, ref, vmax in problems + problems[:1]:
        out = torch.full_like(q, float("nan"))
        kvq.kvq_decode_attention_noalloc(dw.cache, q, dw.block_table, dw.lens, dw.softmax_scale, out)
        torch.cuda.synchronize()
        err = orc.normalized_error(out.float().cpu().numpy().astype(np.float64),
                                   ref.float().cpu().numpy().astype(np.float64), vmax)
        assert err <= TOL, err
        assert kvq.kvq_get_device_status(dw.cache) == (0, 0)
