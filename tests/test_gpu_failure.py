"""Failure paths of decode attention, exercised without faulting or hanging
the GPU.

* A bounded wait that runs out.  The test hook (include/kvq_testing.h) makes
  the grid's first warp arm the barrier of its second chunk without issuing
  that chunk's copies; with the wait limit at 1 ms the warp's wait for the
  chunk runs out with nothing in flight, it sets KVQ_FLAG_TIMEOUT and returns.
  The call completes, kvq_get_device_status reports KVQ_ERR_TIMEOUT, and the
  context stays usable.
* A workspace whose split counters are not zero -- never zero-filled, or left
  non-zero by a call that was cut short.  Every counter word carries a tag of
  the call that wrote it, so the next call that uses the workspace reports
  KVQ_FLAG_BAD_WORKSPACE instead of merging early without a flag; zero-filling
  the workspace again recovers results equal to the oracle's.
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


LENS = [16384, 12000, 16385, 10000]
H = 4


def _problem(fmt, seed):
    # long enough that every warp of the grid has several units (so the first
    # warp fills at least two stages) and every (sequence, head) is cut into pieces
    wl = W.Workload(len(LENS), H, D, LENS, fmt, 1.0, ("per_head", 4, 10.0), "permuted", seed=seed)
    dw = DeviceWorkload(wl)
    dw.prefill()
    q = torch.empty((wl.B, wl.H, D), dtype=torch.float16, device="cuda")
    wl.q_device(q, seed)
    return wl, dw, q


def _oracle_out(wl):
    rb = orc.row_bytes(wl.fmt, D)
    kc = np.zeros((wl.num_pages, wl.H, 64, rb), np.uint8)
    vc = np.zeros_like(kc)
    ks = np.zeros((wl.num_pages, wl.H), np.float32)
    vs = np.zeros_like(ks)
    for b in range(wl.B):
        orc.quantize_into_pages(wl.fmt, wl.kv_host("k", b, 0, int(wl.lens[b])), wl.block_table[b], kc, ks)
        orc.quantize_into_pages(wl.fmt, wl.kv_host("v", b, 0, int(wl.lens[b])), wl.block_table[b], vc, vs)
    ref = orc.decode_attention(wl.fmt, kc, vc, ks, vs, wl.block_table, wl.lens, wl.q_host(wl.seed),
                               np.float32(1 / math.sqrt(D)))
    vmax = orc.value_absmax(wl.fmt, vc, vs, wl.block_table, wl.lens, wl.H, D)
    return ref, vmax


def _decode(dw, q, workspace=None):
    out = torch.full_like(q, float("nan"))
    kvq.kvq_decode_attention(dw.cache, q, dw.block_table, dw.lens, dw.softmax_scale, out,
                             dw.workspace if workspace is None else workspace)
    torch.cuda.synchronize()
    return out


def _err(out, ref, vmax):
    return orc.normalized_error(out.float().cpu().numpy().astype(np.float64), ref, vmax)


@pytest.fixture
def fault_hook():
    yield kvq.kvq_testing_set_decode_fault
    kvq.kvq_testing_set_decode_fault(0, -1)


@pytest.mark.parametrize("fmt", [kvq.KVQ_INT4_B64, kvq.KVQ_INT8_PAGE])
def test_bounded_wait_runs_out_and_reports_timeout(cuda_ok, fault_hook, fmt):
    wl, dw, q = _problem(fmt, 11)
    ref, vmax = _oracle_out(wl)
    assert _err(_decode(dw, q), ref, vmax) <= TOL
    assert kvq.kvq_get_device_status(dw.cache) == (0, 0)

    fault_hook(1000, 1)  # 1 ms limit; warp 0's second chunk gets no copies
    _decode(dw, q)
    fault_hook(0, -1)
    rc, flags = kvq.kvq_get_device_status(dw.cache)
    assert flags & kvq.KVQ_FLAG_TIMEOUT, flags
    assert rc == 5  # KVQ_ERR_TIMEOUT

    # the cut-short call left the workspace's counters non-zero: the next call
    # on it reports that instead of merging with them
    _decode(dw, q)
    rc, flags = kvq.kvq_get_device_status(dw.cache)
    assert flags & kvq.KVQ_FLAG_BAD_WORKSPACE, flags
    # zero-filled again, the workspace gives the oracle's results, twice in a row
    dw.workspace.zero_()
    for _ in range(2):
        assert _err(_decode(dw, q), ref, vmax) <= TOL
        assert kvq.kvq_get_device_status(dw.cache) == (0, 0)


def test_skip_beyond_the_warps_chunks_changes_nothing(cuda_ok, fault_hook):
    wl, dw, q = _problem(kvq.KVQ_INT4_B64, 12)
    ref, vmax = _oracle_out(wl)
    fault_hook(1000, 1 << 30)
    out = _decode(dw, q)
    fault_hook(0, -1)
    assert kvq.kvq_get_device_status(dw.cache) == (0, 0)
    assert _err(out, ref, vmax) <= TOL


def _counter_word_of_first_head():
    """The counter word that counts (sequence 0, head 0) of the int4 problem:
    the split gives warp w the units [U w / GW, U (w+1) / GW) with U = the
    units of all (sequence, head)s (32 tokens each, sequence-major), GW =
    min(SMs x 12, ceil(U / 2)); a split (sequence, head) is counted in the
    word of the warp that holds its last unit."""
    units = [(L + 31) // 32 for L in LENS]
    U = H * sum(units)
    GW = min(torch.cuda.get_device_properties(0).multi_processor_count * 12, (U + 1) // 2)
    last = units[0] - 1
    return ((last + 1) * GW - 1) // U


@pytest.mark.parametrize("pattern", ["one_word", "every_word", "garbage"])
def test_dirty_workspace_is_reported(cuda_ok, pattern):
    """The workspace starts with one counter word per warp of the grid, which
    counts the units of split (sequence, head)s.  A stale count of 1 in the
    word that (sequence 0, head 0) uses, in every word, or arbitrary bytes
    everywhere, must raise KVQ_FLAG_BAD_WORKSPACE."""
    wl, dw, q = _problem(kvq.KVQ_INT4_B64, 13)
    ref, vmax = _oracle_out(wl)
    ws = dw.workspace
    words = ws.view(torch.int64)
    if pattern == "one_word":
        words[_counter_word_of_first_head()] = 1
    elif pattern == "every_word":
        sms = torch.cuda.get_device_properties(0).multi_processor_count
        words[:sms * 16] = 1  # every counter the grid can use
    else:
        g = torch.Generator(device="cuda").manual_seed(5)
        ws.copy_(torch.randint(0, 256, ws.shape, dtype=torch.uint8, device="cuda", generator=g))
    _decode(dw, q)
    rc, flags = kvq.kvq_get_device_status(dw.cache)
    assert flags & kvq.KVQ_FLAG_BAD_WORKSPACE and rc == 6, (rc, flags)
    ws.zero_()
    assert _err(_decode(dw, q), ref, vmax) <= TOL
    assert kvq.kvq_get_device_status(dw.cache) == (0, 0)
