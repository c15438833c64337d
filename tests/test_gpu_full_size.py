"""Parity at the workloads' full sizes, in the launch configuration the
benchmark times: every (sequence, head) of every workload is checked.

For each sequence the oracle regenerates the K and V history from the host
twin of the generator, quantizes it with its own codec and compares every code
block and both scale arrays with the pages the CUDA path wrote (bit-exact);
then it attends over its own cache with the same query, in binary64, and
compares every query head's output (max-abs error normalised by max|v^| of
that (sequence, cache head) <= 2e-3).  Sequences are checked one per worker
thread (the oracle and the generator release the GIL), so only a few
sequences' histories are on the host at a time.

  llama2-7b-layer      B=8, H=32, L=8192 int4: prefill, then three decode steps
                       (append one token per sequence + attend), as timed
  long-context         B=16, H=32, L=32768 int4 (2.1 GB packed): decode
  paged-int8           64 seqs, L ~ U[512, 16384], int8, permuted pages: decode
  prefill-append       64 x 4096 tokens, H=32, int4 into permuted pages (codes
                       and scales only: no attention in this workload)
  llama3-8b-layer-gqa  B=32, 8 cache heads x 4 query heads, L=8192 int4:
                       decode steps through kvq_decode_attention_gqa, as timed
  llama2-7b-layer-fp8  B=8, H=32, L=8192, FP8 E4M3: decode steps, as timed
  mqa-32k              B=64, 1 cache head x 32 query heads, L=32768 int4,
                       permuted pages: decode steps, as timed
  llama3-70b-layer-gqa B=32, 8 cache heads x 8 query heads, L=8192 int4:
                       decode steps, as timed (and the same over FP8:
                       llama3-70b-layer-gqa-fp8)
"""
import concurrent.futures as cf
import math
import os

import numpy as np
import pytest
import torch

from oracle import oracle as orc
from quantized_kv_cache_09_gb300 import kvq
from quantized_kv_cache_09_gb300.runner import DecodeStep, DeviceWorkload
from quantized_kv_cache_09_gb300.synth import workloads as W

pytestmark = pytest.mark.gpu
TOL = 2e-3
D = 128
CHUNK = 4096  # tokens regenerated and quantized at a time (a multiple of 64)


def _oracle_sequence(wl, which, b, L):
    """The oracle's codes [nb][H][64][rb] and scales [nb][H] of one sequence's
    K or V history, quantized CHUNK tokens (whole blocks) at a time."""
    codes, scales = [], []
    for t0 in range(0, L, CHUNK):
        c, s = orc.quantize(wl.fmt, wl.kv_host(which, b, t0, min(L, t0 + CHUNK)))
        codes.append(c)
        scales.append(s)
    return np.concatenate(codes), np.concatenate(scales)


def _check_sequence(wl, b, L, gpu, q_row, out_row):
    """gpu: this sequence's pages as the CUDA path left them (k/v codes and
    scales in block order).  Returns the worst normalised attention error over
    its query heads (0 when no output is checked)."""
    kc, ks = _oracle_sequence(wl, "k", b, L)
    vc, vs = _oracle_sequence(wl, "v", b, L)
    gkc, gks, gvc, gvs = gpu
    for name, a, o in (("k codes", gkc, kc), ("v codes", gvc, vc)):
        if not np.array_equal(a, o):
            bad = np.argwhere(a != o)[0]
            raise AssertionError(f"sequence {b}: {name} differ first at block/head/row/byte {tuple(bad)}")
    for name, a, o in (("k scales", gks, ks), ("v scales", gvs, vs)):
        if not np.array_equal(a.view(np.uint32), o.view(np.uint32)):
            bad = np.argwhere(a.view(np.uint32) != o.view(np.uint32))[0]
            raise AssertionError(f"sequence {b}: {name} differ first at block/head {tuple(bad)}")
    if out_row is None:
        return 0.0
    bt = np.arange(kc.shape[0], dtype=np.int32)[None, :]
    ref = orc.decode_attention(wl.fmt, kc, vc, ks, vs, bt, np.array([L], np.int32), q_row[None],
                               np.float32(1 / math.sqrt(D)))[0]
    vmax = orc.value_absmax(wl.fmt, vc, vs, bt, np.array([L], np.int32), wl.H, D)[0]
    g = wl.Hq // wl.H
    err = orc.normalized_error(out_row.astype(np.float64), ref, np.repeat(vmax, g))
    if not err <= TOL:
        raise AssertionError(f"sequence {b}: normalised attention error {err:.3e} > {TOL}")
    return err


def _verify_all(dw, lens, q_bits=None, out=None):
    """Every sequence of a device workload against the oracle (see the module doc)."""
    wl = dw.wl
    got = None if out is None else out.float().cpu().numpy()
    workers = max(1, min(16, os.cpu_count() or 1))
    worst = 0.0
    with cf.ThreadPoolExecutor(max_workers=workers) as ex:
        futs = []
        for b in range(wl.B):
            L = int(lens[b])
            nb = (L + 63) // 64
            pages = torch.from_numpy(np.ascontiguousarray(wl.block_table[b, :nb])).long().to(dw.cache.k_codes.device)
            gpu = (dw.cache.k_codes[pages].cpu().numpy(), dw.cache.k_scales[pages].cpu().numpy(),
                   dw.cache.v_codes[pages].cpu().numpy(), dw.cache.v_scales[pages].cpu().numpy())
            futs.append(ex.submit(_check_sequence, wl, b, L, gpu, None if q_bits is None else q_bits[b],
                                  None if got is None else got[b]))
            if len(futs) >= 2 * workers:  # bound the host memory in flight
                worst = max(worst, futs.pop(0).result())
        for f in futs:
            worst = max(worst, f.result())
    return worst


@pytest.mark.parametrize("cfg", [2, 6, 7, 9, 10, 11])
def test_layer_decode_steps(cuda_ok, cfg):
    """llama2-7b-layer (int4), llama3-8b-layer-gqa, llama2-7b-layer-fp8,
    mqa-32k, llama3-70b-layer-gqa (int4, FP8): three timed-style steps, then every sequence's pages and every
    (sequence, query head) output against the oracle."""
    wl = W.make_workload(cfg, extra_tokens=64)
    dw = DeviceWorkload(wl)
    dw.prefill()
    step = DecodeStep(dw)
    lens = wl.lens.copy()
    for s in range(3):
        k1, v1, q = dw.new_token_tensors(s)
        before = torch.from_numpy(lens).cuda()
        after = torch.from_numpy(lens + 1).cuda()
        out = step.run(before, after, k1, v1, q)
        lens = lens + 1
    torch.cuda.synchronize()
    assert kvq.kvq_get_device_status(dw.cache) == (0, 0)
    _verify_all(dw, lens, wl.q_host(2), out)


def test_long_context_decode(cuda_ok):
    wl = W.make_workload(3)
    dw = DeviceWorkload(wl)
    dw.prefill(max_tokens_per_call=1 << 16)
    q = torch.empty((wl.B, wl.H, D), dtype=torch.float16, device="cuda")
    wl.q_device(q, 0)
    out = torch.empty_like(q)
    kvq.kvq_decode_attention(dw.cache, q, dw.block_table, dw.lens, dw.softmax_scale, out, dw.workspace)
    torch.cuda.synchronize()
    assert kvq.kvq_get_device_status(dw.cache) == (0, 0)
    _verify_all(dw, wl.lens, wl.q_host(0), out)


def test_paged_int8_decode(cuda_ok):
    wl = W.make_workload(4)
    dw = DeviceWorkload(wl)
    dw.prefill(max_tokens_per_call=1 << 18)
    q = torch.empty((wl.B, wl.H, D), dtype=torch.float16, device="cuda")
    wl.q_device(q, 0)
    out = torch.empty_like(q)
    kvq.kvq_decode_attention(dw.cache, q, dw.block_table, dw.lens, dw.softmax_scale, out, dw.workspace)
    torch.cuda.synchronize()
    assert kvq.kvq_get_device_status(dw.cache) == (0, 0)
    _verify_all(dw, wl.lens, wl.q_host(0), out)


def test_prefill_append_every_sequence(cuda_ok):
    wl = W.make_workload(5)
    dw = DeviceWorkload(wl)
    # one call with all 262144 tokens, as timed
    dw.prefill(max_tokens_per_call=1 << 20)
    assert kvq.kvq_get_device_status(dw.cache) == (0, 0)
    _verify_all(dw, wl.lens)


@pytest.mark.parametrize("cfg,fmt,seqs", [(2, W.INT4, None), (2, W.INT8, None), (7, W.FP8, None), (3, W.INT4, (0, 5, 10, 15))])
def test_stateless_quantize_full_size(cuda_ok, cfg, fmt, seqs):
    """kvq_quantize as the quantize workloads time it: the whole K history of
    the workload's sequences as one [B*L][H][D] tensor (sequences back to
    back), then V; every code block and both scale arrays of the checked
    sequences bit-exact against the oracle (long-context: four of its 16
    sequences, the first and the last among them)."""
    wl = W.make_workload(cfg)
    wl.fmt = fmt
    L = int(wl.lens[0])
    T = wl.B * L
    nb = L // 64
    res = []
    for which in ("k", "v"):
        x = torch.empty((T, wl.H, D), dtype=torch.float16, device="cuda")
        for b in range(wl.B):
            wl.kv_device(which, b, 0, L, x[b * L:(b + 1) * L])
        codes = torch.empty((T // 64, wl.H, 64, wl.row_bytes), dtype=torch.uint8, device="cuda")
        scales = torch.empty((T // 64, wl.H), dtype=torch.float32, device="cuda")
        kvq.kvq_quantize(fmt, x, codes, scales)
        del x
        res.append((codes, scales))
    torch.cuda.synchronize()
    (kc, ks), (vc, vs) = res
    check = range(wl.B) if seqs is None else seqs
    workers = max(1, min(8, os.cpu_count() or 1))
    with cf.ThreadPoolExecutor(max_workers=workers) as ex:
        futs = [ex.submit(_check_sequence, wl, b, L,
                          (kc[b * nb:(b + 1) * nb].cpu().numpy(), ks[b * nb:(b + 1) * nb].cpu().numpy(),
                           vc[b * nb:(b + 1) * nb].cpu().numpy(), vs[b * nb:(b + 1) * nb].cpu().numpy()),
                          None, None) for b in check]
        for f in futs:
            f.result()
