"""Parity at the workloads' full sizes, in the launch configuration the
benchmark times, on sampled outputs the oracle computes one (sequence, head)
at a time from the host twin of the generator.

  llama2-7b-layer  B=8, H=32, L=8192 int4: prefill, then decode steps
                   (append one token per sequence + attend), as timed
  long-context     B=16, H=32, L=32768 int4 (2.1 GB packed): decode
  paged-int8       64 seqs, L ~ U[512, 16384], int8, permuted pages: decode
  prefill-append   64 x 4096 tokens, H=32, int4 into permuted pages
  llama3-8b-layer-gqa  B=32, 8 cache heads x 4 query heads, L=8192 int4:
                   decode steps through kvq_decode_attention_gqa, as timed
  llama2-7b-layer-fp8  B=8, H=32, L=8192, FP8 E4M3: decode steps, as timed
"""
import math

import numpy as np
import pytest
import torch

from oracle import oracle as orc
from quantized_kv_cache_09_gb300 import kvq
from quantized_kv_cache_09_gb300.runner import DecodeStep, DeviceWorkload
from quantized_kv_cache_09_gb300.synth import workloads as W
from quantized_kv_cache_09_gb300.synth import synth_sample_heads

pytestmark = pytest.mark.gpu
TOL = 2e-3
D = 128


def _oracle_one(wl, b, h, L, q_bits, hq=None):
    """oracle codes/scales and attention output of one (sequence, cache head h),
    for query head hq (default h)."""
    hq = h if hq is None else hq
    k = np.ascontiguousarray(wl.kv_host("k", b, 0, L)[:, h:h + 1, :])
    v = np.ascontiguousarray(wl.kv_host("v", b, 0, L)[:, h:h + 1, :])
    kc, ks = orc.quantize(wl.fmt, k)
    vc, vs = orc.quantize(wl.fmt, v)
    nb = kc.shape[0]
    bt = np.arange(nb, dtype=np.int32)[None, :]
    q = np.ascontiguousarray(q_bits[b:b + 1, hq:hq + 1, :])
    ref = orc.decode_attention(wl.fmt, kc, vc, ks, vs, bt, np.array([L]), q, np.float32(1 / math.sqrt(D)))
    vmax = orc.value_absmax(wl.fmt, vc, vs, bt, np.array([L]), 1, D)
    return kc, ks, vc, vs, ref[0, 0], vmax[0, 0]


def _check_pairs(dw, lens, q_bits, out, pairs):
    """pairs: (sequence, query head); query head i reads cache head i // g"""
    wl = dw.wl
    g = wl.Hq // wl.H
    got = out.float().cpu().numpy()
    worst = 0.0
    for b, hq in pairs:
        L = int(lens[b])
        h = hq // g
        kc, ks, vc, vs, ref, vmax = _oracle_one(wl, b, h, L, q_bits, hq)
        pages = wl.block_table[b, :kc.shape[0]]
        gk = dw.cache.k_codes[torch.from_numpy(pages).long().cuda(), h].cpu().numpy()
        gv = dw.cache.v_codes[torch.from_numpy(pages).long().cuda(), h].cpu().numpy()
        assert np.array_equal(gk, kc[:, 0]), (b, h)
        assert np.array_equal(gv, vc[:, 0]), (b, h)
        gks = dw.cache.k_scales[torch.from_numpy(pages).long().cuda(), h].cpu().numpy()
        assert np.array_equal(gks.view(np.uint32), ks[:, 0].view(np.uint32)), (b, h)
        err = np.max(np.abs(got[b, hq] - ref)) / vmax
        assert err <= TOL, (b, hq, err)
        worst = max(worst, err)
    return worst


@pytest.mark.parametrize("cfg", [2, 6, 7])
def test_layer_decode_steps(cuda_ok, cfg):
    """llama2-7b-layer (int4), llama3-8b-layer-gqa, llama2-7b-layer-fp8: three
    timed-style steps, then sampled (sequence, query head) outputs and their
    cache pages against the oracle."""
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
    _check_pairs(dw, lens, wl.q_host(2), out, synth_sample_heads(wl.B, wl.Hq, 6, seed=1))


def test_long_context_decode(cuda_ok):
    wl = W.make_workload(3)
    dw = DeviceWorkload(wl)
    dw.prefill(max_tokens_per_call=1 << 16)
    q = torch.empty((wl.B, wl.H, D), dtype=torch.float16, device="cuda")
    wl.q_device(q, 0)
    out = torch.empty_like(q)
    kvq.kvq_decode_attention(dw.cache, q, dw.block_table, dw.lens, dw.softmax_scale, out, dw.workspace)
    torch.cuda.synchronize()
    _check_pairs(dw, wl.lens, wl.q_host(0), out, synth_sample_heads(wl.B, wl.H, 3, seed=2))


def test_paged_int8_decode(cuda_ok):
    wl = W.make_workload(4)
    dw = DeviceWorkload(wl)
    dw.prefill(max_tokens_per_call=1 << 18)
    q = torch.empty((wl.B, wl.H, D), dtype=torch.float16, device="cuda")
    wl.q_device(q, 0)
    out = torch.empty_like(q)
    kvq.kvq_decode_attention(dw.cache, q, dw.block_table, dw.lens, dw.softmax_scale, out, dw.workspace)
    torch.cuda.synchronize()
    pairs = synth_sample_heads(wl.B, wl.H, 4, seed=3)
    pairs.append((int(np.argmax(wl.lens)), 5))
    pairs.append((int(np.argmin(wl.lens)), 30))
    _check_pairs(dw, wl.lens, wl.q_host(0), out, pairs)


def test_prefill_append_sampled_sequences(cuda_ok):
    wl = W.make_workload(5)
    dw = DeviceWorkload(wl)
    # one call with all 262144 tokens, as timed
    dw.prefill(max_tokens_per_call=1 << 20)
    assert kvq.kvq_get_device_status(dw.cache) == (0, 0)
    for b in (0, 37, 63):
        for which, codes, scales in (("k", dw.cache.k_codes, dw.cache.k_scales),
                                     ("v", dw.cache.v_codes, dw.cache.v_scales)):
            oc, os_ = orc.quantize(wl.fmt, wl.kv_host(which, b, 0, int(wl.lens[b])))
            pages = torch.from_numpy(wl.block_table[b, :oc.shape[0]]).long().cuda()
            assert np.array_equal(codes[pages].cpu().numpy(), oc)
            assert np.array_equal(scales[pages].cpu().numpy().view(np.uint32), os_.view(np.uint32))
