"""GPU parity of decode attention over the quantized paged cache against the
binary64 oracle: the normalised error max|o - o_ref| / max|v^| of every
(sequence, head) must stay within 2e-3, the bound the target states.

The cache is built by the CUDA path (kvq_append) and must first be
bit-identical to the oracle's quantization; the oracle then attends over its
own cache.  Paging: ddd.cn section 4; decode over a quantized cache:
aicoding.csdn.net section 3.1."""
import math

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


def _oracle_cache(wl, lens, fmt=None):
    fmt = wl.fmt if fmt is None else fmt
    rb = orc.row_bytes(fmt, D)
    kc = np.zeros((wl.num_pages, wl.H, 64, rb), np.uint8)
    vc = np.zeros_like(kc)
    ks = np.zeros((wl.num_pages, wl.H), np.float32)
    vs = np.zeros_like(ks)
    for b in range(wl.B):
        if lens[b]:
            orc.quantize_into_pages(fmt, wl.kv_host("k", b, 0, lens[b]), wl.block_table[b], kc, ks)
            orc.quantize_into_pages(fmt, wl.kv_host("v", b, 0, lens[b]), wl.block_table[b], vc, vs)
    return kc, vc, ks, vs


def _check_decode(wl, lens, q_bits, out_gpu, oc=None, pairs=None):
    kc, vc, ks, vs = _oracle_cache(wl, lens) if oc is None else oc
    sm = 1.0 / math.sqrt(D)
    ref = orc.decode_attention(wl.fmt, kc, vc, ks, vs, wl.block_table, lens, q_bits, np.float32(sm))
    vmax = orc.value_absmax(wl.fmt, vc, vs, wl.block_table, lens, wl.H, D)
    got = out_gpu.float().cpu().numpy().astype(np.float64)
    err = orc.normalized_error(got, ref, vmax)
    assert err <= TOL, f"normalised error {err:.3e} > {TOL}"
    return err


def _device_cache_matches(dw, oc, lens):
    kc, vc, ks, vs = oc
    wl = dw.wl
    used = np.unique(np.concatenate([wl.block_table[b, :(lens[b] + 63) // 64] for b in range(wl.B)]))
    assert np.array_equal(dw.cache.k_codes.cpu().numpy()[used], kc[used])
    assert np.array_equal(dw.cache.v_codes.cpu().numpy()[used], vc[used])
    assert np.array_equal(dw.cache.k_scales.cpu().numpy()[used].view(np.uint32), ks[used].view(np.uint32))
    assert np.array_equal(dw.cache.v_scales.cpu().numpy()[used].view(np.uint32), vs[used].view(np.uint32))


def _run_decode(dw, q_np=None, step=0):
    wl = dw.wl
    q = torch.empty((wl.B, wl.H, D), dtype=torch.float16, device="cuda")
    if q_np is None:
        wl.q_device(q, step)
        q_np = wl.q_host(step)
    else:
        q.copy_(torch.from_numpy(q_np.view(np.float16)))
    out = torch.full_like(q, float("nan"))
    kvq.kvq_decode_attention(dw.cache, q, dw.block_table, dw.lens, dw.softmax_scale, out, dw.workspace)
    torch.cuda.synchronize()
    return q_np, out


def test_tiny_config_quantize_plus_one_decode_step(cuda_ok):
    """tiny: B=2, H=4, L=256, int4, contiguous cache; prefill, then one decode
    step (append token 256, attend over 257) exactly as the benchmark runs it."""
    wl = W.make_workload(1, extra_tokens=64)
    dw = DeviceWorkload(wl)
    dw.prefill()
    oc = _oracle_cache(wl, wl.lens)
    _device_cache_matches(dw, oc, wl.lens)
    k1, v1, q = dw.new_token_tensors(0)
    step = DecodeStep(dw)
    after = dw.lens + 1
    out = step.run(dw.lens, after, k1, v1, q)
    torch.cuda.synchronize()
    lens2 = wl.lens + 1
    oc2 = _oracle_cache(wl, lens2)
    _device_cache_matches(dw, oc2, lens2)
    _check_decode(wl, lens2, wl.q_host(0), out, oc2)
    assert kvq.kvq_get_device_status(dw.cache) == (0, 0)


@pytest.mark.parametrize("fmt", [kvq.KVQ_INT4_B64, kvq.KVQ_INT8_PAGE, kvq.KVQ_FP8_E4M3])
def test_ragged_lengths_and_edges(cuda_ok, fmt):
    """Lengths at every unit/page edge, an empty sequence, a permuted table."""
    lens = [1, 15, 16, 17, 31, 32, 33, 63, 64, 65, 127, 128, 129, 0, 257, 700, 1000]
    wl = W.Workload(len(lens), 6, D, lens, fmt, 1.0, ("per_head", 3, 10.0), "permuted", seed=3)
    dw = DeviceWorkload(wl)
    dw.prefill()
    oc = _oracle_cache(wl, wl.lens)
    _device_cache_matches(dw, oc, wl.lens)
    q_np, out = _run_decode(dw)
    _check_decode(wl, wl.lens, q_np, out, oc)
    got = out.float().cpu().numpy()
    assert np.all(got[lens.index(0)] == 0)
    assert np.isfinite(got).all()


@pytest.mark.parametrize("fmt", [kvq.KVQ_INT4_B64, kvq.KVQ_INT8_PAGE, kvq.KVQ_FP8_E4M3])
def test_batch_context_does_not_change_results(cuda_ok, fmt):
    """The same (sequence, head) attended alone or inside a large batch (so cut
    into different splits and merged) agrees to fp32 rounding."""
    lens = [3000, 77, 4096, 1, 513, 2048, 9000, 64]
    wl = W.Workload(len(lens), 4, D, lens, fmt, 1.0, None, "permuted", seed=4)
    dw = DeviceWorkload(wl)
    dw.prefill()
    q_np, out_all = _run_decode(dw)
    for b in (0, 6):
        q1 = torch.from_numpy(q_np[b:b + 1].view(np.float16)).cuda()
        out1 = torch.empty_like(q1)
        kvq.kvq_decode_attention(dw.cache, q1, dw.block_table[b:b + 1], dw.lens[b:b + 1], dw.softmax_scale,
                                 out1, dw.workspace)
        a = out1.float().cpu().numpy()[0]
        c = out_all.float().cpu().numpy()[b]
        assert np.max(np.abs(a - c)) <= 2e-3 * max(1e-3, np.abs(c).max()), b
    _check_decode(wl, wl.lens, q_np, out_all)


@pytest.mark.parametrize("fmt", [kvq.KVQ_INT4_B64, kvq.KVQ_INT8_PAGE, kvq.KVQ_FP8_E4M3])
def test_more_sequences_than_one_launch(cuda_ok, fmt):
    """700 sequences: the entry point runs them as launches of at most 512
    (each with its own slice of q, out, lengths and block table).  Ragged
    lengths with empty sequences on both sides of the launch boundary; every
    (sequence, query head) against the oracle for multi-head attention and for
    groups of 4 (int4: the spare-column kernel) and 32 (the 16-head tiles and
    their merge launch)."""
    rng = np.random.default_rng(77)
    lens = rng.integers(1, 260, size=700).astype(np.int64)
    lens[[0, 300, 511, 512, 699]] = 0
    wl = W.Workload(len(lens), 2, D, lens.tolist(), fmt, 1.0, None, "permuted", seed=78)
    dw = DeviceWorkload(wl)
    dw.prefill()
    oc = _oracle_cache(wl, wl.lens)
    q_np, out = _run_decode(dw)
    _check_decode(wl, wl.lens, q_np, out, oc)
    got = out.float().cpu().numpy()
    assert np.all(got[[0, 300, 511, 512, 699]] == 0)
    kc, vc, ks, vs = oc
    sm = np.float32(1.0 / math.sqrt(D))
    for g in (4, 32):
        qg = (rng.standard_normal((wl.B, wl.H * g, D))).astype(np.float16).view(np.uint16)
        q = torch.from_numpy(qg.view(np.float16)).cuda()
        og = torch.full_like(q, float("nan"))
        kvq.kvq_decode_attention_gqa(dw.cache, q, dw.block_table, dw.lens, dw.softmax_scale, og,
                                     dw.cache.workspace(wl.H * g))
        torch.cuda.synchronize()
        ref = orc.decode_attention(wl.fmt, kc, vc, ks, vs, wl.block_table, wl.lens, qg, sm)
        vmax = np.repeat(orc.value_absmax(wl.fmt, vc, vs, wl.block_table, wl.lens, wl.H, D), g, axis=1)
        err = orc.normalized_error(og.float().cpu().numpy().astype(np.float64), ref, vmax)
        assert err <= TOL, f"g={g}: normalised error {err:.3e} > {TOL}"
    assert kvq.kvq_get_device_status(dw.cache) == (0, 0)


def test_special_queries(cuda_ok):
    """q = 0 gives the mean of the values; one sequence of one token returns
    that token's value row."""
    lens = [300, 1]
    wl = W.Workload(2, 2, D, lens, kvq.KVQ_INT4_B64, 1.0, None, "contiguous", seed=5)
    dw = DeviceWorkload(wl)
    dw.prefill()
    q_np = np.zeros((2, 2, D), np.uint16)
    q_np, out = _run_decode(dw, q_np)
    _check_decode(wl, wl.lens, q_np, out)


def test_bad_block_table_is_flagged_not_faulted(cuda_ok):
    lens = [200]
    wl = W.Workload(1, 2, D, lens, kvq.KVQ_INT4_B64, 1.0, None, "contiguous", seed=6)
    dw = DeviceWorkload(wl)
    dw.prefill()
    assert kvq.kvq_get_device_status(dw.cache) == (0, 0)
    dw.block_table[0, 2] = 10 ** 6
    _run_decode(dw)
    rc, flags = kvq.kvq_get_device_status(dw.cache)
    assert rc == 4 and flags & kvq.KVQ_FLAG_BAD_PAGE
    dw.block_table[0, 2] = 2
    dw.lens[0] = 10 ** 5
    _run_decode(dw)
    rc, flags = kvq.kvq_get_device_status(dw.cache)
    assert flags & kvq.KVQ_FLAG_BAD_LENGTH


def test_host_rejects_bad_arguments(cuda_ok):
    cache = kvq.PagedKVCache(kvq.KVQ_INT4_B64, 4, 2)
    q = torch.zeros((1, 2, D), dtype=torch.float16, device="cuda")
    bt = torch.zeros((1, 1), dtype=torch.int32, device="cuda")
    sl = torch.ones(1, dtype=torch.int32, device="cuda")
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(kvq.KvqError) as e:
        kvq.kvq_decode_attention(cache, q, bt, sl, 0.1, q.clone(), small)
    assert e.value.status == 6
    x = torch.zeros((64, 2, 64), dtype=torch.float16, device="cuda")
    with pytest.raises(kvq.KvqError) as e:
        kvq.kvq_quantize(kvq.KVQ_INT4_B64, x, torch.empty(8192, dtype=torch.uint8, device="cuda"),
                         torch.empty(4, dtype=torch.float32, device="cuda"))
    assert e.value.status == 2


@pytest.mark.parametrize("fmt", [kvq.KVQ_INT4_B64, kvq.KVQ_INT8_PAGE, kvq.KVQ_FP8_E4M3])
def test_one_head_split_over_the_whole_grid(cuda_ok, fmt):
    """One (sequence, head) long enough to be cut into about a thousand pieces:
    the warp that writes the last piece merges them all (more than one round of
    32 lanes).  The zero-filled workspace is reused without clearing (each call
    leaves its piece counters at zero); one that was not zero-filled is
    reported in the status word, and zero-filling it again recovers."""
    lens = [65536 + 17]
    wl = W.Workload(1, 1, D, lens, fmt, 1.0, None, "permuted", seed=8)
    dw = DeviceWorkload(wl)
    dw.prefill()
    q_np, out = _run_decode(dw)
    _check_decode(wl, wl.lens, q_np, out)
    _, out2 = _run_decode(dw, q_np)
    _, out3 = _run_decode(dw, q_np)
    assert torch.equal(out, out2) and torch.equal(out, out3)
    assert kvq.kvq_get_device_status(dw.cache) == (0, 0)
    dw.workspace.fill_(0x7F)
    _run_decode(dw, q_np)
    rc, flags = kvq.kvq_get_device_status(dw.cache)
    assert flags & kvq.KVQ_FLAG_BAD_WORKSPACE and rc == 6
    dw.workspace.zero_()
    _, out4 = _run_decode(dw, q_np)
    assert torch.equal(out, out4)
    assert kvq.kvq_get_device_status(dw.cache) == (0, 0)
