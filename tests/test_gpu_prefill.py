"""GPU parity of chunked-prefill attention (kvq_prefill_attention) against the
binary64 oracle: the chunk of each sequence attends causally over the
quantized paged cache that already holds it, and every (query, query head)
must stay within 2e-3 of the oracle, normalised by max|v^| of its (sequence,
cache head).  Chunked attention: "R1 performance overview"
(aicoding.csdn.net); paging: ddd.cn section 4."""
import math

import numpy as np
import pytest
import torch

from oracle import oracle as orc
from quantized_kv_cache_09_gb300 import kvq
from quantized_kv_cache_09_gb300.runner import DeviceWorkload
from quantized_kv_cache_09_gb300.synth import workloads as W
from quantized_kv_cache_09_gb300.synth import synth_sample_heads

pytestmark = pytest.mark.gpu
TOL = 2e-3
D = 128
SM = 1.0 / math.sqrt(D)


def _oracle_cache(wl):
    rb = orc.row_bytes(wl.fmt, D)
    kc = np.zeros((wl.num_pages, wl.H, 64, rb), np.uint8)
    vc = np.zeros_like(kc)
    ks = np.zeros((wl.num_pages, wl.H), np.float32)
    vs = np.zeros_like(ks)
    for b in range(wl.B):
        if wl.lens[b]:
            orc.quantize_into_pages(wl.fmt, wl.kv_host("k", b, 0, wl.lens[b]), wl.block_table[b], kc, ks)
            orc.quantize_into_pages(wl.fmt, wl.kv_host("v", b, 0, wl.lens[b]), wl.block_table[b], vc, vs)
    return kc, vc, ks, vs


def _counters_zero(ws):
    """The workspace opens with one uint32 count per split unit (padded to 256
    bytes), then 2 x 256 x 132 floats of partials per unit; the counts must be
    back at zero after a call."""
    per_unit = 2 * 256 * 132 * 4
    n = ws.numel()
    units = next(u for u in range(1, n // per_unit + 1) if -(-4 * u // 256) * 256 + u * per_unit == n)
    return not ws[:-(-4 * units // 256) * 256].any()


def _run(dw, chunks, q_bits, max_q=None, split=False):
    """split: with a workspace, so the units of the grid's last wave (here every
    unit: these grids are smaller than one wave) run as two key halves merged
    through it."""
    cu = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
    q = torch.from_numpy(q_bits.view(np.float16)).cuda()
    out = torch.full_like(q, float("nan"))
    mq = max(chunks) if max_q is None else max_q
    ws = kvq.prefill_workspace(q.shape[1], len(chunks), mq) if split else None
    kvq.kvq_prefill_attention(dw.cache, q, torch.from_numpy(cu).cuda(), mq, dw.block_table, dw.lens,
                              dw.softmax_scale, out, workspace=ws)
    torch.cuda.synchronize()
    if split:
        assert _counters_zero(ws)
    return cu, out.float().cpu().numpy().astype(np.float64)


def _check(wl, oc, cu, q_bits, got):
    kc, vc, ks, vs = oc
    ref = orc.prefill_attention(wl.fmt, kc, vc, ks, vs, wl.block_table, wl.lens, cu, q_bits, np.float32(SM))
    vmax = orc.value_absmax(wl.fmt, vc, vs, wl.block_table, wl.lens, wl.H, D)
    g = wl.Hq // wl.H
    worst = 0.0
    for b in range(wl.B):
        for r in range(cu[b], cu[b + 1]):
            for hq in range(wl.Hq):
                err = np.max(np.abs(got[r, hq] - ref[r, hq])) / vmax[b, hq // g]
                assert err <= TOL, (b, r - cu[b], hq, err)
                worst = max(worst, err)
    return worst


@pytest.mark.parametrize("split", [False, True])
@pytest.mark.parametrize("fmt", [kvq.KVQ_INT4_B64, kvq.KVQ_INT8_PAGE, kvq.KVQ_FP8_E4M3])
def test_prefill_ragged_chunks(cuda_ok, fmt, split):
    """Chunks of 1, 64, 65, 37, 130, 64, 200 and 300 tokens after histories of
    0 to 2000 tokens (query tiles and pages cut anywhere), and an empty chunk
    whose output rows do not exist."""
    hist = [0, 0, 0, 100, 63, 500, 1, 77, 2000]
    chunks = [1, 64, 65, 37, 130, 64, 200, 0, 300]
    lens = [h + n for h, n in zip(hist, chunks)]
    wl = W.Workload(len(lens), 4, D, lens, fmt, 1.0, ("per_head", 3, 10.0), "permuted", seed=61)
    dw = DeviceWorkload(wl)
    dw.prefill()
    oc = _oracle_cache(wl)
    q = (np.random.default_rng(62).standard_normal((sum(chunks), 4, D))).astype(np.float16).view(np.uint16)
    cu, got = _run(dw, chunks, q, split=split)
    assert np.isfinite(got).all()
    _check(wl, oc, cu, q, got)
    assert kvq.kvq_get_device_status(dw.cache) == (0, 0)


@pytest.mark.parametrize("split", [False, True])
def test_prefill_grouped_heads(cuda_ok, split):
    """8 query heads over 2 cache heads (g = 4): query head i reads cache head i // 4."""
    hist, chunks = [300, 0, 64], [100, 129, 64]
    lens = [h + n for h, n in zip(hist, chunks)]
    wl = W.Workload(3, 2, D, lens, kvq.KVQ_INT4_B64, 1.0, None, "permuted", seed=63, q_heads=8)
    dw = DeviceWorkload(wl)
    dw.prefill()
    q = (np.random.default_rng(64).standard_normal((sum(chunks), 8, D)) * 2).astype(np.float16).view(np.uint16)
    cu, got = _run(dw, chunks, q, split=split)
    _check(wl, _oracle_cache(wl), cu, q, got)


def test_prefill_bad_lengths_are_flagged(cuda_ok):
    """A chunk longer than its sequence, or than max_q_per_seq, is skipped and
    flagged; the other sequences are still computed."""
    lens = [100, 50]
    wl = W.Workload(2, 2, D, lens, kvq.KVQ_INT4_B64, 1.0, None, "contiguous", seed=65)
    dw = DeviceWorkload(wl)
    dw.prefill()
    chunks = [60, 70]  # the second chunk (70) is longer than its sequence (50)
    q = np.random.default_rng(66).standard_normal((130, 2, D)).astype(np.float16).view(np.uint16)
    cu, got = _run(dw, chunks, q)
    rc, flags = kvq.kvq_get_device_status(dw.cache)
    assert rc == 7 and flags & kvq.KVQ_FLAG_BAD_LENGTH
    assert np.isnan(got[60:]).all() and np.isfinite(got[:60]).all()
    with pytest.raises(kvq.KvqError) as e:
        kvq.kvq_prefill_attention(dw.cache, torch.zeros((4, 3, D), dtype=torch.float16, device="cuda"),
                                  torch.tensor([0, 4, 4], dtype=torch.int32, device="cuda"), 4, dw.block_table,
                                  dw.lens, SM, torch.zeros((4, 3, D), dtype=torch.float16, device="cuda"))
    assert e.value.status == 1   # 3 query heads over 2 cache heads
    small = torch.zeros(64, dtype=torch.uint8, device="cuda")
    q2 = torch.zeros((130, 2, D), dtype=torch.float16, device="cuda")
    with pytest.raises(kvq.KvqError) as e:
        kvq.kvq_prefill_attention(dw.cache, q2, torch.tensor([0, 60, 130], dtype=torch.int32, device="cuda"), 70,
                                  dw.block_table, dw.lens, SM, torch.zeros_like(q2), workspace=small)
    assert e.value.status == 6   # workspace too small


@pytest.mark.parametrize("split", [False, True])
def test_prefill_full_size_sampled(cuda_ok, split):
    """The chunked-prefill workload (B=8, H=32, the last 512 of 8192 tokens):
    sampled (sequence, query, head) outputs against the oracle, one query at a
    time over its causal prefix; with a workspace (as benchmarked) the grid's
    last wave runs as key halves."""
    wl = W.make_workload(8)
    dw = DeviceWorkload(wl)
    dw.prefill(max_tokens_per_call=1 << 16)
    n = wl.chunk
    q = torch.empty((wl.B * n, wl.Hq, D), dtype=torch.float16, device="cuda")
    for b in range(wl.B):
        wl.chunk_q_device(q[b * n:(b + 1) * n], b)
    out = torch.empty_like(q)
    cu = torch.arange(0, wl.B * n + 1, n, dtype=torch.int32, device="cuda")
    ws = kvq.prefill_workspace(wl.Hq, wl.B, n) if split else None
    kvq.kvq_prefill_attention(dw.cache, q, cu, n, dw.block_table, dw.lens, dw.softmax_scale, out, workspace=ws)
    torch.cuda.synchronize()
    assert kvq.kvq_get_device_status(dw.cache) == (0, 0)
    if split:
        assert _counters_zero(ws)
    got = out.float().cpu().numpy()
    rng = np.random.default_rng(67)
    for b, h in synth_sample_heads(wl.B, wl.H, 4, seed=5):
        L = int(wl.lens[b])
        k = np.ascontiguousarray(wl.kv_host("k", b, 0, L)[:, h:h + 1, :])
        v = np.ascontiguousarray(wl.kv_host("v", b, 0, L)[:, h:h + 1, :])
        kc, ks = orc.quantize(wl.fmt, k)
        vc, vs = orc.quantize(wl.fmt, v)
        bt = np.arange(kc.shape[0], dtype=np.int32)[None, :]
        vmax = orc.value_absmax(wl.fmt, vc, vs, bt, np.array([L]), 1, D)[0, 0]
        for i in sorted(set([0, 1, 63, 64, n - 1] + rng.integers(0, n, 4).tolist())):
            qi = wl.chunk_q_host(b, i, i + 1)[:, h:h + 1, :]
            ref = orc.decode_attention(wl.fmt, kc, vc, ks, vs, bt, np.array([L - n + i + 1]), qi, np.float32(SM))
            err = np.max(np.abs(got[b * n + i, h] - ref[0, 0])) / vmax
            assert err <= TOL, (b, h, i, err)


@pytest.mark.parametrize("split", [False, True])
@pytest.mark.parametrize("fmt", [kvq.KVQ_INT4_B64, kvq.KVQ_FP8_E4M3])
def test_prefill_zero_pages_and_negative_scale(cuda_ok, fmt, split):
    """A page whose keys and values are all zero (scales 0) inside the causal
    range, and a negative softmax scale: both as the oracle defines them."""
    H, L, n = 2, 200, 100
    rng = np.random.default_rng(71)
    k = rng.standard_normal((L, H, D)).astype(np.float16)
    v = rng.standard_normal((L, H, D)).astype(np.float16)
    k[64:128] = 0
    v[64:128] = 0
    k[150:160, 1] = 0  # a partly zero page too
    cache = kvq.PagedKVCache(fmt, 4, H, max_seqs=1)
    bt = torch.tensor([[2, 0, 3, 1]], dtype=torch.int32, device="cuda")
    kvq.kvq_append(cache, torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(),
                   torch.tensor([0, L], dtype=torch.int32, device="cuda"), bt,
                   torch.zeros(1, dtype=torch.int32, device="cuda"), L)
    lens = torch.tensor([L], dtype=torch.int32, device="cuda")
    q = (rng.standard_normal((n, H, D)) * 3).astype(np.float16)
    cu = np.array([0, n], dtype=np.int32)
    rb = orc.row_bytes(fmt, D)
    kc = np.zeros((4, H, 64, rb), np.uint8)
    vc = np.zeros_like(kc)
    ks = np.zeros((4, H), np.float32)
    vs = np.zeros_like(ks)
    bt_np = bt.cpu().numpy()
    orc.quantize_into_pages(fmt, k.view(np.uint16), bt_np[0], kc, ks)
    orc.quantize_into_pages(fmt, v.view(np.uint16), bt_np[0], vc, vs)
    assert np.array_equal(cache.k_codes.cpu().numpy(), kc) and np.array_equal(cache.v_codes.cpu().numpy(), vc)
    vmax = orc.value_absmax(fmt, vc, vs, bt_np, np.array([L]), H, D)
    for sm_scale in (SM, -0.05):
        out = torch.full((n, H, D), float("nan"), dtype=torch.float16, device="cuda")
        ws = kvq.prefill_workspace(H, 1, n) if split else None
        kvq.kvq_prefill_attention(cache, torch.from_numpy(q).cuda(), torch.from_numpy(cu).cuda(), n, bt, lens,
                                  sm_scale, out, workspace=ws)
        torch.cuda.synchronize()
        assert kvq.kvq_get_device_status(cache) == (0, 0)
        ref = orc.prefill_attention(fmt, kc, vc, ks, vs, bt_np, np.array([L]), cu, q.view(np.uint16),
                                    np.float32(sm_scale))
        got = out.float().cpu().numpy().astype(np.float64)
        err = orc.normalized_error(got, ref, np.repeat(vmax, n, axis=0))
        assert err <= TOL, (sm_scale, err)
