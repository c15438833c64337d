"""GPU parity of decode attention with grouped query heads (kvq_decode_attention_gqa)
against the binary64 oracle: q holds g query heads per cache head, query head i
reads cache head i // g (multi-query decode of MLA absorbed into MQA, "DeepSeek
R1 performance tips", ddd.cn section 2), and the normalised error of every
(sequence, query head) stays within 2e-3."""
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
SM = 1.0 / math.sqrt(D)


def _oracle_cache(wl, lens):
    rb = orc.row_bytes(wl.fmt, D)
    kc = np.zeros((wl.num_pages, wl.H, 64, rb), np.uint8)
    vc = np.zeros_like(kc)
    ks = np.zeros((wl.num_pages, wl.H), np.float32)
    vs = np.zeros_like(ks)
    for b in range(wl.B):
        if lens[b]:
            orc.quantize_into_pages(wl.fmt, wl.kv_host("k", b, 0, lens[b]), wl.block_table[b], kc, ks)
            orc.quantize_into_pages(wl.fmt, wl.kv_host("v", b, 0, lens[b]), wl.block_table[b], vc, vs)
    return kc, vc, ks, vs


def _queries(B, Hq, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((B, Hq, D)) * scale).astype(np.float16).view(np.uint16)


def _run(dw, q_bits, g, workspace=None):
    q = torch.from_numpy(q_bits.view(np.float16)).cuda()
    out = torch.full_like(q, float("nan"))
    ws = dw.cache.workspace(q.shape[1]) if workspace is None else workspace
    kvq.kvq_decode_attention_gqa(dw.cache, q, dw.block_table, dw.lens, dw.softmax_scale, out, ws)
    torch.cuda.synchronize()
    return out.float().cpu().numpy().astype(np.float64)


def _check(wl, lens, q_bits, got, g, oc=None):
    kc, vc, ks, vs = _oracle_cache(wl, lens) if oc is None else oc
    ref = orc.decode_attention(wl.fmt, kc, vc, ks, vs, wl.block_table, lens, q_bits, np.float32(SM))
    vmax = np.repeat(orc.value_absmax(wl.fmt, vc, vs, wl.block_table, lens, wl.H, D), g, axis=1)
    err = orc.normalized_error(got, ref, vmax)
    assert err <= TOL, f"normalised error {err:.3e} > {TOL}"
    return err


FMTS = {"int4": kvq.KVQ_INT4_B64, "int8": kvq.KVQ_INT8_PAGE, "fp8": kvq.KVQ_FP8_E4M3}
# (format, g): every g <= 8 uses a column kernel (int4: g = 2; 3, 4 on the
# 4-column one, whose columns past g carry zero queries; 5 .. 8 on the
# 8-column one; int8 / FP8: 2 .. 8 on their 8-column one); every larger g the
# 16-query-head tile kernel (20 and 24: a full and a partial tile, 32: two
# tiles, 48: three)
GROUPS = [("int4", 2), ("int4", 4), ("int4", 3), ("int4", 5), ("int4", 6), ("int4", 7), ("int4", 8), ("int4", 16),
          ("int4", 20), ("int4", 32), ("int4", 48), ("int8", 2), ("int8", 5), ("int8", 8), ("int8", 24), ("int8", 32),
          ("fp8", 3), ("fp8", 7),
          ("fp8", 4), ("fp8", 8), ("fp8", 16), ("fp8", 32)]


@pytest.mark.parametrize("fmt,g", GROUPS)
def test_grouped_heads_ragged_lengths(cuda_ok, fmt, g):
    """Lengths at every unit/page edge, an empty sequence, a permuted table,
    outlier channels; 3 cache heads x g query heads."""
    lens = [1, 15, 16, 17, 31, 32, 33, 63, 64, 65, 127, 128, 129, 0, 257, 700, 1000]
    wl = W.Workload(len(lens), 3, D, lens, FMTS[fmt], 1.0, ("per_head", 3, 10.0), "permuted", seed=31)
    dw = DeviceWorkload(wl)
    dw.prefill()
    q = _queries(wl.B, 3 * g, 32 + g)
    got = _run(dw, q, g)
    _check(wl, wl.lens, q, got, g)
    assert np.all(got[lens.index(0)] == 0)
    assert kvq.kvq_get_device_status(dw.cache) == (0, 0)


@pytest.mark.parametrize("fmt", ["int4", "int8", "fp8"])
@pytest.mark.parametrize("g", [32, 64])
def test_multi_query_one_cache_head(cuda_ok, fmt, g):
    """Multi-query decode (the pages' MLA decode absorbed into MQA): one cache
    head serves all g query heads; ragged lengths in a permuted table, long
    enough that every sequence is split over many warps."""
    lens = [9000, 1, 4100, 0, 333, 12000]
    wl = W.Workload(len(lens), 1, D, lens, FMTS[fmt], 1.0, ("per_head", 4, 10.0), "permuted", seed=40 + g)
    dw = DeviceWorkload(wl)
    dw.prefill()
    q = _queries(wl.B, g, 41 + g, scale=1.5)
    got = _run(dw, q, g)
    _check(wl, wl.lens, q, got, g)
    assert np.all(got[lens.index(0)] == 0)
    assert kvq.kvq_get_device_status(dw.cache) == (0, 0)


@pytest.mark.parametrize("fmt,g", [("int4", 2), ("int4", 4), ("int4", 8), ("int4", 32), ("int8", 32), ("fp8", 16)])
def test_grouped_heads_one_long_sequence_many_pieces(cuda_ok, fmt, g):
    """One cache head long enough to be cut into about a thousand split pieces:
    the merge combines them all (several rounds of 32 lanes); the workspace is
    reused without clearing and gives the same bits."""
    wl = W.Workload(1, 1, D, [65536 + 40], FMTS[fmt], 1.0, None, "permuted", seed=33)
    dw = DeviceWorkload(wl)
    dw.prefill()
    q = _queries(1, g, 34, scale=2.0)
    ws = dw.cache.workspace(g)
    got = _run(dw, q, g, ws)
    _check(wl, wl.lens, q, got, g)
    again = _run(dw, q, g, ws)
    assert np.array_equal(got, again)
    assert kvq.kvq_get_device_status(dw.cache) == (0, 0)


def test_group_of_one_is_multi_head_attention(cuda_ok):
    """kvq_decode_attention_gqa with as many query heads as cache heads is
    kvq_decode_attention, bit for bit."""
    wl = W.Workload(4, 4, D, [300, 77, 1, 4096], kvq.KVQ_INT4_B64, 1.0, None, "permuted", seed=35)
    dw = DeviceWorkload(wl)
    dw.prefill()
    q = torch.from_numpy(_queries(4, 4, 36).view(np.float16)).cuda()
    a = torch.empty_like(q)
    b = torch.empty_like(q)
    kvq.kvq_decode_attention(dw.cache, q, dw.block_table, dw.lens, dw.softmax_scale, a, dw.workspace)
    kvq.kvq_decode_attention_gqa(dw.cache, q, dw.block_table, dw.lens, dw.softmax_scale, b, dw.workspace)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_grouped_heads_share_the_cache_pass(cuda_ok):
    """Every query head of a group equals the same head attended alone through
    a multi-head call over a cache whose heads repeat the cache head (to the
    attention tolerance: the two paths order their fp32 sums differently)."""
    g = 4
    lens = [900, 64, 333]
    wl = W.Workload(3, 2, D, lens, kvq.KVQ_INT4_B64, 1.0, None, "permuted", seed=37)
    dw = DeviceWorkload(wl)
    dw.prefill()
    q = _queries(3, 2 * g, 38)
    got = _run(dw, q, g)
    cache2 = kvq.PagedKVCache(kvq.KVQ_INT4_B64, dw.cache.num_pages, 2 * g, max_seqs=3)
    idx = torch.arange(2 * g, device="cuda") // g
    for name in ("k_codes", "v_codes", "k_scales", "v_scales"):
        getattr(cache2, name).copy_(getattr(dw.cache, name)[:, idx])
    qt = torch.from_numpy(q.view(np.float16)).cuda()
    out2 = torch.empty_like(qt)
    kvq.kvq_decode_attention(cache2, qt, dw.block_table, dw.lens, dw.softmax_scale, out2, cache2.workspace())
    torch.cuda.synchronize()
    mha = out2.float().cpu().numpy().astype(np.float64)
    kc, vc, ks, vs = _oracle_cache(wl, wl.lens)
    vmax = np.repeat(orc.value_absmax(wl.fmt, vc, vs, wl.block_table, wl.lens, wl.H, D), g, axis=1)
    assert orc.normalized_error(got, mha, vmax) <= TOL


def test_grouped_heads_argument_checks(cuda_ok):
    cache4 = kvq.PagedKVCache(kvq.KVQ_INT4_B64, 4, 2)
    bt = torch.zeros((1, 1), dtype=torch.int32, device="cuda")
    sl = torch.ones(1, dtype=torch.int32, device="cuda")
    ws = torch.zeros(1 << 22, dtype=torch.uint8, device="cuda")
    q3 = torch.zeros((1, 3, D), dtype=torch.float16, device="cuda")
    with pytest.raises(kvq.KvqError) as e:   # not a multiple of the cache heads
        kvq.kvq_decode_attention_gqa(cache4, q3, bt, sl, 0.1, q3.clone(), ws)
    assert e.value.status == 1
    q_big = torch.zeros((1, 2 * 2048, D), dtype=torch.float16, device="cuda")
    with pytest.raises(kvq.KvqError) as e:   # g = 2048 is beyond the largest group
        kvq.kvq_decode_attention_gqa(cache4, q_big, bt, sl, 0.1, q_big.clone(), ws)
    assert e.value.status == 2
    w1 = kvq.kvq_decode_workspace_bytes_gqa(kvq.KVQ_INT4_B64, 8, 8)
    w4 = kvq.kvq_decode_workspace_bytes_gqa(kvq.KVQ_INT4_B64, 8, 32)
    assert w1 == kvq.kvq_decode_workspace_bytes(kvq.KVQ_INT4_B64, 8) and 3 * w1 < w4 < 4 * w1
    # tiles of 16 query heads: the partials hold 16 rows whatever the group
    w16 = kvq.kvq_decode_workspace_bytes_gqa(kvq.KVQ_INT8_PAGE, 8, 128)
    assert w16 > 0 and w16 == kvq.kvq_decode_workspace_bytes_gqa(kvq.KVQ_INT8_PAGE, 1, 32)
    # the 8-column kernels: 8 rows per partial for every g from 2 to 8 (int4: 5 to 8)
    w8 = kvq.kvq_decode_workspace_bytes_gqa(kvq.KVQ_INT8_PAGE, 8, 64)
    assert w8 > 0 and w8 == kvq.kvq_decode_workspace_bytes_gqa(kvq.KVQ_INT8_PAGE, 1, 2)
    assert kvq.kvq_decode_workspace_bytes_gqa(kvq.KVQ_INT4_B64, 1, 5) == kvq.kvq_decode_workspace_bytes_gqa(
        kvq.KVQ_INT4_B64, 2, 16)
    assert kvq.kvq_decode_workspace_bytes_gqa(kvq.KVQ_INT4_B64, 1, 2048) == 0


OFFSET_CASES = [("int4", 1), ("int4", 2), ("int4", 4), ("int4", 8), ("int4", 32), ("int8", 1), ("fp8", 1), ("fp8", 8)]


@pytest.mark.parametrize("fmt,g", OFFSET_CASES)
@pytest.mark.parametrize("qmean", [4.0, 12.0])
def test_query_with_a_large_common_offset(cuda_ok, fmt, g, qmean):
    """q ~ N(qmean, 1) on every element, over heads with outlier channels, so
    that the K scales of a head's pages differ and its softmax is peaked.  The
    int4 kernels take a share of every score that depends on q alone out after
    the contraction, scaled by each page's K scale: an error in that share does
    not cancel across pages, and this case makes it show."""
    lens = [1, 33, 64, 700, 3000, 8192, 20000, 5]
    wl = W.Workload(len(lens), 4, D, lens, FMTS[fmt], 1.0, ("per_head", 4, 10.0), "permuted", seed=8)
    dw = DeviceWorkload(wl)
    dw.prefill()
    rng = np.random.default_rng(80 + g)
    q = (rng.standard_normal((wl.B, 4 * g, D)) + qmean).astype(np.float16).view(np.uint16)
    got = _run(dw, q, g)
    _check(wl, wl.lens, q, got, g)
    assert kvq.kvq_get_device_status(dw.cache) == (0, 0)
