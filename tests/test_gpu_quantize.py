"""GPU parity of the fused quantize kernel (kvq_quantize, kvq_append) against
the CPU oracle: codes and scales must be bit-exact.  Definition: quantize_block
(jsqmd.com/news/887038 section 2.1), the per-chunk INT8 variant
(aicoding.csdn.net section 2.2) and FP8 E4M3 with the scale set by max|x|
(jsqmd.com/news/887038 section 2.2)."""
import numpy as np
import pytest
import torch

from oracle import oracle as orc
from quantized_kv_cache_09_gb300 import kvq
from quantized_kv_cache_09_gb300.synth import workloads as W

pytestmark = pytest.mark.gpu
FMTS = [kvq.KVQ_INT4_B64, kvq.KVQ_INT8_PAGE, kvq.KVQ_FP8_E4M3]
D = 128


def _gpu_quantize(fmt, x_bits):
    T, H, _ = x_bits.shape
    nb = (T + 63) // 64
    rb = 64 if fmt == kvq.KVQ_INT4_B64 else 128
    x = torch.from_numpy(x_bits.view(np.float16)).cuda()
    codes = torch.full((nb, H, 64, rb), 0xA5, dtype=torch.uint8, device="cuda")  # poison
    scales = torch.full((nb, H), -1.0, dtype=torch.float32, device="cuda")
    kvq.kvq_quantize(fmt, x, codes, scales)
    torch.cuda.synchronize()
    return codes.cpu().numpy(), scales.cpu().numpy()


def _assert_same(fmt, x_bits):
    gc, gs = _gpu_quantize(fmt, x_bits)
    oc, os_ = orc.quantize(fmt, x_bits)
    assert np.array_equal(gs.view(np.uint32), os_.view(np.uint32)), "scales differ"
    if not np.array_equal(gc, oc):
        bad = np.argwhere(gc != oc)
        raise AssertionError(f"{len(bad)} code bytes differ, first at {bad[0].tolist()}")


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("T", [1, 63, 64, 65, 64 * 3 + 17])
def test_random_tensors_bit_exact(cuda_ok, fmt, T):
    rng = np.random.default_rng(T + 100 * fmt)
    x = rng.standard_normal((T, 5, D)) * rng.uniform(0.01, 20.0)
    x[rng.random(x.shape) < 0.01] *= 10
    _assert_same(fmt, x.astype(np.float16).view(np.uint16))


@pytest.mark.parametrize("fmt", FMTS[:2])
def test_exact_rounding_ties_bit_exact(cuda_ok, fmt):
    """Blocks whose quotients are exact half-integers (x = k/2 with max|x| = 7.5
    or 127, scale = 1): every tie must round to even, as the oracle does."""
    rng = np.random.default_rng(5)
    top = 7.5 if fmt == kvq.KVQ_INT4_B64 else 127.0
    x = rng.integers(-int(2 * top), int(2 * top) + 1, (64 * 6, 3, D)).astype(np.float64) / 2
    x[::64, :, 0] = top
    _assert_same(fmt, x.astype(np.float16).view(np.uint16))


@pytest.mark.parametrize("fmt", FMTS[:2])
def test_values_nearest_the_ties_of_random_scales_bit_exact(cuda_ok, fmt):
    """Whole blocks take the quantizer's unchecked fast path when no binary16
    value can lie within its error window of a half-integer quotient t.  Each
    block here holds +-a and, for every half-integer t below the largest code,
    the binary16 value nearest t * scale and its two neighbours, both signs,
    for 4096 random scales: the values the block test must find, wherever the
    scale puts them."""
    rng = np.random.default_rng(23 + fmt)
    n = 4096
    div = np.float32(7.5 if fmt == kvq.KVQ_INT4_B64 else 127.0)
    ts = np.arange(7 if fmt == kvq.KVQ_INT4_B64 else 127, dtype=np.float32) + np.float32(0.5)
    a = np.exp(rng.uniform(np.log(1e-3), np.log(6e4), n)).astype(np.float16)
    a = a[np.isfinite(a) & (a > 0)]
    x = np.zeros((64 * a.size, 1, D), dtype=np.float16)
    for i, ai in enumerate(a):
        s = np.float32(ai) / div
        v = (ts * s).astype(np.float16)
        cand = np.concatenate([v, np.nextafter(v, np.float16(np.inf)), np.nextafter(v, np.float16(0))])
        cand = cand[np.abs(cand.astype(np.float32)) <= np.float32(ai)]
        vals = np.concatenate([[ai, -ai], cand, -cand])
        blk = x[64 * i:64 * i + 64, 0, :].reshape(-1)
        blk[:vals.size] = vals
        fill = np.clip(rng.standard_normal(blk.size - vals.size) * 0.3, -0.9, 0.9) * np.float32(ai)
        blk[vals.size:] = fill.astype(np.float16)
        x[64 * i:64 * i + 64, 0, :] = blk.reshape(64, D)
    _assert_same(fmt, x.view(np.uint16))


def test_fp8_grid_midpoints_and_signed_zeros_bit_exact(cuda_ok):
    """Blocks with max|x| = 448 (scale 1) whose elements are E4M3 values, the
    midpoints between neighbours (ties to even), one binary16 step either side
    of them, -0.0 and negatives that round to zero (code 0x80), under other
    scales too (max|x| = 448 * 2^k, still exact quotients)."""
    vals = np.array([orc.e4m3_to_float(c) for c in range(127)])
    mids = (vals[:-1] + vals[1:]) / 2
    pool = np.concatenate([vals, mids]).astype(np.float16)
    pool = np.concatenate([pool, np.nextafter(pool, np.float16(np.inf)), np.nextafter(pool, np.float16(-np.inf))])
    pool = pool[np.isfinite(pool) & (np.abs(pool) <= 448)]
    rng = np.random.default_rng(9)
    x = rng.choice(pool, (64 * 8, 3, D)) * rng.choice([-1.0, 1.0], (64 * 8, 3, D))
    x[::64, :, 0] = 448.0
    x[1::64, :, :4] = [-0.0, -2.0 ** -11, -2.0 ** -12, 2.0 ** -11]
    for k, blk in enumerate(range(4, 8)):   # scales 2^-3 .. 2^0 times larger quotients stay exact
        x[64 * blk:64 * blk + 64] *= 2.0 ** (-k - 1)
    _assert_same(kvq.KVQ_FP8_E4M3, x.astype(np.float16).view(np.uint16))


def test_fp8_values_nearest_the_midpoints_of_random_scales_bit_exact(cuda_ok):
    """The FP8 fast path brackets RN(x / scale) between y' (1 -+ 2^-21) and
    keeps the code when both ends convert alike.  Each block here holds +-a
    and, for every midpoint m of the E4M3 grid below 448, the binary16 value
    nearest m * scale and its two neighbours, both signs, for 2048 random
    absmax values a (scale = a / 448 inexact): the elements whose groups the
    check must send to the exact division."""
    rng = np.random.default_rng(31)
    vals = np.array([orc.e4m3_to_float(c) for c in range(127)])
    mids = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)
    a = np.exp(rng.uniform(np.log(1e-3), np.log(6e4), 2048)).astype(np.float16)
    a = a[np.isfinite(a) & (a > 0)]
    x = np.zeros((64 * a.size, 1, D), dtype=np.float16)
    for i, ai in enumerate(a):
        s = np.float32(ai) / np.float32(448.0)
        v = (mids * s).astype(np.float16)
        cand = np.concatenate([v, np.nextafter(v, np.float16(np.inf)), np.nextafter(v, np.float16(0))])
        cand = cand[np.isfinite(cand) & (np.abs(cand.astype(np.float32)) <= np.float32(ai))]
        vals_blk = np.concatenate([[ai, -ai], cand, -cand])[:64 * D]
        blk = x[64 * i:64 * i + 64, 0, :].reshape(-1)
        blk[:vals_blk.size] = vals_blk
        fill = np.clip(rng.standard_normal(blk.size - vals_blk.size) * 0.3, -0.9, 0.9) * np.float32(ai)
        blk[vals_blk.size:] = fill.astype(np.float16)
        x[64 * i:64 * i + 64, 0, :] = blk.reshape(64, D)
    _assert_same(kvq.KVQ_FP8_E4M3, x.view(np.uint16))


@pytest.mark.parametrize("fmt", FMTS)
def test_every_fp16_absmax_bit_exact(cuda_ok, fmt):
    """One block per positive finite fp16 magnitude a, row 0 = (a, -a, a/3, ...):
    scale and the codes of +-a (where the binary32 quotient decides between -8
    and -7 for int4) match the oracle for all 31743 magnitudes."""
    mags = np.arange(1, 0x7C00, dtype=np.uint16)
    n = mags.size
    x = np.zeros((64 * n, 1, D), dtype=np.uint16)
    x[0::64, 0, 0] = mags
    x[0::64, 0, 1] = mags | 0x8000
    af = mags.view(np.float16).astype(np.float32)
    for k, frac in enumerate([1 / 3, -0.5, 0.2, -0.7333, 1 / 15, 0.4667]):
        x[0::64, 0, 2 + k] = (af * np.float32(frac)).astype(np.float16).view(np.uint16)
    _assert_same(fmt, x)


@pytest.mark.parametrize("fmt", FMTS)
def test_zero_and_tiny_blocks(cuda_ok, fmt):
    x = np.zeros((64 * 3, 2, D), dtype=np.float16)
    x[64:128, 1, 5] = np.float16(6e-8)       # smallest subnormal
    x[128:, 0, :] = np.float16(-3e-5)
    _assert_same(fmt, x.view(np.uint16))


def test_llama_layer_sequence_bit_exact(cuda_ok):
    """One full sequence of the 7B-layer workload (8192 tokens x 32 heads, 4 x10
    outlier channels per head), generated on the device and quantized there;
    the oracle regenerates the same bits on the host."""
    wl = W.make_workload(2)
    x = torch.empty((8192, 32, D), dtype=torch.float16, device="cuda")
    wl.kv_device("k", 3, 0, 8192, x)
    codes = torch.empty((128, 32, 64, 64), dtype=torch.uint8, device="cuda")
    scales = torch.empty((128, 32), dtype=torch.float32, device="cuda")
    kvq.kvq_quantize(kvq.KVQ_INT4_B64, x, codes, scales)
    oc, os_ = orc.quantize(orc.INT4, wl.kv_host("k", 3, 0, 8192))
    assert np.array_equal(scales.cpu().numpy().view(np.uint32), os_.view(np.uint32))
    assert np.array_equal(codes.cpu().numpy(), oc)


@pytest.mark.parametrize("fmt", FMTS)
def test_append_chunkings_equal_full_history(cuda_ok, fmt):
    """Any sequence of appends (ragged chunks, single tokens, whole blocks,
    block-crossing chunks) leaves the paged cache byte-identical to the oracle's
    quantize_block of each sequence's full history."""
    H = 3
    B = 3
    chunks = [[37, 1, 64, 100, 1, 27, 65, 129],   # ends at 424
              [64, 64, 1, 63, 200],                # 392
              [1] * 70 + [5]]                      # 75
    lens = [sum(c) for c in chunks]
    maxb = max((L + 63) // 64 for L in lens)
    wl = W.Workload(B, H, D, lens, fmt, 1.3, None, "permuted", seed=9)
    bt = torch.from_numpy(wl.block_table.copy()).cuda()
    cache = kvq.PagedKVCache(fmt, wl.num_pages, H, max_seqs=B)
    done = [0] * B
    step = 0
    while any(step < len(c) for c in chunks):
        adds = [c[step] if step < len(c) else 0 for c in chunks]
        cu = np.concatenate([[0], np.cumsum(adds)]).astype(np.int32)
        k = np.concatenate([wl.kv_host("k", b, done[b], done[b] + adds[b]) for b in range(B)])
        v = np.concatenate([wl.kv_host("v", b, done[b], done[b] + adds[b]) for b in range(B)])
        kvq.kvq_append(cache, torch.from_numpy(k.view(np.float16)).cuda(),
                       torch.from_numpy(v.view(np.float16)).cuda(), torch.from_numpy(cu).cuda(), bt,
                       torch.tensor(done, dtype=torch.int32, device="cuda"), max(adds))
        done = [done[b] + adds[b] for b in range(B)]
        step += 1
    rc, flags = kvq.kvq_get_device_status(cache)
    assert rc == 0 and flags == 0
    ko = np.zeros_like(cache.k_codes.cpu().numpy())
    vo = np.zeros_like(ko)
    kso = np.zeros((wl.num_pages, H), np.float32)
    vso = np.zeros_like(kso)
    for b in range(B):
        orc.quantize_into_pages(fmt, wl.kv_host("k", b, 0, lens[b]), wl.block_table[b], ko, kso)
        orc.quantize_into_pages(fmt, wl.kv_host("v", b, 0, lens[b]), wl.block_table[b], vo, vso)
    used = np.unique(np.concatenate([wl.block_table[b, :(lens[b] + 63) // 64] for b in range(B)]))
    assert np.array_equal(cache.k_scales.cpu().numpy()[used].view(np.uint32), kso[used].view(np.uint32))
    assert np.array_equal(cache.v_scales.cpu().numpy()[used].view(np.uint32), vso[used].view(np.uint32))
    assert np.array_equal(cache.k_codes.cpu().numpy()[used], ko[used])
    assert np.array_equal(cache.v_codes.cpu().numpy()[used], vo[used])
    # the tail buffers hold the originals of each open block
    for b in range(B):
        r = lens[b] % 64
        if r:
            want = wl.kv_host("k", b, lens[b] - r, lens[b]).transpose(1, 0, 2)
            got = cache.k_tail[b, :, :r].cpu().numpy().view(np.uint16)
            assert np.array_equal(got, want)


@pytest.mark.parametrize("n", [10, 100])
def test_append_reports_device_problems(cuda_ok, n):
    """A block-table entry out of range, a length beyond the table, an open
    block without a tail buffer: flagged in the status word, nothing faults.
    n = 10 takes the short-append kernel, n = 100 the persistent one."""
    fmt = kvq.KVQ_INT4_B64
    cache = kvq.PagedKVCache(fmt, 4, 2, max_seqs=0, with_tail=False)
    k = torch.zeros((n, 2, D), dtype=torch.float16, device="cuda")
    cu = torch.tensor([0, n], dtype=torch.int32, device="cuda")
    bt = torch.tensor([[7, 1]], dtype=torch.int32, device="cuda")
    kvq.kvq_append(cache, k, k, cu, bt, torch.tensor([0], dtype=torch.int32, device="cuda"), n)
    assert kvq.kvq_get_device_status(cache)[0] == 4
    kvq.kvq_append(cache, k, k, cu, bt, torch.tensor([120], dtype=torch.int32, device="cuda"), n)
    assert kvq.kvq_get_device_status(cache)[0] == 7
    bt2 = torch.tensor([[0, 1]], dtype=torch.int32, device="cuda")
    kvq.kvq_append(cache, k, k, cu, bt2, torch.tensor([5], dtype=torch.int32, device="cuda"), n)
    rc, flags = kvq.kvq_get_device_status(cache)
    assert flags & kvq.KVQ_FLAG_NO_TAIL
    assert kvq.kvq_get_device_status(cache) == (0, 0)   # the word was cleared


@pytest.mark.parametrize("fmt", FMTS)
def test_single_token_appends_keep_or_raise_scale(cuda_ok, fmt):
    """Decode-style appends, one token per sequence per call, through two whole
    blocks: tokens that raise the block's max|x|, tie it exactly, or stay below
    it (where only the new row's codes change).  After every call the open
    block's codes and scale equal the oracle's quantize_block of the history."""
    H, B, steps = 4, 3, 130
    rng = np.random.default_rng(17 + fmt)
    hist = rng.standard_normal((B, steps, H, D)) * np.array([0.5, 2.0, 8.0])[:, None, None, None]
    # sequence 0: magnitudes grow every token (the scale moves every call);
    # sequence 1: token 5 sets a max that tokens 9, 20 and 40 repeat exactly
    hist[0] *= np.linspace(0.1, 3.0, steps)[:, None, None]
    hist[1, 5, :, 7] = 30.0
    for t in (9, 20, 40):
        hist[1, t, :, 3] = -30.0
    bits = hist.astype(np.float16).view(np.uint16)
    wl = W.Workload(B, H, D, [steps] * B, fmt, 1.0, None, "permuted", seed=21)
    bt = torch.from_numpy(wl.block_table.copy()).cuda()
    cache = kvq.PagedKVCache(fmt, wl.num_pages, H, max_seqs=B)
    cu = torch.arange(B + 1, dtype=torch.int32, device="cuda")
    for t in range(steps):
        k = torch.from_numpy(np.ascontiguousarray(bits[:, t]).view(np.float16)).cuda()
        v = torch.from_numpy(np.ascontiguousarray(bits[:, t, :, ::-1]).view(np.float16)).cuda()
        before = torch.full((B,), t, dtype=torch.int32, device="cuda")
        kvq.kvq_append(cache, k, v, cu, bt, before, 1)
        if t % 13 != 12 and t != steps - 1:
            continue
        L = t + 1
        torch.cuda.synchronize()
        for b in range(B):
            pages = wl.block_table[b, :(L + 63) // 64]
            kc = np.zeros_like(cache.k_codes.cpu().numpy())
            ks = np.zeros((wl.num_pages, H), np.float32)
            orc.quantize_into_pages(fmt, np.ascontiguousarray(bits[b, :L]), wl.block_table[b], kc, ks)
            vc = np.zeros_like(kc)
            vs = np.zeros_like(ks)
            orc.quantize_into_pages(fmt, np.ascontiguousarray(bits[b, :L, :, ::-1]), wl.block_table[b], vc, vs)
            assert np.array_equal(cache.k_scales.cpu().numpy()[pages].view(np.uint32), ks[pages].view(np.uint32)), (t, b)
            assert np.array_equal(cache.v_scales.cpu().numpy()[pages].view(np.uint32), vs[pages].view(np.uint32)), (t, b)
            assert np.array_equal(cache.k_codes.cpu().numpy()[pages], kc[pages]), (t, b)
            assert np.array_equal(cache.v_codes.cpu().numpy()[pages], vc[pages]), (t, b)
    assert kvq.kvq_get_device_status(cache) == (0, 0)
