"""The seeded synthetic-input generator, host build (CPU only): binary16
rounding, distribution, determinism, sub-range consistency and the workload
recipes (outlier channels, permuted block tables, length ranges)."""
import numpy as np

from quantized_kv_cache_09_gb300 import synth
from quantized_kv_cache_09_gb300.synth import workloads as W


def test_f32_to_f16_matches_numpy_rounding():
    rng = np.random.default_rng(0)
    bits = rng.integers(0, 2 ** 32, 20000, dtype=np.uint64).astype(np.uint32)
    vals = bits.view(np.float32)
    vals = vals[np.isfinite(vals)]
    edge = np.array([0.0, -0.0, 65504.0, 65519.99, 65520.0, 2.0 ** -24, 2.0 ** -25, 2.0 ** -25 * 1.0001,
                     2.0 ** -14, 2.0 ** -14 * (1 - 2 ** -12), 1.0 + 2 ** -11, 1.0 + 3 * 2 ** -11, -7.5,
                     1e-9, 3e-8, 6e-8, 1e5], dtype=np.float32)
    for v in np.concatenate([vals[:4000], edge, (rng.standard_normal(4000) * 4).astype(np.float32)]):
        with np.errstate(over="ignore"):  # values past the fp16 range round to infinity: part of what is checked
            want = np.array([v], dtype=np.float32).astype(np.float16).view(np.uint16)[0]
        assert synth.f32_to_f16_bits(v) == want, v


def test_normal_moments_and_bounds():
    x = synth.fill_f16_host(1 << 20, 7, synth.stream_id(synth.K_HIST, 0), 0, 1.5).view(np.float16)
    x = x.astype(np.float64)
    assert abs(x.mean()) < 0.01
    assert abs(x.std() - 1.5) < 0.01
    assert np.abs(x).max() <= 6 * 1.5 + 1e-3
    # roughly normal tails: ~0.27% beyond 3 sigma (Irwin-Hall(12) is slightly lighter)
    frac = np.mean(np.abs(x) > 3 * 1.5)
    assert 0.0015 < frac < 0.0035


def test_subrange_and_determinism():
    s = synth.stream_id(synth.V_HIST, 3)
    full = synth.fill_f16_host(5000, 1, s, 0, 1.0)
    part = synth.fill_f16_host(1000, 1, s, 1234, 1.0)
    assert np.array_equal(full[1234:2234], part)
    assert np.array_equal(full, synth.fill_f16_host(5000, 1, s, 0, 1.0))
    assert not np.array_equal(full, synth.fill_f16_host(5000, 2, s, 0, 1.0))
    assert not np.array_equal(full, synth.fill_f16_host(5000, 1, s + 1, 0, 1.0))


def test_outlier_masks():
    m = synth.outliers_per_head(32, 128, 4, 0, synth.stream_id(synth.K_OUTLIER))
    assert m.shape == (32, 128) and np.all(m.sum(axis=1) == 4)
    m2 = synth.outliers_per_head(32, 128, 4, 0, synth.stream_id(synth.V_OUTLIER))
    assert not np.array_equal(m, m2)
    b = synth.outliers_bernoulli(32, 128, 0.01, 0, synth.stream_id(synth.K_OUTLIER))
    assert 10 <= b.sum() <= 80


def test_outliers_scale_the_marked_channels():
    wl = W.make_workload(2)
    x = wl.kv_host("k", 0, 0, 64).view(np.float16).astype(np.float64)   # [64][32][128]
    sd = x.std(axis=0)
    assert np.all(sd[wl.k_mask == 1] > 5) and np.all(sd[wl.k_mask == 0] < 2)


def test_workload_recipes():
    wl4 = W.make_workload(4)
    assert wl4.lens.min() >= 512 and wl4.lens.max() <= 16384
    assert sorted(wl4.block_table.reshape(-1).tolist()) == list(range(wl4.num_pages))
    wl2 = W.make_workload(2, extra_tokens=64)
    assert wl2.max_blocks == 129
    assert np.array_equal(wl2.block_table.reshape(-1), np.arange(wl2.num_pages))
    # the decode working set of the 7B-layer shape (int4): 2 * 8*32*8192 * 64 B codes + scales + q/out
    assert wl2.decode_bytes() == 268435456 + 262144 + 131072
    wl5 = W.make_workload(5)
    assert wl5.quantize_bytes(4096) * 64 == 4294967296 + 1073741824 + 1048576
    # the same token of a history is the same value whichever range it is generated in
    a = wl2.kv_host("v", 5, 100, 103)
    b = wl2.kv_host("v", 5, 101, 102)
    assert np.array_equal(a[1], b[0])
