"""Host logic of the benchmark that needs no GPU: the lookup that ties a
committed DRAM-traffic figure to the kernel sources it was captured on, and
the summary of the nvidia-smi clock samples taken during the timed region
(median SM clock, throttle reasons, samples outside the window ignored)."""
import os
import shutil
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _tree(tmp_path):
    """A copy of the kernel sources and an empty profiles folder, so that the
    lookup can be exercised without touching the committed files."""
    src = os.path.join(ROOT, "quantized_kv_cache_09_gb300", "csrc")
    dst = tmp_path / "quantized_kv_cache_09_gb300" / "csrc"
    dst.mkdir(parents=True)
    for files in bench.KERNEL_SOURCES.values():
        for f in files:
            shutil.copy(os.path.join(src, f), dst / f)
    (tmp_path / "profiles").mkdir()
    return tmp_path


def test_traffic_is_reported_only_for_the_sources_it_was_captured_on(tmp_path, monkeypatch):
    root = _tree(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(root))
    d_dec = bench.source_digest("decode_split_kernel")
    d_pre = bench.source_digest("prefill_attn_tc_kernel")
    assert d_dec != d_pre and len(d_dec) == 16
    (root / "profiles" / "ncu_traffic.txt").write_text(
        "# header line with kernel=decode_split_kernel workload=x dram_bytes_per_launch=1 source_sha256=" + d_dec + "\n"
        "kernel=decode_split_kernel workload=a dram_bytes_per_launch=123 source_sha256=" + d_dec + "\n"
        "kernel=decode_split_kernel workload=b dram_bytes_per_launch=456 source_sha256=0000000000000000\n"
        "kernel=prefill_attn_tc_kernel workload=a dram_bytes_per_launch=789 source_sha256=" + d_pre + "\n"
        "\n")
    assert bench.ncu_traffic("decode_split_kernel", "a") == 123.0
    assert bench.ncu_traffic("prefill_attn_tc_kernel", "a") == 789.0
    assert bench.ncu_traffic("decode_split_kernel", "b") is None      # other sources
    assert bench.ncu_traffic("decode_split_kernel", "x") is None      # comment lines are not data
    assert bench.ncu_traffic("append_kernel", "a") is None            # no line for the kernel
    # any change to a source the kernel is built from (a comment too) retires its figure,
    # and leaves the figures of kernels built from other sources alone
    p = root / "quantized_kv_cache_09_gb300" / "csrc" / "kvq_decode.cu"
    p.write_bytes(p.read_bytes() + b"\n// changed\n")
    assert bench.ncu_traffic("decode_split_kernel", "a") is None
    assert bench.ncu_traffic("prefill_attn_tc_kernel", "a") == 789.0
    # a shared header retires every kernel built from it
    h = root / "quantized_kv_cache_09_gb300" / "csrc" / "kvq_internal.h"
    h.write_bytes(h.read_bytes() + b"\n")
    assert bench.ncu_traffic("prefill_attn_tc_kernel", "a") is None


def test_traffic_without_a_summary_file(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(_tree(tmp_path)))
    assert bench.ncu_traffic("decode_split_kernel", "long-context") is None


def test_every_kernel_is_hashed_over_existing_sources():
    for kernel in bench.KERNEL_SOURCES:
        assert len(bench.source_digest(kernel)) == 16


def _row(mhz, mx=2070, hw="Not Active", hwt="Not Active", swt="Not Active", cap="Not Active"):
    return [str(mhz), str(mx), "900.0", hw, hwt, swt, cap]


def test_clock_summary_reads_the_window_only():
    s = bench.ClockSampler(0)
    s.samples = [(0.5, _row(1000, hw="Active")),    # before the window: ignored
                 (1.0, _row(2070)), (1.5, _row(2055)), (2.0, _row(2070, cap="Active")),
                 (3.5, _row(300, hwt="Active"))]    # after the window: ignored
    s.window = (1.0, 2.0)
    r = s.summary()
    assert r["sm_mhz"] == 2070.0 and r["sm_max_mhz"] == 2070.0
    assert r["reasons"] == ["sw_power_cap"]
    assert r["samples"] == 3 and r["samples_in_window"] == 3


def test_clock_summary_reasons_and_unparsable_rows():
    s = bench.ClockSampler(0)
    s.samples = [(1.0, _row(1980, hw="Active")), (1.1, ["[N/A]", "2070", "", "", "", "", ""]),
                 (1.2, _row(1990, swt="Active")), (1.3, _row(2000, hwt="Active"))]
    s.window = (0.0, 5.0)
    r = s.summary()
    assert r["sm_mhz"] == 1990.0
    assert r["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"]


def test_clock_summary_without_samples_in_the_window_uses_all_and_says_so():
    s = bench.ClockSampler(0)
    s.samples = [(10.0, _row(2070))]
    s.window = (0.0, 1.0)
    r = s.summary()
    assert r["sm_mhz"] == 2070.0 and r["samples"] == 1 and r["samples_in_window"] == 0
    s.samples = []
    assert bench.ClockSampler(0).summary()["sm_mhz"] is None
