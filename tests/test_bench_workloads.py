"""Host logic of the benchmark's workload table (no GPU): every workload has a
config, the stateless-codec workloads carry the codec they name, and their
algorithmic bytes are the per-element figures of the codec -- fp16 read (2 B)
plus the code written (0.5 B int4, 1 B int8 / FP8) per element, and one fp32
scale per (64-token block, head) -- for K and V."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_every_workload_has_a_config():
    for name, (kind, _) in bench.WORKLOADS.items():
        cfg = bench.workload_config(name)
        assert cfg["workload"] == name
        assert kind in ("decode", "append", "prefill", "quantize")


def test_quantize_workloads_bytes_per_element():
    per_elem = {"int4-b64": 2.5, "int8-page": 3.0, "fp8-e4m3-page": 3.0}
    seen = set()
    for name, (kind, _) in bench.WORKLOADS.items():
        if kind != "quantize":
            continue
        cfg = bench.workload_config(name)
        wl = bench._make(name, 0)
        L = int(wl.lens[0])
        assert (wl.lens == L).all() and L % 64 == 0  # whole blocks, sequences back to back
        elems = 2 * wl.B * L * wl.H * wl.D  # K and V
        scales = 2 * wl.B * (L // 64) * wl.H * 4
        assert wl.quantize_bytes(L) * wl.B == per_elem[cfg["format"]] * elems + scales
        seen.add((cfg["format"], cfg["tokens"]))
    # the 7B layer's history in all three codecs and the long-context history in int4
    assert seen == {("int4-b64", 65536), ("int8-page", 65536), ("fp8-e4m3-page", 65536), ("int4-b64", 524288)}


def test_reference_arm_of_a_quantize_workload():
    rate, cores, desc, unit = bench.oracle_rate("quantize-7b-layer-int8", 0.3, 0)
    assert unit == "GB/s" and rate > 0 and cores >= 1
    assert "int8" in desc and "quantize-7b-layer-int8" in desc


def test_decode_workloads_bytes_per_unit():
    """The decode rooflines' numerator: 128 B per token-head for int4 (64 B of K
    codes and 64 of V) and 256 B for int8 / FP8, 8 B per (page, cache head) for
    its two scales, and 256 B each for a query row read and an output row
    written -- per decode call over the lengths the benchmark decodes at."""
    per_tok = {"int4-b64": 128, "int8-page": 256, "fp8-e4m3-page": 256}
    for name, (kind, _) in bench.WORKLOADS.items():
        if kind != "decode":
            continue
        cfg = bench.workload_config(name)
        wl = bench._make(name, 0)
        lens = wl.lens + 1  # one appended token per sequence, as a decode step
        pages = ((lens + 63) // 64).sum()
        expect = (int(lens.sum()) * wl.H * per_tok[cfg["format"]] + int(pages) * wl.H * 8
                  + 2 * wl.B * wl.Hq * wl.D * 2)
        assert wl.decode_bytes(lens) == expect, name


def test_reference_arm_line_keeps_the_contract():
    """`bench.py --impl reference` (the oracle on the host's cores) prints one
    JSON line with the keys a bench line carries, `impl: reference`, a
    cpu_baseline describing the run and an e2e with no host copies."""
    import json
    import subprocess

    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                          "llama2-7b-layer", "--cpu-seconds", "0.5", "--steps", "3", "--warmup", "3"],
                         capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [x for x in out.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "higher_is_better", "scaling", "vs_baseline",
              "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["n_gpus"] == 1 and d["value"] > 0
    assert d["config"] == bench.workload_config("llama2-7b-layer")
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
