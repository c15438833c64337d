#!/usr/bin/env python3
"""Benchmark of the quantized-KV decode path on one GB300 (or N, as replicas).

Headline workload (long-context): B=16 sequences, H=32 heads, D=128, context
32768, int4 64-token blocks, K/V ~ N(0,1) with each (head, channel) an outlier
x10 with probability 0.01, inputs generated in HBM by the seeded generator
(2.15 GB of packed codes, far larger than L2).  One step = the whole hot path
once: append one token per sequence (re-quantizing each open block from its
fp16 originals: absmax, scale, quantize, pack) and decode attention of the
step's query over every sequence (one split-K launch that also merges).  The
decode position cycles through one 64-token block, so the context stays
32769..32832 tokens.

Every other workload of the path runs after it, each with its own roofline,
under "workloads" in the same JSON line: tiny, llama2-7b-layer, paged-int8,
prefill-append (quantize GB/s), llama3-8b-layer-gqa, llama2-7b-layer-fp8,
chunked-prefill (tensor-core attention, TFLOP/s), mqa-32k (one cache head
serving 32 query heads), llama3-70b-layer-gqa and llama3-70b-layer-gqa-fp8
(8 query heads per cache head, int4 and FP8) and the stateless codec (kvq_quantize, GB/s) over the
whole K and V history of the 7B layer (int4, int8, FP8) and of long-context
(int4).

value    decode tokens/s = sequences advanced one token through one layer's
         attention per second, summed over ranks (weak scaling: every rank runs
         its own batch; no collective on the data path)
e2e      the same steps through the C ABI with host buffers: each step's new
         K/V rows and query are copied from pinned host memory and its output
         back, on a copy stream one step ahead of the compute stream
roofline the split decode kernel's algorithmic bytes / its CUDA-event time
cpu_baseline / --impl reference: the CPU oracle timed on host cores on a
         bounded sample of the same step
"""
import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "quantized-KV decode attention tokens/s and KV GB/s vs HBM roofline; quantize GB/s"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_TFLOPS = 1900.0
L2_BYTES = 129e6
DEFAULT_WORKLOAD = "long-context"

# name -> (kind, workload number in synth/workloads.py)
WORKLOADS = {
    "tiny": ("decode", 1),
    "llama2-7b-layer": ("decode", 2),
    "long-context": ("decode", 3),
    "paged-int8": ("decode", 4),
    "prefill-append": ("append", 5),
    "llama3-8b-layer-gqa": ("decode", 6),
    "llama2-7b-layer-fp8": ("decode", 7),
    "chunked-prefill": ("prefill", 8),
    "mqa-32k": ("decode", 9),
    "llama3-70b-layer-gqa": ("decode", 10),
    "llama3-70b-layer-gqa-fp8": ("decode", 11),
    "quantize-7b-layer": ("quantize", 2),
    "quantize-long-context": ("quantize", 3),
    "quantize-7b-layer-int8": ("quantize", 2),
    "quantize-7b-layer-fp8": ("quantize", 7),
}
# stateless-codec workloads whose format is not their history's
QUANT_FORMAT = {"quantize-7b-layer-int8": 1}
FORMAT_NAMES = {0: ("int4", "int4-b64"), 1: ("int8", "int8-page"), 2: ("fp8-e4m3", "fp8-e4m3-page")}


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=list(WORKLOADS))
    ap.add_argument("--prefill-seqs", type=int, default=64)
    ap.add_argument("--sub-steps", type=int, default=100, help="timed steps of each further workload")
    ap.add_argument("--no-extras", dest="extras", action="store_false", help="the headline workload only")
    return ap.parse_args(argv)


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def rank_seed(base_seed, rank):
    """Weak scaling: every rank runs its own batch, drawn with its own seed."""
    return int(base_seed) + int(rank)


def max_over_ranks(pg, x, device):
    """The slowest rank's time (every rank gets it); x unchanged without a group."""
    if pg is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world, units_per_rank, seconds):
    """Units all ranks processed per second of the slowest rank."""
    return world * units_per_rank / seconds


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f)
    except Exception:
        return None


def measured_peak():
    """HBM GB/s: the measured copy bandwidth, else the fallback."""
    p = _peaks()
    if p and "hbm_gbs" in p:
        return float(p["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def measured_tensor_peak():
    """Dense fp16/bf16 tensor peak in TFLOP/s: the measured cuBLAS bf16 burst
    figure (fp16 and bf16 have the same nominal rate), else the fallback."""
    p = _peaks()
    if p and "bf16_tflops" in p:
        return float(p["bf16_tflops"]), "measured (bf16 burst; fp16 same nominal rate)"
    return FALLBACK_TFLOPS, "fallback"


KERNEL_SOURCES = {
    "decode_split_kernel": ("kvq_decode.cu", "kvq_device.cuh", "kvq_internal.h"),
    "append_kernel": ("kvq_quantize.cu", "kvq_device.cuh", "kvq_internal.h"),
    "quantize_contig_kernel": ("kvq_quantize.cu", "kvq_device.cuh", "kvq_internal.h"),
    "prefill_attn_tc_kernel": ("kvq_prefill.cu", "kvq_device.cuh", "kvq_internal.h"),
}


def source_digest(kernel):
    """Digest of the sources a kernel is built from (ties a profile to them)."""
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "quantized_kv_cache_09_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel, workload):
    """dram bytes per launch of `kernel` on `workload` from the committed ncu
    summary, or None when the summary is missing or was taken on other kernel
    sources."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    if not os.path.exists(path):
        return None
    digest = source_digest(kernel)
    with open(path) as f:
        for line in f:
            if line.startswith("#") or "=" not in line:
                continue
            kv = dict(p.split("=", 1) for p in line.split())
            if (kv.get("kernel") == kernel and kv.get("workload") == workload
                    and kv.get("source_sha256") == digest):
                return float(kv["dram_bytes_per_launch"])
    return None


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index, period_ms=20):
        self.index = index
        self.period_ms = period_ms
        self.samples = []
        self.proc = None
        self.thread = None
        self.window = (0.0, 0.0)

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", str(self.period_ms), "-i", str(self.index)], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [p.strip() for p in line.split(",")]))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        t0, t1 = self.window
        inside = [s for t, s in self.samples if t0 <= t <= t1]
        use = inside if inside else [s for _, s in self.samples]
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        sm = []
        mx = None
        for s in use:
            try:
                sm.append(float(s[0]))
                mx = float(s[1])
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, s[3:7]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(use), "samples_in_window": len(inside),
                "window": "the headline's warm-up cycle, timed passes, graph replays and e2e pass (GPU busy)"}


# --------------------------------------------------------------------------
# workload descriptions shared by both arms (the same `config` dict)
# --------------------------------------------------------------------------
def _make(name, seed, prefill_seqs=64):
    from quantized_kv_cache_09_gb300.synth import workloads as W
    kind, cfg = WORKLOADS[name]
    if kind == "decode":
        return W.make_workload(cfg, seed=seed, extra_tokens=64)
    if kind == "append":
        c = W.RECIPES[5]
        return W.Workload(prefill_seqs, c["H"], c["D"], [c["L"]] * prefill_seqs, c["fmt"], c["sigma"], None,
                          "permuted", seed, 0, c["name"])
    wl = W.make_workload(cfg, seed=seed)
    if kind == "quantize" and name in QUANT_FORMAT:
        wl.fmt = QUANT_FORMAT[name]
    return wl


def decode_context(wl):
    """The context range the decode steps run over (steps cycle through one block)."""
    lens = wl.lens
    if bool((lens % 64 == 0).all()) and lens.min() == lens.max():
        return f"{int(lens[0]) + 1}..{int(lens[0]) + 64}"
    return f"{int(lens.min()) + 1}..{int(lens.max()) + 1} (sum {int(lens.sum()) + len(lens)})"


def decode_ctx_lens(wl, step):
    """Lengths after the append of decode step `step` (the cycle of measure_decode)."""
    aligned = bool((wl.lens % 64 == 0).all())
    return wl.lens + ((step % 64) if aligned else 0) + 1


def workload_config(name, world=1, seed=0, prefill_seqs=64):
    kind, _ = WORKLOADS[name]
    wl = _make(name, seed, prefill_seqs)
    par = f"replicas x{world} (sequence-sharded, no collective)"
    if kind == "decode":
        dec_bytes = wl.decode_bytes(wl.lens + 1)
        return {"workload": name, "B": wl.B, "H": wl.H, "Hq": wl.Hq, "D": wl.D, "context": decode_context(wl),
                "format": FORMAT_NAMES[wl.fmt][1], "table": wl.table, "step": "append 1 token + decode attention",
                "parallelism": par,
                "l2": "inputs larger than L2" if dec_bytes > L2_BYTES else "fits in L2 (no flush; latency only)"}
    if kind == "append":
        return {"workload": name, "new_tokens": int(wl.lens.sum()), "H": wl.H, "D": wl.D, "format": "int4-b64",
                "table": wl.table, "step": "one kvq_append of all new tokens", "parallelism": par,
                "l2": "inputs larger than L2"}
    if kind == "quantize":
        return {"workload": name, "tokens": int(wl.lens.sum()), "B": wl.B, "H": wl.H, "D": wl.D,
                "format": FORMAT_NAMES[wl.fmt][1],
                "step": "kvq_quantize of the K history, then of V ([tokens][H][D] each, sequences back to back)",
                "parallelism": par, "l2": "inputs larger than L2"}
    return {"workload": name, "B": wl.B, "H": wl.H, "Hq": wl.Hq, "D": wl.D, "context": int(wl.lens[0]),
            "chunk": wl.chunk, "format": FORMAT_NAMES[wl.fmt][1], "step": "one kvq_prefill_attention of every chunk query",
            "parallelism": par, "l2": "codes (268 MB) larger than L2"}


# --------------------------------------------------------------------------
# the CPU oracle on bounded samples of a workload
# --------------------------------------------------------------------------
def _threads():
    return max(1, min(16, os.cpu_count() or 1))


def oracle_decode_rate(name, seconds, seed, threads=None):
    """Oracle decode steps on (sequence, cache head) samples of a decode
    workload: each sample re-quantizes its open block with the appended token
    (oracle codec) and attends over L + 1 tokens with the g query heads of that
    cache head in binary64.  One thread per sample (the oracle releases the
    GIL).  A token of a sequence needs every cache head, so tokens/s =
    sample-steps/s / H.  Returns (tokens/s, threads, description)."""
    import numpy as np

    from oracle import oracle as orc

    wl = _make(name, seed)
    n = threads or _threads()
    g = wl.Hq // wl.H
    sm = np.float32(1.0 / math.sqrt(wl.D))
    units = [(i % wl.B, (i * 5 + i // wl.B) % wl.H) for i in range(n)]

    def setup(u):  # untimed: the oracle's cache of one (sequence, head) history and the step's inputs
        b, h = u
        L = int(wl.lens[b])
        o = (L // 64) * 64  # first row of the block the new token goes to
        kc, ks = orc.quantize(wl.fmt, wl.kv_host_head("k", b, h, 0, L)) if L else (None, None)
        vc, vs = orc.quantize(wl.fmt, wl.kv_host_head("v", b, h, 0, L)) if L else (None, None)
        nb_full = o // 64
        rb = orc.row_bytes(wl.fmt, wl.D)
        kcp = np.zeros((nb_full + 1, 1, 64, rb), np.uint8)
        vcp = np.zeros_like(kcp)
        ksp = np.zeros((nb_full + 1, 1), np.float32)
        vsp = np.zeros_like(ksp)
        if nb_full:
            kcp[:nb_full], vcp[:nb_full], ksp[:nb_full], vsp[:nb_full] = kc[:nb_full], vc[:nb_full], ks[:nb_full], vs[:nb_full]
        k_open = wl.kv_host_head("k", b, h, o, L + 1)
        v_open = wl.kv_host_head("v", b, h, o, L + 1)
        q = np.ascontiguousarray(wl.q_host(0)[b:b + 1, h * g:(h + 1) * g])
        return (kcp, vcp, ksp, vsp, nb_full, k_open, v_open, q, L)

    # (sequentially: the per-token generator calls hold the interpreter lock between calls)
    caches = [setup(u) for u in units]

    done = [0] * n
    stop = time.time() + seconds

    def work(i):
        kc, vc, ks, vs, nbf, k_open, v_open, q, L = caches[i]
        bt = np.arange(nbf + 1, dtype=np.int32)[None, :]
        while time.time() < stop:
            c, s = orc.quantize(wl.fmt, k_open)   # the open block with the new token, re-quantized
            kc[nbf], ks[nbf] = c[0], s[0]
            c, s = orc.quantize(wl.fmt, v_open)
            vc[nbf], vs[nbf] = c[0], s[0]
            orc.decode_attention(wl.fmt, kc, vc, ks, vs, bt, np.array([L + 1]), q, sm)
            done[i] += 1

    t0 = time.time()
    ths = [threading.Thread(target=work, args=(i,)) for i in range(n)]
    for t in ths:
        t.start()
    for t in ths:
        t.join()
    el = time.time() - t0
    steps = sum(done)
    heads = f"{g} query head{'s' if g > 1 else ''}"
    desc = (f"{steps} oracle (sequence, cache head) steps of {name} (re-quantize the open block with the new "
            f"token + binary64 attention of {heads} over its L+1 tokens), {n} samples on {n} threads for "
            f"{el:.1f} s; tokens/s = steps/s / {wl.H} cache heads")
    return steps / el / wl.H, n, desc


def oracle_append_rate(seconds, seed, threads=None, name="prefill-append"):
    """The oracle codec on samples of a quantize workload (prefill-append or a
    stateless quantize): each thread quantizes 1024-token x H-head K and V
    chunks of its own sequence; GB/s of fp16 read + codes + scales written, as
    for the GPU.  Returns (GB/s, threads, desc)."""
    from oracle import oracle as orc

    wl = _make(name, seed)
    n = threads or _threads()
    xs = []
    for i in range(n):
        b = i % wl.B
        xs.append((wl.kv_host("k", b, 0, 1024), wl.kv_host("v", b, 0, 1024)))
    done = [0] * n
    stop = time.time() + seconds

    def work(i):
        k, v = xs[i]
        while time.time() < stop:
            orc.quantize(wl.fmt, k)
            orc.quantize(wl.fmt, v)
            done[i] += 1

    t0 = time.time()
    ths = [threading.Thread(target=work, args=(i,)) for i in range(n)]
    for t in ths:
        t.start()
    for t in ths:
        t.join()
    el = time.time() - t0
    nbytes = sum(done) * wl.quantize_bytes(1024)
    return nbytes / el / 1e9, n, (f"{sum(done)} oracle {FORMAT_NAMES[wl.fmt][0]} quantizations of 1024-token x "
                                  f"{wl.H}-head K+V chunks of {name} on {n} threads, {el:.1f} s")


def oracle_prefill_rate(seconds, seed):
    """The oracle's chunked-prefill rate on a sample of the workload: queries of
    sequence 0, every head, each over its causal prefix (binary64), one thread."""
    import numpy as np

    from oracle import oracle as orc

    wl = _make("chunked-prefill", seed)
    L, n = int(wl.lens[0]), wl.chunk
    kc, ks = orc.quantize(wl.fmt, wl.kv_host("k", 0, 0, L))
    vc, vs = orc.quantize(wl.fmt, wl.kv_host("v", 0, 0, L))
    bt = np.arange(kc.shape[0], dtype=np.int32)[None, :]
    t0 = time.time()
    done = 0
    while time.time() - t0 < seconds and done < n:
        i = n - 1 - done
        orc.decode_attention(wl.fmt, kc, vc, ks, vs, bt, np.array([L - n + i + 1]),
                             wl.chunk_q_host(0, i, i + 1), np.float32(1.0 / np.sqrt(wl.D)))
        done += 1
    el = time.time() - t0
    return done / el, 1, (f"{done} chunk queries of sequence 0 (all {wl.Hq} heads, causal prefixes of ~{L} tokens, "
                          f"binary64) in {el:.1f} s")


def oracle_rate(name, seconds, seed):
    kind, _ = WORKLOADS[name]
    if kind == "decode":
        return oracle_decode_rate(name, seconds, seed) + ("tokens/s",)
    if kind == "append":
        return oracle_append_rate(seconds, seed) + ("GB/s",)
    if kind == "quantize":
        return oracle_append_rate(seconds, seed, name=name) + ("GB/s",)
    return oracle_prefill_rate(seconds, seed) + ("tokens/s",)


def run_reference(args):
    world, rank, _ = dist_env()
    if world > 1 and rank != 0:
        return
    name = args.workload
    rate, cores, desc, unit = oracle_rate(name, args.cpu_seconds, args.seed)
    line = {"metric": METRIC if WORKLOADS[name][0] != "prefill" else PREFILL_METRIC, "value": rate, "unit": unit,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": None, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64 attention, f32 codec", "data": "synthetic",
            "config": workload_config(name, world, args.seed, args.prefill_seqs),
            "impl": "reference",
            "cpu_baseline": {"value": rate, "unit": unit, "cores": cores, "kind": "oracle", "sample": desc},
            "e2e": {"value": rate, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


PREFILL_METRIC = "chunked-prefill attention tokens/s over the quantized cache (tensor roofline)"


# --------------------------------------------------------------------------
# GPU measurements
# --------------------------------------------------------------------------
def _sync_all(pg, dev):
    import torch
    torch.cuda.synchronize(dev)
    if pg:
        pg.barrier()


def measure_decode(name, K, Wm, seed, dev, pg, clocks=None, graph=True):
    """Decode steps (append one token per sequence + decode attention) on a
    decode workload.  64-aligned histories cycle the appended position through
    one block (a real decode progression); ragged histories re-append the token
    at their end every step, which leaves the cache in the same state."""
    import numpy as np
    import torch

    from quantized_kv_cache_09_gb300 import kvq
    from quantized_kv_cache_09_gb300.runner import DecodeStep, DeviceWorkload

    wl = _make(name, seed)
    dw = DeviceWorkload(wl, device=dev)
    dw.prefill(max_tokens_per_call=1 << 18)
    B, H, D, Hq = wl.B, wl.H, wl.D, wl.Hq
    aligned = bool(np.all(wl.lens % 64 == 0))
    step = DecodeStep(dw)
    NS = 64
    k_steps, v_steps, q_steps, lens_b, lens_a = [], [], [], [], []
    for s in range(NS):
        k1, v1, q = dw.new_token_tensors(s if aligned else 0)
        if not aligned:
            wl.q_device(q, s)
        k_steps.append(k1)
        v_steps.append(v1)
        q_steps.append(q)
        off = s if aligned else 0
        lens_b.append(torch.from_numpy(wl.lens + off).to(dev))
        lens_a.append(torch.from_numpy(wl.lens + off + 1).to(dev))
    t_busy0 = time.time()  # the clock window: from here to the end of the e2e pass, the GPU runs these steps
    for s in range(NS):   # one full cycle establishes the open block's tail rows
        step.run(lens_b[s], lens_a[s], k_steps[s], v_steps[s], q_steps[s])
    for i in range(Wm):
        s = i % NS
        step.run(lens_b[s], lens_a[s], k_steps[s], v_steps[s], q_steps[s])
    torch.cuda.synchronize(dev)
    rc, flags = kvq.kvq_get_device_status(dw.cache)
    if rc != 0:
        raise RuntimeError(f"{name}: device status {rc} flags {flags:#x} after warm-up")

    stream = torch.cuda.current_stream(dev)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    _sync_all(pg, dev)
    # (1) the headline: K whole steps back to back, events only around them, so
    # each launch overlaps the previous one's tail as in a serving loop
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for i in range(K):
        s = (Wm + i) % NS
        kvq.kvq_append(dw.cache, k_steps[s], v_steps[s], step.cu, dw.block_table, lens_b[s], 1)
        kvq.kvq_decode_attention_gqa(dw.cache, q_steps[s], dw.block_table, lens_a[s], dw.softmax_scale, step.out,
                                     dw.workspace)
    end.record(stream)
    _sync_all(pg, dev)
    total_ms = start.elapsed_time(end)
    # (2) the same K steps again with an event before, between and after the two
    # calls: each call's own duration (the events serialise the launches)
    for i in range(K):
        s = (Wm + K + i) % NS
        e0, e1, e2 = ev[i]
        e0.record(stream)
        kvq.kvq_append(dw.cache, k_steps[s], v_steps[s], step.cu, dw.block_table, lens_b[s], 1)
        e1.record(stream)
        kvq.kvq_decode_attention_gqa(dw.cache, q_steps[s], dw.block_table, lens_a[s], dw.softmax_scale, step.out,
                                     dw.workspace)
        e2.record(stream)
    _sync_all(pg, dev)
    app_ms = sum(ev[i][0].elapsed_time(ev[i][1]) for i in range(K)) / K
    dec_ms = sum(ev[i][1].elapsed_time(ev[i][2]) for i in range(K)) / K
    split_ms = ev[0][0].elapsed_time(ev[K - 1][2])
    rc, flags = kvq.kvq_get_device_status(dw.cache)
    if rc != 0:
        raise RuntimeError(f"{name}: device status {rc} flags {flags:#x} after timed steps")
    dec_bytes = sum(wl.decode_bytes(decode_ctx_lens(wl, Wm + K + i)) for i in range(K)) / K

    graph_ms = None
    if graph:
        # (3) the steps replayed from one CUDA graph holding the 64-step input
        # cycle (kvq_step_graph, captured before the timing): ceil(K / 64) replays
        g = kvq.StepGraph([step.graph_step(lens_b[s], lens_a[s], k_steps[s], v_steps[s], q_steps[s])
                           for s in range(NS)])
        g.launch()
        _sync_all(pg, dev)
        reps = -(-K // NS)
        g_s = torch.cuda.Event(enable_timing=True)
        g_e = torch.cuda.Event(enable_timing=True)
        g_s.record(stream)
        for _ in range(reps):
            g.launch()
        g_e.record(stream)
        _sync_all(pg, dev)
        graph_ms = g_s.elapsed_time(g_e) * K / (reps * NS)  # per K steps
        g.close()
        rc, flags = kvq.kvq_get_device_status(dw.cache)
        if rc != 0:
            raise RuntimeError(f"{name}: device status {rc} flags {flags:#x} after graph steps")

    # (4) end to end through the C ABI with host buffers.  A copy stream runs one
    # step ahead: it brings step i+1's new rows and query from pinned memory
    # (one copy: each step's K rows, V rows and query packed back to back)
    # while step i computes, and copies step i's output back once it is done; the
    # compute stream waits only for events, so consecutive kernels keep their
    # programmatic-launch overlap.  Inputs and outputs are double-buffered.
    nk, nq = k_steps[0].numel(), q_steps[0].numel()
    pin_in = [torch.cat([k_steps[s].reshape(-1), v_steps[s].reshape(-1), q_steps[s].reshape(-1)]).cpu().pin_memory()
              for s in range(NS)]
    pin_o = [torch.empty((B, Hq, D), dtype=torch.float16).pin_memory() for _ in range(2)]
    d_in = [torch.empty(2 * nk + nq, dtype=torch.float16, device=dev) for _ in range(2)]
    dk = [x[:nk].view(k_steps[0].shape) for x in d_in]
    dv = [x[nk:2 * nk].view(v_steps[0].shape) for x in d_in]
    dq = [x[2 * nk:].view(q_steps[0].shape) for x in d_in]
    outs = [torch.empty((B, Hq, D), dtype=torch.float16, device=dev) for _ in range(2)]
    copy = torch.cuda.Stream(dev)
    h2d = [torch.cuda.Event() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]
    d2h = [torch.cuda.Event() for _ in range(2)]
    Ke = K
    base = Wm + 2 * K

    def stage(i, slot):
        s = (base + i) % NS
        with torch.cuda.stream(copy):
            d_in[slot].copy_(pin_in[s], non_blocking=True)
            h2d[slot].record(copy)

    _sync_all(pg, dev)
    e2e_s = torch.cuda.Event(enable_timing=True)
    e2e_e = torch.cuda.Event(enable_timing=True)
    e2e_s.record(stream)
    copy.wait_event(e2e_s)
    stage(0, 0)
    for i in range(Ke):
        slot = i & 1
        s = (base + i) % NS
        if i + 1 < Ke:
            if i >= 1:
                copy.wait_event(done[1 - slot])  # step i-1 is done with that slot's inputs
            stage(i + 1, 1 - slot)
        stream.wait_event(h2d[slot])
        if i >= 2:
            stream.wait_event(d2h[slot])  # step i-2's output has been read back
        kvq.kvq_append(dw.cache, dk[slot], dv[slot], step.cu, dw.block_table, lens_b[s], 1)
        kvq.kvq_decode_attention_gqa(dw.cache, dq[slot], dw.block_table, lens_a[s], dw.softmax_scale, outs[slot],
                                     dw.workspace)
        done[slot].record(stream)
        copy.wait_event(done[slot])
        with torch.cuda.stream(copy):
            pin_o[slot].copy_(outs[slot], non_blocking=True)
            d2h[slot].record(copy)
    stream.wait_stream(copy)
    e2e_e.record(stream)
    _sync_all(pg, dev)
    e2e_ms = e2e_s.elapsed_time(e2e_e)
    if clocks is not None:
        clocks.window = (t_busy0, time.time())
    rc, flags = kvq.kvq_get_device_status(dw.cache)
    if rc != 0:
        raise RuntimeError(f"{name}: device status {rc} flags {flags:#x} after end-to-end steps")

    res = dict(wl=wl, B=B, H=H, D=D, Hq=Hq, aligned=aligned, total_ms=total_ms, app_ms=app_ms, dec_ms=dec_ms,
               graph_ms=graph_ms, e2e_ms=e2e_ms, Ke=Ke, dec_bytes=dec_bytes, split_ms=split_ms,
               h2d=(2 * H + Hq) * B * D * 2, d2h=B * Hq * D * 2, launches=(1 + -(-B // 512)) * K)
    del dw
    torch.cuda.empty_cache()
    return res


def measure_append(K, Wm, seed, dev, nseqs=64):
    """prefill-append: one kvq_append of nseqs x 4096 new tokens (H=32) into
    randomly permuted empty pages; repeated calls write the same bytes."""
    import torch

    from quantized_kv_cache_09_gb300 import kvq
    from quantized_kv_cache_09_gb300.runner import DeviceWorkload

    wl = _make("prefill-append", seed, nseqs)
    dw = DeviceWorkload(wl, device=dev)
    L = int(wl.lens[0])
    k_new = torch.empty((nseqs * L, wl.H, wl.D), dtype=torch.float16, device=dev)
    v_new = torch.empty_like(k_new)
    for b in range(nseqs):
        wl.kv_device("k", b, 0, L, k_new[b * L:(b + 1) * L])
        wl.kv_device("v", b, 0, L, v_new[b * L:(b + 1) * L])
    cu = torch.arange(0, nseqs * L + 1, L, dtype=torch.int32, device=dev)
    zero = torch.zeros(nseqs, dtype=torch.int32, device=dev)
    for _ in range(Wm):
        kvq.kvq_append(dw.cache, k_new, v_new, cu, dw.block_table, zero, L)
    stream = torch.cuda.current_stream(dev)
    torch.cuda.synchronize(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for i in range(K):
        ev[i][0].record(stream)
        kvq.kvq_append(dw.cache, k_new, v_new, cu, dw.block_table, zero, L)
        ev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    ms = sum(a.elapsed_time(b) for a, b in ev) / K
    rc, flags = kvq.kvq_get_device_status(dw.cache)
    if rc != 0:
        raise RuntimeError(f"prefill-append: device status {rc} flags {flags:#x}")
    nbytes = wl.quantize_bytes(L) * nseqs
    del k_new, v_new, dw
    torch.cuda.empty_cache()
    return dict(ms=ms, bytes=nbytes, tokens=nseqs * L)


def measure_quantize(name, K, Wm, seed, dev):
    """A stateless-codec workload: kvq_quantize of the whole K history of the
    workload's sequences ([B*L][H][D], sequences back to back, so every 64-row
    block is one (sequence, head, block) of quantize_block), then of V."""
    import torch

    from quantized_kv_cache_09_gb300 import kvq

    wl = _make(name, seed)
    L = int(wl.lens[0])
    if not bool((wl.lens == L).all()) or L % 64:
        raise ValueError(f"{name}: the stateless quantize workloads need equal, block-aligned lengths")
    T = wl.B * L
    xs, codes, scales = [], [], []
    for which in ("k", "v"):
        x = torch.empty((T, wl.H, wl.D), dtype=torch.float16, device=dev)
        for b in range(wl.B):
            wl.kv_device(which, b, 0, L, x[b * L:(b + 1) * L])
        xs.append(x)
        codes.append(torch.empty((T // 64, wl.H, 64, wl.row_bytes), dtype=torch.uint8, device=dev))
        scales.append(torch.empty((T // 64, wl.H), dtype=torch.float32, device=dev))

    def step():
        for i in range(2):
            kvq.kvq_quantize(wl.fmt, xs[i], codes[i], scales[i])

    for _ in range(Wm):
        step()
    stream = torch.cuda.current_stream(dev)
    torch.cuda.synchronize(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for i in range(K):
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    ms = sum(a.elapsed_time(b) for a, b in ev) / K
    nbytes = wl.quantize_bytes(L) * wl.B
    del xs, codes, scales
    torch.cuda.empty_cache()
    return dict(ms=ms, bytes=nbytes, tokens=T, fmt=wl.fmt)


def measure_chunked_prefill(K, Wm, seed, dev):
    """chunked-prefill: kvq_prefill_attention of the last 512 of 8192 tokens of
    8 sequences (H=32, int4) over the cache that holds them."""
    import torch

    from quantized_kv_cache_09_gb300 import kvq
    from quantized_kv_cache_09_gb300.runner import DeviceWorkload

    wl = _make("chunked-prefill", seed)
    dw = DeviceWorkload(wl, device=dev)
    dw.prefill(max_tokens_per_call=1 << 16)
    n = wl.chunk
    q = torch.empty((wl.B * n, wl.Hq, wl.D), dtype=torch.float16, device=dev)
    for b in range(wl.B):
        wl.chunk_q_device(q[b * n:(b + 1) * n], b)
    out = torch.empty_like(q)
    cu = torch.arange(0, wl.B * n + 1, n, dtype=torch.int32, device=dev)
    # the grid's last wave of 256-row units runs as key halves merged in this workspace
    ws = kvq.prefill_workspace(wl.Hq, wl.B, n, device=dev)
    for _ in range(Wm):
        kvq.kvq_prefill_attention(dw.cache, q, cu, n, dw.block_table, dw.lens, dw.softmax_scale, out, workspace=ws)
    torch.cuda.synchronize(dev)
    stream = torch.cuda.current_stream(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for i in range(K):
        ev[i][0].record(stream)
        kvq.kvq_prefill_attention(dw.cache, q, cu, n, dw.block_table, dw.lens, dw.softmax_scale, out, workspace=ws)
        ev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    ms = sum(a.elapsed_time(b) for a, b in ev) / K
    # end to end: the chunk's queries from pinned host memory, the output back
    pin_q = q.cpu().pin_memory()
    pin_o = torch.empty_like(pin_q).pin_memory()
    e_s, e_e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e_s.record(stream)
    for _ in range(K):
        q.copy_(pin_q, non_blocking=True)
        kvq.kvq_prefill_attention(dw.cache, q, cu, n, dw.block_table, dw.lens, dw.softmax_scale, out, workspace=ws)
        pin_o.copy_(out, non_blocking=True)
    e_e.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = e_s.elapsed_time(e_e) / K
    rc, flags = kvq.kvq_get_device_status(dw.cache)
    if rc != 0:
        raise RuntimeError(f"chunked-prefill: device status {rc} flags {flags:#x}")
    res = dict(ms=ms, e2e_ms=e2e_ms, flops=wl.prefill_flops(), tokens=wl.B * n, qbytes=q.numel() * 2)
    del dw, q, out
    torch.cuda.empty_cache()
    return res


# --------------------------------------------------------------------------
# result lines
# --------------------------------------------------------------------------
def _decode_kernels(wl):
    """The kernels one decode call launches (the roofline's event time covers them all)."""
    g = wl.Hq // wl.H
    if g == 1 or (wl.fmt == 0 and g in (2, 4)):
        return "kvq_decode_attention (decode_split_kernel, split merge in the same launch)"
    return "kvq_decode_attention_gqa (decode_split_kernel on 16-query-head tiles + decode_tile_merge_kernel)"


def decode_result(name, r, world, pg, dev, K, Wm, peak, peak_kind, cfg_seed=0):
    total_ms = max_over_ranks(pg, r["total_ms"], dev)
    e2e_ms = max_over_ranks(pg, r["e2e_ms"], dev)
    dec_ms = max_over_ranks(pg, r["dec_ms"], dev)
    app_ms = max_over_ranks(pg, r["app_ms"], dev)
    B = r["B"]
    achieved = r["dec_bytes"] / (dec_ms * 1e-3) / 1e9
    out = {"metric": METRIC, "value": whole_job_rate(world, B * K, total_ms * 1e-3), "unit": "tokens/s",
           "n_gpus": world, "steps": K, "warmup": Wm, "ms_per_step": total_ms / K, "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": FORMAT_NAMES[r["wl"].fmt][0] + " codes, fp32 math",
           "data": "synthetic (seeded generator in HBM)",
           "config": workload_config(name, world, cfg_seed),
           "kv_gb_per_s": achieved, "decode_us": dec_ms * 1e3, "append_us": app_ms * 1e3,
           "step_us_events_between_calls": r["split_ms"] / K * 1e3,
           "roofline": {"kernel": _decode_kernels(r["wl"]), "bound": "hbm",
                        "achieved": achieved, "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                        "frac": achieved / peak, "traffic": ncu_traffic("decode_split_kernel", name),
                        "algorithmic_bytes_per_launch": r["dec_bytes"],
                        "timing": "mean CUDA-event time of one kvq_decode_attention call (events on the launching "
                                  "stream between calls)"},
           "e2e": {"value": whole_job_rate(world, B * r["Ke"], e2e_ms * 1e-3), "unit": "tokens/s",
                   "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"],
                   "how": "pinned host -> device copies of each step's new K/V rows and query and the output back, "
                          "on a copy stream one step ahead"},
           "gpu_launches": r["launches"]}
    if r["graph_ms"] is not None:
        graph_ms = max_over_ranks(pg, r["graph_ms"], dev)
        out["graph"] = {"ms_per_step": graph_ms / K, "value": whole_job_rate(world, B * K, graph_ms * 1e-3),
                        "unit": "tokens/s", "how": "one kvq_step_graph of 64 steps (append + decode each), replayed"}
    return out


def append_result(r, world, pg, dev, K, Wm, peak, peak_kind, cfg_seed=0, prefill_seqs=64):
    ms = max_over_ranks(pg, r["ms"], dev)
    gbs = r["bytes"] / (ms * 1e-3) / 1e9
    return {"metric": METRIC, "value": whole_job_rate(world, r["bytes"] / 1e9, ms * 1e-3), "unit": "GB/s",
            "n_gpus": world, "steps": K, "warmup": Wm, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "fp16 in, int4 codes out, fp32 math",
            "data": "synthetic (seeded generator in HBM)", "config": workload_config("prefill-append", world, cfg_seed, prefill_seqs),
            "roofline": {"kernel": "append_kernel", "bound": "hbm", "achieved": gbs, "peak": peak,
                         "peak_kind": peak_kind, "unit": "GB/s", "frac": gbs / peak,
                         "traffic": ncu_traffic("append_kernel", "prefill-append"),
                         "algorithmic_bytes_per_launch": r["bytes"]},
            "gpu_launches": K}


def quantize_result(name, r, world, pg, dev, K, Wm, peak, peak_kind, cfg_seed=0):
    ms = max_over_ranks(pg, r["ms"], dev)
    gbs = r["bytes"] / (ms * 1e-3) / 1e9
    return {"metric": METRIC, "value": whole_job_rate(world, r["bytes"] / 1e9, ms * 1e-3), "unit": "GB/s",
            "n_gpus": world, "steps": K, "warmup": Wm, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": f"fp16 in, {FORMAT_NAMES[r['fmt']][0]} codes out, fp32 math",
            "data": "synthetic (seeded generator in HBM)", "config": workload_config(name, world, cfg_seed),
            "roofline": {"kernel": "quantize_contig_kernel", "bound": "hbm", "achieved": gbs, "peak": peak,
                         "peak_kind": peak_kind, "unit": "GB/s", "frac": gbs / peak,
                         "traffic": ncu_traffic("quantize_contig_kernel", name),
                         "algorithmic_bytes_per_launch": r["bytes"] / 2,
                         "timing": "mean CUDA-event time of one step = two kvq_quantize calls (K, V)"},
            "gpu_launches": 2 * K}


def prefill_result(r, world, pg, dev, K, Wm, cfg_seed=0):
    ms = max_over_ranks(pg, r["ms"], dev)
    e2e_ms = max_over_ranks(pg, r["e2e_ms"], dev)
    tflops = r["flops"] / (ms * 1e-3) / 1e12
    tpeak, tkind = measured_tensor_peak()
    return {"metric": PREFILL_METRIC, "value": whole_job_rate(world, r["tokens"], ms * 1e-3), "unit": "tokens/s",
            "n_gpus": world, "steps": K, "warmup": Wm, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "int4 codes, fp16 MMA operands, fp32 accumulation",
            "data": "synthetic (seeded generator in HBM)", "config": workload_config("chunked-prefill", world, cfg_seed),
            "tflops": tflops,
            "roofline": {"kernel": "prefill_attn_tc_kernel", "bound": "tensor", "achieved": tflops, "peak": tpeak,
                         "peak_kind": tkind, "unit": "TFLOP/s", "frac": tflops / tpeak,
                         "traffic": ncu_traffic("prefill_attn_tc_kernel", "chunked-prefill"),
                         "algorithmic_flops_per_launch": r["flops"]},
            "e2e": {"value": whole_job_rate(world, r["tokens"], e2e_ms * 1e-3), "unit": "tokens/s",
                    "h2d_bytes_per_step": r["qbytes"], "d2h_bytes_per_step": r["qbytes"]},
            "gpu_launches": K}


def measure(name, K, Wm, seed, dev, pg, world, clocks=None, prefill_seqs=64, cfg_seed=0):
    """One workload's result dict.  seed: this rank's inputs; cfg_seed: the
    base seed the `config` is described with (the same in both arms)."""
    peak, peak_kind = measured_peak()
    kind, _ = WORKLOADS[name]
    if kind == "decode":
        r = measure_decode(name, K, Wm, seed, dev, pg, clocks=clocks)
        return decode_result(name, r, world, pg, dev, K, Wm, peak, peak_kind, cfg_seed)
    if kind == "append":
        r = measure_append(K, max(Wm, 1), seed, dev, prefill_seqs)
        return append_result(r, world, pg, dev, K, Wm, peak, peak_kind, cfg_seed, prefill_seqs)
    if kind == "quantize":
        r = measure_quantize(name, K, max(Wm, 1), seed, dev)
        return quantize_result(name, r, world, pg, dev, K, Wm, peak, peak_kind, cfg_seed)
    r = measure_chunked_prefill(K, max(Wm, 1), seed, dev)
    return prefill_result(r, world, pg, dev, K, Wm, cfg_seed)


SUB_KEYS = ("value", "unit", "ms_per_step", "steps", "decode_us", "append_us", "kv_gb_per_s", "tflops", "roofline",
            "e2e", "graph", "config")


def run_ours(args):
    import torch

    world, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA device")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist
    seed = rank_seed(args.seed, rank)
    K, Wm = args.steps, args.warmup

    clocks = ClockSampler(dev.index or 0)
    clocks.start()
    time.sleep(0.3)
    t0 = time.time()
    line = measure(args.workload, K, Wm, seed, dev, pg, world, clocks=clocks, prefill_seqs=args.prefill_seqs,
                   cfg_seed=args.seed)
    if clocks.window == (0.0, 0.0):
        clocks.window = (t0, time.time())
    clocks.stop()
    line["clocks"] = clocks.summary()

    if args.extras:
        subs = {}
        Ks = max(args.sub_steps, 3)
        for name in WORKLOADS:
            if name == args.workload:
                continue
            r = measure(name, Ks, max(Wm, 3), seed, dev, pg, world, prefill_seqs=args.prefill_seqs,
                        cfg_seed=args.seed)
            subs[name] = {k: r[k] for k in SUB_KEYS if k in r}
        line["workloads"] = subs
    if rank == 0 and not args.no_cpu_baseline:
        rate, cores, desc, unit = oracle_rate(args.workload, args.cpu_seconds, args.seed)
        line["cpu_baseline"] = {"value": rate, "unit": unit, "cores": cores, "kind": "oracle", "sample": desc}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if pg:
        pg.barrier()
        pg.destroy_process_group()


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
