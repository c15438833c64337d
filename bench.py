#!/usr/bin/env python3
"""Benchmark of the quantized-KV decode step on one GB300 (or N, as replicas).

Workload (llama2-7b-layer): B=8 sequences, H=32 heads, D=128, context 8192,
int4 64-token blocks, K/V ~ N(0,1) with 4 outlier channels per head x10,
inputs generated in HBM by the seeded generator.  One step = the whole hot
path once: append one token per sequence (re-quantizing each open block from
its fp16 originals: absmax, scale, quantize, pack) and decode attention of the
step's query over every sequence (one split-K launch that also merges).  The decode
position cycles through one 64-token block, so the context stays 8193..8256
tokens and the working set (~270 MB of codes) stays larger than L2 (129 MB).

value    decode tokens/s = sequences advanced one token through one layer's
         attention per second, summed over ranks (weak scaling: every rank runs
         its own batch; no collective on the data path)
e2e      the same steps through the C ABI with host buffers: each step copies its
         new K/V rows and query from pinned host memory and its output back
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

CONFIG = 2
METRIC = "quantized-KV decode attention tokens/s and KV GB/s vs HBM roofline; quantize GB/s"
FALLBACK_HBM_GBS = 6800.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--workload", default="llama2-7b-layer",
                    choices=["tiny", "llama2-7b-layer", "long-context", "paged-int8", "prefill-append",
                             "llama3-8b-layer-gqa", "llama2-7b-layer-fp8", "chunked-prefill"])
    ap.add_argument("--prefill-seqs", type=int, default=64)
    ap.add_argument("--no-extras", dest="extras", action="store_false")
    return ap.parse_args()


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


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def measured_tensor_peak():
    """Dense fp16/bf16 tensor peak in TFLOP/s: the measured cuBLAS bf16 burst
    figure (fp16 and bf16 have the same nominal rate), else the fallback."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured (bf16 burst; fp16 same nominal rate)"
    except Exception:
        return 1900.0, "fallback"


KERNEL_SOURCES = {
    "decode_split_kernel": ("kvq_decode.cu", "kvq_device.cuh", "kvq_internal.h"),
    "append_kernel": ("kvq_quantize.cu", "kvq_device.cuh", "kvq_internal.h"),
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
    """nvidia-smi samples (every 100 ms) of SM clock and throttle reasons."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.samples = []
        self.proc = None
        self.thread = None
        self.window = (0.0, 0.0)

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "100", "-i", str(self.index)], stdout=subprocess.PIPE,
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
            except ValueError:
                continue
            for n, v in zip(names, s[3:7]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(use), "samples_in_timed_region": len(inside)}


# --------------------------------------------------------------------------
# the CPU oracle on a bounded sample of the same step
# --------------------------------------------------------------------------
def oracle_step_rate(seconds, seed, threads=None, cfg=None):
    """Oracle decode steps of a uniform-length decode workload (default: the 7B
    layer): for each sampled sequence, re-quantize its open block (oracle
    quantize of the 64-token block holding the new token) and attend over its
    L + 1 tokens, every query head, binary64.
    Threads run independent sequences (the oracle releases the GIL).
    Returns (steps per second, threads, description)."""
    import numpy as np

    from oracle import oracle as orc
    from quantized_kv_cache_09_gb300.synth import workloads as W

    wl = W.make_workload(cfg or CONFIG, seed=seed, extra_tokens=64)
    threads = threads or max(1, min(16, os.cpu_count() or 1))
    L = int(wl.lens[0])
    sm = np.float32(1.0 / math.sqrt(wl.D))

    # untimed setup: the oracle's cache of each sampled sequence's history
    nseq = min(wl.B, threads)
    caches = []
    for b in range(nseq):
        kc, ks = orc.quantize(wl.fmt, wl.kv_host("k", b, 0, L))
        vc, vs = orc.quantize(wl.fmt, wl.kv_host("v", b, 0, L))
        nb = kc.shape[0]
        kc = np.concatenate([kc, np.zeros_like(kc[:1])])
        vc = np.concatenate([vc, np.zeros_like(vc[:1])])
        ks = np.concatenate([ks, np.zeros_like(ks[:1])])
        vs = np.concatenate([vs, np.zeros_like(vs[:1])])
        k_new = wl.kv_host("k", b, L, L + 1)
        v_new = wl.kv_host("v", b, L, L + 1)
        q = wl.q_host(0)[b:b + 1]
        caches.append((kc, vc, ks, vs, nb, k_new, v_new, q))

    done = [0] * nseq
    stop = time.time() + seconds

    def work(i):
        kc, vc, ks, vs, nb, k_new, v_new, q = caches[i]
        bt = np.arange(nb + 1, dtype=np.int32)[None, :]
        while time.time() < stop:
            # append: the new token opens block nb; re-quantize it
            c, s = orc.quantize(wl.fmt, k_new)
            kc[nb], ks[nb] = c[0], s[0]
            c, s = orc.quantize(wl.fmt, v_new)
            vc[nb], vs[nb] = c[0], s[0]
            orc.decode_attention(wl.fmt, kc, vc, ks, vs, bt, np.array([L + 1]), q, sm)
            done[i] += 1

    t0 = time.time()
    ths = [threading.Thread(target=work, args=(i,)) for i in range(nseq)]
    for t in ths:
        t.start()
    for t in ths:
        t.join()
    el = time.time() - t0
    steps = sum(done)
    heads = f"{wl.H} heads" if wl.Hq == wl.H else f"{wl.Hq} query heads over {wl.H} cache heads"
    desc = (f"{steps} oracle sequence-steps (append 1 token + binary64 attention over {L + 1} tokens x "
            f"{heads}), {nseq} sequences on {nseq} threads for {el:.1f} s")
    return steps / el, nseq, desc


# --------------------------------------------------------------------------
def run_reference(args):
    world, rank, _ = dist_env()
    if world > 1 and rank != 0:
        return
    from quantized_kv_cache_09_gb300.synth import workloads as W
    name = args.workload if args.workload in ORACLE_WORKLOADS else "llama2-7b-layer"
    cfg = W.CONFIGS[ORACLE_WORKLOADS[name]]
    rate, cores, desc = oracle_step_rate(args.cpu_seconds, args.seed, cfg=ORACLE_WORKLOADS[name])
    line = {"metric": METRIC, "value": rate, "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1000.0 / rate if rate else None, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": name, "B": cfg["B"], "H": cfg["H"], "Hq": cfg.get("Hq", cfg["H"]), "D": 128,
                       "context": cfg["L"], "format": "int4-b64", "step": "append 1 token + decode attention"},
            "impl": "reference",
            "cpu_baseline": {"value": rate, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": desc},
            "e2e": {"value": rate, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


DECODE_WORKLOADS = {"tiny": 1, "llama2-7b-layer": 2, "long-context": 3, "paged-int8": 4,
                    "llama3-8b-layer-gqa": 6, "llama2-7b-layer-fp8": 7}
FORMAT_NAMES = {0: ("int4", "int4-b64"), 1: ("int8", "int8-page"), 2: ("fp8-e4m3", "fp8-e4m3-page")}
# workloads whose cpu_baseline / reference arm samples their own shape (uniform lengths)
ORACLE_WORKLOADS = {"llama2-7b-layer": 2, "llama3-8b-layer-gqa": 6}


def _sync_all(pg, dev):
    import torch
    torch.cuda.synchronize(dev)
    if pg:
        pg.barrier()


def measure_decode(name, K, Wm, seed, dev, pg):
    """Decode steps (append one token per sequence + decode attention) on a
    decode workload.  64-aligned histories cycle the appended position through
    one block (a real decode progression); ragged histories re-append the token
    at their end every step, which leaves the cache in the same state."""
    import numpy as np
    import torch

    from quantized_kv_cache_09_gb300 import kvq
    from quantized_kv_cache_09_gb300.runner import DecodeStep, DeviceWorkload
    from quantized_kv_cache_09_gb300.synth import workloads as W

    wl = W.make_workload(DECODE_WORKLOADS[name], seed=seed, extra_tokens=64)
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
    for s in range(NS):   # one full cycle establishes the open block's tail rows
        step.run(lens_b[s], lens_a[s], k_steps[s], v_steps[s], q_steps[s])
    for i in range(Wm):
        s = i % NS
        step.run(lens_b[s], lens_a[s], k_steps[s], v_steps[s], q_steps[s])
    torch.cuda.synchronize(dev)
    rc, flags = kvq.kvq_get_device_status(dw.cache)
    if rc != 0:
        raise RuntimeError(f"device status {rc} flags {flags:#x} after warm-up")

    stream = torch.cuda.current_stream(dev)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    clocks = ClockSampler(dev.index or 0)
    clocks.start()
    time.sleep(0.3)
    _sync_all(pg, dev)
    t_wall0 = time.time()
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
    clocks.window = (t_wall0, time.time())
    app_ms = sum(ev[i][0].elapsed_time(ev[i][1]) for i in range(K)) / K
    dec_ms = sum(ev[i][1].elapsed_time(ev[i][2]) for i in range(K)) / K
    split_ms = ev[0][0].elapsed_time(ev[K - 1][2])
    rc, flags = kvq.kvq_get_device_status(dw.cache)
    if rc != 0:
        raise RuntimeError(f"device status {rc} flags {flags:#x} after timed steps")
    # (3) the steps replayed from one CUDA graph holding the 64-step input cycle
    # (kvq_step_graph, captured before the timed loop): ceil(K / 64) replays
    graph = kvq.StepGraph([step.graph_step(lens_b[s], lens_a[s], k_steps[s], v_steps[s], q_steps[s])
                           for s in range(NS)])
    graph.launch()
    _sync_all(pg, dev)
    reps = -(-K // NS)
    g_s = torch.cuda.Event(enable_timing=True)
    g_e = torch.cuda.Event(enable_timing=True)
    g_s.record(stream)
    for i in range(reps):
        graph.launch()
    g_e.record(stream)
    _sync_all(pg, dev)
    graph_ms = g_s.elapsed_time(g_e) * K / (reps * NS)  # per K steps
    graph.close()
    rc, flags = kvq.kvq_get_device_status(dw.cache)
    if rc != 0:
        raise RuntimeError(f"device status {rc} flags {flags:#x} after graph steps")

    # end to end through the C ABI with host buffers
    pin_k = [k.cpu().pin_memory() for k in k_steps]
    pin_v = [v.cpu().pin_memory() for v in v_steps]
    pin_q = [q.cpu().pin_memory() for q in q_steps]
    pin_o = torch.empty((B, Hq, D), dtype=torch.float16).pin_memory()
    dk, dv, dq = (torch.empty_like(k_steps[0]), torch.empty_like(v_steps[0]), torch.empty_like(q_steps[0]))
    Ke = max(1, K // 2)
    _sync_all(pg, dev)
    e2e_s = torch.cuda.Event(enable_timing=True)
    e2e_e = torch.cuda.Event(enable_timing=True)
    e2e_s.record(stream)
    for i in range(Ke):
        s = (Wm + 2 * K + i) % NS
        dk.copy_(pin_k[s], non_blocking=True)
        dv.copy_(pin_v[s], non_blocking=True)
        dq.copy_(pin_q[s], non_blocking=True)
        kvq.kvq_append(dw.cache, dk, dv, step.cu, dw.block_table, lens_b[s], 1)
        kvq.kvq_decode_attention_gqa(dw.cache, dq, dw.block_table, lens_a[s], dw.softmax_scale, step.out,
                                     dw.workspace)
        pin_o.copy_(step.out, non_blocking=True)
    e2e_e.record(stream)
    _sync_all(pg, dev)
    e2e_ms = e2e_s.elapsed_time(e2e_e)
    clocks.stop()

    ctx = [(wl.lens + ((Wm + K + i) % NS if aligned else 0) + 1) for i in range(K)]
    dec_bytes = sum(wl.decode_bytes(c) for c in ctx) / K
    res = dict(wl=wl, B=B, H=H, D=D, aligned=aligned, total_ms=total_ms, app_ms=app_ms, dec_ms=dec_ms, graph_ms=graph_ms,
               e2e_ms=e2e_ms, Ke=Ke, dec_bytes=dec_bytes, clocks=clocks.summary(), split_ms=split_ms,
               h2d=(2 * H + Hq) * B * D * 2, d2h=B * Hq * D * 2, launches=(1 + -(-B // 512)) * K, Hq=Hq)
    del dw
    torch.cuda.empty_cache()
    return res


def measure_prefill(K, Wm, seed, dev, nseqs=64):
    """prefill-append: one kvq_append of nseqs x 4096 new tokens (H=32) into
    randomly permuted empty pages; repeated calls write the same bytes."""
    import torch

    from quantized_kv_cache_09_gb300 import kvq
    from quantized_kv_cache_09_gb300.runner import DeviceWorkload
    from quantized_kv_cache_09_gb300.synth import workloads as W

    c = W.CONFIGS[5]
    wl = W.Workload(nseqs, c["H"], c["D"], [c["L"]] * nseqs, c["fmt"], c["sigma"], None, "permuted", seed,
                    0, c["name"])
    dw = DeviceWorkload(wl, device=dev)
    L = c["L"]
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
        raise RuntimeError(f"device status {rc} flags {flags:#x} in prefill-append")
    nbytes = wl.quantize_bytes(L) * nseqs
    del k_new, v_new, dw
    torch.cuda.empty_cache()
    return dict(ms=ms, bytes=nbytes, tokens=nseqs * L)


def measure_chunked_prefill(K, Wm, seed, dev):
    """chunked-prefill: kvq_prefill_attention of the last 512 of 8192 tokens of
    8 sequences (H=32, int4) over the cache that holds them."""
    import torch

    from quantized_kv_cache_09_gb300 import kvq
    from quantized_kv_cache_09_gb300.runner import DeviceWorkload
    from quantized_kv_cache_09_gb300.synth import workloads as W

    wl = W.make_workload(8, seed=seed)
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
    clocks = ClockSampler(dev.index or 0)
    clocks.start()
    time.sleep(0.3)
    t_wall0 = time.time()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for i in range(K):
        ev[i][0].record(stream)
        kvq.kvq_prefill_attention(dw.cache, q, cu, n, dw.block_table, dw.lens, dw.softmax_scale, out, workspace=ws)
        ev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    clocks.window = (t_wall0, time.time())
    ms = sum(a.elapsed_time(b) for a, b in ev) / K
    # end to end: the chunk's queries from pinned host memory, the output back
    pin_q = q.cpu().pin_memory()
    pin_o = torch.empty_like(pin_q).pin_memory()
    e_s, e_e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    Ke = max(1, K // 2)
    e_s.record(stream)
    for _ in range(Ke):
        q.copy_(pin_q, non_blocking=True)
        kvq.kvq_prefill_attention(dw.cache, q, cu, n, dw.block_table, dw.lens, dw.softmax_scale, out, workspace=ws)
        pin_o.copy_(out, non_blocking=True)
    e_e.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = e_s.elapsed_time(e_e) / Ke
    clocks.stop()
    rc, flags = kvq.kvq_get_device_status(dw.cache)
    if rc != 0:
        raise RuntimeError(f"device status {rc} flags {flags:#x} in chunked-prefill")
    res = dict(ms=ms, e2e_ms=e2e_ms, flops=wl.prefill_flops(), tokens=wl.B * n, B=wl.B, H=wl.H, Hq=wl.Hq, n=n,
               L=int(wl.lens[0]), qbytes=q.numel() * 2, clocks=clocks.summary())
    del dw, q, out
    torch.cuda.empty_cache()
    return res


def oracle_prefill_rate(seconds, seed):
    """The oracle's chunked-prefill rate on a sample of the workload: queries of
    sequence 0, every head, each over its causal prefix (binary64), one thread."""
    import numpy as np

    from oracle import oracle as orc
    from quantized_kv_cache_09_gb300.synth import workloads as W

    wl = W.make_workload(8, seed=seed)
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
    return done / el, 1, f"{done} chunk queries of sequence 0 (all {wl.Hq} heads, causal prefixes of ~{L} tokens, binary64) in {el:.1f} s"


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
    peak, peak_kind = measured_peak()

    K, Wm = args.steps, args.warmup
    if args.workload == "prefill-append":
        r = measure_prefill(K, max(Wm, 1), seed, dev, args.prefill_seqs)
        ms = max_over_ranks(pg, r["ms"], dev)
        gbs = r["bytes"] / (ms * 1e-3) / 1e9
        line = {"metric": METRIC, "value": whole_job_rate(world, r["bytes"] / 1e9, ms * 1e-3), "unit": "GB/s", "n_gpus": world, "steps": K, "warmup": Wm,
                "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "fp16 in, int4 codes out, fp32 math", "data": "synthetic (seeded generator in HBM)",
                "config": {"workload": "prefill-append", "new_tokens": r["tokens"], "H": 32, "D": 128,
                           "format": "int4-b64", "step": "one kvq_append of all new tokens"},
                "roofline": {"kernel": "append_kernel", "bound": "hbm", "achieved": gbs, "peak": peak,
                             "peak_kind": peak_kind, "unit": "GB/s", "frac": gbs / peak,
                             "traffic": ncu_traffic("append_kernel", "prefill-append"), "algorithmic_bytes_per_launch": r["bytes"]},
                "gpu_launches": K}
        if rank == 0:
            print(json.dumps(line), flush=True)
        if pg:
            pg.destroy_process_group()
        return

    if args.workload == "chunked-prefill":
        r = measure_chunked_prefill(K, max(Wm, 1), seed, dev)
        ms = max_over_ranks(pg, r["ms"], dev)
        e2e_ms = max_over_ranks(pg, r["e2e_ms"], dev)
        tflops = r["flops"] / (ms * 1e-3) / 1e12
        tpeak, tkind = measured_tensor_peak()
        line = {"metric": "chunked-prefill attention tokens/s over the quantized cache (tensor roofline)",
                "value": whole_job_rate(world, r["tokens"], ms * 1e-3), "unit": "tokens/s", "n_gpus": world,
                "steps": K, "warmup": Wm, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "int4 codes, fp16 MMA operands, fp32 accumulation",
                "data": "synthetic (seeded generator in HBM)",
                "config": {"workload": "chunked-prefill", "B": r["B"], "H": r["H"], "Hq": r["Hq"], "D": 128,
                           "context": r["L"], "chunk": r["n"], "format": "int4-b64",
                           "step": "one kvq_prefill_attention of every chunk query",
                           "l2": "codes (268 MB) larger than L2"},
                "tflops": tflops,
                "roofline": {"kernel": "prefill_attn_tc_kernel", "bound": "tensor", "achieved": tflops, "peak": tpeak,
                             "peak_kind": tkind, "unit": "TFLOP/s", "frac": tflops / tpeak,
                             "traffic": ncu_traffic("prefill_attn_tc_kernel", "chunked-prefill"),
                             "algorithmic_flops_per_launch": r["flops"]},
                "e2e": {"value": whole_job_rate(world, r["tokens"], e2e_ms * 1e-3), "unit": "tokens/s",
                        "h2d_bytes_per_step": r["qbytes"], "d2h_bytes_per_step": r["qbytes"]},
                "gpu_launches": K, "clocks": r["clocks"]}
        if rank == 0 and not args.no_cpu_baseline:
            rate, cores, desc = oracle_prefill_rate(args.cpu_seconds, args.seed)
            line["cpu_baseline"] = {"value": rate, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                                    "sample": desc}
        if rank == 0:
            print(json.dumps(line), flush=True)
        if pg:
            pg.destroy_process_group()
        return

    r = measure_decode(args.workload, K, Wm, seed, dev, pg)
    total_ms = max_over_ranks(pg, r["total_ms"], dev)
    e2e_ms = max_over_ranks(pg, r["e2e_ms"], dev)
    dec_ms = max_over_ranks(pg, r["dec_ms"], dev)
    app_ms = max_over_ranks(pg, r["app_ms"], dev)
    graph_ms = max_over_ranks(pg, r["graph_ms"], dev)
    B = r["B"]
    wl = r["wl"]
    achieved = r["dec_bytes"] / (dec_ms * 1e-3) / 1e9
    value = whole_job_rate(world, B * K, total_ms * 1e-3)
    lens = wl.lens
    ctx = (f"{int(lens[0]) + 1}..{int(lens[0]) + 64}" if r["aligned"] and lens.min() == lens.max()
           else f"{int(lens.min()) + 1}..{int(lens.max()) + 1} (sum {int(lens.sum()) + len(lens)})")
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K, "warmup": Wm,
            "ms_per_step": total_ms / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": FORMAT_NAMES[wl.fmt][0] + " codes, fp32 math",
            "data": "synthetic (seeded generator in HBM)",
            "config": {"workload": args.workload, "B": B, "H": r["H"], "Hq": r["Hq"], "D": r["D"], "context": ctx,
                       "format": FORMAT_NAMES[wl.fmt][1],
                       "step": "append 1 token + decode attention",
                       "parallelism": f"replicas x{world} (sequence-sharded, no collective)",
                       "l2": "inputs larger than L2" if r["dec_bytes"] > 129e6 else "fits in L2 (no flush)"},
            "kv_gb_per_s": achieved, "decode_us": dec_ms * 1e3, "append_us": app_ms * 1e3,
            "step_us_events_between_calls": r["split_ms"] / K * 1e3,
            "graph": {"ms_per_step": graph_ms / K, "value": whole_job_rate(world, B * K, graph_ms * 1e-3),
                      "unit": "tokens/s", "how": "one kvq_step_graph of 64 steps (append + decode each), replayed"},
            "roofline": {"kernel": "kvq_decode_attention (decode_split_kernel, merge fused)", "bound": "hbm",
                         "achieved": achieved, "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": ncu_traffic("decode_split_kernel", args.workload),
                         "algorithmic_bytes_per_launch": r["dec_bytes"]},
            "e2e": {"value": whole_job_rate(world, B * r["Ke"], e2e_ms * 1e-3), "unit": "tokens/s",
                    "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"]},
            "gpu_launches": r["launches"], "clocks": r["clocks"]}
    if args.extras and args.workload == "llama2-7b-layer":
        q = measure_prefill(5, 2, seed, dev, args.prefill_seqs)
        qms = max_over_ranks(pg, q["ms"], dev)
        qg = q["bytes"] / (qms * 1e-3) / 1e9
        line["quantize"] = {"workload": "prefill-append", "new_tokens": q["tokens"], "gb_per_s": qg,
                            "frac": qg / peak, "ms": qms}
    if rank == 0 and not args.no_cpu_baseline:
        rate, cores, desc = oracle_step_rate(args.cpu_seconds, args.seed, cfg=ORACLE_WORKLOADS.get(args.workload))
        line["cpu_baseline"] = {"value": rate, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": desc}
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
