"""The multi-rank path of the benchmark on CPU (gloo, world size 2).

Decode attention shards by sequence: every rank owns its own batch (weak
scaling, seed = base + rank) and no data-path step exchanges anything; the
only collective is the timing reduction (max over ranks).  Two gloo ranks
each run the oracle on their own small batch, reduce their times, and check
that (a) both ranks agree on the slowest time, (b) the whole-job rate counts
every rank's units, and (c) each rank's outputs equal those of a single
process that computes the same seed alone -- i.e. sharding changes nothing.
"""
import math
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_batch(seed):
    from oracle import oracle as orc
    from quantized_kv_cache_09_gb300.synth import workloads as W
    wl = W.Workload(2, 3, 128, [70, 129], 0, 1.0, None, "permuted", seed=seed)
    rb = orc.row_bytes(wl.fmt, wl.D)
    kc = np.zeros((wl.num_pages, wl.H, 64, rb), np.uint8)
    vc = np.zeros_like(kc)
    ks = np.zeros((wl.num_pages, wl.H), np.float32)
    vs = np.zeros_like(ks)
    for b in range(wl.B):
        orc.quantize_into_pages(wl.fmt, wl.kv_host("k", b, 0, int(wl.lens[b])), wl.block_table[b], kc, ks)
        orc.quantize_into_pages(wl.fmt, wl.kv_host("v", b, 0, int(wl.lens[b])), wl.block_table[b], vc, vs)
    return orc.decode_attention(wl.fmt, kc, vc, ks, vs, wl.block_table, wl.lens, wl.q_host(0),
                                1 / math.sqrt(wl.D))


def _worker(rank, world, port, results):
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        seed = bench.rank_seed(5, rank)
        out = _rank_batch(seed)
        my_ms = 10.0 + 5.0 * rank                # a stand-in time per rank
        slowest = bench.max_over_ranks(dist, my_ms, "cpu")
        rate = bench.whole_job_rate(world, 2 * 7, slowest * 1e-3)
        results[rank] = (seed, out, slowest, rate)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_shard_by_sequence():
    world = 2
    port = _free_port()
    mgr = mp.Manager()
    results = mgr.dict()
    mp.spawn(_worker, args=(world, port, results), nprocs=world, join=True)
    assert sorted(results.keys()) == [0, 1]
    seeds = [results[r][0] for r in range(world)]
    assert seeds == [5, 6]
    for r in range(world):
        seed, out, slowest, rate = results[r]
        assert slowest == 15.0                   # every rank sees the slowest rank's time
        assert rate == pytest.approx(world * 14 / 15e-3)
        np.testing.assert_array_equal(out, _rank_batch(seed))   # sharding changes nothing
    assert not np.array_equal(results[0][1], results[1][1])


def test_single_process_helpers():
    assert bench.max_over_ranks(None, 3.5, "cpu") == 3.5
    assert bench.whole_job_rate(1, 8, 0.5) == 16.0
    assert bench.rank_seed(0, 3) == 3
