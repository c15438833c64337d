"""The device build of the input generator produces the same bits as the host
build (so full-size inputs generated in HBM are the ones the oracle sees)."""
import numpy as np
import pytest
import torch

from quantized_kv_cache_09_gb300 import synth
from quantized_kv_cache_09_gb300.synth import workloads as W

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("cfg", [1, 2, 3, 5])
def test_device_equals_host(cuda_ok, cfg):
    wl = W.make_workload(cfg)
    for which in ("k", "v"):
        for b, t0, t1 in ((0, 0, 70), (wl.B - 1, 1000, 1003)):
            x = torch.empty((t1 - t0, wl.H, wl.D), dtype=torch.float16, device="cuda")
            wl.kv_device(which, b, t0, t1, x)
            assert np.array_equal(x.cpu().numpy().view(np.uint16), wl.kv_host(which, b, t0, t1))
    q = torch.empty((wl.B, wl.H, wl.D), dtype=torch.float16, device="cuda")
    wl.q_device(q, 7)
    assert np.array_equal(q.cpu().numpy().view(np.uint16), wl.q_host(7))


def test_large_fill_matches(cuda_ok):
    n = 3 * (1 << 22) + 5
    s = synth.stream_id(synth.K_HIST, 11)
    x = torch.empty(n, dtype=torch.float16, device="cuda")
    synth.fill_f16_device(x, 4, s, 12345, 1.5)
    assert np.array_equal(x.cpu().numpy().view(np.uint16), synth.fill_f16_host(n, 4, s, 12345, 1.5))
