"""The binding's optional NVTX ranges: with KVQ_NVTX set at import, every entry
point that launches work is wrapped (a range named after its C function);
without it the entry points are the plain functions.  CPU only: wrapping is
decided at import, nothing is launched."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
LAUNCHING = ("kvq_quantize", "kvq_append", "kvq_decode_attention", "kvq_decode_attention_gqa",
             "kvq_decode_attention_noalloc", "kvq_prefill_attention")


def _probe(env_value):
    env = dict(os.environ)
    env.pop("KVQ_NVTX", None)
    if env_value is not None:
        env["KVQ_NVTX"] = env_value
    code = ("from quantized_kv_cache_09_gb300 import kvq\n"
            f"names = {LAUNCHING!r}\n"
            "w = [hasattr(getattr(kvq, n), '__wrapped__') for n in names]\n"
            "w.append(hasattr(kvq.StepGraph.launch, '__wrapped__'))\n"
            "print(int(kvq.NVTX), sum(w), len(w), kvq.kvq_append.__name__)\n")
    out = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True, text=True, check=True)
    return out.stdout.split()


def test_entry_points_wrapped_with_kvq_nvtx():
    on, wrapped, total, name = _probe("1")
    assert on == "1" and wrapped == total and name == "kvq_append"


def test_entry_points_plain_without_kvq_nvtx():
    for value in (None, "0"):
        on, wrapped, _, _ = _probe(value)
        assert on == "0" and wrapped == "0"


_RUN = """
import sys, numpy as np, torch
from quantized_kv_cache_09_gb300 import kvq
from quantized_kv_cache_09_gb300.runner import DeviceWorkload
from quantized_kv_cache_09_gb300.synth import workloads as W
wl = W.make_workload(1, extra_tokens=64)
dw = DeviceWorkload(wl)
dw.prefill()
q = torch.empty((wl.B, wl.H, 128), dtype=torch.float16, device="cuda")
wl.q_device(q, 0)
out = torch.empty_like(q)
kvq.kvq_decode_attention(dw.cache, q, dw.block_table, dw.lens, dw.softmax_scale, out, dw.workspace)
torch.cuda.synchronize()
np.save(sys.argv[1], out.cpu().numpy())
"""



@pytest.mark.gpu
def test_ranges_around_real_calls_change_nothing(cuda_ok, tmp_path):
    """The tiny workload's decode with and without the NVTX ranges gives the same bits."""
    import numpy as np
    outs = []
    for value in ("1", None):
        env = dict(os.environ)
        env.pop("KVQ_NVTX", None)
        if value is not None:
            env["KVQ_NVTX"] = value
        f = tmp_path / f"out{len(outs)}.npy"
        subprocess.run([sys.executable, "-c", _RUN, str(f)], cwd=ROOT, env=env, check=True)
        outs.append(np.load(f))
    assert np.array_equal(outs[0], outs[1]) and np.isfinite(outs[0].astype(np.float32)).all()
