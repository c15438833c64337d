"""The C ABI without a GPU: the library loads, exports every function
include/kvq.h declares, and rejects bad arguments on the host before any
CUDA call."""
import ctypes
import os
import re

import pytest

from quantized_kv_cache_09_gb300 import build, kvq

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions(header="kvq.h"):
    with open(os.path.join(ROOT, "include", header)) as fh:
        src = fh.read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(kvq_[a-z_0-9]+)\s*\(", src)))


def test_library_builds_and_exports_every_declared_symbol():
    build.build()
    lib = kvq.lib()
    names = _declared_functions()
    assert set(names) == set(kvq.EXPORTS), names
    testing = _declared_functions("kvq_testing.h")
    assert set(testing) == set(kvq.TESTING_EXPORTS), testing
    headers = sorted(f for f in os.listdir(os.path.join(ROOT, "include")) if f.endswith(".h"))
    assert headers == ["kvq.h", "kvq_testing.h"], headers
    for n in names + testing:
        assert hasattr(lib, n), n
    assert kvq.kvq_version() == 100


def test_testing_hook_validates_on_the_host():
    lib = kvq.lib()
    assert lib.kvq_testing_set_decode_fault(0, -2) == 1
    assert lib.kvq_testing_set_decode_fault(0, -1) == 0   # the defaults


def test_status_strings():
    for s in range(8):
        assert kvq.kvq_status_string(s) != "unknown status"
    assert kvq.kvq_status_string(99) == "unknown status"


def test_host_validation_without_gpu():
    lib = kvq.lib()
    # unsupported head_dim, unknown format, bad sizes, null pointers: no CUDA call is made
    assert lib.kvq_quantize(0, ctypes.c_void_p(16), 64, 2, 64, ctypes.c_void_p(16), ctypes.c_void_p(16), None) == 2
    assert lib.kvq_quantize(7, ctypes.c_void_p(16), 64, 2, 128, ctypes.c_void_p(16), ctypes.c_void_p(16), None) == 2
    assert lib.kvq_quantize(0, None, 64, 2, 128, ctypes.c_void_p(16), ctypes.c_void_p(16), None) == 1
    assert lib.kvq_quantize(0, ctypes.c_void_p(8), 64, 2, 128, ctypes.c_void_p(16), ctypes.c_void_p(16), None) == 1
    assert lib.kvq_quantize(0, None, 0, 2, 128, None, None, None) == 0   # empty is a no-op
    assert lib.kvq_quantize(0, None, -1, 2, 128, None, None, None) == 1
    c = kvq.kvq_cache(0, 2, 128, 64, 4, 1, 16, 16, 16, 16, None, None, None)
    assert lib.kvq_append(ctypes.byref(c), None, None, None, None, 1, None, 1, 0, 1, None) == 1
    c2 = kvq.kvq_cache(0, 2, 96, 64, 4, 1, 16, 16, 16, 16, None, None, None)
    assert lib.kvq_append(ctypes.byref(c2), None, None, None, None, 1, None, 1, 0, 1, None) == 2
    c3 = kvq.kvq_cache(0, 2, 128, 32, 4, 1, 16, 16, 16, 16, None, None, None)
    assert lib.kvq_decode_attention(ctypes.byref(c3), None, None, 1, None, 1, 0.1, None, None, 0, None) == 2
    assert lib.kvq_decode_attention(None, None, None, 1, None, 1, 0.1, None, None, 0, None) == 1
    assert lib.kvq_decode_workspace_bytes(0, 2, 64) == 0
    # tails given for K only
    c4 = kvq.kvq_cache(0, 2, 128, 64, 4, 1, 16, 16, 16, 16, 32, None, None)
    assert lib.kvq_append(ctypes.byref(c4), None, None, None, None, 1, None, 1, 0, 1, None) == 1


def test_oracle_and_product_share_no_code():
    """The oracle directory and the CUDA library sources include nothing of each other."""
    csrc = os.path.join(ROOT, "quantized_kv_cache_09_gb300", "csrc")
    for f in os.listdir(csrc):
        with open(os.path.join(csrc, f)) as fh:
            text = fh.read()
        assert "oracle" not in text.lower(), f
    for f in os.listdir(os.path.join(ROOT, "oracle")):
        if f.endswith((".c", ".py")):
            with open(os.path.join(ROOT, "oracle", f)) as fh:
                text = fh.read()
            assert "quantized_kv_cache_09_gb300" not in text and "kvq_synth" not in text, f


def _cache(fmt=0, H=2, D=128, page=64, pages=4, k=16, v=16, ks=16, vs=16, kt=None, vt=None):
    return kvq.kvq_cache(fmt, H, D, page, pages, 1, k, v, ks, vs, kt, vt, None)


def test_grouped_decode_host_validation_without_gpu():
    """kvq_decode_attention_gqa and its workspace query reject bad arguments on
    the host, before any CUDA call: the cache description, the group (query
    heads a multiple of the cache heads, at most 1024 per cache head), sizes,
    the softmax scale, null and misaligned buffers; zero sequences is a no-op."""
    lib = kvq.lib()
    d = lib.kvq_decode_attention_gqa
    P = ctypes.c_void_p(16)

    def call(c, hq, mb=4, n=1, scale=0.1, q=P, out=P):
        return d(ctypes.byref(c), q, hq, P, mb, P, n, scale, out, P, 1 << 20, None)

    c = _cache(H=2)
    assert call(c, 3) == 1                      # 3 query heads over 2 cache heads
    assert call(c, 0) == 1
    assert call(c, -2) == 1
    assert call(c, 2 * 1025) == 2               # 1025 query heads per cache head
    assert call(c, 2, scale=float("inf")) == 1
    assert call(c, 2, scale=float("nan")) == 1
    assert call(c, 2, mb=0) == 1
    assert call(c, 2, mb=(1 << 22) + 1) == 2    # the split's 24-bit unit count
    assert call(c, 2, mb=1 << 22, n=64) == 2    # one launch's units in 32 bits
    assert call(c, 2, n=-1) == 1
    assert call(c, 2, n=0, q=None, out=None) == 0
    assert call(c, 2, q=None) == 1
    assert call(c, 2, q=ctypes.c_void_p(24)) == 1
    assert call(c, 2, out=ctypes.c_void_p(40)) == 1
    assert call(c, 16, q=None) == 1             # grouped heads take the same checks
    # the cache description
    assert call(_cache(fmt=7), 2) == 2
    assert call(_cache(D=64), 2) == 2
    assert call(_cache(page=32), 2) == 2
    assert call(_cache(pages=0), 2) == 1
    assert call(_cache(H=0), 2) == 1
    assert call(_cache(k=None), 2) == 1
    assert call(_cache(vs=None), 2) == 1
    assert call(_cache(v=24), 2) == 1           # misaligned codes
    assert call(_cache(kt=32, vt=None), 2) == 1
    assert call(_cache(kt=32, vt=40), 2) == 1   # misaligned tail
    assert d(None, P, 2, P, 4, P, 1, 0.1, P, P, 1 << 20, None) == 1
    # workspace sizes: 0 for anything unsupported, without asking the device
    w = lib.kvq_decode_workspace_bytes_gqa
    assert w(0, 2, 3, 128) == 0
    assert w(0, 2, 2 * 1025, 128) == 0
    assert w(0, 0, 2, 128) == 0
    assert w(9, 2, 2, 128) == 0
    assert w(1, 2, 4, 96) == 0


def test_prefill_host_validation_without_gpu():
    lib = kvq.lib()
    f = lib.kvq_prefill_attention
    P = ctypes.c_void_p(16)

    def call(c, hq, total=8, max_q=8, mb=4, n=1, scale=0.1, q=P, out=P):
        return f(ctypes.byref(c), q, hq, P, total, max_q, P, mb, P, n, scale, out, None, 0, None)

    c = _cache(H=2)
    assert call(c, 3) == 1
    assert call(c, 0) == 1
    assert call(c, 2, total=-1) == 1
    assert call(c, 2, max_q=-1) == 1
    assert call(c, 2, n=-1) == 1
    assert call(c, 2, mb=0) == 1
    assert call(c, 2, scale=float("nan")) == 1
    assert call(c, 2, total=0, q=None, out=None) == 0
    assert call(c, 2, n=0, q=None, out=None) == 0
    assert call(c, 2, max_q=0, q=None, out=None) == 0
    assert call(c, 2, q=None) == 1
    assert call(c, 2, out=ctypes.c_void_p(8)) == 1
    assert call(c, 2, n=65536) == 2
    assert call(_cache(fmt=5), 2) == 2
    assert call(_cache(page=128), 2) == 2
    assert lib.kvq_prefill_workspace_bytes(0, 1, 1) == 0
    assert lib.kvq_prefill_workspace_bytes(2, 0, 1) == 0
    assert lib.kvq_prefill_workspace_bytes(2, 1, -1) == 0


def test_graph_and_noalloc_null_handles_without_gpu():
    lib = kvq.lib()
    c = _cache()
    a = kvq.kvq_step_args()
    h = ctypes.c_void_p(0)
    assert lib.kvq_step_graph_create(ctypes.byref(c), ctypes.byref(a), 1, None) == 1
    assert lib.kvq_step_graph_create(ctypes.byref(c), ctypes.byref(a), 0, ctypes.byref(h)) == 1
    assert h.value is None                      # nothing handed out on a rejected call
    assert lib.kvq_step_graph_create(None, ctypes.byref(a), 1, ctypes.byref(h)) == 1
    assert lib.kvq_step_graph_update(None, ctypes.byref(c), ctypes.byref(a), 1) == 1
    assert lib.kvq_step_graph_launch(None, None) == 1
    assert lib.kvq_step_graph_destroy(None) == 0
    assert lib.kvq_decode_attention_noalloc(None, None, None, 1, None, 1, 0.1, None, None) == 1
    flags = ctypes.c_int32(0)
    assert lib.kvq_get_device_status(None, None, ctypes.byref(flags)) == 1
