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
