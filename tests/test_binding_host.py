"""The Python binding without a GPU: there is no CPU fallback anywhere on the
product path.  Host (CPU) tensors are refused before the library is called,
wrong dtypes and shapes are refused, and a missing CUDA library is an error on
first use rather than a silent switch to other code."""
import pytest
import torch

from quantized_kv_cache_09_gb300 import kvq


def _h(*shape, dtype=torch.float16):
    return torch.zeros(*shape, dtype=dtype)


def test_host_tensors_are_refused():
    x = _h(64, 2, 128)
    i32 = _h(2, dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA"):
        kvq.kvq_quantize(kvq.KVQ_INT4_B64, x, _h(1, 2, 64, 64, dtype=torch.uint8), _h(1, 2, dtype=torch.float32))
    with pytest.raises(ValueError, match="CUDA"):
        kvq.kvq_append(None, x, x, _h(3, dtype=torch.int32), _h(2, 1, dtype=torch.int32), i32, 1)
    q = _h(2, 2, 128)
    for fn in (kvq.kvq_decode_attention, kvq.kvq_decode_attention_gqa):
        with pytest.raises(ValueError, match="CUDA"):
            fn(None, q, _h(2, 1, dtype=torch.int32), i32, 0.1, q.clone(), _h(16, dtype=torch.uint8))
    with pytest.raises(ValueError, match="CUDA"):
        kvq.kvq_decode_attention_noalloc(None, q, _h(2, 1, dtype=torch.int32), i32, 0.1, q.clone())
    with pytest.raises(ValueError, match="CUDA"):
        kvq.kvq_prefill_attention(None, q, _h(3, dtype=torch.int32), 1, _h(2, 1, dtype=torch.int32), i32, 0.1,
                                  q.clone())


def test_missing_library_is_an_error(monkeypatch, tmp_path):
    monkeypatch.setattr(kvq, "_lib", None)
    monkeypatch.setattr(kvq, "library_path", lambda: str(tmp_path / "libkvq.so"))
    with pytest.raises(RuntimeError, match="not built"):
        kvq.lib()
    with pytest.raises(RuntimeError, match="not built"):
        kvq.kvq_version()
