"""Block-quantized KV cache and decode attention for one GB300 GPU.

The compute path is the CUDA library behind include/kvq.h (lib/libkvq.so);
`kvq` is its Python binding and `synth` the seeded synthetic-input generator.
"""
from . import kvq  # noqa: F401
from .kvq import (KVQ_FP8_E4M3, KVQ_INT4_B64, KVQ_INT8_PAGE, PagedKVCache, StepGraph, kvq_append,  # noqa: F401
                  kvq_decode_attention, kvq_decode_attention_gqa, kvq_decode_workspace_bytes,
                  kvq_decode_workspace_bytes_gqa, kvq_get_device_status, kvq_prefill_attention,
                  kvq_prefill_workspace_bytes, kvq_quantize, prefill_workspace)
