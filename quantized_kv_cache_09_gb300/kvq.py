"""Python binding of the kvq C ABI (include/kvq.h): ctypes over lib/libkvq.so.

Argument marshalling only -- torch tensors in, raw device pointers, sizes and
the current CUDA stream out; every step of the work runs in the CUDA kernels.
There is no fallback: if the library is missing the first call raises.

With KVQ_NVTX set (to anything but 0) when this module is imported, every
entry point that launches work is wrapped in an NVTX range named after its C
function, for profilers that filter by range (ncu --nvtx --nvtx-include ...);
unset, the wrappers are the plain functions.
"""
import ctypes
import functools
import os

import torch

from . import build as _build

KVQ_INT4_B64 = 0
KVQ_INT8_PAGE = 1
KVQ_FP8_E4M3 = 2
HEAD_DIM = 128
PAGE_TOKENS = 64

KVQ_FLAG_BAD_PAGE = 0x1
KVQ_FLAG_BAD_LENGTH = 0x2
KVQ_FLAG_TIMEOUT = 0x4
KVQ_FLAG_NO_TAIL = 0x8
KVQ_FLAG_BAD_APPEND = 0x10
KVQ_FLAG_BAD_WORKSPACE = 0x20

STATUS_NAMES = {0: "KVQ_OK", 1: "KVQ_ERR_INVALID_ARG", 2: "KVQ_ERR_UNSUPPORTED", 3: "KVQ_ERR_CUDA",
                4: "KVQ_ERR_BAD_BLOCK_TABLE", 5: "KVQ_ERR_TIMEOUT", 6: "KVQ_ERR_WORKSPACE",
                7: "KVQ_ERR_BAD_LENGTH"}

# every symbol include/kvq.h declares
EXPORTS = ("kvq_quantize", "kvq_append", "kvq_decode_workspace_bytes", "kvq_decode_attention",
           "kvq_decode_workspace_bytes_gqa", "kvq_decode_attention_gqa",
           "kvq_decode_attention_noalloc", "kvq_prefill_workspace_bytes", "kvq_prefill_attention",
           "kvq_step_graph_create", "kvq_step_graph_update",
           "kvq_step_graph_launch", "kvq_step_graph_destroy", "kvq_get_device_status", "kvq_status_string",
           "kvq_version")
# every symbol include/kvq_testing.h declares (test hooks)
TESTING_EXPORTS = ("kvq_testing_set_decode_fault",)
NOALLOC_SCRATCH_BYTES = 4 << 20


NVTX = os.environ.get("KVQ_NVTX", "") not in ("", "0")


def _nvtx(fn=None, *, name=None):
    """The entry point inside an NVTX range named after its C function (only with KVQ_NVTX set)."""
    if fn is None:
        return lambda f: _nvtx(f, name=name)
    if not NVTX:
        return fn
    label = name or fn.__name__

    @functools.wraps(fn)
    def ranged(*args, **kwargs):
        torch.cuda.nvtx.range_push(label)
        try:
            return fn(*args, **kwargs)
        finally:
            torch.cuda.nvtx.range_pop()

    return ranged


class KvqError(RuntimeError):
    def __init__(self, status, what):
        self.status = status
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)} ({kvq_status_string(status)})")


class kvq_cache(ctypes.Structure):
    _fields_ = [("fmt", ctypes.c_int32), ("num_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("page_tokens", ctypes.c_int32), ("num_pages", ctypes.c_int32), ("max_seqs", ctypes.c_int32),
                ("k_codes", ctypes.c_void_p), ("v_codes", ctypes.c_void_p), ("k_scales", ctypes.c_void_p),
                ("v_scales", ctypes.c_void_p), ("k_tail", ctypes.c_void_p), ("v_tail", ctypes.c_void_p),
                ("status", ctypes.c_void_p)]


class kvq_step_args(ctypes.Structure):
    _fields_ = [("k_new", ctypes.c_void_p), ("v_new", ctypes.c_void_p), ("cu_seqlens", ctypes.c_void_p),
                ("seq_lens_before", ctypes.c_void_p), ("total_new_tokens", ctypes.c_int64),
                ("max_new_tokens", ctypes.c_int32), ("block_table", ctypes.c_void_p),
                ("max_blocks_per_seq", ctypes.c_int32), ("num_seqs", ctypes.c_int32), ("q", ctypes.c_void_p),
                ("num_q_heads", ctypes.c_int32), ("seq_lens", ctypes.c_void_p), ("softmax_scale", ctypes.c_float),
                ("out", ctypes.c_void_p), ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t)]


_lib = None


def library_path():
    return _build.LIB_KVQ


def lib():
    """The loaded C library; raises if it has not been built."""
    global _lib
    if _lib is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"kvq CUDA library not built ({path}); run __graft_entry__.build()")
        L = ctypes.CDLL(path)
        vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
        cp = ctypes.POINTER(kvq_cache)
        L.kvq_quantize.argtypes = [ctypes.c_int, vp, i64, i32, i32, vp, vp, vp]
        L.kvq_quantize.restype = ctypes.c_int
        L.kvq_append.argtypes = [cp, vp, vp, vp, vp, i32, vp, i32, i64, i32, vp]
        L.kvq_append.restype = ctypes.c_int
        L.kvq_decode_workspace_bytes.argtypes = [ctypes.c_int, i32, i32]
        L.kvq_decode_workspace_bytes.restype = sz
        L.kvq_decode_attention.argtypes = [cp, vp, vp, i32, vp, i32, ctypes.c_float, vp, vp, sz, vp]
        L.kvq_decode_attention.restype = ctypes.c_int
        L.kvq_decode_workspace_bytes_gqa.argtypes = [ctypes.c_int, i32, i32, i32]
        L.kvq_decode_workspace_bytes_gqa.restype = sz
        L.kvq_decode_attention_gqa.argtypes = [cp, vp, i32, vp, i32, vp, i32, ctypes.c_float, vp, vp, sz, vp]
        L.kvq_decode_attention_gqa.restype = ctypes.c_int
        L.kvq_decode_attention_noalloc.argtypes = [cp, vp, vp, i32, vp, i32, ctypes.c_float, vp, vp]
        L.kvq_decode_attention_noalloc.restype = ctypes.c_int
        L.kvq_prefill_workspace_bytes.argtypes = [i32, i32, i32]
        L.kvq_prefill_workspace_bytes.restype = sz
        L.kvq_prefill_attention.argtypes = [cp, vp, i32, vp, i64, i32, vp, i32, vp, i32, ctypes.c_float, vp, vp, sz,
                                            vp]
        L.kvq_prefill_attention.restype = ctypes.c_int
        ap = ctypes.POINTER(kvq_step_args)
        L.kvq_step_graph_create.argtypes = [cp, ap, i32, ctypes.POINTER(vp)]
        L.kvq_step_graph_create.restype = ctypes.c_int
        L.kvq_step_graph_update.argtypes = [vp, cp, ap, i32]
        L.kvq_step_graph_update.restype = ctypes.c_int
        L.kvq_step_graph_launch.argtypes = [vp, vp]
        L.kvq_step_graph_launch.restype = ctypes.c_int
        L.kvq_step_graph_destroy.argtypes = [vp]
        L.kvq_step_graph_destroy.restype = ctypes.c_int
        L.kvq_get_device_status.argtypes = [cp, vp, ctypes.POINTER(i32)]
        L.kvq_get_device_status.restype = ctypes.c_int
        L.kvq_status_string.argtypes = [ctypes.c_int]
        L.kvq_status_string.restype = ctypes.c_char_p
        L.kvq_version.argtypes = []
        L.kvq_version.restype = i32
        L.kvq_testing_set_decode_fault.argtypes = [ctypes.c_uint32, i32]
        L.kvq_testing_set_decode_fault.restype = ctypes.c_int
        _lib = L
    return _lib


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream, device=None):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _check(rc, what):
    if rc != 0:
        raise KvqError(rc, what)


def _cuda(t, dtype, name):
    if not (t.is_cuda and t.is_contiguous() and t.dtype == dtype):
        raise ValueError(f"{name} must be a contiguous CUDA {dtype} tensor")


def kvq_status_string(status):
    return lib().kvq_status_string(int(status)).decode()


def kvq_version():
    return lib().kvq_version()


def kvq_testing_set_decode_fault(wait_limit_us=0, skip_chunk=-1):
    """Test hook (include/kvq_testing.h): every later decode launch of the
    process waits at most wait_limit_us per copy (0: the default 0.5 s) and,
    when skip_chunk >= 0, leaves the copies of that chunk of the grid's first
    warp unissued, so its bounded wait runs out; (0, -1) restores the defaults."""
    _check(lib().kvq_testing_set_decode_fault(int(wait_limit_us), int(skip_chunk)), "kvq_testing_set_decode_fault")


@_nvtx
def kvq_quantize(fmt, x, codes, scales, stream=None):
    """x fp16 [T][H][128] -> codes uint8 [ceil(T/64)][H][64][64 or 128], scales fp32 [ceil(T/64)][H]."""
    _cuda(x, torch.float16, "x")
    _cuda(codes, torch.uint8, "codes")
    _cuda(scales, torch.float32, "scales")
    T, H, D = x.shape
    nb = (T + PAGE_TOKENS - 1) // PAGE_TOKENS
    rb = D // 2 if fmt == KVQ_INT4_B64 else D
    if codes.numel() < nb * H * PAGE_TOKENS * rb or scales.numel() < nb * H:
        raise ValueError("codes or scales too small")
    _check(lib().kvq_quantize(int(fmt), _ptr(x), T, H, D, _ptr(codes), _ptr(scales), _stream(stream, x.device)),
           "kvq_quantize")


@_nvtx
def kvq_append(cache, k_new, v_new, cu_seqlens, block_table, seq_lens_before, max_new_tokens, stream=None):
    """Append the rows of k_new/v_new fp16 [total][H][128] to every sequence (see kvq.h)."""
    _cuda(k_new, torch.float16, "k_new")
    _cuda(v_new, torch.float16, "v_new")
    for t, n in ((cu_seqlens, "cu_seqlens"), (block_table, "block_table"), (seq_lens_before, "seq_lens_before")):
        _cuda(t, torch.int32, n)
    B = seq_lens_before.numel()
    if cu_seqlens.numel() != B + 1 or block_table.dim() != 2 or block_table.shape[0] != B:
        raise ValueError("cu_seqlens must have num_seqs + 1 entries and block_table num_seqs rows")
    if k_new.shape != v_new.shape or k_new.dim() != 3:
        raise ValueError("k_new and v_new must both be [total][H][128]")
    _check(lib().kvq_append(ctypes.byref(cache.struct), _ptr(k_new), _ptr(v_new), _ptr(cu_seqlens),
                            _ptr(block_table), block_table.shape[1], _ptr(seq_lens_before), B,
                            k_new.shape[0], int(max_new_tokens), _stream(stream, k_new.device)), "kvq_append")


def kvq_decode_workspace_bytes(fmt, num_heads, head_dim=HEAD_DIM):
    return int(lib().kvq_decode_workspace_bytes(int(fmt), int(num_heads), int(head_dim)))


@_nvtx
def kvq_decode_attention(cache, q, block_table, seq_lens, softmax_scale, out, workspace, stream=None):
    """out fp16 [B][H][128] = decode attention of q fp16 [B][H][128] over the cache."""
    _cuda(q, torch.float16, "q")
    _cuda(out, torch.float16, "out")
    _cuda(block_table, torch.int32, "block_table")
    _cuda(seq_lens, torch.int32, "seq_lens")
    _cuda(workspace, torch.uint8, "workspace")
    B = q.shape[0]
    if out.shape != q.shape or seq_lens.numel() != B or block_table.dim() != 2 or block_table.shape[0] != B:
        raise ValueError("q/out/seq_lens/block_table shapes disagree")
    _check(lib().kvq_decode_attention(ctypes.byref(cache.struct), _ptr(q), _ptr(block_table), block_table.shape[1],
                                      _ptr(seq_lens), B, float(softmax_scale), _ptr(out), _ptr(workspace),
                                      workspace.numel(), _stream(stream, q.device)), "kvq_decode_attention")


def kvq_decode_workspace_bytes_gqa(fmt, num_kv_heads, num_q_heads, head_dim=HEAD_DIM):
    return int(lib().kvq_decode_workspace_bytes_gqa(int(fmt), int(num_kv_heads), int(num_q_heads), int(head_dim)))


@_nvtx
def kvq_decode_attention_gqa(cache, q, block_table, seq_lens, softmax_scale, out, workspace, stream=None):
    """out fp16 [B][Hq][128] = decode attention of q fp16 [B][Hq][128] over the
    cache, Hq = g * cache heads, query head i reading cache head i // g."""
    _cuda(q, torch.float16, "q")
    _cuda(out, torch.float16, "out")
    _cuda(block_table, torch.int32, "block_table")
    _cuda(seq_lens, torch.int32, "seq_lens")
    _cuda(workspace, torch.uint8, "workspace")
    B = q.shape[0]
    if out.shape != q.shape or seq_lens.numel() != B or block_table.dim() != 2 or block_table.shape[0] != B:
        raise ValueError("q/out/seq_lens/block_table shapes disagree")
    _check(lib().kvq_decode_attention_gqa(ctypes.byref(cache.struct), _ptr(q), q.shape[1], _ptr(block_table),
                                          block_table.shape[1], _ptr(seq_lens), B, float(softmax_scale), _ptr(out),
                                          _ptr(workspace), workspace.numel(), _stream(stream, q.device)),
           "kvq_decode_attention_gqa")


@_nvtx
def kvq_decode_attention_noalloc(cache, q, block_table, seq_lens, softmax_scale, out, stream=None):
    """kvq_decode_attention without a workspace, for callers that cannot
    allocate device memory when they run decode attention (a plugin whose
    execute step must not allocate, memory reserved up front by another
    allocator, a loop that cannot afford cudaMalloc's synchronisation): the
    scratch is a fixed 4 MiB array inside the library, shared by every call, so
    calls that may overlap on the GPU must be serialised by the caller; each
    call clears the array's split counters first on the same stream."""
    _cuda(q, torch.float16, "q")
    _cuda(out, torch.float16, "out")
    _cuda(block_table, torch.int32, "block_table")
    _cuda(seq_lens, torch.int32, "seq_lens")
    B = q.shape[0]
    if out.shape != q.shape or seq_lens.numel() != B or block_table.dim() != 2 or block_table.shape[0] != B:
        raise ValueError("q/out/seq_lens/block_table shapes disagree")
    _check(lib().kvq_decode_attention_noalloc(ctypes.byref(cache.struct), _ptr(q), _ptr(block_table),
                                              block_table.shape[1], _ptr(seq_lens), B, float(softmax_scale),
                                              _ptr(out), _stream(stream, q.device)), "kvq_decode_attention_noalloc")


def kvq_prefill_workspace_bytes(num_q_heads, num_seqs, max_q_per_seq):
    """Bytes of the optional kvq_prefill_attention workspace for these sizes
    on the current device (0: nothing to split)."""
    return int(lib().kvq_prefill_workspace_bytes(int(num_q_heads), int(num_seqs), int(max_q_per_seq)))


def prefill_workspace(num_q_heads, num_seqs, max_q_per_seq, device="cuda"):
    """A zero-filled workspace for kvq_prefill_attention (reusable by calls of
    at most these sizes, one call at a time)."""
    n = kvq_prefill_workspace_bytes(num_q_heads, num_seqs, max_q_per_seq)
    return torch.zeros(max(n, 16), dtype=torch.uint8, device=device)


@_nvtx
def kvq_prefill_attention(cache, q, cu_seqlens_q, max_q_per_seq, block_table, seq_lens, softmax_scale, out,
                          workspace=None, stream=None):
    """out fp16 [total][Hq][128] = causal attention of the chunk queries q fp16
    [total][Hq][128] over the cache: sequence b's chunk is its last
    cu[b+1] - cu[b] tokens (already appended); query i sits at position
    seq_lens[b] - n_b + i.  Hq = g * cache heads.  workspace (optional,
    prefill_workspace): the grid's last wave runs as key halves merged there."""
    _cuda(q, torch.float16, "q")
    _cuda(out, torch.float16, "out")
    for t, n in ((cu_seqlens_q, "cu_seqlens_q"), (block_table, "block_table"), (seq_lens, "seq_lens")):
        _cuda(t, torch.int32, n)
    B = seq_lens.numel()
    if (out.shape != q.shape or q.dim() != 3 or cu_seqlens_q.numel() != B + 1 or block_table.dim() != 2 or
            block_table.shape[0] != B):
        raise ValueError("q/out/cu_seqlens_q/seq_lens/block_table shapes disagree")
    _check(lib().kvq_prefill_attention(ctypes.byref(cache.struct), _ptr(q), q.shape[1], _ptr(cu_seqlens_q),
                                       q.shape[0], int(max_q_per_seq), _ptr(block_table), block_table.shape[1],
                                       _ptr(seq_lens), B, float(softmax_scale), _ptr(out),
                                       None if workspace is None else _ptr(workspace),
                                       0 if workspace is None else workspace.numel() * workspace.element_size(),
                                       _stream(stream, q.device)), "kvq_prefill_attention")


class StepGraph:
    """kvq_step_graph_*: a sequence of decode steps -- each appends one chunk of
    new tokens per sequence, then runs decode attention over the grown
    sequences -- captured once into one CUDA graph bound to these tensors;
    launch() replays them with whatever the tensors hold then.  Per-step inputs
    are written into the same tensors.

    steps: a list of tuples (cache, k_new, v_new, cu_seqlens, block_table,
    seq_lens_before, max_new_tokens, q, seq_lens, softmax_scale, out,
    workspace), run in order (e.g. a model's layers)."""

    def __init__(self, steps):
        self._h = None
        caches, args, keep = self._pack(steps)
        h = ctypes.c_void_p()
        _check(lib().kvq_step_graph_create(caches, args, len(steps), ctypes.byref(h)), "kvq_step_graph_create")
        self._h, self._caches, self._args, self._keep = h, caches, args, keep
        self._device = steps[0][7].device

    @staticmethod
    def _pack(steps):
        if not steps:
            raise ValueError("no steps")
        n = len(steps)
        caches = (kvq_cache * n)()
        args = (kvq_step_args * n)()
        keep = []
        for i, st in enumerate(steps):
            (cache, k_new, v_new, cu_seqlens, block_table, seq_lens_before, max_new_tokens, q, seq_lens,
             softmax_scale, out, workspace) = st
            for t, dt, name in ((k_new, torch.float16, "k_new"), (v_new, torch.float16, "v_new"),
                                (cu_seqlens, torch.int32, "cu_seqlens"), (block_table, torch.int32, "block_table"),
                                (seq_lens_before, torch.int32, "seq_lens_before"), (q, torch.float16, "q"),
                                (seq_lens, torch.int32, "seq_lens"), (out, torch.float16, "out"),
                                (workspace, torch.uint8, "workspace")):
                _cuda(t, dt, name)
            B = q.shape[0]
            if (out.shape != q.shape or seq_lens.numel() != B or seq_lens_before.numel() != B or
                    cu_seqlens.numel() != B + 1 or block_table.dim() != 2 or block_table.shape[0] != B or
                    k_new.shape != v_new.shape or k_new.dim() != 3):
                raise ValueError(f"step {i}: tensor shapes disagree")
            caches[i] = cache.struct
            args[i] = kvq_step_args(k_new.data_ptr(), v_new.data_ptr(), cu_seqlens.data_ptr(),
                                    seq_lens_before.data_ptr(), k_new.shape[0], int(max_new_tokens),
                                    block_table.data_ptr(), block_table.shape[1], B, q.data_ptr(), q.shape[1],
                                    seq_lens.data_ptr(), float(softmax_scale), out.data_ptr(), workspace.data_ptr(),
                                    workspace.numel())
            keep.append(st)
        return caches, args, keep

    def update(self, steps):
        """Rebind to other tensors (cudaGraphExecUpdate, or a new instance when the launches differ)."""
        caches, args, keep = self._pack(steps)
        _check(lib().kvq_step_graph_update(self._h, caches, args, len(steps)), "kvq_step_graph_update")
        self._caches, self._args, self._keep = caches, args, keep

    @_nvtx(name="kvq_step_graph_launch")
    def launch(self, stream=None):
        _check(lib().kvq_step_graph_launch(self._h, _stream(stream, self._device)), "kvq_step_graph_launch")

    def close(self):
        if self._h is not None:
            torch.cuda.synchronize(self._device)
            _check(lib().kvq_step_graph_destroy(self._h), "kvq_step_graph_destroy")
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def kvq_get_device_status(cache, stream=None):
    """(status, flags): reads and clears the cache's device status word (synchronises the stream)."""
    flags = ctypes.c_int32(0)
    rc = lib().kvq_get_device_status(ctypes.byref(cache.struct), _stream(stream), ctypes.byref(flags))
    return rc, flags.value


class PagedKVCache:
    """Device buffers of one paged cache (allocated with torch) and the
    kvq_cache descriptor that points at them."""

    def __init__(self, fmt, num_pages, num_heads, max_seqs=0, device="cuda", with_tail=True):
        self.fmt = int(fmt)
        self.num_pages = int(num_pages)
        self.num_heads = int(num_heads)
        self.max_seqs = int(max_seqs)
        rb = HEAD_DIM // 2 if self.fmt == KVQ_INT4_B64 else HEAD_DIM
        self.row_bytes = rb
        shape = (self.num_pages, self.num_heads, PAGE_TOKENS, rb)
        self.k_codes = torch.zeros(shape, dtype=torch.uint8, device=device)
        self.v_codes = torch.zeros(shape, dtype=torch.uint8, device=device)
        self.k_scales = torch.zeros((self.num_pages, self.num_heads), dtype=torch.float32, device=device)
        self.v_scales = torch.zeros((self.num_pages, self.num_heads), dtype=torch.float32, device=device)
        if with_tail and self.max_seqs > 0:
            tshape = (self.max_seqs, self.num_heads, PAGE_TOKENS, HEAD_DIM)
            self.k_tail = torch.zeros(tshape, dtype=torch.float16, device=device)
            self.v_tail = torch.zeros(tshape, dtype=torch.float16, device=device)
        else:
            self.k_tail = self.v_tail = None
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        self.struct = kvq_cache(self.fmt, self.num_heads, HEAD_DIM, PAGE_TOKENS, self.num_pages, self.max_seqs,
                                self.k_codes.data_ptr(), self.v_codes.data_ptr(), self.k_scales.data_ptr(),
                                self.v_scales.data_ptr(),
                                None if self.k_tail is None else self.k_tail.data_ptr(),
                                None if self.v_tail is None else self.v_tail.data_ptr(),
                                self.status.data_ptr())

    def rows_from(self, b0):
        """A descriptor of the same cache whose tail rows start at sequence row b0,
        for an append call that covers sequences b0, b0+1, ... of a larger batch."""
        view = type("PagedKVCacheRows", (), {})()
        step = self.num_heads * PAGE_TOKENS * HEAD_DIM * 2
        s = self.struct
        view.struct = kvq_cache(s.fmt, s.num_heads, s.head_dim, s.page_tokens, s.num_pages,
                                max(0, self.max_seqs - b0), s.k_codes, s.v_codes, s.k_scales, s.v_scales,
                                None if s.k_tail is None else s.k_tail + b0 * step,
                                None if s.v_tail is None else s.v_tail + b0 * step, s.status)
        return view

    def workspace(self, num_q_heads=None):
        n = kvq_decode_workspace_bytes_gqa(self.fmt, self.num_heads, num_q_heads or self.num_heads)
        if n <= 0:
            raise RuntimeError("kvq_decode_workspace_bytes returned 0")
        return torch.zeros(n, dtype=torch.uint8, device=self.k_codes.device)  # zero-filled before first use

    def bytes(self):
        t = [self.k_codes, self.v_codes, self.k_scales, self.v_scales]
        return sum(x.numel() * x.element_size() for x in t)


__all__ = ["KVQ_INT4_B64", "KVQ_INT8_PAGE", "KVQ_FP8_E4M3", "HEAD_DIM", "PAGE_TOKENS", "EXPORTS", "KvqError", "kvq_cache",
           "PagedKVCache", "lib", "library_path", "kvq_quantize", "kvq_append", "kvq_decode_workspace_bytes",
           "kvq_decode_attention", "kvq_decode_attention_noalloc", "kvq_get_device_status", "kvq_status_string",
           "kvq_version", "StepGraph", "kvq_step_args", "kvq_prefill_attention"]
