"""The synthetic workloads: shapes, value distributions and structure.

  tiny             B=2, H=4, L=256, int4, K/V/q ~ N(0,1), contiguous cache,
                   quantize then one decode step (append 1 token, attend over 257)
  llama2-7b-layer  B=8, H=32, L=8192, int4, K/V ~ N(0,1) with 4 channels per
                   head (separately for K and V, the same for every token and
                   sequence) scaled x10, contiguous cache; decode
  long-context     B=16, H=32, L=32768, int4, each (head, channel) an outlier
                   x10 with probability 0.01, contiguous cache; decode
  paged-int8       64 sequences, L uniform in [512, 16384], H=32, int8 with a
                   per-(page, head) scale, 64-token pages in a randomly
                   permuted block table; decode
  prefill-append   262144 new tokens as 64 sequences x 4096, H=32, K/V ~
                   N(0, 1.5^2), int4, randomly permuted pages; append/quantize
  llama3-8b-layer-gqa  B=32, 8 cache heads, 32 query heads (groups of 4),
                   L=8192, int4, otherwise as llama2-7b-layer; decode with
                   grouped query heads.  The batch of 32 puts the same KV
                   bytes as llama2-7b-layer behind one step (268 MB, more
                   than L2)
  llama2-7b-layer-fp8  as llama2-7b-layer, FP8 E4M3 codes (one byte per
                   element, 537 MB of K and V per step); decode
  chunked-prefill  B=8, H=32, L=8192 of which the last 512 tokens are a new
                   chunk (already appended), int4, K/V as llama2-7b-layer,
                   chunk queries ~ N(0,1); causal attention of the chunk
  mqa-32k          B=64, 1 cache head, 32 query heads (multi-query decode, the
                   pages' MLA decode absorbed into MQA), L=32768, int4, K/V as
                   llama2-7b-layer, randomly permuted pages; 268 MB of codes

D = 128 and 64-token blocks throughout.  q ~ N(0, 1).  All values are fp16.
"""
import numpy as np

from . import (BLOCK_TABLE, CHUNK_QUERY, K_HIST, K_OUTLIER, LENGTHS, QUERY, V_HIST, V_OUTLIER, fill_f16_device,
               fill_f16_host, outliers_bernoulli, outliers_per_head, permutation, stream_id,
               uniform_int)

INT4 = 0
INT8 = 1
FP8 = 2
PAGE = 64

RECIPES = {
    1: dict(name="tiny", B=2, H=4, D=128, L=256, fmt=INT4, sigma=1.0, outliers=None, table="contiguous"),
    2: dict(name="llama2-7b-layer", B=8, H=32, D=128, L=8192, fmt=INT4, sigma=1.0,
            outliers=("per_head", 4, 10.0), table="contiguous"),
    3: dict(name="long-context", B=16, H=32, D=128, L=32768, fmt=INT4, sigma=1.0,
            outliers=("bernoulli", 0.01, 10.0), table="contiguous"),
    4: dict(name="paged-int8", B=64, H=32, D=128, L=("uniform", 512, 16384), fmt=INT8, sigma=1.0,
            outliers=None, table="permuted"),
    5: dict(name="prefill-append", B=64, H=32, D=128, L=4096, fmt=INT4, sigma=1.5, outliers=None,
            table="permuted"),
    # grouped query heads: 32 query heads
    # over 8 cache heads, the Llama-3-8B attention shape
    6: dict(name="llama3-8b-layer-gqa", B=32, H=8, Hq=32, D=128, L=8192, fmt=INT4, sigma=1.0,
            outliers=("per_head", 4, 10.0), table="contiguous"),
    # the FP8 E4M3 cache on the 7B-layer shape
    7: dict(name="llama2-7b-layer-fp8", B=8, H=32, D=128, L=8192, fmt=FP8, sigma=1.0,
            outliers=("per_head", 4, 10.0), table="contiguous"),
    # chunked prefill: the last 512 of 8192 tokens attend causally over the cache
    8: dict(name="chunked-prefill", B=8, H=32, D=128, L=8192, chunk=512, fmt=INT4, sigma=1.0,
            outliers=("per_head", 4, 10.0), table="contiguous"),
    # multi-query decode (MLA absorbed into MQA): one cache head serves 32 query
    # heads; 64 sequences of 32K tokens put 268 MB of codes behind one step
    9: dict(name="mqa-32k", B=64, H=1, Hq=32, D=128, L=32768, fmt=INT4, sigma=1.0,
            outliers=("per_head", 4, 10.0), table="permuted"),
    # 64 query heads over 8 cache heads (g = 8), the Llama-3-70B attention shape,
    # with the 8B layer's batch and context: the same 268 MB of codes per step
    10: dict(name="llama3-70b-layer-gqa", B=32, H=8, Hq=64, D=128, L=8192, fmt=INT4, sigma=1.0,
             outliers=("per_head", 4, 10.0), table="contiguous"),
    # the same shape over an FP8 E4M3 cache (537 MB of codes per step)
    11: dict(name="llama3-70b-layer-gqa-fp8", B=32, H=8, Hq=64, D=128, L=8192, fmt=FP8, sigma=1.0,
             outliers=("per_head", 4, 10.0), table="contiguous"),
}


class Workload:
    """One seeded instance of a workload.

    lens[b]      tokens already in the cache for sequence b (the decode history,
                 or for prefill-append the tokens to append)
    extra_tokens room reserved per sequence beyond lens (decode steps)
    block_table  int32 [B][max_blocks]; num_pages = B * max_blocks
    """

    def __init__(self, B, H, D, lens, fmt, sigma=1.0, outliers=None, table="contiguous", seed=0,
                 extra_tokens=0, name="custom", q_heads=None, chunk=0):
        self.name = name
        self.chunk = int(chunk)  # new tokens per sequence for chunked prefill (the last `chunk` of lens)
        self.B, self.H, self.D = int(B), int(H), int(D)
        self.Hq = self.H if q_heads is None else int(q_heads)  # query heads (a multiple of the cache heads H)
        self.lens = np.asarray(lens, dtype=np.int32).reshape(self.B)
        self.fmt = int(fmt)
        self.sigma = float(sigma)
        self.seed = int(seed)
        self.extra_tokens = int(extra_tokens)
        cap = int(self.lens.max(initial=0)) + self.extra_tokens
        self.max_blocks = max(1, (cap + PAGE - 1) // PAGE)
        self.num_pages = self.B * self.max_blocks
        if table == "contiguous":
            self.block_table = np.arange(self.num_pages, dtype=np.int32).reshape(self.B, self.max_blocks)
        elif table == "permuted":
            self.block_table = permutation(self.num_pages, self.seed,
                                           stream_id(BLOCK_TABLE)).reshape(self.B, self.max_blocks)
        else:
            raise ValueError(table)
        self.table = table
        self.outlier_mult = 1.0
        self.k_mask = self.v_mask = None
        if outliers is not None:
            kind, param, mult = outliers
            self.outlier_mult = float(mult)
            if kind == "per_head":
                self.k_mask = outliers_per_head(self.H, self.D, int(param), self.seed, stream_id(K_OUTLIER))
                self.v_mask = outliers_per_head(self.H, self.D, int(param), self.seed, stream_id(V_OUTLIER))
            elif kind == "bernoulli":
                self.k_mask = outliers_bernoulli(self.H, self.D, float(param), self.seed, stream_id(K_OUTLIER))
                self.v_mask = outliers_bernoulli(self.H, self.D, float(param), self.seed, stream_id(V_OUTLIER))
            else:
                raise ValueError(kind)
        self._dev_masks = {}

    # ---- host (numpy) -------------------------------------------------
    def kv_host(self, which, b, t0, t1):
        """fp16 bits [t1-t0][H][D] of the key ('k') or value ('v') history of sequence b."""
        kind, mask = (K_HIST, self.k_mask) if which == "k" else (V_HIST, self.v_mask)
        n = (t1 - t0) * self.H * self.D
        x = fill_f16_host(n, self.seed, stream_id(kind, b), t0 * self.H * self.D, self.sigma, mask,
                          self.outlier_mult)
        return x.reshape(t1 - t0, self.H, self.D)

    def kv_host_head(self, which, b, h, t0, t1):
        """fp16 bits [t1-t0][1][D] of head h alone of the key ('k') or value ('v')
        history of sequence b: the same bits as kv_host(...)[:, h:h+1, :],
        generated one D-element row per token."""
        kind, mask = (K_HIST, self.k_mask) if which == "k" else (V_HIST, self.v_mask)
        out = np.empty((t1 - t0, 1, self.D), dtype=np.uint16)
        sid = stream_id(kind, b)
        for t in range(t0, t1):
            out[t - t0, 0] = fill_f16_host(self.D, self.seed, sid, (t * self.H + h) * self.D, self.sigma, mask,
                                           self.outlier_mult)
        return out

    def q_host(self, step=0):
        """fp16 bits [B][Hq][D] of the query of decode step `step`."""
        n = self.B * self.Hq * self.D
        return fill_f16_host(n, self.seed, stream_id(QUERY, step), 0, 1.0).reshape(self.B, self.Hq, self.D)

    # ---- device (torch) -----------------------------------------------
    def _mask_dev(self, which, device):
        import torch
        key = (which, str(device))
        mask = self.k_mask if which == "k" else self.v_mask
        if mask is None:
            return None
        if key not in self._dev_masks:
            self._dev_masks[key] = torch.from_numpy(mask.reshape(-1).copy()).to(device)
        return self._dev_masks[key]

    def kv_device(self, which, b, t0, t1, out):
        """Fill out (CUDA, 2-byte elements, (t1-t0)*H*D elements) with the same bits as kv_host."""
        kind = K_HIST if which == "k" else V_HIST
        assert out.numel() == (t1 - t0) * self.H * self.D
        return fill_f16_device(out, self.seed, stream_id(kind, b), t0 * self.H * self.D, self.sigma,
                               self._mask_dev(which, out.device), self.outlier_mult)

    def chunk_q_host(self, b, i0, i1):
        """fp16 bits [i1-i0][Hq][D] of queries i0 .. i1-1 of sequence b's prefill chunk."""
        n = (i1 - i0) * self.Hq * self.D
        return fill_f16_host(n, self.seed, stream_id(CHUNK_QUERY, b), i0 * self.Hq * self.D,
                             1.0).reshape(i1 - i0, self.Hq, self.D)

    def chunk_q_device(self, out, b, i0=0):
        """Fill out (fp16, [n][Hq][D]) with queries i0 .. i0+n-1 of sequence b's prefill chunk."""
        return fill_f16_device(out, self.seed, stream_id(CHUNK_QUERY, b), i0 * self.Hq * self.D, 1.0)

    def prefill_flops(self, chunk=None):
        """Algorithmic flops of chunked-prefill attention: 4 D per (query head,
        causal key) -- QK and PV, a multiply and an add each -- summed over the
        last `chunk` queries of every sequence (query i sees L - n + i + 1 keys)."""
        n = self.chunk if chunk is None else int(chunk)
        keys = sum(int(L) * n - n * (n - 1) // 2 for L in self.lens)
        return 4 * self.D * self.Hq * keys

    def q_device(self, out, step=0):
        assert out.numel() == self.B * self.Hq * self.D
        return fill_f16_device(out, self.seed, stream_id(QUERY, step), 0, 1.0)

    # ---- sizes ---------------------------------------------------------
    @property
    def row_bytes(self):
        return self.D // 2 if self.fmt == INT4 else self.D

    def page_bytes(self):
        return PAGE * self.H * self.row_bytes

    def decode_bytes(self, lens=None):
        """Algorithmic HBM bytes of one decode-attention call over lengths `lens`:
        K and V codes of every valid token, one K and one V scale per touched
        (page, head), the query read and the output written."""
        lens = self.lens if lens is None else np.asarray(lens)
        tok = int(lens.sum())
        pages = int(((lens + PAGE - 1) // PAGE).sum())
        return (2 * tok * self.H * self.row_bytes + 2 * pages * self.H * 4 +
                2 * self.B * self.Hq * self.D * 2)

    def quantize_bytes(self, ntok):
        """Algorithmic bytes of quantizing ntok tokens of K and V into full blocks:
        fp16 read, codes written, one scale per (block, head)."""
        blocks = (ntok + PAGE - 1) // PAGE
        return 2 * (ntok * self.H * self.D * 2 + ntok * self.H * self.row_bytes + blocks * self.H * 4)


def make_workload(cfg, seed=0, extra_tokens=0):
    c = RECIPES[cfg]
    B = c["B"]
    if isinstance(c["L"], tuple):
        _, lo, hi = c["L"]
        lens = uniform_int(B, lo, hi, seed, stream_id(LENGTHS))
    else:
        lens = np.full(B, c["L"], dtype=np.int32)
    return Workload(B, c["H"], c["D"], lens, c["fmt"], c["sigma"], c["outliers"], c["table"], seed,
                    extra_tokens, c["name"], c.get("Hq"), c.get("chunk", 0))
