"""Drive the CUDA path on a synthetic workload: fill a paged cache from a
workload's fp16 history (generated in HBM), run decode steps.  Used by the GPU
tests, the smoke check and the benchmark; every arithmetic step runs in the
kvq kernels, this module only moves tensors and calls the C ABI."""
import math

import numpy as np
import torch

from . import kvq
from .synth import workloads as W


class DeviceWorkload:
    """The device-side state of one workload: cache, block table, lengths."""

    def __init__(self, wl, device="cuda"):
        self.wl = wl
        self.device = device
        self.cache = kvq.PagedKVCache(wl.fmt, wl.num_pages, wl.H, max_seqs=wl.B, device=device)
        self.block_table = torch.from_numpy(np.ascontiguousarray(wl.block_table)).to(device)
        self.lens = torch.from_numpy(wl.lens.copy()).to(device)
        self.lens_host = wl.lens.copy()
        self.workspace = self.cache.workspace(wl.Hq)
        self.softmax_scale = 1.0 / math.sqrt(wl.D)

    def prefill(self, max_tokens_per_call=1 << 21):
        """Append every sequence's history [0, lens[b]) in calls of whole sequences
        holding at most max_tokens_per_call tokens (generated on the device)."""
        wl = self.wl
        H, D = wl.H, wl.D
        b = 0
        while b < wl.B:
            group = [b]
            tot = int(wl.lens[b])
            while group[-1] + 1 < wl.B and tot + int(wl.lens[group[-1] + 1]) <= max_tokens_per_call:
                group.append(group[-1] + 1)
                tot += int(wl.lens[group[-1]])
            k_new = torch.empty((max(tot, 1), H, D), dtype=torch.float16, device=self.device)
            v_new = torch.empty_like(k_new)
            cu = [0]
            for g in group:
                L = int(wl.lens[g])
                if L:
                    wl.kv_device("k", g, 0, L, k_new[cu[-1]:cu[-1] + L])
                    wl.kv_device("v", g, 0, L, v_new[cu[-1]:cu[-1] + L])
                cu.append(cu[-1] + L)
            b0, b1 = group[0], group[-1] + 1
            cu_t = torch.tensor(cu, dtype=torch.int32, device=self.device)
            before = torch.zeros(b1 - b0, dtype=torch.int32, device=self.device)
            mx = int(max(wl.lens[b0:b1].max(), 1))
            kvq.kvq_append(self.cache.rows_from(b0), k_new, v_new, cu_t, self.block_table[b0:b1], before, mx)
            del k_new, v_new
            b = b1
        torch.cuda.current_stream().synchronize()

    def new_token_tensors(self, step):
        """fp16 K/V rows of the token each sequence appends at decode step `step`
        (position lens_host[b] + step of its history) and the step's query."""
        wl = self.wl
        k = torch.empty((wl.B, wl.H, wl.D), dtype=torch.float16, device=self.device)
        v = torch.empty_like(k)
        for b in range(wl.B):
            t = int(self.lens_host[b]) + step
            wl.kv_device("k", b, t, t + 1, k[b:b + 1])
            wl.kv_device("v", b, t, t + 1, v[b:b + 1])
        q = torch.empty((wl.B, wl.Hq, wl.D), dtype=torch.float16, device=self.device)
        wl.q_device(q, step)
        return k, v, q


class DecodeStep:
    """One decode step of the whole batch: append one token per sequence
    (re-quantizing each open block from its fp16 originals), then attend with
    the step's query over every sequence's history including that token."""

    def __init__(self, dw):
        self.dw = dw
        B = dw.wl.B
        self.cu = torch.arange(B + 1, dtype=torch.int32, device=dw.device)
        self.out = torch.empty((B, dw.wl.Hq, dw.wl.D), dtype=torch.float16, device=dw.device)

    def run(self, lens_before, lens_after, k1, v1, q, stream=None):
        dw = self.dw
        kvq.kvq_append(dw.cache, k1, v1, self.cu, dw.block_table, lens_before, 1, stream)
        kvq.kvq_decode_attention_gqa(dw.cache, q, dw.block_table, lens_after, dw.softmax_scale, self.out,
                                     dw.workspace, stream)
        return self.out

    def graph_step(self, lens_before, lens_after, k1, v1, q):
        """This step's entry of a kvq.StepGraph (bound to these tensors and self.out)."""
        dw = self.dw
        return (dw.cache, k1, v1, self.cu, dw.block_table, lens_before, 1, q, lens_after, dw.softmax_scale,
                self.out, dw.workspace)

    def graph(self, lens_before, lens_after, k1, v1, q):
        """The step as a one-step kvq.StepGraph."""
        return kvq.StepGraph([self.graph_step(lens_before, lens_after, k1, v1, q)])


def kernel_names():
    """Substrings of the kernel names the CUDA path launches."""
    return ["quantize_contig_kernel", "append_kernel", "append_short_kernel", "decode_split_kernel"]


__all__ = ["DeviceWorkload", "DecodeStep", "kernel_names", "W"]
