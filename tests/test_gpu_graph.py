"""GPU tests of the decode step captured as a CUDA graph (kvq_step_graph_*;
CUDA Graph instance reuse, jsqmd.com/news/887038 section 4.1): replaying the
graph must give bit-identical outputs and caches to the eager calls it
records, with per-step inputs written into the bound tensors, and its outputs
must match the binary64 oracle's attention over the oracle's own cache of the
grown histories (2e-3 of max|v^|); rebinding with kvq_step_graph_update must
move the step to the new tensors; rejected arguments must be reported as the
eager calls report them."""
import math

import numpy as np
import pytest
import torch

from oracle import oracle as orc
from quantized_kv_cache_09_gb300 import kvq
from quantized_kv_cache_09_gb300.runner import DecodeStep, DeviceWorkload
from quantized_kv_cache_09_gb300.synth import workloads as W

pytestmark = pytest.mark.gpu
D = 128


def _pair(fmt, lens, H=4, Hq=None, seed=41):
    wl = W.Workload(len(lens), H, D, lens, fmt, 1.0, ("per_head", 2, 10.0), "permuted", seed=seed,
                    extra_tokens=80, q_heads=Hq)
    a, b = DeviceWorkload(wl), DeviceWorkload(wl)
    a.prefill()
    b.prefill()
    return wl, a, b


TOL = 2e-3


def _oracle_check(wl, lens_after, q_bits, out):
    """The graph's output of one step against the oracle: quantize every
    sequence's history up to lens_after with the oracle's codec, attend with
    the step's query in binary64."""
    rb = orc.row_bytes(wl.fmt, D)
    kc = np.zeros((wl.num_pages, wl.H, 64, rb), np.uint8)
    vc = np.zeros_like(kc)
    ks = np.zeros((wl.num_pages, wl.H), np.float32)
    vs = np.zeros_like(ks)
    for b in range(wl.B):
        L = int(lens_after[b])
        orc.quantize_into_pages(wl.fmt, wl.kv_host("k", b, 0, L), wl.block_table[b], kc, ks)
        orc.quantize_into_pages(wl.fmt, wl.kv_host("v", b, 0, L), wl.block_table[b], vc, vs)
    ref = orc.decode_attention(wl.fmt, kc, vc, ks, vs, wl.block_table, lens_after, q_bits,
                               np.float32(1 / math.sqrt(D)))
    vmax = np.repeat(orc.value_absmax(wl.fmt, vc, vs, wl.block_table, lens_after, wl.H, D), wl.Hq // wl.H, axis=1)
    err = orc.normalized_error(out.float().cpu().numpy().astype(np.float64), ref, vmax)
    assert err <= TOL, err
    return err


def _same_cache(a, b):
    for name in ("k_codes", "v_codes", "k_scales", "v_scales", "k_tail", "v_tail"):
        assert torch.equal(getattr(a.cache, name), getattr(b.cache, name)), name


@pytest.mark.parametrize("fmt,H,Hq", [(kvq.KVQ_INT4_B64, 4, None), (kvq.KVQ_INT8_PAGE, 4, None),
                                      (kvq.KVQ_FP8_E4M3, 4, None), (kvq.KVQ_INT4_B64, 2, 8),
                                      (kvq.KVQ_INT8_PAGE, 2, 16), (kvq.KVQ_INT4_B64, 1, 32)])
def test_graph_replay_equals_eager(cuda_ok, fmt, H, Hq):
    """70 steps (every sequence crosses a page boundary): the graph, fed
    through its bound slots, and the eager calls give identical bits."""
    lens = [100, 63, 64, 300, 1]
    wl, ea, gr = _pair(fmt, lens, H, Hq)
    st_e, st_g = DecodeStep(ea), DecodeStep(gr)
    k0, v0, q0 = gr.new_token_tensors(0)
    slot_k, slot_v, slot_q = torch.empty_like(k0), torch.empty_like(v0), torch.empty_like(q0)
    slot_lb = torch.empty(len(lens), dtype=torch.int32, device="cuda")
    slot_la = torch.empty_like(slot_lb)
    g = st_g.graph(slot_lb, slot_la, slot_k, slot_v, slot_q)
    base = torch.from_numpy(wl.lens.copy()).cuda()
    for s in range(70):
        k1, v1, q = ea.new_token_tensors(s)
        out_e = st_e.run(base + s, base + s + 1, k1, v1, q).clone()
        slot_k.copy_(k1)
        slot_v.copy_(v1)
        slot_q.copy_(q)
        slot_lb.copy_(base + s)
        slot_la.copy_(base + s + 1)
        g.launch()
        torch.cuda.synchronize()
        assert torch.equal(out_e, st_g.out), s
        if s % 23 == 0 or s == 69:  # the replay against the oracle, not only against eager calls
            _oracle_check(wl, wl.lens + s + 1, wl.q_host(s), st_g.out)
    g.close()
    _same_cache(ea, gr)
    assert kvq.kvq_get_device_status(ea.cache) == (0, 0)
    assert kvq.kvq_get_device_status(gr.cache) == (0, 0)


def test_graph_of_layers_and_steps_equals_eager(cuda_ok):
    """One graph holding 3 layers (3 caches of different formats) x 5 steps
    each, in layer-major order per step as a model runs them, against the
    same calls made eagerly; the graph is replayed twice (the lengths start on
    page boundaries, so a replay re-opens the same blocks and repeats the
    same states)."""
    lens = [128, 64, 192, 640]
    fmts = [kvq.KVQ_INT4_B64, kvq.KVQ_FP8_E4M3, kvq.KVQ_INT8_PAGE]
    layers = [_pair(f, lens, seed=50 + i) for i, f in enumerate(fmts)]
    base = torch.from_numpy(layers[0][0].lens.copy()).cuda()
    eager = [DecodeStep(e) for _, e, _ in layers]
    graphed = [DecodeStep(g) for _, _, g in layers]
    outs_e, steps = [], []
    inputs = [[gdw.new_token_tensors(s) for s in range(5)] for _, _, gdw in layers]
    lb = [base + s for s in range(5)]
    la = [base + s + 1 for s in range(5)]
    g_outs = []
    for s in range(5):
        for li in range(3):
            out = torch.empty_like(graphed[li].out)
            g_outs.append(out)
            k1, v1, q = inputs[li][s]
            st = graphed[li].graph_step(lb[s], la[s], k1, v1, q)
            steps.append(st[:10] + (out,) + st[11:])
            outs_e.append(eager[li].run(lb[s], la[s], k1, v1, q).clone())
    g = kvq.StepGraph(steps)
    for rep_ in range(2):
        for o in g_outs:
            o.fill_(float("nan"))
        g.launch()
        torch.cuda.synchronize()
        for i, (a, b) in enumerate(zip(outs_e, g_outs)):
            assert torch.equal(a, b), (rep_, i)
    for s in (0, 4):  # the replayed outputs of the first and last step of every layer against the oracle
        for li in range(3):
            wl = layers[li][0]
            _oracle_check(wl, wl.lens + s + 1, wl.q_host(s), g_outs[3 * s + li])
    g.close()
    for _, e, gdw in layers:
        _same_cache(e, gdw)
        assert kvq.kvq_get_device_status(gdw.cache) == (0, 0)


def test_graph_update_rebinds_tensors(cuda_ok):
    """After kvq_step_graph_update to other q / out / length tensors the replay
    writes the new output tensor and leaves the old one alone."""
    lens = [500, 77, 64]
    wl, ea, gr = _pair(kvq.KVQ_INT4_B64, lens)
    st_e, st_g = DecodeStep(ea), DecodeStep(gr)
    base = torch.from_numpy(wl.lens.copy()).cuda()
    k1, v1, q = gr.new_token_tensors(0)
    g = st_g.graph(base.clone(), base + 1, k1, v1, q)
    g.launch()
    out0 = st_e.run(base, base + 1, *ea.new_token_tensors(0)).clone()
    torch.cuda.synchronize()
    assert torch.equal(out0, st_g.out)
    k2, v2, q2 = gr.new_token_tensors(1)
    out_new = torch.full_like(st_g.out, float("nan"))
    old = st_g.out.clone()
    g.update([(gr.cache, k2, v2, st_g.cu, gr.block_table, base + 1, 1, q2, base + 2, gr.softmax_scale, out_new,
               gr.workspace)])
    g.launch()
    out1 = st_e.run(base + 1, base + 2, *ea.new_token_tensors(1)).clone()
    torch.cuda.synchronize()
    assert torch.equal(out1, out_new)
    assert torch.equal(old, st_g.out)
    g.close()
    _same_cache(ea, gr)


def test_graph_update_to_another_format(cuda_ok):
    """Rebinding to a cache of another format changes the kernels: the graph is
    instantiated anew and still matches the eager step."""
    lens = [200, 65]
    wl4, _, g4 = _pair(kvq.KVQ_INT4_B64, lens)
    wl8, e8, g8 = _pair(kvq.KVQ_INT8_PAGE, lens)
    base = torch.from_numpy(wl4.lens.copy()).cuda()
    s4, s8, se = DecodeStep(g4), DecodeStep(g8), DecodeStep(e8)
    g = s4.graph(base, base + 1, *g4.new_token_tensors(0))
    k1, v1, q = g8.new_token_tensors(0)
    g.update([s8.graph_step(base, base + 1, k1, v1, q)])
    g.launch()
    ref = se.run(base, base + 1, *e8.new_token_tensors(0)).clone()
    torch.cuda.synchronize()
    assert torch.equal(ref, s8.out)
    g.close()
    _same_cache(e8, g8)


def test_graph_rejects_bad_arguments(cuda_ok):
    lens = [70, 10]
    wl, a, _ = _pair(kvq.KVQ_INT4_B64, lens)
    st = DecodeStep(a)
    base = torch.from_numpy(wl.lens.copy()).cuda()
    k1, v1, q = a.new_token_tensors(0)
    with pytest.raises(kvq.KvqError) as e:  # workspace too small
        kvq.StepGraph([(a.cache, k1, v1, st.cu, a.block_table, base, 1, q, base + 1, a.softmax_scale, st.out,
                        a.workspace[:64])])
    assert e.value.status == 6
    q3 = torch.zeros((2, 3, D), dtype=torch.float16, device="cuda")
    with pytest.raises(kvq.KvqError) as e:  # 3 query heads over 4 cache heads, in the second step
        kvq.StepGraph([st.graph_step(base, base + 1, k1, v1, q),
                       (a.cache, k1, v1, st.cu, a.block_table, base, 1, q3, base + 1, a.softmax_scale, q3.clone(),
                        a.workspace)])
    assert e.value.status == 1
    # nothing ran: the cache is as the prefill left it
    assert kvq.kvq_get_device_status(a.cache) == (0, 0)
