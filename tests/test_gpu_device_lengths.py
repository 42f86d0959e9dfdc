"""Decode steps that take their positions from the device lengths
(qa_decode_step_device_lengths), and their capture in a CUDA graph: one graph
of a multi-layer decode step replays at every position because the kernel
reads and advances the lengths on the device."""
import numpy as np
import pytest
import torch

from gpu_util import GpuCache, assert_parity, bits, dev, f64
from gqa_attention_preallocated_qa_gb300.inputs import bf16_bits_to_f64 as F
from gqa_attention_preallocated_qa_gb300.inputs import layer_inputs

pytestmark = pytest.mark.gpu

HQ, HKV, D = 32, 8, 128


@pytest.fixture(scope="module")
def qa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gqa_attention_preallocated_qa_gb300 import _build
    _build.build()
    from gqa_attention_preallocated_qa_gb300 import binding
    return binding


def prefilled(qa, layers, prompt, cap, inps):
    c = GpuCache(qa, layers, len(prompt), HQ, HKV, D, cap)
    for l, inp in enumerate(inps):
        q, k, v, wq, wk = (dev(a) for a in (inp.q, inp.k, inp.v, inp.wq, inp.wk))
        out = torch.empty_like(q)
        qa.qa_prefill(c.h, l, list(prompt), q, k, v, wq, wk, out)
    torch.cuda.synchronize()
    return c


def test_device_lengths_step_equals_host_position_step(qa, oracle_mod):
    prompt, steps, cap = (300, 129, 1, 512), 5, 600
    inp = layer_inputs(81, prompt, HQ, HKV, D, steps)
    wq, wk = dev(inp.wq), dev(inp.wk)
    a = prefilled(qa, 1, prompt, cap, [inp])
    b = prefilled(qa, 1, prompt, cap, [inp])
    lay = oracle_mod.OracleLayer(oracle_mod.Geometry(4, HQ, HKV, D, cap))
    lay.prefill(prompt, F(inp.q), F(inp.k), F(inp.v), F(inp.wq), F(inp.wk))
    # the same split plan on both sides makes the two sums bit-comparable:
    # device-length steps plan for a full cache, host-position steps for the
    # current lengths, and one launch at a time fits the same split count here
    qa.qa_cache_set_decode_overlap(a.h, 1)
    qa.qa_cache_set_decode_overlap(b.h, 1)
    try:
        for s in range(steps):
            dq, dk, dv = dev(inp.dq[s]), dev(inp.dk[s]), dev(inp.dv[s])
            oa, ob = torch.empty_like(dq), torch.empty_like(dq)
            qa.qa_decode_step(a.h, 0, 4, dq, dk, dv, wq, wk, oa)
            qa.qa_decode_step_device_lengths(b.h, 0, 4, dq, dk, dv, wq, wk, ob)
            torch.cuda.synchronize()
            np.testing.assert_array_equal(bits(oa), bits(ob))
            _, want = lay.decode(F(inp.dq[s]), F(inp.dk[s]), F(inp.dv[s]), F(inp.wq), F(inp.wk))
            assert_parity(f64(ob), want, f"device-length step {s}")
        final = [n + steps for n in prompt]
        assert list(b.views()[2].cpu().numpy()) == final
        assert qa.qa_cache_lengths(b.h, 0, 4) == list(prompt)  # host copy not advanced
        qa.qa_cache_sync_lengths(b.h, 0)
        assert qa.qa_cache_lengths(b.h, 0, 4) == final
        Ka, Va, _ = a.views()
        Kb, Vb, _ = b.views()
        np.testing.assert_array_equal(bits(Ka), bits(Kb))
        np.testing.assert_array_equal(bits(Va), bits(Vb))
        # after the sync, host-position steps continue where the device ones left off
        qa.qa_cache_set_decode_overlap(b.h, 1)
        dq, dk, dv = dev(inp.dq[0]), dev(inp.dk[0]), dev(inp.dv[0])
        oa, ob = torch.empty_like(dq), torch.empty_like(dq)
        qa.qa_decode_step(a.h, 0, 4, dq, dk, dv, wq, wk, oa)
        qa.qa_decode_step(b.h, 0, 4, dq, dk, dv, wq, wk, ob)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(bits(oa), bits(ob))
        assert a.device_error() == (0, 0) and b.device_error() == (0, 0)
    finally:
        a.free()
        b.free()


def test_cuda_graph_of_a_two_layer_decode_step_replays_at_every_position(qa, oracle_mod):
    prompt, cap, replays = (200, 77, 512, 129), 560, 4
    inps = [layer_inputs(83 + l, prompt, HQ, HKV, D, replays) for l in range(2)]
    ws = [(dev(i.wq), dev(i.wk)) for i in inps]
    g_cache = prefilled(qa, 2, prompt, cap, inps)
    e_cache = prefilled(qa, 2, prompt, cap, inps)
    # the oracle follows both layers step by step: every replay is checked against it
    lays = []
    for inp in inps:
        lay = oracle_mod.OracleLayer(oracle_mod.Geometry(4, HQ, HKV, D, cap))
        lay.prefill(prompt, F(inp.q), F(inp.k), F(inp.v), F(inp.wq), F(inp.wk))
        lays.append(lay)

    def oracle_step(s):
        return [lays[l].decode(F(inps[l].dq[s]), F(inps[l].dk[s]), F(inps[l].dv[s]),
                               F(inps[l].wq), F(inps[l].wk))[1] for l in range(2)]
    try:
        # static buffers of the captured step
        sq = [torch.empty((4, HQ, D), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
        sk = [torch.empty((4, HKV, D), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
        sv = [torch.empty((4, HKV, D), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
        so = [torch.empty((4, HQ, D), dtype=torch.bfloat16, device="cuda") for _ in range(2)]

        def load(s):
            for l in range(2):
                sq[l].copy_(dev(inps[l].dq[s]))
                sk[l].copy_(dev(inps[l].dk[s]))
                sv[l].copy_(dev(inps[l].dv[s]))

        def step(h):
            for l in range(2):
                qa.qa_decode_step_device_lengths(h, l, 4, sq[l], sk[l], sv[l], *ws[l], so[l])

        # step 0 eagerly on both caches (configures the kernel outside capture)
        load(0)
        step(g_cache.h)
        torch.cuda.synchronize()
        want = [[f64(so[l])] for l in range(2)]
        orc = oracle_step(0)
        for l in range(2):
            assert_parity(want[l][0], orc[l], f"eager device-length step 0, layer {l}")
        step(e_cache.h)
        torch.cuda.synchronize()
        for l in range(2):
            np.testing.assert_array_equal(f64(so[l]), want[l][0])
        graph = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            with torch.cuda.graph(graph):
                step(g_cache.h)
        torch.cuda.current_stream().wait_stream(side)
        for s in range(1, replays):
            load(s)
            step(e_cache.h)  # eager reference of step s
            torch.cuda.synchronize()
            ref = [f64(so[l]) for l in range(2)]
            load(s)
            graph.replay()
            torch.cuda.synchronize()
            orc = oracle_step(s)
            for l in range(2):
                np.testing.assert_array_equal(f64(so[l]), ref[l], err_msg=f"replay {s} layer {l}")
                assert_parity(f64(so[l]), orc[l], f"graph replay {s}, layer {l}")
        final = [n + replays for n in prompt]
        for l in range(2):
            assert list(g_cache.views(l)[2].cpu().numpy()) == final
            Kg, Vg, _ = g_cache.views(l)
            Ke, Ve, _ = e_cache.views(l)
            np.testing.assert_array_equal(bits(Kg), bits(Ke))
            np.testing.assert_array_equal(bits(Vg), bits(Ve))
        assert g_cache.device_error() == (0, 0) and e_cache.device_error() == (0, 0)
    finally:
        g_cache.free()
        e_cache.free()


def test_device_lengths_capacity_is_checked_on_the_device(qa):
    prompt, cap = (40, 63), 64
    inp = layer_inputs(89, prompt, HQ, HKV, D, 2)
    wq, wk = dev(inp.wq), dev(inp.wk)
    c = prefilled(qa, 1, prompt, cap, [inp])
    try:
        for s in range(2):
            dq, dk, dv = dev(inp.dq[s]), dev(inp.dk[s]), dev(inp.dv[s])
            o = torch.empty_like(dq)
            qa.qa_decode_step_device_lengths(c.h, 0, 2, dq, dk, dv, wq, wk, o)
        torch.cuda.synchronize()
        # sequence 1 reached the capacity at the first step; the second found it full
        assert list(c.views()[2].cpu().numpy()) == [42, 64]
        st, word = c.device_error()
        assert st == 8 and word != 0  # QA_ERR_DEVICE_BOUNDS
    finally:
        c.free()


def test_multi_layer_device_length_loop_reads_settled_positions_early(qa, oracle_mod):
    # Six layers decoded step by step, as a model's layer loop does: when a step
    # of layer l is launched, no launch still running writes layer l (the ones in
    # flight are other layers'), so the kernel reads its positions at once and
    # overlaps the previous launch.  Every output is checked against the oracle, and
    # the device lengths advance exactly.
    layers, prompt, cap, steps = 6, (300, 700), 800, 3
    inps = [layer_inputs(91 + l, prompt, HQ, HKV, D, steps) for l in range(layers)]
    c = prefilled(qa, layers, prompt, cap, inps)
    lays = []
    for inp in inps:
        lay = oracle_mod.OracleLayer(oracle_mod.Geometry(2, HQ, HKV, D, cap))
        lay.prefill(prompt, F(inp.q), F(inp.k), F(inp.v), F(inp.wq), F(inp.wk))
        lays.append(lay)
    try:
        ins = [[(dev(i.dq[s]), dev(i.dk[s]), dev(i.dv[s])) for s in range(steps)] for i in inps]
        ws = [(dev(i.wq), dev(i.wk)) for i in inps]
        outs = [[torch.empty((2, HQ, D), dtype=torch.bfloat16, device="cuda")
                 for _ in range(steps)] for _ in range(layers)]
        torch.cuda.synchronize()
        for s in range(steps):
            for l in range(layers):
                qa.qa_decode_step_device_lengths(c.h, l, 2, *ins[l][s], *ws[l], outs[l][s])
        torch.cuda.synchronize()
        for l in range(layers):
            for s in range(steps):
                i = inps[l]
                _, want = lays[l].decode(F(i.dq[s]), F(i.dk[s]), F(i.dv[s]), F(i.wq), F(i.wk))
                assert_parity(f64(outs[l][s]), want, f"layer {l} step {s}")
            assert list(c.views(l)[2].cpu().numpy()) == [n + steps for n in prompt]
        assert c.device_error() == (0, 0)
    finally:
        c.free()
