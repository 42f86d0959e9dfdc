"""Sliding-window attention (qa_cache_set_window): a token at position i
attends to keys max(0, i + 1 - W) .. i, in prefill (also chunked) and in the
decode steps.  Expected values: the oracle's attention over exactly those
cached keys (the window only narrows the key range of the definition)."""
import numpy as np
import pytest
import torch

from gpu_util import GpuCache, assert_parity, bits, dev, f64
from gqa_attention_preallocated_qa_gb300.inputs import bf16_bits_to_f64 as F
from gqa_attention_preallocated_qa_gb300.inputs import layer_inputs
from test_gpu_chunked_prefill import ChunkOracle

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


class WindowOracle(ChunkOracle):
    def __init__(self, *a, window, **kw):
        super().__init__(*a, **kw)
        self.W = window

    def out_row(self, b, pos, h, q_row):
        om = self.om
        qp = om.rope(om.rmsnorm(q_row, self.wq, self.eps), pos, self.theta)
        lo = max(0, pos + 1 - self.W)
        g = h // self.G
        return om.attend(qp, self.K[b, g, lo:pos + 1], self.V[b, g, lo:pos + 1])[0]


@pytest.mark.parametrize("window", [64, 200])
def test_window_prefill_chunks_and_decode(qa, oracle_mod, window):
    chunks = [(300, 129, 1, 700), (50, 0, 140, 3)]
    steps, cap = 3, 900
    inps = [layer_inputs(97 + n, lens, HQ, HKV, D, steps if n == 1 else 0)
            for n, lens in enumerate(chunks)]
    wq, wk = inps[0].wq, inps[0].wk
    B = len(chunks[0])
    c = GpuCache(qa, 1, B, HQ, HKV, D, cap)
    orc = WindowOracle(oracle_mod, B, HQ, HKV, D, cap, wq, wk, window=window)
    rng = np.random.default_rng(window)
    try:
        qa.qa_cache_set_window(c.h, 0, window)
        wq_d, wk_d = dev(wq), dev(wk)
        for n, (lens, inp) in enumerate(zip(chunks, inps)):
            q, k, v = dev(inp.q), dev(inp.k), dev(inp.v)
            out = torch.empty_like(q)
            start = list(orc.lens)
            qa.qa_prefill(c.h, 0, list(lens), q, k, v, wq_d, wk_d, out)
            torch.cuda.synchronize()
            got, qf = f64(out), F(inp.q)
            want, have, t0 = [], [], 0
            for b, L in enumerate(lens):
                orc.append(b, F(inp.k[t0:t0 + L]), F(inp.v[t0:t0 + L]))
                if L:
                    # rows around tile and window boundaries, plus random ones
                    rows = {0, L - 1, min(L - 1, 127), min(L - 1, 128), min(L - 1, window),
                            min(L - 1, window + 130)}
                    rows |= set(rng.integers(0, L, size=10).tolist())
                    for i in sorted(rows):
                        for h in (0, 7, 16, 31):
                            want.append(orc.out_row(b, start[b] + i, h, qf[t0 + i, h]))
                            have.append(got[t0 + i, h])
                t0 += L
            assert_parity(np.array(have), np.array(want), f"window {window} chunk {n}")
        inp = inps[1]
        for s in range(steps):
            dq, dk, dv = dev(inp.dq[s]), dev(inp.dk[s]), dev(inp.dv[s])
            o = torch.empty_like(dq)
            qa.qa_decode_step(c.h, 0, B, dq, dk, dv, wq_d, wk_d, o)
            torch.cuda.synchronize()
            want = []
            for b in range(B):
                orc.append(b, F(inp.dk[s][b][None]), F(inp.dv[s][b][None]))
                want.append([orc.out_row(b, orc.lens[b] - 1, h, F(inp.dq[s][b, h]))
                             for h in range(HQ)])
            assert_parity(f64(o), np.array(want), f"window {window} decode step {s}")
        assert c.device_error() == (0, 0)
    finally:
        c.free()


def test_window_longer_than_every_sequence_is_full_attention(qa):
    prompt, steps, cap = (300, 129, 1, 700), 3, 720
    inp = layer_inputs(101, prompt, HQ, HKV, D, steps)
    q, k, v, wq, wk = (dev(a) for a in (inp.q, inp.k, inp.v, inp.wq, inp.wk))
    res = []
    for window in (0, cap):
        c = GpuCache(qa, 1, 4, HQ, HKV, D, cap)
        try:
            qa.qa_cache_set_window(c.h, 0, window)
            out = torch.empty_like(q)
            qa.qa_prefill(c.h, 0, list(prompt), q, k, v, wq, wk, out)
            outs = [bits(out)]
            for s in range(steps):
                o = torch.empty((4, HQ, D), dtype=torch.bfloat16, device="cuda")
                qa.qa_decode_step(c.h, 0, 4, dev(inp.dq[s]), dev(inp.dk[s]), dev(inp.dv[s]), wq, wk, o)
                outs.append(bits(o))
            torch.cuda.synchronize()
            res.append(outs)
            assert c.device_error() == (0, 0)
        finally:
            c.free()
    for a, b in zip(*res):
        np.testing.assert_array_equal(a, b)


def test_window_1024_over_2048_prompts_and_decode(qa, oracle_mod):
    # The sliding window of the A10G reproduction repo's stack (1024 keys) over
    # prompts of 2048 and 1500 tokens, then decode steps past the prompt: rows
    # around the tile and window boundaries, on three heads, and every decode
    # output against attention over exactly the window's keys.
    window, prompt, steps = 1024, (2048, 1500), 3
    cap = max(prompt) + steps
    inp = layer_inputs(107, prompt, HQ, HKV, D, steps)
    B = len(prompt)
    c = GpuCache(qa, 1, B, HQ, HKV, D, cap)
    orc = WindowOracle(oracle_mod, B, HQ, HKV, D, cap, inp.wq, inp.wk, window=window)
    rng = np.random.default_rng(1024)
    try:
        qa.qa_cache_set_window(c.h, 0, window)
        q, k, v, wq, wk = (dev(a) for a in (inp.q, inp.k, inp.v, inp.wq, inp.wk))
        out = torch.empty_like(q)
        qa.qa_prefill(c.h, 0, list(prompt), q, k, v, wq, wk, out)
        torch.cuda.synchronize()
        got, qf = f64(out), F(inp.q)
        want, have, t0 = [], [], 0
        for b, L in enumerate(prompt):
            orc.append(b, F(inp.k[t0:t0 + L]), F(inp.v[t0:t0 + L]))
            rows = {0, 127, 128, 1022, 1023, 1024, 1025, 1151, 1152, L - 129, L - 1}
            rows |= set(rng.integers(0, L, size=8).tolist())
            for i in sorted(r for r in rows if r < L):
                for h in (0, 13, 31):
                    want.append(orc.out_row(b, i, h, qf[t0 + i, h]))
                    have.append(got[t0 + i, h])
            t0 += L
        assert_parity(np.array(have), np.array(want), "window 1024 prefill")
        for s in range(steps):
            dq, dk, dv = dev(inp.dq[s]), dev(inp.dk[s]), dev(inp.dv[s])
            o = torch.empty_like(dq)
            qa.qa_decode_step(c.h, 0, B, dq, dk, dv, wq, wk, o)
            torch.cuda.synchronize()
            want = []
            for b in range(B):
                orc.append(b, F(inp.dk[s][b][None]), F(inp.dv[s][b][None]))
                want.append([orc.out_row(b, orc.lens[b] - 1, h, F(inp.dq[s][b, h]))
                             for h in range(HQ)])
            assert_parity(f64(o), np.array(want), f"window 1024 decode step {s}")
        assert c.device_error() == (0, 0)
    finally:
        c.free()
