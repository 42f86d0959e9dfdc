"""The attention epilogue, fused (GPU).

On this path the attention epilogue is what stands between the attention sum
and the output projection of a Qwen3-style layer: dividing the accumulated
P.V by the softmax denominator, casting to the activation type (bf16), and
laying the heads out token-major, as the [T, Hq*D] matrix the output
projection multiplies (the module transposes its [B, Hq, T, D] attention
output to [B, T, Hq, D] and makes it contiguous before that GEMM).  The
prefill and decode kernels do all three in their output stage.  Checked here:
  - no kernel besides the attention kernels runs (launch counters), and every
    element of the output buffer is written (it is poisoned first);
  - the output, read as the [T, Hq*D] matrix, is the oracle's attention output
    in token-major order, and multiplying it by an output-projection weight
    gives the oracle's projected rows within the bound the parity bar implies.
"""
import numpy as np
import pytest
import torch

from gpu_util import GpuCache, MAX_ABS, assert_parity, dev, f64
from gqa_attention_preallocated_qa_gb300.inputs import bf16_bits_to_f64 as F
from gqa_attention_preallocated_qa_gb300.inputs import layer_inputs

pytestmark = pytest.mark.gpu

HQ, HKV, D = 32, 8, 128
NAN_BITS = np.int16(0x7FC1)


@pytest.fixture(scope="module")
def qa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gqa_attention_preallocated_qa_gb300 import _build
    _build.build()
    from gqa_attention_preallocated_qa_gb300 import binding
    return binding


def _projection_check(got, want, rng, what):
    # out [T, Hq*D] @ W [Hq*D, 64]: |row error . W| <= sum_i |err_i| |W_i|, and
    # each |err_i| is within the parity bar, so every projected element lies
    # within MAX_ABS * sum|W_col| of the oracle's.
    T = got.shape[0]
    W = rng.standard_normal((HQ * D, 64)) / np.sqrt(HQ * D)
    g, w = got.reshape(T, HQ * D) @ W, want.reshape(T, HQ * D) @ W
    bound = MAX_ABS * np.abs(W).sum(axis=0)
    assert (np.abs(g - w) <= bound[None, :]).all(), what


def test_prefill_and_decode_outputs_need_no_epilogue_kernel(qa, oracle_mod):
    prompt, steps, cap = (300, 129), 3, 440
    inp = layer_inputs(113, prompt, HQ, HKV, D, steps)
    B, T = len(prompt), sum(prompt)
    rng = np.random.default_rng(5)
    c = GpuCache(qa, 1, B, HQ, HKV, D, cap)
    lay = oracle_mod.OracleLayer(oracle_mod.Geometry(B, HQ, HKV, D, cap))
    try:
        q, k, v, wq, wk = (dev(a) for a in (inp.q, inp.k, inp.v, inp.wq, inp.wk))
        out = torch.empty_like(q)
        out.view(torch.int16).fill_(NAN_BITS)
        before = qa.qa_stats(c.h)
        qa.qa_prefill(c.h, 0, list(prompt), q, k, v, wq, wk, out)
        torch.cuda.synchronize()
        after = qa.qa_stats(c.h)
        assert {n: after[n] - before[n] for n in after} == {
            "norm_rope_append": 1, "prefill_attn": 1, "decode_attn": 0, "reset": 0}
        got = f64(out)
        assert np.isfinite(got).all(), "an output element was left unwritten"
        _, want = lay.prefill(prompt, F(inp.q), F(inp.k), F(inp.v), F(inp.wq), F(inp.wk))
        assert_parity(got.reshape(T, HQ * D), want.reshape(T, HQ * D), "prefill [T, Hq*D]")
        _projection_check(got, want, rng, "prefill projected")
        for s in range(steps):
            o = torch.empty((B, HQ, D), dtype=torch.bfloat16, device="cuda")
            o.view(torch.int16).fill_(NAN_BITS)
            before = qa.qa_stats(c.h)
            qa.qa_decode_step(c.h, 0, B, dev(inp.dq[s]), dev(inp.dk[s]), dev(inp.dv[s]), wq, wk, o)
            torch.cuda.synchronize()
            after = qa.qa_stats(c.h)
            assert {n: after[n] - before[n] for n in after} == {
                "norm_rope_append": 0, "prefill_attn": 0, "decode_attn": 1, "reset": 0}
            g = f64(o)
            assert np.isfinite(g).all(), "an output element was left unwritten"
            _, w2 = lay.decode(F(inp.dq[s]), F(inp.dk[s]), F(inp.dv[s]), F(inp.wq), F(inp.wk))
            assert_parity(g.reshape(B, HQ * D), w2.reshape(B, HQ * D), f"decode {s} [B, Hq*D]")
            _projection_check(g, w2, rng, f"decode {s} projected")
        assert c.device_error() == (0, 0)
    finally:
        c.free()
