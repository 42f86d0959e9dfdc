"""Failure detection on the GPU without a GPU fault: every wait of the
kernels is bounded, and a wait that runs out is reported, not hung on.

The library's test hook (qa_debug_arm_wait_timeout) makes the next launch of a
kernel withhold one tile copy in its first thread block (both CTAs of the
first pair in the CTA-pair prefill), so a wait for that tile can never
succeed, and gives the launch's waits a short limit.  The
kernel records QA_ERR_DEVICE_TIMEOUT in the error word, waits for its own
copies in flight (and, in the decode kernel's clusters, for what its peers
send it), frees its tensor memory and exits.  The host reads the status; the
context stays usable: the next calls on the same cache match the oracle.
Nothing here faults, traps or hangs the GPU.
"""
import numpy as np
import pytest
import torch

from gpu_util import GpuCache, assert_parity, dev, f64
from gqa_attention_preallocated_qa_gb300.inputs import bf16_bits_to_f64 as F
from gqa_attention_preallocated_qa_gb300.inputs import layer_inputs

pytestmark = pytest.mark.gpu

QA_KERNEL_PREFILL_ATTN, QA_KERNEL_DECODE_ATTN = 1, 2
TIMEOUT, K2, K3 = 1, 2, 3


@pytest.fixture(scope="module")
def qa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gqa_attention_preallocated_qa_gb300 import _build
    _build.build()
    from gqa_attention_preallocated_qa_gb300 import binding
    return binding


def _check_word(st, word, kernel):
    assert st == 7, (st, hex(word))  # QA_ERR_DEVICE_TIMEOUT
    assert (word & 0xff) == TIMEOUT and ((word >> 8) & 0xff) == kernel, hex(word)


# The first geometry runs the one-CTA prefill (10 four-head items, fewer than
# the device holds pairs); the second the CTA-pair prefill (128 items).
@pytest.mark.parametrize("lens,Hq,Hkv,D,cap,steps", [((300, 129), 8, 2, 128, 440, 2),
                                                     ((1024, 900), 32, 8, 128, 1030, 2)])
def test_prefill_wait_that_runs_out_is_reported_and_the_cache_stays_usable(qa, oracle_mod, lens, Hq,
                                                                           Hkv, D, cap, steps):
    inp = layer_inputs(61, lens, Hq, Hkv, D, steps)
    c = GpuCache(qa, 1, len(lens), Hq, Hkv, D, cap)
    try:
        q, k, v, wq, wk = (dev(a) for a in (inp.q, inp.k, inp.v, inp.wq, inp.wk))
        out = torch.empty_like(q)
        qa.qa_debug_arm_wait_timeout(QA_KERNEL_PREFILL_ATTN, 20000)  # 20 ms
        qa.qa_prefill(c.h, 0, list(lens), q, k, v, wq, wk, out)
        st, word = c.device_error()
        _check_word(st, word, K2)
        assert c.device_error() == (0, 0)  # reading cleared it
        # a new generate call on the same cache: prefill and decode match the oracle
        qa.qa_cache_reset(c.h)
        qa.qa_prefill(c.h, 0, list(lens), q, k, v, wq, wk, out)
        torch.cuda.synchronize()
        lay = oracle_mod.OracleLayer(oracle_mod.Geometry(len(lens), Hq, Hkv, D, cap))
        _, want = lay.prefill(lens, F(inp.q), F(inp.k), F(inp.v), F(inp.wq), F(inp.wk))
        assert_parity(f64(out), want, "prefill after a timeout")
        for s in range(steps):
            dq, dk, dv = (dev(a) for a in (inp.dq[s], inp.dk[s], inp.dv[s]))
            o = torch.empty_like(dq)
            qa.qa_decode_step(c.h, 0, len(lens), dq, dk, dv, wq, wk, o)
            torch.cuda.synchronize()
            _, w2 = lay.decode(F(inp.dq[s]), F(inp.dk[s]), F(inp.dv[s]), F(inp.wq), F(inp.wk))
            assert_parity(f64(o), w2, f"decode step {s} after a timeout")
        assert c.device_error() == (0, 0)
    finally:
        qa.qa_debug_arm_wait_timeout(-1, 0)
        c.free()


def test_decode_wait_that_runs_out_is_reported_and_the_next_step_is_correct(qa, oracle_mod):
    lens, Hq, Hkv, D, cap = (700, 1100), 32, 8, 128, 1200
    inp = layer_inputs(67, lens, Hq, Hkv, D, 2)
    c = GpuCache(qa, 1, len(lens), Hq, Hkv, D, cap)
    try:
        q, k, v, wq, wk = (dev(a) for a in (inp.q, inp.k, inp.v, inp.wq, inp.wk))
        out = torch.empty_like(q)
        qa.qa_prefill(c.h, 0, list(lens), q, k, v, wq, wk, out)
        torch.cuda.synchronize()
        lay = oracle_mod.OracleLayer(oracle_mod.Geometry(len(lens), Hq, Hkv, D, cap))
        lay.prefill(lens, F(inp.q), F(inp.k), F(inp.v), F(inp.wq), F(inp.wk))
        assert c.device_error() == (0, 0)
        dq, dk, dv = (dev(a) for a in (inp.dq[0], inp.dk[0], inp.dv[0]))
        o = torch.empty_like(dq)
        qa.qa_debug_arm_wait_timeout(QA_KERNEL_DECODE_ATTN, 20000)
        qa.qa_decode_step(c.h, 0, len(lens), dq, dk, dv, wq, wk, o)
        st, word = c.device_error()
        _check_word(st, word, K3)
        # the appended slot and the lengths are those of a completed step
        assert qa.qa_cache_lengths(c.h, 0, 2) == [n + 1 for n in lens]
        assert list(c.views()[2].cpu().numpy()) == [n + 1 for n in lens]
        lay.decode(F(inp.dq[0]), F(inp.dk[0]), F(inp.dv[0]), F(inp.wq), F(inp.wk))
        dq, dk, dv = (dev(a) for a in (inp.dq[1], inp.dk[1], inp.dv[1]))
        qa.qa_decode_step(c.h, 0, len(lens), dq, dk, dv, wq, wk, o)
        torch.cuda.synchronize()
        _, want = lay.decode(F(inp.dq[1]), F(inp.dk[1]), F(inp.dv[1]), F(inp.wq), F(inp.wk))
        assert_parity(f64(o), want, "decode step after a timeout")
        assert c.device_error() == (0, 0)
    finally:
        qa.qa_debug_arm_wait_timeout(-1, 0)
        c.free()


def test_arming_rejects_bad_arguments(qa):
    for kernel, us in ((0, 100), (3, 100), (QA_KERNEL_DECODE_ATTN, 0),
                       (QA_KERNEL_DECODE_ATTN, 2000001)):
        with pytest.raises(qa.QaError) as e:
            qa.qa_debug_arm_wait_timeout(kernel, us)
        assert e.value.status == 1
    qa.qa_debug_arm_wait_timeout(-1, 0)
