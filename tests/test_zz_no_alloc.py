"""The allocation-free decode step (GPU), through the C ABI.

qa_decode_step_noalloc serves callers that cannot allocate device memory
(engines that own every byte of the GPU through their own arena, plug-ins in a
framework that owns the allocator): it takes the cache memory and the
positions from the caller and keeps its only scratch, an error word, in a
fixed array of the library.  Here a regular cache is prefilled, its K/V are
copied into caller-owned buffers, and two decode calls in a row go through
both entry points with the same inputs.  With the same split plan (the regular
cache planned for one launch at a time, as the allocation-free step does) both
run the same kernel body, so outputs and appended slots must be bit-identical;
the outputs must also meet the oracle's parity bar.  The error word must read
clean.  A second test makes one of the step's bounded waits run out (the
library's test hook withholds a tile copy) and checks that the error is
reported through the allocation-free error accessor and that the next call is
correct again.  This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

from gpu_util import assert_parity, bits, dev, f64
from gqa_attention_preallocated_qa_gb300.inputs import bf16_bits_to_f64 as F
from gqa_attention_preallocated_qa_gb300.inputs import layer_inputs

pytestmark = pytest.mark.gpu

QA_KERNEL_DECODE_ATTN = 2


@pytest.fixture(scope="module")
def qa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gqa_attention_preallocated_qa_gb300 import _build
    _build.build()
    from gqa_attention_preallocated_qa_gb300 import binding
    return binding


def _setup(qa, oracle_mod, lens, Hq, Hkv, D, cap, steps):
    B = len(lens)
    inp = layer_inputs(71 + sum(lens), lens, Hq, Hkv, D, steps)
    h = qa.qa_cache_alloc(1, B, Hq, Hkv, D, cap)
    # the allocation-free step plans its splits for one launch at a time
    qa.qa_cache_set_decode_overlap(h, 1)
    q, k, v, wq, wk = (dev(a) for a in (inp.q, inp.k, inp.v, inp.wq, inp.wk))
    out = torch.empty_like(q)
    qa.qa_prefill(h, 0, list(lens), q, k, v, wq, wk, out)
    K, V, _ = qa.cache_tensors(h, 0, B, Hkv, cap, D)
    K2, V2 = K.clone(), V.clone()  # caller-owned cache memory
    lay = oracle_mod.OracleLayer(oracle_mod.Geometry(B, Hq, Hkv, D, cap))
    lay.prefill(lens, F(inp.q), F(inp.k), F(inp.v), F(inp.wq), F(inp.wk))
    return inp, h, (K, V), (K2, V2), (wq, wk), lay


@pytest.mark.parametrize("lens,Hq,Hkv,D,cap", [((300, 517), 32, 8, 128, 530),
                                               ((64,), 2, 1, 64, 72),
                                               ((40, 3, 90), 16, 2, 64, 100)])
def test_noalloc_decode_matches_regular_decode_and_oracle(qa, oracle_mod, lens, Hq, Hkv, D, cap):
    B = len(lens)
    inp, h, (K, V), (K2, V2), (wq, wk), lay = _setup(qa, oracle_mod, lens, Hq, Hkv, D, cap, 2)
    try:
        cfg = qa.qa_config(1, B, Hq, Hkv, D, cap, 1e6, 1e-6)
        assert qa.qa_noalloc_get_device_error() == (0, 0)
        positions = list(lens)
        for s in range(2):  # two calls in a row
            dq, dk, dv = (dev(a) for a in (inp.dq[s], inp.dk[s], inp.dv[s]))
            o_ref = torch.empty_like(dq)
            o_na = torch.empty_like(dq)
            qa.qa_decode_step(h, 0, B, dq, dk, dv, wq, wk, o_ref)
            qa.qa_decode_step_noalloc(cfg, positions, K2, V2, dq, dk, dv, wq, wk, o_na)
            torch.cuda.synchronize()
            np.testing.assert_array_equal(bits(o_na), bits(o_ref), err_msg=f"call {s}")
            _, want = lay.decode(F(inp.dq[s]), F(inp.dk[s]), F(inp.dv[s]), F(inp.wq), F(inp.wk))
            assert_parity(f64(o_na), want, f"no-alloc call {s}")
            for bi, pos in enumerate(positions):
                assert torch.equal(K2[bi, :, pos], K[bi, :, pos])
                assert torch.equal(V2[bi, :, pos], V[bi, :, pos])
            positions = [p + 1 for p in positions]
        assert qa.qa_noalloc_get_device_error() == (0, 0)
        assert qa.qa_get_device_error(h) == (0, 0)
    finally:
        qa.qa_cache_free(h)


def test_noalloc_reports_a_bounded_wait_that_ran_out(qa, oracle_mod):
    lens, Hq, Hkv, D, cap = (300, 517), 32, 8, 128, 530
    B = len(lens)
    inp, h, _, (K2, V2), (wq, wk), lay = _setup(qa, oracle_mod, lens, Hq, Hkv, D, cap, 2)
    try:
        cfg = qa.qa_config(1, B, Hq, Hkv, D, cap, 1e6, 1e-6)
        assert qa.qa_noalloc_get_device_error() == (0, 0)
        dq, dk, dv = (dev(a) for a in (inp.dq[0], inp.dk[0], inp.dv[0]))
        o = torch.empty_like(dq)
        qa.qa_debug_arm_wait_timeout(QA_KERNEL_DECODE_ATTN, 20000)  # 20 ms
        qa.qa_decode_step_noalloc(cfg, list(lens), K2, V2, dq, dk, dv, wq, wk, o)
        st, word = qa.qa_noalloc_get_device_error()
        assert st == 7, (st, hex(word))               # QA_ERR_DEVICE_TIMEOUT
        assert (word & 0xff) == 1 and ((word >> 8) & 0xff) == 3  # timeout, decode kernel
        assert qa.qa_noalloc_get_device_error() == (0, 0)  # reading cleared it
        # the context stays usable: the same step again is correct
        qa.qa_decode_step_noalloc(cfg, list(lens), K2, V2, dq, dk, dv, wq, wk, o)
        torch.cuda.synchronize()
        _, want = lay.decode(F(inp.dq[0]), F(inp.dk[0]), F(inp.dv[0]), F(inp.wq), F(inp.wk))
        assert_parity(f64(o), want, "no-alloc after a timeout")
        assert qa.qa_noalloc_get_device_error() == (0, 0)
    finally:
        qa.qa_debug_arm_wait_timeout(-1, 0)
        qa.qa_cache_free(h)


def test_noalloc_rejects_sizes_beyond_its_limits(qa):
    cfg = qa.qa_config(1, 32, 32, 8, 128, 64, 1e6, 1e-6)
    t = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(qa.QaError) as e:   # 17 sequences: above the parameter block
        qa.qa_decode_step_noalloc(cfg, [0] * 17, t, t, t, t, t, t, t, t)
    assert e.value.status == 2
    with pytest.raises(qa.QaError) as e:   # no free slot left
        qa.qa_decode_step_noalloc(cfg, [64], t, t, t, t, t, t, t, t)
    assert e.value.status == 4
