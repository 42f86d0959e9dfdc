"""The allocation-free decode step against the regular one (GPU).

qa_decode_step_noalloc serves callers that cannot allocate device memory; it
takes the cache memory and the positions from the caller and keeps its own
scratch in a fixed array of the library.  Here a regular cache is prefilled,
its K/V are copied into caller-owned buffers, and two decode calls in a row go
through both entry points with the same inputs: outputs must agree within the
parity bar of the other tests, and the appended slots within the bf16 rounding
bound.  This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

from gpu_util import MAX_ABS, MEAN_ABS, dev, f64, rope_pair_tolerance
from gqa_attention_preallocated_qa_gb300.inputs import layer_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def qa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gqa_attention_preallocated_qa_gb300 import _build
    _build.build()
    from gqa_attention_preallocated_qa_gb300 import binding
    return binding


@pytest.mark.parametrize("lens,Hq,Hkv,D,cap", [((300, 517), 32, 8, 128, 530),
                                               ((64,), 2, 1, 64, 72),
                                               ((40, 3, 90), 16, 2, 64, 100)])
def test_noalloc_decode_matches_regular_decode(qa, lens, Hq, Hkv, D, cap):
    B = len(lens)
    inp = layer_inputs(71 + sum(lens), lens, Hq, Hkv, D, 2)
    h = qa.qa_cache_alloc(1, B, Hq, Hkv, D, cap)
    try:
        q, k, v, wq, wk = (dev(a) for a in (inp.q, inp.k, inp.v, inp.wq, inp.wk))
        out = torch.empty_like(q)
        qa.qa_prefill(h, 0, list(lens), q, k, v, wq, wk, out)
        K, V, _ = qa.cache_tensors(h, 0, B, Hkv, cap, D)
        K2, V2 = K.clone(), V.clone()  # caller-owned cache memory
        cfg = qa.qa_config(1, B, Hq, Hkv, D, cap, 1e6, 1e-6)
        positions = list(lens)
        for s in range(2):
            dq, dk, dv = (dev(a) for a in (inp.dq[s], inp.dk[s], inp.dv[s]))
            o_ref = torch.empty_like(dq)
            o_na = torch.empty_like(dq)
            qa.qa_decode_step(h, 0, B, dq, dk, dv, wq, wk, o_ref)
            qa.qa_decode_step_noalloc(cfg, positions, K2, V2, dq, dk, dv, wq, wk, o_na)
            torch.cuda.synchronize()
            a, b = f64(o_na), f64(o_ref)
            d = np.abs(a - b)
            assert np.isfinite(a).all()
            assert d.max() <= MAX_ABS and d.mean() <= MEAN_ABS, (s, d.max(), d.mean())
            for bi, pos in enumerate(positions):
                ka, kb = f64(K2[bi, :, pos]), f64(K[bi, :, pos])
                assert (np.abs(ka - kb) <= 2 * rope_pair_tolerance(kb)).all()
                assert torch.equal(V2[bi, :, pos], V[bi, :, pos])
            positions = [p + 1 for p in positions]
        assert qa.qa_get_device_error(h) == (0, 0)
    finally:
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
