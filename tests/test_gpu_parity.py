"""GPU parity of the CUDA path (called through the C ABI) against the fp64
oracle, on the same seeded inputs.

Bar: attention outputs max-abs <= 2e-2 and mean-abs <= 2e-3; cache slot
indexing, positions and lengths bit-exact; V copied bit-exactly; K within the
bf16 rounding bound of the normed + rotated keys; slots past a sequence's
length never touched (they hold a NaN sentinel that would poison any read).
"""
import numpy as np
import pytest
import torch

from gpu_util import (GpuCache, MAX_ABS, assert_parity, bits, dev, errors, f64,
                      rope_pair_tolerance)
from gqa_attention_preallocated_qa_gb300.configs import TINY, QWEN3_4B_B1
from gqa_attention_preallocated_qa_gb300.inputs import bf16_bits_to_f64 as F
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


def _oracle_layer(oracle_mod, B, Hq, Hkv, D, cap):
    return oracle_mod.OracleLayer(oracle_mod.Geometry(B=B, Hq=Hq, Hkv=Hkv, D=D, cap=cap))


def _check_cache(c, lay, lens, D, layer=0):
    """K within the rounding bound, V bit-exact, slots >= len untouched, lens exact."""
    K, V, L = c.views(layer)
    Kh, Vh = K.view(torch.int16).cpu().numpy().view(np.uint16), \
        V.view(torch.int16).cpu().numpy().view(np.uint16)
    assert list(L.cpu().numpy()[: len(lens)]) == list(lens)
    for b, n in enumerate(lens):
        got = F(Kh[b, :, :n])
        want = lay.Kc[b, :, :n]
        assert (np.abs(got - want) <= rope_pair_tolerance(want)).all(), f"K slots of seq {b}"
        vwant = lay.Vc[b, :, :n]
        np.testing.assert_array_equal(F(Vh[b, :, :n]), vwant)
        if n < c.cap:
            assert (Kh[b, :, n:] == 0x7FC1).all() and (Vh[b, :, n:] == 0x7FC1).all(), \
                f"seq {b}: slot at or past its length was written"


# ------------------------------------------------------------------ K1 alone
# The last three have token row counts (q, k and v heads) that are not a whole
# number of a warp's passes, and q rows that end mid-pass.
@pytest.mark.parametrize("lens,Hq,Hkv,D,cap", [((64,), 2, 1, 64, 72), ((512,), 32, 8, 128, 544),
                                               ((3, 130, 1, 64), 8, 2, 128, 140),
                                               ((7, 33), 16, 2, 128, 40), ((50,), 12, 6, 64, 56),
                                               ((9, 2), 4, 1, 64, 12)])
def test_k1_transform_matches_oracle(qa, oracle_mod, lens, Hq, Hkv, D, cap):
    inp = layer_inputs(11, lens, Hq, Hkv, D, steps=0)
    c = GpuCache(qa, 1, len(lens), Hq, Hkv, D, cap)
    try:
        c.poison()
        q, k, v, wq, wk = (dev(a) for a in (inp.q, inp.k, inp.v, inp.wq, inp.wk))
        qp = torch.empty_like(q)
        qa.qa_prefill_transform(c.h, 0, list(lens), q, k, v, wq, wk, qp)
        torch.cuda.synchronize()
        lay = _oracle_layer(oracle_mod, len(lens), Hq, Hkv, D, cap)
        want = lay.prefill_transform(lens, F(inp.q), F(inp.k), F(inp.v), F(inp.wq), F(inp.wk))
        got = f64(qp)
        assert (np.abs(got - want) <= rope_pair_tolerance(want)).all()
        # position 0 is the identity rotation: q' there is bf16(w * bf16(x_hat)) exactly
        _check_cache(c, lay, lens, D)
        assert qa.qa_cache_lengths(c.h, 0, len(lens)) == list(lens)
        assert c.device_error() == (0, 0)
    finally:
        c.free()


# ------------------------------------------------------------------ decode on a filled cache
@pytest.mark.parametrize("B,L,Hq,Hkv,D", [(1, 40, 2, 1, 64), (2, 300, 32, 8, 128),
                                          (4, 2048, 32, 8, 128), (1, 5000, 8, 1, 64),
                                          (3, 1000, 16, 2, 64), (2, 333, 4, 4, 128)])
def test_decode_on_prefilled_cache(qa, oracle_mod, B, L, Hq, Hkv, D):
    from gqa_attention_preallocated_qa_gb300.inputs import prefilled_cache_inputs
    inp = prefilled_cache_inputs(21 + L, B, L, Hq, Hkv, D)
    cap = L + 1
    c = GpuCache(qa, 1, B, Hq, Hkv, D, cap)
    try:
        c.poison()
        K, V, _ = c.views()
        K[:, :, :L] = dev(inp.cache_k)
        V[:, :, :L] = dev(inp.cache_v)
        qa.qa_cache_set_lengths(c.h, 0, [L] * B)
        q, k, v, wq, wk = (dev(a) for a in (inp.dq[0], inp.dk[0], inp.dv[0], inp.wq, inp.wk))
        out = torch.empty_like(q)
        qa.qa_decode_step(c.h, 0, B, q, k, v, wq, wk, out)
        torch.cuda.synchronize()
        lay = _oracle_layer(oracle_mod, B, Hq, Hkv, D, cap)
        Kf = np.zeros((B, Hkv, cap, D)); Vf = np.zeros_like(Kf)
        Kf[:, :, :L] = F(inp.cache_k); Vf[:, :, :L] = F(inp.cache_v)
        lay.set_cache(Kf, Vf, [L] * B)
        _, want = lay.decode(F(inp.dq[0]), F(inp.dk[0]), F(inp.dv[0]), F(inp.wq), F(inp.wk))
        assert_parity(f64(out), want, f"decode B={B} L={L}")
        _check_cache(c, lay, [L + 1] * B, D)
        assert c.device_error() == (0, 0)
    finally:
        c.free()


# ------------------------------------------------------------------ prefill + decode, small
@pytest.mark.parametrize("lens,Hq,Hkv,D,steps,cap", [
    (TINY.prompt_lens, TINY.Hq, TINY.Hkv, TINY.D, TINY.steps, TINY.cap),
    (QWEN3_4B_B1.prompt_lens, 32, 8, 128, QWEN3_4B_B1.steps, QWEN3_4B_B1.cap),  # all 32 steps
    ((200, 77, 300, 1, 129), 32, 8, 128, 3, 310),      # ragged, tails of 1 and 127 rows
    ((130, 5), 16, 2, 64, 2, 140),                      # group 8 (two head groups per kv head)
    ((100, 256), 4, 4, 128, 2, 260),                    # group 1 (multi-head)
    (tuple(range(1, 45, 4)), 4, 2, 64, 2, 50),          # 11 sequences: several prefill launches
    # CTA-pair prefill (144 four-head items) with sequence ends inside a warp's
    # 32 rows (direct stores) next to whole warps (TMA stores of the output)
    ((700, 333, 1100), 32, 8, 128, 2, 1110),
    ((1100, 700), 32, 4, 128, 2, 1110),                 # group 8 on CTA pairs (120 items)
])
def test_prefill_then_decode_matches_oracle(qa, oracle_mod, lens, Hq, Hkv, D, steps, cap):
    B = len(lens)
    inp = layer_inputs(31 + sum(lens), lens, Hq, Hkv, D, steps)
    c = GpuCache(qa, 1, B, Hq, Hkv, D, cap)
    try:
        c.poison()
        q, k, v, wq, wk = (dev(a) for a in (inp.q, inp.k, inp.v, inp.wq, inp.wk))
        out = torch.empty_like(q)
        qa.qa_prefill(c.h, 0, list(lens), q, k, v, wq, wk, out)
        torch.cuda.synchronize()
        lay = _oracle_layer(oracle_mod, B, Hq, Hkv, D, cap)
        _, want = lay.prefill(lens, F(inp.q), F(inp.k), F(inp.v), F(inp.wq), F(inp.wk))
        got = f64(out)
        assert_parity(got, want, f"prefill {lens}")
        # Row 0 of every sequence is v_0 of its kv head, bit for bit.
        t0 = 0
        for L in lens:
            if L:
                for h in range(Hq):
                    np.testing.assert_array_equal(got[t0, h], F(inp.v)[t0, h // (Hq // Hkv)])
            t0 += L
        _check_cache(c, lay, lens, D)
        for s in range(steps):
            dq, dk, dv = (dev(a) for a in (inp.dq[s], inp.dk[s], inp.dv[s]))
            o = torch.empty_like(dq)
            qa.qa_decode_step(c.h, 0, B, dq, dk, dv, wq, wk, o)
            torch.cuda.synchronize()
            _, w2 = lay.decode(F(inp.dq[s]), F(inp.dk[s]), F(inp.dv[s]), F(inp.wq), F(inp.wk))
            assert_parity(f64(o), w2, f"decode step {s}")
        _check_cache(c, lay, [L + steps for L in lens], D)
        st = qa.qa_stats(c.h)
        assert st["decode_attn"] == steps and st["prefill_attn"] >= 1
        assert c.device_error() == (0, 0)
    finally:
        c.free()


def test_prefill_is_causal_bit_exact(qa):
    lens, Hq, Hkv, D = (300,), 8, 2, 128
    inp = layer_inputs(41, lens, Hq, Hkv, D, 0)
    outs = []
    for perturb in (False, True):
        k, v = inp.k.copy(), inp.v.copy()
        if perturb:
            k[150:] ^= 0x0040
            v[150:] ^= 0x0040
        c = GpuCache(qa, 1, 1, Hq, Hkv, D, 300)
        try:
            q = dev(inp.q)
            out = torch.empty_like(q)
            qa.qa_prefill(c.h, 0, list(lens), q, dev(k), dev(v), dev(inp.wq), dev(inp.wk), out)
            outs.append(bits(out))
        finally:
            c.free()
    np.testing.assert_array_equal(outs[0][:150], outs[1][:150])
    assert (outs[0][150:] != outs[1][150:]).any()


def test_ragged_batch_equals_sequences_alone_bit_exact(qa):
    lens, Hq, Hkv, D = (70, 300, 129), 32, 8, 128
    inp = layer_inputs(43, lens, Hq, Hkv, D, 0)
    c = GpuCache(qa, 1, 3, Hq, Hkv, D, 300)
    try:
        q = dev(inp.q)
        out = torch.empty_like(q)
        qa.qa_prefill(c.h, 0, list(lens), q, dev(inp.k), dev(inp.v), dev(inp.wq), dev(inp.wk), out)
        full = bits(out)
    finally:
        c.free()
    t0 = 0
    for L in lens:
        c = GpuCache(qa, 1, 1, Hq, Hkv, D, 300)
        try:
            q = dev(inp.q[t0:t0 + L])
            out = torch.empty_like(q)
            qa.qa_prefill(c.h, 0, [L], q, dev(inp.k[t0:t0 + L]), dev(inp.v[t0:t0 + L]),
                          dev(inp.wq), dev(inp.wk), out)
            np.testing.assert_array_equal(bits(out), full[t0:t0 + L])
        finally:
            c.free()
        t0 += L


def test_decode_reproduces_prefill_row_on_gpu(qa):
    # decode at position t == row t of a prefill of t+1 tokens (different kernels: tolerance)
    t, Hq, Hkv, D = 200, 32, 8, 128
    inp = layer_inputs(47, (t + 1,), Hq, Hkv, D, 0)
    q, k, v, wq, wk = (dev(a) for a in (inp.q, inp.k, inp.v, inp.wq, inp.wk))
    c1 = GpuCache(qa, 1, 1, Hq, Hkv, D, t + 1)
    c2 = GpuCache(qa, 1, 1, Hq, Hkv, D, t + 1)
    try:
        full = torch.empty_like(q)
        qa.qa_prefill(c1.h, 0, [t + 1], q, k, v, wq, wk, full)
        part = torch.empty_like(q[:t])
        qa.qa_prefill(c2.h, 0, [t], q[:t].contiguous(), k[:t].contiguous(), v[:t].contiguous(),
                      wq, wk, part)
        o = torch.empty_like(q[t:t + 1])
        qa.qa_decode_step(c2.h, 0, 1, q[t:t + 1].contiguous(), k[t:t + 1].contiguous(),
                          v[t:t + 1].contiguous(), wq, wk, o)
        torch.cuda.synchronize()
        d = (o.float() - full[t:t + 1].float()).abs().max().item()
        assert d <= MAX_ABS
        np.testing.assert_array_equal(bits(part), bits(full[:t]))
    finally:
        c1.free()
        c2.free()


# ------------------------------------------------------------------ edge cases and errors
def test_empty_prompt_then_decode_attends_to_itself(qa):
    lens, Hq, Hkv, D = (0, 17), 4, 2, 64
    inp = layer_inputs(51, lens, Hq, Hkv, D, 1)
    c = GpuCache(qa, 1, 2, Hq, Hkv, D, 20)
    try:
        c.poison()
        q, k, v, wq, wk = (dev(a) for a in (inp.q, inp.k, inp.v, inp.wq, inp.wk))
        out = torch.empty_like(q)
        qa.qa_prefill(c.h, 0, list(lens), q, k, v, wq, wk, out)
        assert qa.qa_cache_lengths(c.h, 0, 2) == [0, 17]
        dq, dk, dv = (dev(a) for a in (inp.dq[0], inp.dk[0], inp.dv[0]))
        o = torch.empty_like(dq)
        qa.qa_decode_step(c.h, 0, 2, dq, dk, dv, wq, wk, o)
        torch.cuda.synchronize()
        # sequence 0 has one key: the output is its own v exactly
        got = bits(o)
        for h in range(Hq):
            np.testing.assert_array_equal(got[0, h], inp.dv[0][0, h // 2])
        assert list(c.views()[2].cpu().numpy()) == [1, 18]
        assert c.device_error() == (0, 0)
    finally:
        c.free()


def test_errors_leave_state_unchanged(qa):
    Hq, Hkv, D = 4, 2, 64
    inp = layer_inputs(53, (8,), Hq, Hkv, D, 2)
    c = GpuCache(qa, 2, 1, Hq, Hkv, D, 8)
    try:
        q, k, v, wq, wk = (dev(a) for a in (inp.q, inp.k, inp.v, inp.wq, inp.wk))
        out = torch.empty_like(q)
        with pytest.raises(qa.QaError) as e:
            qa.qa_prefill(c.h, 0, [9], q, k, v, wq, wk, out)
        assert e.value.status == 4  # capacity
        qa.qa_prefill(c.h, 0, [8], q, k, v, wq, wk, out)  # exactly the capacity
        launched = qa.qa_stats(c.h)  # every call below fails and launches nothing
        with pytest.raises(qa.QaError) as e:
            qa.qa_prefill(c.h, 0, [1], q[:1], k[:1], v[:1], wq, wk, out[:1])
        assert e.value.status == 4  # a further chunk would pass the capacity
        dq, dk, dv = (dev(a) for a in (inp.dq[0], inp.dk[0], inp.dv[0]))
        o = torch.empty_like(dq)
        with pytest.raises(qa.QaError) as e:
            qa.qa_decode_step(c.h, 0, 1, dq, dk, dv, wq, wk, o)
        assert e.value.status == 4  # full: no eviction
        with pytest.raises(qa.QaError) as e:
            qa.qa_decode_step(c.h, 2, 1, dq, dk, dv, wq, wk, o)
        assert e.value.status == 1  # no such layer
        with pytest.raises(qa.QaError) as e:
            qa.qa_decode_step(c.h, 1, 1, dq.data_ptr() + 2, dk, dv, wq, wk, o)
        assert e.value.status == 3  # misaligned
        torch.cuda.synchronize()
        assert qa.qa_cache_lengths(c.h, 0, 1) == [8]
        assert int(c.views(0)[2][0].item()) == 8
        assert qa.qa_stats(c.h) == launched
        assert c.device_error() == (0, 0)
    finally:
        c.free()


def test_reset_rerun_is_bit_identical_and_matches_fresh_cache(qa):
    lens, Hq, Hkv, D, steps = (300, 200), 32, 8, 128, 6
    inp = layer_inputs(57, lens, Hq, Hkv, D, steps)
    q, k, v, wq, wk = (dev(a) for a in (inp.q, inp.k, inp.v, inp.wq, inp.wk))

    def run(c):
        out = torch.empty_like(q)
        qa.qa_prefill(c.h, 0, list(lens), q, k, v, wq, wk, out)
        res = [bits(out)]
        for s in range(steps):
            dq, dk, dv = (dev(a) for a in (inp.dq[s], inp.dk[s], inp.dv[s]))
            o = torch.empty_like(dq)
            qa.qa_decode_step(c.h, 0, 2, dq, dk, dv, wq, wk, o)
            res.append(bits(o))
        return res

    c = GpuCache(qa, 1, 2, Hq, Hkv, D, 320)
    try:
        first = run(c)
        for _ in range(2):
            qa.qa_cache_reset(c.h)
            again = run(c)
            for a, b in zip(first, again):
                np.testing.assert_array_equal(a, b)
    finally:
        c.free()
    c = GpuCache(qa, 1, 2, Hq, Hkv, D, 320)
    try:
        fresh = run(c)
        for a, b in zip(first, fresh):
            np.testing.assert_array_equal(a, b)
    finally:
        c.free()
