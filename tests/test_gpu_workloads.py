"""Full-size workloads on the GPU, checked against the oracle on sampled
outputs (the oracle computes them one by one) and on properties that hold at
any size.

- B=4, prompts of 2048, 128 decode steps, capacity 2176 (the benchmark's
  launch configuration), run three times with a cache reset in between.
- B=4 ragged prompts (512, 1024, 1536, 2048), 64 decode steps, 36 independent
  layer caches: every layer's decode steps 0 and 63 on one head per kv group,
  and layers 0, 17 and 35 in full (every prompt row on one head plus sampled
  rows on two more, every decode step on every head, the cache slots).
- Decode sweep: B in {1, 4} x cache length in {512, 2048, 8192, 16384}, cache
  filled with raw N(0,1) keys/values, one decode step, every head checked.
"""
import numpy as np
import pytest
import torch

from gpu_util import (GpuCache, SENTINEL_BITS, assert_parity, bits, dev, f64,
                      rope_pair_tolerance)
from gqa_attention_preallocated_qa_gb300.configs import DECODE_SWEEP, QWEN3_4B_B4, RAGGED_36L
from gqa_attention_preallocated_qa_gb300.inputs import bf16_bits_to_f64 as F

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def qa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gqa_attention_preallocated_qa_gb300 import _build
    _build.build()
    from gqa_attention_preallocated_qa_gb300 import binding
    return binding


def sample_rows(L, rng, extra=12):
    rows = {0, 1, 2, 63, 64, 127, 128, 129, 255, 256, 511, 512, 1023, 1024, 1535, 2046, 2047,
            4095, 4096, 6143, 8190, 8191}
    rows = {r for r in rows if r < L} | {L - 1}
    rows |= set(rng.integers(0, L, size=extra).tolist())
    return sorted(rows)


def check_prefill_rows(lay, w, qp, got, lens, rng, heads):
    t0 = 0
    for b, L in enumerate(lens):
        want_rows, got_rows = [], []
        for i in sample_rows(L, rng):
            for h in heads:
                want_rows.append(lay.prefill_row(b, h, i, qp[t0 + i, h]))
                got_rows.append(got[t0 + i, h])
        assert_parity(np.array(got_rows), np.array(want_rows), f"prefill seq {b}")
        t0 += L


def check_cache(c, lay, lens, layer=0):
    K, V, Ld = c.views(layer)
    assert list(Ld.cpu().numpy()[: len(lens)]) == list(lens)
    Kh = K.view(torch.int16).cpu().numpy().view(np.uint16)
    Vh = V.view(torch.int16).cpu().numpy().view(np.uint16)
    for b, n in enumerate(lens):
        want = lay.Kc[b, :, :n]
        assert (np.abs(F(Kh[b, :, :n]) - want) <= rope_pair_tolerance(want)).all(), f"K of seq {b}"
        np.testing.assert_array_equal(F(Vh[b, :, :n]), lay.Vc[b, :, :n])
        if n < c.cap:
            assert (Kh[b, :, n:] == SENTINEL_BITS).all() and (Vh[b, :, n:] == SENTINEL_BITS).all()


def test_b4_prompt2048_128_steps_with_reset_reruns(qa, oracle_mod):
    w = QWEN3_4B_B4
    inp = w.inputs()
    rng = np.random.default_rng(123)
    c = GpuCache(qa, 1, w.B, w.Hq, w.Hkv, w.D, w.cap)
    try:
        c.poison()
        q, k, v, wq, wk = (dev(a) for a in (inp.q, inp.k, inp.v, inp.wq, inp.wk))
        dq, dk, dv = dev(inp.dq), dev(inp.dk), dev(inp.dv)
        runs = []
        for run in range(w.reruns):
            if run:
                qa.qa_cache_reset(c.h)
            out = torch.empty_like(q)
            qa.qa_prefill(c.h, 0, list(w.prompt_lens), q, k, v, wq, wk, out)
            douts = torch.empty((w.steps, w.B, w.Hq, w.D), dtype=torch.bfloat16, device="cuda")
            for s in range(w.steps):
                qa.qa_decode_step(c.h, 0, w.B, dq[s], dk[s], dv[s], wq, wk, douts[s])
            torch.cuda.synchronize()
            runs.append((bits(out), bits(douts)))
        for pre, dec in runs[1:]:  # reset state is clean: reruns are bit-identical
            np.testing.assert_array_equal(pre, runs[0][0])
            np.testing.assert_array_equal(dec, runs[0][1])
        got_pre = F(runs[0][0])
        got_dec = F(runs[0][1])
        lay = oracle_mod.OracleLayer(oracle_mod.Geometry(w.B, w.Hq, w.Hkv, w.D, w.cap))
        qp = lay.prefill_transform(w.prompt_lens, F(inp.q), F(inp.k), F(inp.v), F(inp.wq),
                                   F(inp.wk))
        check_prefill_rows(lay, w, qp, got_pre, w.prompt_lens, rng, heads=(0, 3, 4, 17, 31))
        for s in range(w.steps):  # every decode step, every head
            qd = lay.decode_transform(F(inp.dq[s]), F(inp.dk[s]), F(inp.dv[s]), F(inp.wq),
                                      F(inp.wk))
            want = np.array([[lay.attend_cached(b, h, qd[b, h]) for h in range(w.Hq)]
                             for b in range(w.B)])
            assert_parity(got_dec[s], want, f"decode step {s}")
        check_cache(c, lay, [w.cap] * w.B)
        assert c.device_error() == (0, 0)
    finally:
        c.free()


def check_all_prefill_rows(lay, qp, got, lens, head):
    """Every prompt row of every sequence on one head."""
    want_rows, got_rows = [], []
    t0 = 0
    for b, L in enumerate(lens):
        for i in range(L):
            want_rows.append(lay.prefill_row(b, head, i, qp[t0 + i, head]))
            got_rows.append(got[t0 + i, head])
        t0 += L
    assert_parity(np.array(got_rows), np.array(want_rows), f"all prompt rows, head {head}")


def test_ragged_prompts_36_layers(qa, oracle_mod):
    w = RAGGED_36L
    rng = np.random.default_rng(7)
    tracked = (0, 17, 35)
    every_layer_steps = (0, w.steps - 1)
    c = GpuCache(qa, w.layers, w.B, w.Hq, w.Hkv, w.D, w.cap)
    try:
        c.poison(tracked)
        layers = {}
        dec = []
        for l in range(w.layers):
            inp = w.inputs(l)
            q, k, v, wq, wk = (dev(a) for a in (inp.q, inp.k, inp.v, inp.wq, inp.wk))
            out = torch.empty_like(q)
            qa.qa_prefill(c.h, l, list(w.prompt_lens), q, k, v, wq, wk, out)
            dec.append((dev(inp.dq), dev(inp.dk), dev(inp.dv), wq, wk))
            if l in tracked:
                torch.cuda.synchronize()
                layers[l] = F(bits(out))
            del q, k, v, out, inp
        douts = {l: torch.empty((w.steps, w.B, w.Hq, w.D), dtype=torch.bfloat16, device="cuda")
                 for l in tracked}
        # steps 0 and 63 of every layer
        souts = torch.empty((len(every_layer_steps), w.layers, w.B, w.Hq, w.D), dtype=torch.bfloat16,
                            device="cuda")
        scratch = torch.empty((w.B, w.Hq, w.D), dtype=torch.bfloat16, device="cuda")
        for s in range(w.steps):          # the generate loop: every layer, step by step
            for l in range(w.layers):
                dq, dk, dv, wq, wk = dec[l]
                if l in tracked:
                    o = douts[l][s]
                elif s in every_layer_steps:
                    o = souts[every_layer_steps.index(s), l]
                else:
                    o = scratch
                qa.qa_decode_step(c.h, l, w.B, dq[s], dk[s], dv[s], wq, wk, o)
                if l in tracked and s in every_layer_steps:
                    souts[every_layer_steps.index(s), l].copy_(o)
        torch.cuda.synchronize()
        final = [L + w.steps for L in w.prompt_lens]
        for l in range(w.layers):
            assert qa.qa_cache_lengths(c.h, l, w.B) == final
            assert list(c.views(l)[2].cpu().numpy()) == final
        got_steps = f64(souts)
        G = w.Hq // w.Hkv
        for l in range(w.layers):
            inp = w.inputs(l)
            lay = oracle_mod.OracleLayer(oracle_mod.Geometry(w.B, w.Hq, w.Hkv, w.D, w.cap))
            qp = lay.prefill_transform(w.prompt_lens, F(inp.q), F(inp.k), F(inp.v), F(inp.wq),
                                       F(inp.wk))
            if l in tracked:
                check_all_prefill_rows(lay, qp, layers[l], w.prompt_lens, head=(l % w.Hq))
                check_prefill_rows(lay, w, qp, layers[l], w.prompt_lens, rng, heads=(1, 30))
                got_dec = f64(douts[l])
            for s in range(w.steps):
                qd = lay.decode_transform(F(inp.dq[s]), F(inp.dk[s]), F(inp.dv[s]), F(inp.wq),
                                          F(inp.wk))
                if l in tracked:  # every step, every head
                    want = np.array([[lay.attend_cached(b, h, qd[b, h]) for h in range(w.Hq)]
                                     for b in range(w.B)])
                    assert_parity(got_dec[s], want, f"layer {l} decode step {s}")
                if s in every_layer_steps:  # one head per kv group, rotating with the layer
                    heads = [kvh * G + (l + kvh) % G for kvh in range(w.Hkv)]
                    want = np.array([[lay.attend_cached(b, h, qd[b, h]) for h in heads]
                                     for b in range(w.B)])
                    got = got_steps[every_layer_steps.index(s), l][:, heads]
                    assert_parity(got, want, f"layer {l} decode step {s}")
            if l in tracked:
                check_cache(c, lay, final, layer=l)
        assert c.device_error() == (0, 0)
        assert qa.qa_stats(c.h)["decode_attn"] == w.layers * w.steps
    finally:
        c.free()


@pytest.mark.parametrize("pt", DECODE_SWEEP, ids=lambda p: p.name)
def test_decode_sweep_point(qa, oracle_mod, pt):
    inp = pt.inputs()
    c = GpuCache(qa, 1, pt.B, pt.Hq, pt.Hkv, pt.D, pt.cap)
    try:
        K, V, _ = c.views()
        K[:, :, : pt.L] = dev(inp.cache_k)
        V[:, :, : pt.L] = dev(inp.cache_v)
        qa.qa_cache_set_lengths(c.h, 0, [pt.L] * pt.B)
        q, k, v, wq, wk = (dev(a) for a in (inp.dq[0], inp.dk[0], inp.dv[0], inp.wq, inp.wk))
        out = torch.empty_like(q)
        qa.qa_decode_step(c.h, 0, pt.B, q, k, v, wq, wk, out)
        torch.cuda.synchronize()
        got = f64(out)
        wq_, wk_ = F(inp.wq), F(inp.wk)
        G = pt.Hq // pt.Hkv
        want = np.empty_like(got)
        Kh = K.view(torch.int16).cpu().numpy().view(np.uint16)
        for b in range(pt.B):
            for kvh in range(pt.Hkv):
                kn = oracle_mod.rope(oracle_mod.rmsnorm(F(inp.dk[0][b, kvh]), wk_, pt.eps), pt.L,
                                     pt.theta)
                Kf = np.concatenate([F(inp.cache_k[b, kvh]), kn[None]])
                Vf = np.concatenate([F(inp.cache_v[b, kvh]), F(inp.dv[0][b, kvh])[None]])
                got_k = F(Kh[b, kvh, pt.L])
                assert (np.abs(got_k - kn) <= rope_pair_tolerance(kn)).all()
                for g in range(G):
                    h = kvh * G + g
                    qn = oracle_mod.rope(oracle_mod.rmsnorm(F(inp.dq[0][b, h]), wq_, pt.eps),
                                         pt.L, pt.theta)
                    want[b, h] = oracle_mod.attend(qn, Kf, Vf)[0]
        assert_parity(got, want, pt.name)
        assert qa.qa_cache_lengths(c.h, 0, pt.B) == [pt.L + 1] * pt.B
        assert c.device_error() == (0, 0)
    finally:
        c.free()


# Long prompts: up to 64 key tiles per query block, so every ring and Q slot of
# the prefill goes through many phases.  The first geometry runs the CTA-pair
# prefill (704 four-head items), the second the one-CTA form (head_dim 64).
@pytest.mark.parametrize("lens,Hq,Hkv,D", [((8192, 3000), 32, 8, 128), ((6000,), 16, 2, 64)])
def test_long_prompts_sampled_rows_and_decode(qa, oracle_mod, lens, Hq, Hkv, D):
    from gqa_attention_preallocated_qa_gb300.inputs import layer_inputs
    steps = 2
    cap = max(lens) + steps
    inp = layer_inputs(91, lens, Hq, Hkv, D, steps)
    rng = np.random.default_rng(91)
    c = GpuCache(qa, 1, len(lens), Hq, Hkv, D, cap)
    try:
        c.poison()
        q, k, v, wq, wk = (dev(a) for a in (inp.q, inp.k, inp.v, inp.wq, inp.wk))
        out = torch.empty_like(q)
        qa.qa_prefill(c.h, 0, list(lens), q, k, v, wq, wk, out)
        douts = []
        for s in range(steps):
            o = torch.empty_like(dev(inp.dq[s]))
            qa.qa_decode_step(c.h, 0, len(lens), dev(inp.dq[s]), dev(inp.dk[s]), dev(inp.dv[s]),
                              wq, wk, o)
            douts.append(o)
        torch.cuda.synchronize()
        lay = oracle_mod.OracleLayer(oracle_mod.Geometry(len(lens), Hq, Hkv, D, cap))
        qp = lay.prefill_transform(lens, F(inp.q), F(inp.k), F(inp.v), F(inp.wq), F(inp.wk))
        check_prefill_rows(lay, None, qp, f64(out), lens, rng, heads=(0, Hq // 2 - 1, Hq - 1))
        for s in range(steps):
            qd = lay.decode_transform(F(inp.dq[s]), F(inp.dk[s]), F(inp.dv[s]), F(inp.wq),
                                      F(inp.wk))
            want = np.array([[lay.attend_cached(b, h, qd[b, h]) for h in range(Hq)]
                             for b in range(len(lens))])
            assert_parity(f64(douts[s]), want, f"decode step {s} after long prompts")
        check_cache(c, lay, [L + steps for L in lens])
        assert c.device_error() == (0, 0)
    finally:
        c.free()
