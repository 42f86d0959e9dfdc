"""Short chunks (at most 8 new tokens per sequence: the verify step of
speculative decoding, or a short append) run as the decode kernel's
multi-token form: every (sequence, kv head) streams its cache once for all of
its new tokens, token t attends to the cache and to new tokens 0..t.

Expected values come from the oracle's primitives one token at a time
(ChunkOracle, WindowOracle): the definition does not depend on which kernel
serves a chunk.  The last test runs steps back to back on one layer with no
host synchronisation in between (each launch overlapping the previous one) and
requires the outputs of the same steps run one at a time, bit for bit.
"""
import numpy as np
import pytest
import torch

from gpu_util import GpuCache, assert_parity, bits, dev, f64
from gqa_attention_preallocated_qa_gb300.inputs import bf16_bits_to_f64 as F
from gqa_attention_preallocated_qa_gb300.inputs import layer_inputs
from test_gpu_chunked_prefill import ChunkOracle, run_chunks
from test_gpu_window import WindowOracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def qa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gqa_attention_preallocated_qa_gb300 import _build
    _build.build()
    from gqa_attention_preallocated_qa_gb300 import binding
    return binding


def test_short_chunks_qwen3_geometry(qa, oracle_mod):
    # A long first chunk (prefill kernels), then short ones that take each
    # multi-token shape: 8 tokens (1 head x 8 tokens per CTA), 2 (4 x 2),
    # 3 and 4 (2 x 4), 1; sequences without new tokens in between.
    chunks = [(300, 129, 1, 700), (3, 8, 0, 1), (2, 2, 2, 2), (4, 1, 3, 0), (1, 1, 1, 1)]
    run_chunks(qa, oracle_mod, chunks, 32, 8, 128, 740, seed=131, decode_steps=2,
               heads=tuple(range(32)), rows_per_chunk=8)


def test_short_chunks_one_head_per_group(qa, oracle_mod):
    # G = 1 (one head per CTA, 8 token rows), D = 64; the first chunks start
    # from an empty cache (no cache keys: only the new tokens).
    chunks = [(5, 0), (8, 7), (1, 2), (10, 3)]
    run_chunks(qa, oracle_mod, chunks, 2, 2, 64, 64, seed=137, decode_steps=2,
               heads=(0, 1), rows_per_chunk=10)


def test_short_chunks_count_as_decode_launches(qa):
    Hq, Hkv, D = 32, 8, 128
    inp = layer_inputs(139, (40, 3), Hq, Hkv, D, 0)
    c = GpuCache(qa, 1, 2, Hq, Hkv, D, 64)
    try:
        q, k, v, wq, wk = (dev(a) for a in (inp.q, inp.k, inp.v, inp.wq, inp.wk))
        out = torch.empty_like(q)
        qa.qa_prefill(c.h, 0, [40, 3], q, k, v, wq, wk, out)
        s0 = qa.qa_stats(c.h)
        o = torch.empty_like(q[:5])
        qa.qa_prefill(c.h, 0, [3, 2], q[:5], k[:5], v[:5], wq, wk, o)
        torch.cuda.synchronize()
        s1 = qa.qa_stats(c.h)
        assert s1["prefill_attn"] == s0["prefill_attn"]
        assert s1["norm_rope_append"] == s0["norm_rope_append"]
        assert s1["decode_attn"] == s0["decode_attn"] + 1
        assert qa.qa_cache_lengths(c.h, 0, 2) == [43, 5]
        assert c.device_error() == (0, 0)
    finally:
        c.free()


@pytest.mark.parametrize("window", [1, 3, 64])
def test_short_chunks_with_window(qa, oracle_mod, window):
    """Windows narrower than a chunk (1, 3) and wider: token t at pos + t sees
    keys from pos + t + 1 - W, among them the earlier new tokens of its chunk."""
    HQ, HKV, D = 32, 8, 128
    chunks = [(300, 129, 1, 40), (3, 8, 0, 1), (2, 2, 2, 2)]
    steps, cap = 2, 360
    inps = [layer_inputs(149 + n, lens, HQ, HKV, D, steps if n == len(chunks) - 1 else 0)
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
                rows = range(L) if L <= 8 else sorted(
                    {0, L - 1, min(L - 1, window), min(L - 1, 128)} |
                    set(rng.integers(0, L, size=6).tolist()))
                for i in rows:
                    for h in (0, 3, 4, 17, 31):
                        want.append(orc.out_row(b, start[b] + i, h, qf[t0 + i, h]))
                        have.append(got[t0 + i, h])
                t0 += L
            assert_parity(np.array(have), np.array(want), f"window {window} chunk {n}")
        inp = inps[-1]
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


def test_window_of_one_returns_each_tokens_own_value(qa):
    """W = 1: every token attends to itself only, so its output is its own v
    (rounded to bf16: exactly v), through the prefill kernels, the
    multi-token form and the decode step alike."""
    HQ, HKV, D = 32, 8, 128
    G = HQ // HKV
    chunks = [(200, 1, 130), (5, 2, 8)]
    c = GpuCache(qa, 1, 3, HQ, HKV, D, 400)
    try:
        qa.qa_cache_set_window(c.h, 0, 1)
        for n, lens in enumerate(chunks):
            inp = layer_inputs(157 + n, lens, HQ, HKV, D, 2 if n else 0)
            q, k, v, wq, wk = (dev(a) for a in (inp.q, inp.k, inp.v, inp.wq, inp.wk))
            out = torch.empty_like(q)
            qa.qa_prefill(c.h, 0, list(lens), q, k, v, wq, wk, out)
            torch.cuda.synchronize()
            want = np.repeat(F(inp.v), G, axis=1)  # query head h reads kv head h // G
            np.testing.assert_array_equal(f64(out), want)
        for s in range(2):
            dq, dk, dv = dev(inp.dq[s]), dev(inp.dk[s]), dev(inp.dv[s])
            o = torch.empty_like(dq)
            qa.qa_decode_step(c.h, 0, 3, dq, dk, dv, wq, wk, o)
            torch.cuda.synchronize()
            np.testing.assert_array_equal(f64(o), np.repeat(F(inp.dv[s]), G, axis=1))
        assert c.device_error() == (0, 0)
    finally:
        c.free()


def test_back_to_back_steps_equal_synchronised_steps(qa):
    """Decode steps and short chunks on one layer, launched back to back (each
    launch may start while the previous one still runs), give the outputs and
    cache of the same calls with a host synchronisation after each."""
    Hq, Hkv, D, B = 32, 8, 128, 4
    prompt = (63, 64, 95, 33)  # the first slots sit at and next to chunk boundaries
    plan = ["d", "d", 3, "d", 8, "d", "d", 2, "d"] + ["d"] * 24 + [5, "d", "d"]
    ntok = sum(1 if x == "d" else x for x in plan)
    cap = max(prompt) + ntok + 1
    inp = layer_inputs(163, prompt, Hq, Hkv, D, ntok)
    wq, wk = dev(inp.wq), dev(inp.wk)
    # per call: q, k, v of its tokens (decode: [B, H, D]; chunk: [B * x, H, D])
    calls, t = [], 0
    for x in plan:
        n = 1 if x == "d" else x
        sl = slice(t, t + n)
        tq = np.ascontiguousarray(inp.dq[sl].transpose(1, 0, 2, 3)).reshape(B * n, Hq, D)
        tk = np.ascontiguousarray(inp.dk[sl].transpose(1, 0, 2, 3)).reshape(B * n, Hkv, D)
        tv = np.ascontiguousarray(inp.dv[sl].transpose(1, 0, 2, 3)).reshape(B * n, Hkv, D)
        calls.append((x, dev(tq), dev(tk), dev(tv), torch.empty((B * n, Hq, D), dtype=torch.bfloat16,
                                                                device="cuda")))
        t += n
    res = []
    for sync in (True, False):
        c = GpuCache(qa, 1, B, Hq, Hkv, D, cap)
        try:
            q, k, v = dev(inp.q), dev(inp.k), dev(inp.v)
            out = torch.empty_like(q)
            qa.qa_prefill(c.h, 0, list(prompt), q, k, v, wq, wk, out)
            torch.cuda.synchronize()
            for x, tq, tk, tv, o in calls:
                if x == "d":
                    qa.qa_decode_step(c.h, 0, B, tq, tk, tv, wq, wk, o)
                else:
                    qa.qa_prefill(c.h, 0, [x] * B, tq, tk, tv, wq, wk, o)
                if sync:
                    torch.cuda.synchronize()
            torch.cuda.synchronize()
            K, V, L = c.views()
            res.append(([bits(o) for *_, o in calls], bits(K), bits(V), list(L.cpu().numpy())))
            assert c.device_error() == (0, 0)
        finally:
            c.free()
    (oa, Ka, Va, La), (ob, Kb, Vb, Lb) = res
    assert La == Lb == [n + ntok for n in prompt]
    for i, (a, b) in enumerate(zip(oa, ob)):
        np.testing.assert_array_equal(a, b, err_msg=f"call {i} ({plan[i]})")
    np.testing.assert_array_equal(Ka, Kb)
    np.testing.assert_array_equal(Va, Vb)


def test_decode_overlap_changes_splits_not_results(qa, oracle_mod):
    """qa_cache_set_decode_overlap only sets how many launches the split plan
    fits on the device at once: fewer splits for more overlap, and the same
    attention (every setting within the parity bar of the oracle)."""
    Hq, Hkv, D, B = 32, 8, 128, 4
    prompt = (600, 700, 520, 650)
    steps, cap = 3, 720
    inp = layer_inputs(167, prompt, Hq, Hkv, D, steps)
    wq, wk = dev(inp.wq), dev(inp.wk)
    splits, outs = {}, {}
    for overlap in (1, 2, 4):
        c = GpuCache(qa, 1, B, Hq, Hkv, D, cap)
        try:
            qa.qa_cache_set_decode_overlap(c.h, overlap)
            q, k, v = dev(inp.q), dev(inp.k), dev(inp.v)
            out = torch.empty_like(q)
            qa.qa_prefill(c.h, 0, list(prompt), q, k, v, wq, wk, out)
            splits[overlap] = qa.qa_decode_splits(c.h, 0, B)
            res = []
            for s in range(steps):
                o = torch.empty((B, Hq, D), dtype=torch.bfloat16, device="cuda")
                qa.qa_decode_step(c.h, 0, B, dev(inp.dq[s]), dev(inp.dk[s]), dev(inp.dv[s]), wq, wk, o)
                res.append(o)
            torch.cuda.synchronize()
            outs[overlap] = np.stack([f64(o) for o in res])
            with pytest.raises(qa.QaError):
                qa.qa_cache_set_decode_overlap(c.h, 0)
            with pytest.raises(qa.QaError):
                qa.qa_cache_set_decode_overlap(c.h, 9)
            assert c.device_error() == (0, 0)
        finally:
            c.free()
    assert splits[1] > splits[4] >= 1 and splits[1] >= splits[2] >= splits[4]
    orc = ChunkOracle(oracle_mod, B, Hq, Hkv, D, cap, inp.wq, inp.wk)
    t0 = 0
    for b, L in enumerate(prompt):
        orc.append(b, F(inp.k[t0:t0 + L]), F(inp.v[t0:t0 + L]))
        t0 += L
    want = []
    for s in range(steps):
        row = []
        for b in range(B):
            orc.append(b, F(inp.dk[s][b][None]), F(inp.dv[s][b][None]))
            row.append([orc.out_row(b, orc.lens[b] - 1, h, F(inp.dq[s][b, h])) for h in (0, 9, 22, 31)])
        want.append(row)
    want = np.array(want)
    for overlap, got in outs.items():
        assert_parity(got[:, :, (0, 9, 22, 31)], want, f"overlap {overlap}")


@pytest.mark.parametrize("Hq,Hkv,D,chunks", [
    (16, 2, 128, [(40, 9), (3, 8), (2, 1), (1, 4)]),    # G = 8: two head groups per kv head
    (4, 2, 64, [(20, 33), (5, 3), (8, 8), (2, 0)]),     # G = 2
])
def test_short_chunks_other_groupings(qa, oracle_mod, Hq, Hkv, D, chunks):
    run_chunks(qa, oracle_mod, chunks, Hq, Hkv, D, 80, seed=173 + Hq, decode_steps=2,
               heads=tuple(range(Hq)), rows_per_chunk=8)


def test_short_chunks_over_64_sequences(qa, oracle_mod):
    """More sequences than one launch carries: several multi-token launches in
    one call (and sequences without new tokens skipped)."""
    B = 80
    rng = np.random.default_rng(179)
    prompt = tuple(int(x) for x in rng.integers(1, 40, size=B))
    short = tuple(0 if i % 10 == 3 else 1 + i % 3 for i in range(B))  # 72 sequences with tokens
    run_chunks(qa, oracle_mod, [prompt, short], 2, 1, 64, 48, seed=181, decode_steps=1,
               heads=(0, 1), rows_per_chunk=3)
