"""Chunked prefill on the GPU: qa_prefill appends each call's tokens after what
the layer already holds, so a prompt can arrive in several chunks (and a
decode step can follow any of them).

Expected values come from the oracle's primitives applied token by token in
the order of the definition: the new token at position pos is normed and
rotated at pos, appended, and attends to the sequence's keys 0..pos.  That a
decode step at position t reproduces prefill row t is pinned in the oracle's
own tests, so this is the oracle's prefill with the first positions already
taken.
"""
import numpy as np
import pytest
import torch

from gpu_util import GpuCache, SENTINEL_BITS, assert_parity, bits, dev, f64, rope_pair_tolerance
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


class ChunkOracle:
    """The cache contents and attention outputs of the definition, one new token
    at a time (fp64, oracle primitives only)."""

    def __init__(self, om, B, Hq, Hkv, D, cap, wq, wk, theta=1e6, eps=1e-6):
        self.om, self.Hq, self.Hkv, self.D = om, Hq, Hkv, D
        self.G = Hq // Hkv
        self.wq, self.wk, self.theta, self.eps = F(wq), F(wk), theta, eps
        self.K = np.zeros((B, Hkv, cap, D))
        self.V = np.zeros((B, Hkv, cap, D))
        self.lens = [0] * B

    def append(self, b, k_rows, v_rows):
        om = self.om
        for i in range(k_rows.shape[0]):
            pos = self.lens[b] + i
            for h in range(self.Hkv):
                self.K[b, h, pos] = om.rope(om.rmsnorm(k_rows[i, h], self.wk, self.eps), pos, self.theta)
                self.V[b, h, pos] = v_rows[i, h]
        self.lens[b] += k_rows.shape[0]

    def out_row(self, b, pos, h, q_row):
        om = self.om
        qp = om.rope(om.rmsnorm(q_row, self.wq, self.eps), pos, self.theta)
        return om.attend(qp, self.K[b, h // self.G, :pos + 1], self.V[b, h // self.G, :pos + 1])[0]


def run_chunks(qa, om, chunks, Hq, Hkv, D, cap, seed, decode_steps, heads, rows_per_chunk):
    B = len(chunks[0])
    inps = [layer_inputs(seed + 7 * n, lens, Hq, Hkv, D, decode_steps if n == len(chunks) - 1 else 0)
            for n, lens in enumerate(chunks)]
    wq, wk = inps[0].wq, inps[0].wk  # one layer: the same norm weights for every chunk
    c = GpuCache(qa, 1, B, Hq, Hkv, D, cap)
    orc = ChunkOracle(om, B, Hq, Hkv, D, cap, wq, wk)
    rng = np.random.default_rng(seed)
    try:
        c.poison()
        wq_d, wk_d = dev(wq), dev(wk)
        for n, (lens, inp) in enumerate(zip(chunks, inps)):
            q, k, v = dev(inp.q), dev(inp.k), dev(inp.v)
            out = torch.empty_like(q)
            start = list(orc.lens)
            qa.qa_prefill(c.h, 0, list(lens), q, k, v, wq_d, wk_d, out)
            torch.cuda.synchronize()
            got = f64(out)
            qf = F(inp.q)
            t0 = 0
            want, have = [], []
            for b, L in enumerate(lens):
                orc.append(b, F(inp.k[t0:t0 + L]), F(inp.v[t0:t0 + L]))
                if L:
                    rows = {0, L - 1} | set(rng.integers(0, L, size=rows_per_chunk).tolist())
                    for i in sorted(rows):
                        for h in heads:
                            want.append(orc.out_row(b, start[b] + i, h, qf[t0 + i, h]))
                            have.append(got[t0 + i, h])
                t0 += L
            if want:
                assert_parity(np.array(have), np.array(want), f"chunk {n} {lens}")
            assert qa.qa_cache_lengths(c.h, 0, B) == orc.lens
        inp = inps[-1]
        for s in range(decode_steps):
            dq, dk, dv = dev(inp.dq[s]), dev(inp.dk[s]), dev(inp.dv[s])
            o = torch.empty_like(dq)
            qa.qa_decode_step(c.h, 0, B, dq, dk, dv, wq_d, wk_d, o)
            torch.cuda.synchronize()
            want = []
            for b in range(B):
                orc.append(b, F(inp.dk[s][b][None]), F(inp.dv[s][b][None]))
                want.append([orc.out_row(b, orc.lens[b] - 1, h, F(inp.dq[s][b, h])) for h in range(Hq)])
            assert_parity(f64(o), np.array(want), f"decode step {s} after chunks")
        # Cache: every written slot against the definition, nothing past a length.
        K, V, Ld = c.views()
        assert list(Ld.cpu().numpy()[:B]) == orc.lens
        Kh = K.view(torch.int16).cpu().numpy().view(np.uint16)
        Vh = V.view(torch.int16).cpu().numpy().view(np.uint16)
        for b, n in enumerate(orc.lens):
            wantk = orc.K[b, :, :n]
            assert (np.abs(F(Kh[b, :, :n]) - wantk) <= rope_pair_tolerance(wantk)).all(), f"K of seq {b}"
            np.testing.assert_array_equal(F(Vh[b, :, :n]), orc.V[b, :, :n])
            if n < cap:
                assert (Kh[b, :, n:] == SENTINEL_BITS).all() and (Vh[b, :, n:] == SENTINEL_BITS).all()
        assert c.device_error() == (0, 0)
    finally:
        c.free()


def test_chunked_prefill_qwen3_geometry(qa, oracle_mod):
    # Chunk starts off and on the 128-row tile grid, an empty first chunk,
    # one-token and zero-token chunks, then decode steps.
    chunks = [(100, 256, 0, 383), (300, 100, 130, 1), (0, 50, 200, 129)]
    run_chunks(qa, oracle_mod, chunks, 32, 8, 128, 600, seed=61, decode_steps=3,
               heads=(0, 5, 17, 31), rows_per_chunk=12)


def test_chunked_prefill_on_cta_pairs(qa, oracle_mod):
    # The second chunk has 96 four-head items (two sequences x 6 query blocks x
    # 8 kv heads): the CTA-pair prefill, at start offsets off the tile grid.
    chunks = [(300, 250), (700, 701)]
    run_chunks(qa, oracle_mod, chunks, 32, 8, 128, 1010, seed=71, decode_steps=2,
               heads=(0, 3, 13, 30), rows_per_chunk=10)


def test_chunked_prefill_one_tile_per_cta(qa, oracle_mod):
    # G = 1: a CTA has a single query tile (no head pair); D = 64.
    chunks = [(10, 0), (60, 7), (2, 130)]
    run_chunks(qa, oracle_mod, chunks, 2, 2, 64, 150, seed=67, decode_steps=2,
               heads=(0, 1), rows_per_chunk=40)


def test_chunked_prefill_matches_one_shot_prefill(qa):
    """The same prompt in one call and in three chunks gives the same cache bit
    for bit (K1 is per token) and attention outputs within the parity bar of
    each other (tile boundaries differ, so the summation order differs)."""
    Hq, Hkv, D, L = 32, 8, 128, 520
    inp = layer_inputs(71, (L,), Hq, Hkv, D, 0)
    q, k, v, wq, wk = (dev(a) for a in (inp.q, inp.k, inp.v, inp.wq, inp.wk))
    outs, caches = [], []
    for parts in ((L,), (129, 255, 136)):
        c = GpuCache(qa, 1, 1, Hq, Hkv, D, L)
        try:
            out = torch.empty_like(q)
            r0 = 0
            for n in parts:
                qa.qa_prefill(c.h, 0, [n], q[r0:r0 + n], k[r0:r0 + n], v[r0:r0 + n], wq, wk,
                              out[r0:r0 + n])
                r0 += n
            torch.cuda.synchronize()
            K, V, _ = c.views()
            outs.append(f64(out))
            caches.append((bits(K), bits(V)))
            assert c.device_error() == (0, 0)
        finally:
            c.free()
    np.testing.assert_array_equal(caches[0][0], caches[1][0])
    np.testing.assert_array_equal(caches[0][1], caches[1][1])
    d = np.abs(outs[0] - outs[1])
    assert d.max() <= 2e-2 and d.mean() <= 2e-3


def test_multi_token_verify_equals_sequential_decode(qa):
    """A k-token query against the cache (the verify step of speculative
    decoding) is a chunked prefill of k tokens: it matches k decode steps of
    the same tokens within the parity bar, and leaves the same cache (V bit for
    bit, K within the rounding bound)."""
    Hq, Hkv, D, B, k = 32, 8, 128, 4, 4
    prompt = (200, 129, 1, 300)
    inp = layer_inputs(73, prompt, Hq, Hkv, D, k)
    q, kk, v, wq, wk = (dev(a) for a in (inp.q, inp.k, inp.v, inp.wq, inp.wk))
    # verify tokens packed per sequence: [B*k] rows, sequence b's k tokens together
    vq = dev(np.ascontiguousarray(inp.dq.transpose(1, 0, 2, 3)).reshape(B * k, Hq, D))
    vk = dev(np.ascontiguousarray(inp.dk.transpose(1, 0, 2, 3)).reshape(B * k, Hkv, D))
    vv = dev(np.ascontiguousarray(inp.dv.transpose(1, 0, 2, 3)).reshape(B * k, Hkv, D))
    res = []
    for mode in ("verify", "decode"):
        c = GpuCache(qa, 1, B, Hq, Hkv, D, 320)
        try:
            out = torch.empty_like(q)
            qa.qa_prefill(c.h, 0, list(prompt), q, kk, v, wq, wk, out)
            if mode == "verify":
                o = torch.empty_like(vq)
                qa.qa_prefill(c.h, 0, [k] * B, vq, vk, vv, wq, wk, o)
                got = f64(o).reshape(B, k, Hq, D)
            else:
                steps = []
                for s in range(k):
                    o = torch.empty((B, Hq, D), dtype=torch.bfloat16, device="cuda")
                    qa.qa_decode_step(c.h, 0, B, dev(inp.dq[s]), dev(inp.dk[s]), dev(inp.dv[s]), wq, wk, o)
                    steps.append(f64(o))
                got = np.stack(steps, axis=1)
            torch.cuda.synchronize()
            K, V, L = c.views()
            res.append((got, bits(K), bits(V), list(L.cpu().numpy()[:B])))
            assert c.device_error() == (0, 0)
        finally:
            c.free()
    (gv, kv_, vv_, lv), (gd, kd, vd, ld) = res
    assert lv == ld == [n + k for n in prompt]
    np.testing.assert_array_equal(vv_, vd)  # v is copied
    # k' comes from K1 on one side and from the decode kernel on the other: the
    # same formula, compiled apart, so equal within the bf16 rounding bound
    for b, n in enumerate(ld):
        kd_b = F(kd[b, :, :n])
        assert (np.abs(F(kv_[b, :, :n]) - kd_b) <= rope_pair_tolerance(kd_b)).all()
    d = np.abs(gv - gd)
    assert d.max() <= 2e-2 and d.mean() <= 2e-3
