"""The GPU tests of chunked prefill, short chunks (verify steps) and attention
windows take their expected values from two builders in the test modules:
ChunkOracle and WindowOracle, the oracle's primitives applied one new token at
a time.  These CPU tests pin the builders: to the oracle's own prefill and
decode (pinned against brute force in test_oracle_pins.py), and to what a
window of W keys must do (a window covering every key is full attention; a
window of one key returns the token's own value; keys outside the window do
not matter, keys inside do)."""
import numpy as np

from gqa_attention_preallocated_qa_gb300.inputs import bf16_bits_to_f64 as F
from gqa_attention_preallocated_qa_gb300.inputs import layer_inputs
from test_gpu_chunked_prefill import ChunkOracle
from test_gpu_window import WindowOracle

HQ, HKV, D = 4, 2, 16


def fill(orc, lens, inp):
    t0 = 0
    for b, L in enumerate(lens):
        orc.append(b, F(inp.k[t0:t0 + L]), F(inp.v[t0:t0 + L]))
        t0 += L


def test_chunk_builder_equals_oracle_prefill_and_decode(oracle_mod):
    lens, steps, cap = (5, 9, 1), 2, 16
    inp = layer_inputs(11, lens, HQ, HKV, D, steps)
    layer = oracle_mod.OracleLayer(oracle_mod.Geometry(len(lens), HQ, HKV, D, cap))
    _, out = layer.prefill(lens, F(inp.q), F(inp.k), F(inp.v), F(inp.wq), F(inp.wk))
    dec = [layer.decode(F(inp.dq[s]), F(inp.dk[s]), F(inp.dv[s]), F(inp.wq), F(inp.wk))[1]
           for s in range(steps)]

    orc = ChunkOracle(oracle_mod, len(lens), HQ, HKV, D, cap, inp.wq, inp.wk)
    fill(orc, lens, inp)
    t0 = 0
    for b, L in enumerate(lens):
        for i in range(L):
            for h in range(HQ):
                np.testing.assert_allclose(orc.out_row(b, i, h, F(inp.q[t0 + i, h])), out[t0 + i, h],
                                           rtol=0, atol=1e-12)
        t0 += L
    for s in range(steps):
        for b in range(len(lens)):
            orc.append(b, F(inp.dk[s][b][None]), F(inp.dv[s][b][None]))
            for h in range(HQ):
                np.testing.assert_allclose(orc.out_row(b, orc.lens[b] - 1, h, F(inp.dq[s][b, h])),
                                           dec[s][b, h], rtol=0, atol=1e-12)
    assert list(layer.lens) == orc.lens
    for b, n in enumerate(orc.lens):
        np.testing.assert_allclose(orc.K[b, :, :n], layer.Kc[b, :, :n], rtol=0, atol=1e-12)
        np.testing.assert_array_equal(orc.V[b, :, :n], layer.Vc[b, :, :n])


def test_chunk_builder_in_pieces_equals_one_piece(oracle_mod):
    """Appending a prompt in chunks leaves the same cache and rows (a chunk's
    tokens take the positions after what the sequence holds)."""
    L, cap = 11, 16
    inp = layer_inputs(13, (L,), HQ, HKV, D, 0)
    whole = ChunkOracle(oracle_mod, 1, HQ, HKV, D, cap, inp.wq, inp.wk)
    whole.append(0, F(inp.k), F(inp.v))
    parts = ChunkOracle(oracle_mod, 1, HQ, HKV, D, cap, inp.wq, inp.wk)
    for a, e in ((0, 3), (3, 4), (4, 11)):
        parts.append(0, F(inp.k[a:e]), F(inp.v[a:e]))
    np.testing.assert_array_equal(whole.K, parts.K)
    np.testing.assert_array_equal(whole.V, parts.V)
    for i in range(L):
        np.testing.assert_array_equal(whole.out_row(0, i, 1, F(inp.q[i, 1])),
                                      parts.out_row(0, i, 1, F(inp.q[i, 1])))


def test_window_covering_every_key_is_full_attention(oracle_mod):
    lens, cap = (7, 12), 16
    inp = layer_inputs(17, lens, HQ, HKV, D, 0)
    full = ChunkOracle(oracle_mod, 2, HQ, HKV, D, cap, inp.wq, inp.wk)
    win = WindowOracle(oracle_mod, 2, HQ, HKV, D, cap, inp.wq, inp.wk, window=cap)
    fill(full, lens, inp)
    fill(win, lens, inp)
    t0 = 0
    for b, L in enumerate(lens):
        for i in range(L):
            for h in range(HQ):
                q = F(inp.q[t0 + i, h])
                np.testing.assert_array_equal(win.out_row(b, i, h, q), full.out_row(b, i, h, q))
        t0 += L


def test_window_of_one_key_returns_the_tokens_own_value(oracle_mod):
    lens, cap = (6,), 8
    inp = layer_inputs(19, lens, HQ, HKV, D, 0)
    win = WindowOracle(oracle_mod, 1, HQ, HKV, D, cap, inp.wq, inp.wk, window=1)
    fill(win, lens, inp)
    G = HQ // HKV
    for i in range(6):
        for h in range(HQ):
            np.testing.assert_array_equal(win.out_row(0, i, h, F(inp.q[i, h])), F(inp.v[i, h // G]))


def test_window_sees_exactly_its_keys(oracle_mod):
    """With a window of W keys, row i depends on keys i + 1 - W .. i only:
    changing a key before the window leaves the row bit-identical, changing one
    inside changes it."""
    L, W, cap, i, h = 12, 4, 16, 9, 2
    inp = layer_inputs(23, (L,), HQ, HKV, D, 0)
    q = F(inp.q[i, h])
    base = WindowOracle(oracle_mod, 1, HQ, HKV, D, cap, inp.wq, inp.wk, window=W)
    fill(base, (L,), inp)
    ref = base.out_row(0, i, h, q)
    g = h // (HQ // HKV)
    for j, inside in ((i - W, False), (0, False), (i + 1 - W, True), (i, True)):
        other = WindowOracle(oracle_mod, 1, HQ, HKV, D, cap, inp.wq, inp.wk, window=W)
        fill(other, (L,), inp)
        other.K[0, g, j] += 1.0
        other.V[0, g, j] -= 1.0
        got = other.out_row(0, i, h, q)
        if inside:
            assert np.abs(got - ref).max() > 1e-6, f"key {j} is inside the window"
        else:
            np.testing.assert_array_equal(got, ref)
