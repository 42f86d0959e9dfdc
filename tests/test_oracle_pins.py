"""Pins of the fp64 oracle to facts outside itself (CPU only).

Each test checks the oracle against a closed form, an invariant, a special
case that reduces to a textbook or library routine, or brute force with an
independent formulation (complex-number rotation, matrix-form softmax from
scipy).  They are chosen so that the plausible mistakes -- eps outside the
square root, sum instead of mean, 1/D instead of 1/sqrt(D), interleaved
instead of rotate-half pairing, a flipped rotation sign, a wrong frequency
exponent, an off-by-one causal mask, a wrong GQA head mapping, positions that
do not restart per sequence -- each fail at least one of them.
"""
import math

import numpy as np
import pytest
from scipy.special import softmax as sp_softmax

from gqa_attention_preallocated_qa_gb300.inputs import bf16_bits_to_f64, layer_inputs

RNG = np.random.default_rng(1234)


# ---------------------------------------------------------------- RMSNorm
def test_rmsnorm_constant_vector_closed_form(oracle_mod):
    # x = c*1: mean(x^2) = c^2, so y = w * c / sqrt(c^2 + eps); with c = 1e-3 and
    # eps = 1e-6 the eps term is as large as the signal, so its placement shows.
    D, c, eps = 8, 1e-3, 1e-6
    w = np.linspace(0.5, 1.5, D)
    y = oracle_mod.rmsnorm(np.full(D, c), w, eps)
    np.testing.assert_allclose(y, w * (1e-3 / math.sqrt(2e-6)), rtol=1e-14)
    np.testing.assert_allclose(y, w * 0.7071067811865476, rtol=1e-14)


def test_rmsnorm_two_element_example(oracle_mod):
    # x = (3, 4): mean of squares 12.5 (not the sum 25), so y = x / 3.5355339...
    y = oracle_mod.rmsnorm([3.0, 4.0], [1.0, 1.0], 0.0)
    np.testing.assert_allclose(y, [0.848528137423857, 1.131370849898476], rtol=1e-14)
    y = oracle_mod.rmsnorm([3.0, 4.0], [2.0, 0.5], 0.0)
    np.testing.assert_allclose(y, [1.697056274847714, 0.565685424949238], rtol=1e-14)


def test_rmsnorm_unit_rms_and_scale_invariance(oracle_mod):
    D = 128
    x = RNG.standard_normal(D)
    y = oracle_mod.rmsnorm(x, np.ones(D), 0.0)
    assert abs(math.sqrt(np.mean(y * y)) - 1.0) < 1e-14
    y2 = oracle_mod.rmsnorm(37.5 * x, np.ones(D), 0.0)
    np.testing.assert_allclose(y2, y, rtol=1e-13)


# ---------------------------------------------------------------- RoPE
def test_rope_position_zero_is_identity(oracle_mod):
    x = RNG.standard_normal(128)
    np.testing.assert_array_equal(oracle_mod.rope(x, 0, 1e6), x)


@pytest.mark.parametrize("D,pos,theta", [(4, 1, 1e6), (64, 7, 1e6), (128, 16383, 1e6),
                                         (128, 5, 1e4)])
def test_rope_matches_complex_rotation(oracle_mod, D, pos, theta):
    # Independent formulation: pair (i, i+D/2) is the complex number x_i + i*x_{i+D/2},
    # multiplied by exp(i * pos * inv_freq_i) with inv_freq_i = theta^(-2i/D).
    x = RNG.standard_normal(D)
    half = D // 2
    z = x[:half] + 1j * x[half:]
    inv_freq = 1.0 / theta ** (np.arange(0, D, 2, dtype=np.float64) / D)
    zr = z * np.exp(1j * pos * inv_freq)
    want = np.concatenate([zr.real, zr.imag])
    np.testing.assert_allclose(oracle_mod.rope(x, pos, theta), want, rtol=1e-10, atol=1e-12)


def test_rope_first_pair_turns_by_one_radian(oracle_mod):
    # inv_freq_0 = theta^0 = 1 for any theta: at pos 1 the first pair turns by
    # exactly 1 rad, counter-clockwise from (x_0, x_{D/2}).
    D = 8
    x = np.zeros(D)
    x[0] = 1.0
    y = oracle_mod.rope(x, 1, 1e6)
    assert abs(y[0] - math.cos(1.0)) < 1e-15 and abs(y[D // 2] - math.sin(1.0)) < 1e-15
    assert np.count_nonzero(y) == 2


def test_rope_frequency_ladder(oracle_mod):
    # Angle of pair i after one position, read back with atan2, is theta^(-2i/D).
    D, theta = 128, 1e6
    for i in (0, 1, 17, 63):
        x = np.zeros(D)
        x[i] = 1.0
        y = oracle_mod.rope(x, 1, theta)
        ang = math.atan2(y[i + D // 2], y[i])
        assert abs(ang - theta ** (-2.0 * i / D)) < 1e-14


def test_rope_preserves_pair_norms_and_composes(oracle_mod):
    D = 128
    x = RNG.standard_normal(D)
    y = oracle_mod.rope(x, 911, 1e6)
    half = D // 2
    np.testing.assert_allclose(np.hypot(y[:half], y[half:]), np.hypot(x[:half], x[half:]),
                               rtol=1e-13)
    # R(m) R(n) = R(m + n)
    np.testing.assert_allclose(oracle_mod.rope(oracle_mod.rope(x, 300, 1e6), 611, 1e6), y,
                               rtol=1e-9, atol=1e-12)


def test_rope_relative_position_property(oracle_mod):
    # <R(m) q, R(n) k> depends on m - n only.
    D = 128
    q, k = RNG.standard_normal(D), RNG.standard_normal(D)
    a = oracle_mod.rope(q, 40, 1e6) @ oracle_mod.rope(k, 15, 1e6)
    b = oracle_mod.rope(q, 1040, 1e6) @ oracle_mod.rope(k, 1015, 1e6)
    assert abs(a - b) < 1e-9


# ---------------------------------------------------------------- attention
def test_attend_single_key_returns_its_value(oracle_mod):
    D = 64
    v = RNG.standard_normal((1, D))
    out, p = oracle_mod.attend(RNG.standard_normal(D), RNG.standard_normal((1, D)), v)
    np.testing.assert_array_equal(out, v[0])
    assert p[0] == 1.0


def test_attend_two_key_sigmoid_and_sqrt_d_scale(oracle_mod):
    # D = 4, q = (2,0,0,0), k0 = 0, k1 = (1,0,0,0): s1 - s0 = 2/sqrt(4) = 1,
    # so p1 = sigmoid(1); a 1/D scale would give sigmoid(0.5).
    q = np.array([2.0, 0, 0, 0])
    K = np.array([[0.0, 0, 0, 0], [1.0, 0, 0, 0]])
    V = np.array([[1.0, 0, 0, 0], [0.0, 1, 0, 0]])
    out, p = oracle_mod.attend(q, K, V)
    assert abs(p[1] - 0.7310585786300049) < 1e-15
    np.testing.assert_allclose(out, [1 - 0.7310585786300049, 0.7310585786300049, 0, 0],
                               rtol=1e-14)


def test_attend_equal_keys_give_mean_and_rows_sum_to_one(oracle_mod):
    D, n = 32, 9
    K = np.tile(RNG.standard_normal(D), (n, 1))
    V = RNG.standard_normal((n, D))
    out, p = oracle_mod.attend(RNG.standard_normal(D), K, V)
    np.testing.assert_allclose(out, V.mean(axis=0), rtol=1e-13, atol=1e-15)
    K = RNG.standard_normal((n, D))
    out, p = oracle_mod.attend(RNG.standard_normal(D), K, np.ones((n, D)))
    assert abs(p.sum() - 1.0) < 1e-15
    np.testing.assert_allclose(out, np.ones(D), rtol=1e-14)


def test_attend_matches_scipy_softmax(oracle_mod):
    D, n = 16, 11
    q, K, V = RNG.standard_normal(D), RNG.standard_normal((n, D)), RNG.standard_normal((n, D))
    p_ref = sp_softmax(K @ q / math.sqrt(D))
    out, p = oracle_mod.attend(q, K, V)
    np.testing.assert_allclose(p, p_ref, rtol=1e-13)
    np.testing.assert_allclose(out, p_ref @ V, rtol=1e-12, atol=1e-14)


# ---------------------------------------------------------------- whole layer
def _brute_force_layer(prompt_lens, q, k, v, wq, wk, Hq, Hkv, theta, eps):
    """Matrix-form restatement: vectorised RMSNorm, complex rotation, repeat_kv,
    masked scores, scipy softmax.  Independent of the oracle's loops."""
    D = q.shape[-1]
    half = D // 2
    inv_freq = 1.0 / theta ** (np.arange(0, D, 2, dtype=np.float64) / D)

    def norm(x, w):
        return w * x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)

    def rot(x, pos):
        z = (x[..., :half] + 1j * x[..., half:]) * np.exp(1j * pos[:, None, None] * inv_freq)
        return np.concatenate([z.real, z.imag], axis=-1)

    outs = []
    t0 = 0
    for L in prompt_lens:
        pos = np.arange(L, dtype=np.float64)
        qs = rot(norm(q[t0:t0 + L], wq), pos)              # [L, Hq, D]
        ks = rot(norm(k[t0:t0 + L], wk), pos)              # [L, Hkv, D]
        vs = v[t0:t0 + L]
        G = Hq // Hkv
        ks = np.repeat(ks, G, axis=1)
        vs = np.repeat(vs, G, axis=1)
        S = np.einsum("ihd,jhd->hij", qs, ks) / math.sqrt(D)
        S = np.where(np.tril(np.ones((L, L), bool))[None], S, -np.inf)
        P = sp_softmax(S, axis=-1)
        outs.append(np.einsum("hij,jhd->ihd", P, vs))
        t0 += L
    return np.concatenate(outs, axis=0)


def _geom(oracle_mod, B, Hq, Hkv, D, cap):
    return oracle_mod.Geometry(B=B, Hq=Hq, Hkv=Hkv, D=D, cap=cap, theta=1e6, eps=1e-6)


def _f(x):
    return bf16_bits_to_f64(x)


@pytest.mark.parametrize("prompt_lens,Hq,Hkv,D", [((5,), 2, 1, 8), ((3, 7, 1), 4, 2, 16),
                                                  ((64,), 2, 1, 64), ((9, 4), 8, 2, 32)])
def test_prefill_matches_brute_force(oracle_mod, prompt_lens, Hq, Hkv, D):
    inp = layer_inputs(99, prompt_lens, Hq, Hkv, D, steps=0)
    g = _geom(oracle_mod, len(prompt_lens), Hq, Hkv, D, max(prompt_lens) + 2)
    lay = oracle_mod.OracleLayer(g)
    qp, out = lay.prefill(prompt_lens, _f(inp.q), _f(inp.k), _f(inp.v), _f(inp.wq), _f(inp.wk))
    want = _brute_force_layer(prompt_lens, _f(inp.q), _f(inp.k), _f(inp.v), _f(inp.wq),
                              _f(inp.wk), Hq, Hkv, 1e6, 1e-6)
    np.testing.assert_allclose(out, want, rtol=1e-10, atol=1e-12)
    assert list(lay.lens) == list(prompt_lens)


def test_prefill_first_row_is_first_value_exactly(oracle_mod):
    lens = (6, 3)
    inp = layer_inputs(5, lens, 4, 2, 16, steps=0)
    lay = oracle_mod.OracleLayer(_geom(oracle_mod, 2, 4, 2, 16, 8))
    _, out = lay.prefill(lens, _f(inp.q), _f(inp.k), _f(inp.v), _f(inp.wq), _f(inp.wk))
    v = _f(inp.v)
    for b, t0 in ((0, 0), (1, 6)):
        for h in range(4):
            np.testing.assert_array_equal(out[t0, h], v[t0, h // 2])


def test_prefill_is_causal(oracle_mod):
    L, i = 12, 5
    inp = layer_inputs(6, (L,), 2, 1, 16, steps=0)
    args = [_f(a) for a in (inp.q, inp.k, inp.v, inp.wq, inp.wk)]
    lay = oracle_mod.OracleLayer(_geom(oracle_mod, 1, 2, 1, 16, L))
    _, out = lay.prefill((L,), *args)
    k2, v2 = args[1].copy(), args[2].copy()
    k2[i + 1:] += 3.0
    v2[i + 1:] -= 7.0
    lay2 = oracle_mod.OracleLayer(_geom(oracle_mod, 1, 2, 1, 16, L))
    _, out2 = lay2.prefill((L,), args[0], k2, v2, args[3], args[4])
    np.testing.assert_array_equal(out2[: i + 1], out[: i + 1])
    assert np.abs(out2[i + 1:] - out[i + 1:]).max() > 1e-3


def test_prefill_gqa_equals_mha_with_repeated_kv(oracle_mod):
    lens, Hq, Hkv, D = (10,), 8, 2, 16
    inp = layer_inputs(7, lens, Hq, Hkv, D, steps=0)
    q, k, v, wq, wk = (_f(a) for a in (inp.q, inp.k, inp.v, inp.wq, inp.wk))
    lay = oracle_mod.OracleLayer(_geom(oracle_mod, 1, Hq, Hkv, D, 10))
    _, out = lay.prefill(lens, q, k, v, wq, wk)
    G = Hq // Hkv
    mha = oracle_mod.OracleLayer(_geom(oracle_mod, 1, Hq, Hq, D, 10))
    _, out2 = mha.prefill(lens, q, np.repeat(k, G, axis=1), np.repeat(v, G, axis=1), wq, wk)
    np.testing.assert_array_equal(out, out2)


def test_ragged_batch_equals_sequences_alone(oracle_mod):
    lens, Hq, Hkv, D = (5, 9, 2), 4, 2, 16
    inp = layer_inputs(8, lens, Hq, Hkv, D, steps=0)
    q, k, v, wq, wk = (_f(a) for a in (inp.q, inp.k, inp.v, inp.wq, inp.wk))
    lay = oracle_mod.OracleLayer(_geom(oracle_mod, 3, Hq, Hkv, D, 9))
    _, out = lay.prefill(lens, q, k, v, wq, wk)
    t0 = 0
    for L in lens:
        one = oracle_mod.OracleLayer(_geom(oracle_mod, 1, Hq, Hkv, D, 9))
        _, o1 = one.prefill((L,), q[t0:t0 + L], k[t0:t0 + L], v[t0:t0 + L], wq, wk)
        np.testing.assert_array_equal(out[t0:t0 + L], o1)
        t0 += L


def test_decode_reproduces_prefill_row(oracle_mod):
    # A prefill of t tokens followed by one decode step of token t gives the same
    # output as row t of a prefill of t+1 tokens.
    t, Hq, Hkv, D = 11, 4, 2, 32
    inp = layer_inputs(9, (t + 1,), Hq, Hkv, D, steps=0)
    q, k, v, wq, wk = (_f(a) for a in (inp.q, inp.k, inp.v, inp.wq, inp.wk))
    full = oracle_mod.OracleLayer(_geom(oracle_mod, 1, Hq, Hkv, D, t + 1))
    _, out_full = full.prefill((t + 1,), q, k, v, wq, wk)
    lay = oracle_mod.OracleLayer(_geom(oracle_mod, 1, Hq, Hkv, D, t + 1))
    lay.prefill((t,), q[:t], k[:t], v[:t], wq, wk)
    qp, out_dec = lay.decode(q[t:t + 1], k[t:t + 1], v[t:t + 1], wq, wk)
    np.testing.assert_allclose(out_dec[0], out_full[t], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(lay.Kc, full.Kc, rtol=0, atol=1e-15)
    assert int(lay.lens[0]) == t + 1


def test_reset_then_rerun_is_identical_and_overflow_is_an_error(oracle_mod):
    lens, Hq, Hkv, D = (4, 6), 2, 1, 16
    inp = layer_inputs(10, lens, Hq, Hkv, D, steps=2)
    args = [_f(a) for a in (inp.q, inp.k, inp.v, inp.wq, inp.wk)]
    lay = oracle_mod.OracleLayer(_geom(oracle_mod, 2, Hq, Hkv, D, 8))
    first = [lay.prefill(lens, *args)[1]]
    for s in range(2):
        first.append(lay.decode(_f(inp.dq[s]), _f(inp.dk[s]), _f(inp.dv[s]), args[3], args[4])[1])
    lay.reset()
    assert list(lay.lens) == [0, 0]
    again = [lay.prefill(lens, *args)[1]]
    for s in range(2):
        again.append(lay.decode(_f(inp.dq[s]), _f(inp.dk[s]), _f(inp.dv[s]), args[3], args[4])[1])
    for a, b in zip(first, again):
        np.testing.assert_array_equal(a, b)
    # lens = (6, 8): the second sequence is full, so the next step must fail.
    with pytest.raises(oracle_mod.OracleError):
        lay.decode(_f(inp.dq[0]), _f(inp.dk[0]), _f(inp.dv[0]), args[3], args[4])
    # a prefill on a non-empty layer is an error too
    with pytest.raises(oracle_mod.OracleError):
        lay.prefill(lens, *args)


def test_attend_cached_after_decode_transform_matches_brute_force_and_decode(oracle_mod):
    # OracleLayer.attend_cached is the expected value of the full-size decode
    # checks (the cache is appended once by decode_transform, then any head is
    # attended on its own).  Pinned two ways: (1) against the matrix-form brute
    # force over each sequence's prompt + decode tokens (decode step s of a
    # sequence is row L_b + s of that concatenation), and (2) against the
    # oracle's own fused decode on a second layer.  A head-mapping slip (h % Hkv
    # instead of h // G) or a length slip (keys :n+1 or :n-1) fails both.
    prompt_lens, Hq, Hkv, D, steps = (6, 1, 9), 8, 2, 16, 3
    inp = layer_inputs(37, prompt_lens, Hq, Hkv, D, steps)
    q, k, v, wq, wk = (_f(a) for a in (inp.q, inp.k, inp.v, inp.wq, inp.wk))
    dq, dk, dv = _f(inp.dq), _f(inp.dk), _f(inp.dv)
    B, cap = len(prompt_lens), max(prompt_lens) + steps
    a = oracle_mod.OracleLayer(_geom(oracle_mod, B, Hq, Hkv, D, cap))
    b = oracle_mod.OracleLayer(_geom(oracle_mod, B, Hq, Hkv, D, cap))
    a.prefill(prompt_lens, q, k, v, wq, wk)
    b.prefill(prompt_lens, q, k, v, wq, wk)
    # brute force over the concatenated tokens of each sequence
    cu = np.concatenate([[0], np.cumsum(prompt_lens)])
    cat = [np.concatenate([x[cu[i]:cu[i + 1]] for i in range(B)] +
                          [d[s, i:i + 1] for s in range(steps) for i in range(B)])
           for x, d in ((q, dq), (k, dk), (v, dv))]
    # reorder into sequence-major packing: sequence i's prompt rows, then its steps
    rows = []
    off = int(cu[-1])
    for i in range(B):
        rows.extend(range(cu[i], cu[i + 1]))
        rows.extend(off + s * B + i for s in range(steps))
    qb, kb, vb = (c[rows] for c in cat)
    brute = _brute_force_layer([L + steps for L in prompt_lens], qb, kb, vb, wq, wk, Hq, Hkv,
                               1e6, 1e-6)
    bcu = np.concatenate([[0], np.cumsum([L + steps for L in prompt_lens])])
    for s in range(steps):
        qp = a.decode_transform(dq[s], dk[s], dv[s], wq, wk)
        _, fused = b.decode(dq[s], dk[s], dv[s], wq, wk)
        for i in range(B):
            for h in range(Hq):
                got = a.attend_cached(i, h, qp[i, h])
                np.testing.assert_allclose(got, fused[i, h], rtol=1e-12, atol=1e-14)
                np.testing.assert_allclose(got, brute[bcu[i] + prompt_lens[i] + s, h],
                                           rtol=1e-9, atol=1e-12)
    assert list(a.lens) == [L + steps for L in prompt_lens]


def test_prefill_transform_outputs_match_brute_force(oracle_mod):
    # The transform the GPU's K1 is judged against: q' rows, the cache's K and V
    # slots and the lengths, each from the complex-rotation formulation above
    # (positions restart at 0 in every sequence; slots past a length untouched).
    lens, Hq, Hkv, D, cap = (3, 6, 1), 4, 2, 16, 8
    inp = layer_inputs(41, lens, Hq, Hkv, D, steps=0)
    q, k, v, wq, wk = (_f(a) for a in (inp.q, inp.k, inp.v, inp.wq, inp.wk))
    lay = oracle_mod.OracleLayer(_geom(oracle_mod, len(lens), Hq, Hkv, D, cap))
    qp = lay.prefill_transform(lens, q, k, v, wq, wk)
    half = D // 2
    inv_freq = 1.0 / 1e6 ** (np.arange(0, D, 2, dtype=np.float64) / D)

    def norm_rot(x, w, L):
        y = w * x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + 1e-6)
        z = (y[..., :half] + 1j * y[..., half:]) * np.exp(1j * np.arange(L)[:, None, None] * inv_freq)
        return np.concatenate([z.real, z.imag], axis=-1)

    t0 = 0
    for b, L in enumerate(lens):
        np.testing.assert_allclose(qp[t0:t0 + L], norm_rot(q[t0:t0 + L], wq, L), rtol=1e-12, atol=1e-14)
        kr = norm_rot(k[t0:t0 + L], wk, L)             # [L, Hkv, D]
        for h in range(Hkv):
            np.testing.assert_allclose(lay.Kc[b, h, :L], kr[:, h], rtol=1e-12, atol=1e-14)
            np.testing.assert_array_equal(lay.Vc[b, h, :L], v[t0:t0 + L, h])
            assert not lay.Kc[b, h, L:].any() and not lay.Vc[b, h, L:].any()
        t0 += L
    assert list(lay.lens) == list(lens)


def test_set_cache_restores_a_layer(oracle_mod):
    # A layer loaded with another layer's cache and lengths decodes the next
    # token exactly as that layer does.
    lens, Hq, Hkv, D, cap = (5, 2), 4, 2, 16, 7
    inp = layer_inputs(43, lens, Hq, Hkv, D, steps=1)
    q, k, v, wq, wk = (_f(a) for a in (inp.q, inp.k, inp.v, inp.wq, inp.wk))
    a = oracle_mod.OracleLayer(_geom(oracle_mod, 2, Hq, Hkv, D, cap))
    a.prefill(lens, q, k, v, wq, wk)
    b = oracle_mod.OracleLayer(_geom(oracle_mod, 2, Hq, Hkv, D, cap))
    b.set_cache(a.Kc, a.Vc, a.lens)
    step = [_f(x[0]) for x in (inp.dq, inp.dk, inp.dv)]
    _, out_a = a.decode(*step, wq, wk)
    _, out_b = b.decode(*step, wq, wk)
    np.testing.assert_array_equal(out_a, out_b)
    np.testing.assert_array_equal(a.Kc, b.Kc)
    assert list(b.lens) == [n + 1 for n in lens]
