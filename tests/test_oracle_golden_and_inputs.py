"""Regression pin of the oracle and checks of the seeded input generator (CPU)."""
import json
import os

import numpy as np
import pytest
import torch

from gqa_attention_preallocated_qa_gb300.inputs import (bf16_bits_to_f64, f32_to_bf16_bits,
                                                        layer_inputs)

HERE = os.path.dirname(os.path.abspath(__file__))


def test_oracle_reproduces_stored_tiny_fixture(oracle_mod):
    import importlib.util
    spec = importlib.util.spec_from_file_location("mk", os.path.join(HERE, "golden",
                                                                     "make_golden.py"))
    mk = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mk)
    got = mk.compute()
    want = json.load(open(os.path.join(HERE, "golden", "tiny_oracle.json")))["values"]
    assert got["final_len"] == want["final_len"] == 72
    np.testing.assert_allclose(got["prefill_sum"], want["prefill_sum"], rtol=1e-12)
    np.testing.assert_allclose(got["prefill_samples"], want["prefill_samples"], rtol=1e-12)
    for a, b in zip(got["decode"], want["decode"]):
        np.testing.assert_allclose([a["sum"], a["first"], a["last"]],
                                   [b["sum"], b["first"], b["last"]], rtol=1e-12)


def test_bf16_rounding_is_nearest_even():
    one = 1.0
    x = np.array([one + 2.0 ** -8, one + 3 * 2.0 ** -8, -2.5, 0.0], np.float32)
    got = bf16_bits_to_f64(f32_to_bf16_bits(x))
    np.testing.assert_array_equal(got, [1.0, 1.0 + 2.0 ** -6, -2.5, 0.0])
    # library routine: torch's fp32 -> bf16 conversion rounds to nearest even
    r = np.random.default_rng(3).standard_normal(100000).astype(np.float32) * 7
    t = torch.from_numpy(r).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(f32_to_bf16_bits(r), t)


def test_layer_inputs_are_seeded_and_shaped():
    a = layer_inputs(3, (5, 2), 4, 2, 16, steps=3)
    b = layer_inputs(3, (5, 2), 4, 2, 16, steps=3)
    assert a.q.shape == (7, 4, 16) and a.k.shape == (7, 2, 16) and a.dq.shape == (3, 2, 4, 16)
    np.testing.assert_array_equal(a.q, b.q)
    np.testing.assert_array_equal(a.dv, b.dv)
    w = bf16_bits_to_f64(a.wq)
    assert 0.5 < w.mean() < 1.5 and 0.02 < w.std() < 0.3
    x = bf16_bits_to_f64(a.q)
    assert abs(x.mean()) < 0.2 and 0.8 < x.std() < 1.2
