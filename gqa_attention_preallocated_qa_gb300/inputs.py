"""Seeded synthetic inputs for the attention hot path.

This module is shared by the CUDA path's tests and benchmark and by the oracle
tests.  It holds none of the method's arithmetic: it only draws numbers and
rounds them to bf16 (round-to-nearest-even), the storage type of every input.

Workloads follow the shapes the pages describe for greedy Qwen3 decoding
(batch 1 and 4, prompts of 512 to 2048 tokens, 32 to 128 generated tokens;
dryft-flash-infer agent guide, "What is measured" and "Where the wins are").
No dataset or model weight is involved: q/k/v are N(0,1), the per-head norm
weights are 1 + N(0, 0.1).

Draw order for one layer, from ``numpy.random.default_rng(seed)`` in fp32:
prompt q [T,Hq,D], k [T,Hkv,D], v [T,Hkv,D]; then w_q [D], w_k [D]; then for
each decode step s: q_s [B,Hq,D], k_s [B,Hkv,D], v_s [B,Hkv,D].
For a pre-filled cache (the decode sweep) the order is: K [B,Hkv,L,D],
V [B,Hkv,L,D], w_q, w_k, then the decode step.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np


def f32_to_bf16_bits(x) -> np.ndarray:
    """Round fp32 values to bf16 (nearest even); returns the uint16 bit patterns."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def bf16_bits_to_f64(b) -> np.ndarray:
    """Exact float64 image of bf16 bit patterns."""
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def bf16_bits_to_f32(b) -> np.ndarray:
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def _normal_bf16(rng: np.random.Generator, shape) -> np.ndarray:
    return f32_to_bf16_bits(rng.standard_normal(shape, dtype=np.float32))


def _weight_bf16(rng: np.random.Generator, D: int) -> np.ndarray:
    w = np.float32(1.0) + np.float32(0.1) * rng.standard_normal(D, dtype=np.float32)
    return f32_to_bf16_bits(w)


@dataclass
class LayerInputs:
    """bf16 bit patterns (uint16) of one layer's inputs."""
    prompt_lens: list
    q: np.ndarray            # [T, Hq, D]
    k: np.ndarray            # [T, Hkv, D]
    v: np.ndarray            # [T, Hkv, D]
    wq: np.ndarray           # [D]
    wk: np.ndarray           # [D]
    dq: np.ndarray           # [steps, B, Hq, D]
    dk: np.ndarray           # [steps, B, Hkv, D]
    dv: np.ndarray           # [steps, B, Hkv, D]
    cache_k: np.ndarray = field(default=None)   # [B, Hkv, L, D] for a pre-filled cache
    cache_v: np.ndarray = field(default=None)


def layer_inputs(seed: int, prompt_lens, Hq: int, Hkv: int, D: int, steps: int) -> LayerInputs:
    rng = np.random.default_rng(seed)
    B = len(prompt_lens)
    T = int(sum(prompt_lens))
    q = _normal_bf16(rng, (T, Hq, D))
    k = _normal_bf16(rng, (T, Hkv, D))
    v = _normal_bf16(rng, (T, Hkv, D))
    wq = _weight_bf16(rng, D)
    wk = _weight_bf16(rng, D)
    dq = np.empty((steps, B, Hq, D), np.uint16)
    dk = np.empty((steps, B, Hkv, D), np.uint16)
    dv = np.empty((steps, B, Hkv, D), np.uint16)
    for s in range(steps):
        dq[s] = _normal_bf16(rng, (B, Hq, D))
        dk[s] = _normal_bf16(rng, (B, Hkv, D))
        dv[s] = _normal_bf16(rng, (B, Hkv, D))
    return LayerInputs(list(prompt_lens), q, k, v, wq, wk, dq, dk, dv)


def prefilled_cache_inputs(seed: int, B: int, L: int, Hq: int, Hkv: int, D: int) -> LayerInputs:
    """A cache already holding L raw N(0,1) keys/values per sequence, plus one decode token."""
    rng = np.random.default_rng(seed)
    ck = _normal_bf16(rng, (B, Hkv, L, D))
    cv = _normal_bf16(rng, (B, Hkv, L, D))
    wq = _weight_bf16(rng, D)
    wk = _weight_bf16(rng, D)
    dq = _normal_bf16(rng, (1, B, Hq, D))
    dk = _normal_bf16(rng, (1, B, Hkv, D))
    dv = _normal_bf16(rng, (1, B, Hkv, D))
    empty_q = np.empty((0, Hq, D), np.uint16)
    empty_kv = np.empty((0, Hkv, D), np.uint16)
    return LayerInputs([0] * B, empty_q, empty_kv, empty_kv.copy(), wq, wk, dq, dk, dv,
                       cache_k=ck, cache_v=cv)
