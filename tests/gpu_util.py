"""Helpers for the GPU parity tests: device transfer of bf16 bit patterns, a
cache handle with torch views, and the error metrics of the parity bar."""
from __future__ import annotations

import numpy as np
import torch

from gqa_attention_preallocated_qa_gb300.inputs import bf16_bits_to_f64

# Parity bar on bf16 attention outputs against the fp64 oracle.
MAX_ABS = 2e-2
MEAN_ABS = 2e-3
# bf16 NaN used to poison cache slots that must never be read.
SENTINEL_BITS = 0x7FC1


def dev(bits: np.ndarray) -> torch.Tensor:
    """uint16 bf16 bit patterns -> bf16 CUDA tensor."""
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)


def f64(t: torch.Tensor) -> np.ndarray:
    return bf16_bits_to_f64(bits(t))


def errors(got: np.ndarray, want: np.ndarray) -> dict:
    d = np.abs(got.astype(np.float64) - want)
    return {"max_abs": float(d.max()) if d.size else 0.0, "mean_abs": float(d.mean()) if d.size else 0.0,
            "p99_abs": float(np.quantile(d, 0.99)) if d.size else 0.0,
            "violations": int((d > MAX_ABS).sum())}


def assert_parity(got: np.ndarray, want: np.ndarray, what: str) -> dict:
    e = errors(got, want)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    assert e["max_abs"] <= MAX_ABS and e["mean_abs"] <= MEAN_ABS, f"{what}: {e}"
    return e


def rope_pair_tolerance(want: np.ndarray) -> np.ndarray:
    """Per-element bound for a normed + rotated head vector rounded like the
    kernels.  bf16 keeps 8 significant bits, so one rounding moves a value by
    at most u = 2^-8 relative.  Two roundings precede the rotation (x_hat, then
    w * x_hat): |dy| <= 2u|y|.  The rotation mixes y_i and its partner, so
    |d out_i| <= 2u(|y_i| + |y_p|) <= 2u * sqrt(2) * |pair|, and the final
    rounding adds u * |pair|, |pair| being the norm of the rotated pair
    (i, i+D/2), which the rotation preserves.  (2*sqrt(2) + 1) * 2^-8 = 0.01495;
    0.016 leaves room for the fp32 cos/sin table and the fp32 reciprocal root."""
    D = want.shape[-1]
    h = D // 2
    pair = np.sqrt(want[..., :h] ** 2 + want[..., h:] ** 2)
    pair = np.concatenate([pair, pair], axis=-1)
    return 0.016 * pair + 1e-6


class GpuCache:
    """A qa cache plus torch views of one layer's K, V and lengths."""

    def __init__(self, qa, layers, max_batch, Hq, Hkv, D, cap, theta=1e6, eps=1e-6):
        self.qa = qa
        self.shape = (layers, max_batch, Hq, Hkv, D, cap)
        self.h = qa.qa_cache_alloc(layers, max_batch, Hq, Hkv, D, cap, theta, eps)
        self.max_batch, self.Hq, self.Hkv, self.D, self.cap = max_batch, Hq, Hkv, D, cap

    def views(self, layer=0):
        return self.qa.cache_tensors(self.h, layer, self.max_batch, self.Hkv, self.cap, self.D)

    def poison(self, layers=None):
        for l in range(self.shape[0]) if layers is None else layers:
            K, V, _ = self.views(l)
            K.view(torch.int16).fill_(np.int16(SENTINEL_BITS))
            V.view(torch.int16).fill_(np.int16(SENTINEL_BITS))
        torch.cuda.synchronize()

    def device_error(self):
        return self.qa.qa_get_device_error(self.h)

    def free(self):
        if self.h:
            self.qa.qa_cache_free(self.h)
            self.h = None
