"""The five synthetic workloads of the attention hot path, as plain data.

Shapes follow the greedy Qwen3 decoding the pages describe: batch 1 and 4,
prompts 512 to 2048, 32 to 128 generated tokens (dryft-flash-infer agent
guide, "What is measured", "Where the wins are"); the geometry is the Qwen3-4B
attention block (32 query heads, 8 KV heads, head_dim 128), RMSNorm eps 1e-6
and RoPE theta 1e6.  Capacity per sequence is prompt + generated tokens, so a
run fills the cache exactly and never evicts.
"""
from __future__ import annotations

from dataclasses import dataclass

from .inputs import layer_inputs, prefilled_cache_inputs


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    D: int
    prompt_lens: tuple
    steps: int
    cap: int
    layers: int = 1
    seed: int = 0
    reruns: int = 1           # generate calls on the same cache, reset in between
    theta: float = 1e6
    eps: float = 1e-6

    @property
    def T(self) -> int:
        return int(sum(self.prompt_lens))

    def layer_seed(self, layer: int) -> int:
        return self.seed if self.layers == 1 else self.seed * 1000 + layer

    def inputs(self, layer: int = 0):
        return layer_inputs(self.layer_seed(layer), self.prompt_lens, self.Hq, self.Hkv, self.D,
                            self.steps)

    def causal_flops(self) -> float:
        """Algorithmic prefill attention flops: 4*Hq*D per causal (query, key) pair."""
        return 4.0 * self.Hq * self.D * sum(L * (L + 1) // 2 for L in self.prompt_lens)


TINY = Workload("tiny_gqa_b1_p64", B=1, Hq=2, Hkv=1, D=64, prompt_lens=(64,), steps=8, cap=72,
                seed=0)
QWEN3_4B_B1 = Workload("qwen3_4b_b1_p512_d32", B=1, Hq=32, Hkv=8, D=128, prompt_lens=(512,),
                       steps=32, cap=544, seed=1)
QWEN3_4B_B4 = Workload("qwen3_4b_b4_p2048_d128", B=4, Hq=32, Hkv=8, D=128,
                       prompt_lens=(2048, 2048, 2048, 2048), steps=128, cap=2176, seed=2,
                       reruns=3)
RAGGED_36L = Workload("qwen3_4b_b4_ragged_36layers", B=4, Hq=32, Hkv=8, D=128,
                      prompt_lens=(512, 1024, 1536, 2048), steps=64, cap=2112, layers=36,
                      seed=3)

WORKLOADS = {w.name: w for w in (TINY, QWEN3_4B_B1, QWEN3_4B_B4, RAGGED_36L)}


@dataclass(frozen=True)
class SweepPoint:
    """Decode-only sweep point: cache pre-filled with L raw N(0,1) keys/values."""
    B: int
    L: int
    Hq: int = 32
    Hkv: int = 8
    D: int = 128
    seed: int = 4
    theta: float = 1e6
    eps: float = 1e-6

    @property
    def cap(self) -> int:
        return self.L + 1

    @property
    def name(self) -> str:
        return f"decode_sweep_b{self.B}_l{self.L}"

    def inputs(self):
        return prefilled_cache_inputs(self.seed * 1000 + self.B * 100000 + self.L, self.B, self.L,
                                      self.Hq, self.Hkv, self.D)

    def kv_bytes(self) -> int:
        """Algorithmic HBM bytes of one decode step: K and V of L+1 positions, bf16."""
        return self.B * self.Hkv * (self.L + 1) * self.D * 2 * 2


DECODE_SWEEP = tuple(SweepPoint(B, L) for B in (1, 4) for L in (512, 2048, 8192, 16384))
