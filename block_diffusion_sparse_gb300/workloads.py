"""Synthetic workload shapes for the HERALD hot path.

Each workload is one attention layer of a block diffusion LLM at a given
context length: batch N, query heads Hq, KV heads Hkv (GQA group G = Hq/Hkv),
head dim d, cached context L, block size B, denoising steps T per block,
stage-1 candidates C, final budget K, sink S and local window W.  The shapes
follow the block-dLLM setting of the HERALD abstracts (block of B tokens
decoded over T steps, budget K=1024, selection reused across the T steps) on
Qwen2.5-7B-like (28/4 heads) and Llama-8B-like (32/8 heads) layers.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace


@dataclass(frozen=True)
class Workload:
    name: str
    N: int
    Hq: int
    Hkv: int
    d: int
    L: int
    B: int
    T: int
    C: int
    K: int
    S: int
    W: int
    layers: int = 1
    kv_on_host: bool = False
    # heavy-hitter structure: "points" (count given by n_planted) or "spans"
    planted: str = "points"
    n_planted: int = 0
    span: int = 64
    sink_boost: float = 1.0   # norm multiplier of the first `n_boost` keys
    n_boost: int = 0
    index: int = 0            # workload number, part of the seed
    extra_rows: int = 0       # cache rows past L (room for appended blocks)

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def R(self) -> int:
        return self.B * self.G

    @property
    def P(self) -> int:
        """Row capacity of the selected-index list and of a pool buffer."""
        return self.K + self.S + self.W

    @property
    def L_max(self) -> int:
        return self.L + self.extra_rows

    def scaled(self, **kw) -> "Workload":
        return replace(self, **kw)


TINY = Workload("tiny", N=1, Hq=4, Hkv=1, d=64, L=2048, B=16, T=4, C=256,
                K=128, S=16, W=64, planted="points", n_planted=8, index=1,
                extra_rows=16)

QWEN_32K = Workload("qwen2.5-7b-layer-32k", N=1, Hq=28, Hkv=4, d=128,
                    L=32768, B=32, T=8, C=4096, K=1024, S=64, W=256,
                    planted="points", n_planted=328, sink_boost=4.0,
                    n_boost=4, index=2, extra_rows=32)

LLAMA_64K = Workload("llama-8b-layer-4x64k", N=4, Hq=32, Hkv=8, d=128,
                     L=65536, B=32, T=16, C=4096, K=1024, S=64, W=256,
                     planted="spans", n_planted=11, span=64, index=3,
                     extra_rows=32)

LONG_128K_HOST = Workload("long-128k-host-kv", N=1, Hq=32, Hkv=8, d=128,
                          L=131072, B=32, T=32, C=8192, K=1024, S=64, W=512,
                          kv_on_host=True, planted="points", n_planted=1311,
                          sink_boost=4.0, n_boost=4, index=4, extra_rows=32)

QWEN_STACK = Workload("qwen2.5-7b-28-layer-stack-8x32k", N=8, Hq=28, Hkv=4,
                      d=128, L=32768, B=32, T=8, C=4096, K=1024, S=64, W=256,
                      layers=28, planted="points", n_planted=328,
                      sink_boost=4.0, n_boost=4, index=5, extra_rows=4 * 32)

ALL = {w.name: w for w in (TINY, QWEN_32K, LLAMA_64K, LONG_128K_HOST, QWEN_STACK)}
