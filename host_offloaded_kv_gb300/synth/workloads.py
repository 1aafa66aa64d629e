"""The named CLO decode workloads (shapes, seeds and distributions).

Each workload is one decode configuration of a GQA attention stack whose full
K/V lives in pinned host memory.  The five workloads follow the CLO abstract's
setting (Llama3-8B and Qwen2.5-14B shaped stacks, top-k = 10 % of the context,
batch up to 64) with seeded synthetic data; see the fields for the exact shapes.
"""
from __future__ import annotations

from dataclasses import dataclass, replace


@dataclass(frozen=True)
class Workload:
    name: str
    n_layers: int
    batch: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    n_tokens: int          # cached tokens per sequence
    topk: int              # >0: fixed k; 0: ceil(topk_ratio * N)
    topk_ratio: float
    decode_steps: int
    rho_lo: float          # AR(1) query coefficient range
    rho_hi: float
    tau_fixed: float | None  # fixed per-head threshold, or None -> warm-up profiling
    n_persist: int         # persistent (fully resident) kv heads per layer
    seed: int
    warmup_steps: int = 16
    tau_offset: float = 0.05
    hh_ratio: float = 0.01

    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads

    @property
    def units(self) -> int:
        return self.n_layers * self.batch * self.n_kv_heads

    def scaled(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS = {
    "tiny": Workload("tiny", 1, 1, 8, 2, 64, 4096, 410, 0.1, 16, 0.6, 0.98, 0.8, 0, seed=0),
    "llama32k": Workload("llama32k", 32, 8, 32, 8, 128, 32768, 0, 0.1, 64, 0.6, 0.98, None, 4, seed=1),
    "llama128k": Workload("llama128k", 32, 16, 32, 8, 128, 131072, 0, 0.1, 32, 0.6, 0.98, None, 0, seed=2),
    "qwen512k": Workload("qwen512k", 48, 1, 40, 8, 128, 524288, 0, 0.1, 32, 0.7, 0.98, None, 6, seed=3),
    "stress": Workload("stress", 32, 64, 32, 8, 128, 32768, 0, 0.1, 32, 0.2, 0.7, 0.8, 0, seed=4),
}


def get_workload(name: str) -> Workload:
    if name not in WORKLOADS:
        raise KeyError(f"unknown workload {name!r}; known: {sorted(WORKLOADS)}")
    return WORKLOADS[name]
