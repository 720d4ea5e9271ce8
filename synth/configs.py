"""The five workloads the boundary is checked and measured on.

All use hidden size D = 5120 (Beam blog pages, "Model architecture": 52-layer
decoder, hidden size 5120) and eps = 1e-6 (the pages give no eps; this is the
value the workloads fix).

  DENSE_DECODE_T4        dense boundary, decode:   T = 4,      n = 2
  DECODE_CHAIN_T64       decode chain:             T = 64,     all 104 boundaries,
                         n = 2 .. 105, fresh branch x and norm weights per boundary
  DENSE_PREFILL_T16384   dense boundary, prefill:  T = 8 x 2048 = 16384, n = 7
  MOE_T16384             MoE combine boundary:     T = 16384,  n = 20,
                         expert outputs ~ N(0,1)
  MOE_STRESS_T131072     MoE combine, stress:      T = 131072, n = 104, expert
                         outputs Student-t(3) at unit variance, 0.1 % of the
                         T*8 expert rows x100

h and x ~ N(0,1); norm weights 1 + 0.1 N(0,1); routing weights are the
logistic of N(0,1) draws, renormalised to sum 1 over the top 8, then x2.5.
Each workload has its own seed (0 .. 4 in the order above).
"""
from __future__ import annotations

from dataclasses import dataclass

# one counter stream per tensor; chain step s adds 16*s to the x / weight streams
STREAMS = {"h": 1, "x": 2, "post_w": 3, "pre_w": 4, "e": 5, "topk": 6, "outlier": 7}


@dataclass(frozen=True)
class Config:
    seed: int
    name: str
    kind: str            # "dense" | "chain" | "moe"
    T: int
    D: int = 5120
    n: int = 2           # residual-add index (first of the chain for "chain")
    steps: int = 1       # boundaries applied in sequence
    eps: float = 1e-6
    K: int = 8           # experts combined per token (MoE)
    route_scale: float = 2.5
    expert_dist: str = "normal"
    outlier_p: float = 0.0
    outlier_scale: float = 1.0

    def bytes_per_token(self) -> int:
        """Algorithmic HBM bytes per token: read h and the branch, write h' and y."""
        if self.kind == "moe":
            return 2 * self.D * (self.K + 1) + 4 * self.K + 2 * 2 * self.D
        return 4 * 2 * self.D

    def bytes_per_launch(self, T: int | None = None) -> int:
        T = self.T if T is None else T
        return T * self.bytes_per_token() + 2 * 2 * self.D  # + the two norm weight vectors


DENSE_DECODE_T4 = Config(0, "dense_decode_T4", "dense", T=4, n=2)
DECODE_CHAIN_T64 = Config(1, "decode_chain_T64", "chain", T=64, n=2, steps=104)
DENSE_PREFILL_T16384 = Config(2, "dense_prefill_T16384", "dense", T=16384, n=7)
MOE_T16384 = Config(3, "moe_T16384", "moe", T=16384, n=20)
MOE_STRESS_T131072 = Config(4, "moe_stress_T131072", "moe", T=131072, n=104,
                            expert_dist="t3_outliers", outlier_p=1e-3, outlier_scale=100.0)

WORKLOADS = {c.name: c for c in (DENSE_DECODE_T4, DECODE_CHAIN_T64, DENSE_PREFILL_T16384,
                                 MOE_T16384, MOE_STRESS_T131072)}
