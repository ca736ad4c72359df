"""The five serving-shaped workloads the verification path is tested and measured on.

Shapes and value distributions (logit scale, Zipf-style frequency bias over a seeded permutation,
draft noise, temperatures, greedy share, ragged draft lengths) follow the workload list this library
is specified against. The pages themselves time no verification step, so these synthetic logits
stand in for real serving traffic.
"""
from __future__ import annotations

from dataclasses import dataclass


@dataclass(frozen=True)
class Config:
    name: str
    B: int
    gamma_max: int
    V: int
    dtype: str                      # "f32" or "bf16": storage type of both logit tensors
    target_std: float               # z_t = target_std * N(0, 1) - zipf * log(rank)
    zipf: float                     # 0 disables the frequency bias
    draft: str                      # "additive": z_d = z_t + sigma * N(0,1); "scaled": see config 2
    sigma: float | tuple = 0.0      # draft noise; a (lo, hi) pair means per-row U[lo, hi]
    temperature: float | tuple = 1.0   # a (lo, hi) pair means per-row U[lo, hi]
    greedy: str = "none"            # "none", "odd" (odd rows greedy), or "frac:<f>" (seeded subset)
    ragged: bool = False            # draft_len ~ U{1..gamma_max} per row
    seed: int = 0

    @property
    def n_positions_padded(self) -> int:
        return self.B * (self.gamma_max + 1)


# Draft noise of the V=128256 workload: the value that puts the mean acceptance rate near 0.7
# (found by oracle/calibrate_sigma.py with the fp64 oracle on 16 seeded rows).
SIGMA_CFG3 = 0.90

CONFIGS = [
    # 1: tiny fp32 case; drafts sampled from q (the tests draw them with the oracle's sampler).
    Config("b1_g4_v256_f32", B=1, gamma_max=4, V=256, dtype="f32", target_std=2.0, zipf=0.0,
           draft="additive", sigma=0.5, temperature=1.0, seed=0),
    # 2: bf16, half the rows greedy (odd b), T = 0.8 elsewhere; z_d = 0.9 z_t + 0.44 * 3 * N(0,1).
    Config("b8_g4_v32000_bf16", B=8, gamma_max=4, V=32000, dtype="bf16", target_std=3.0, zipf=1.1,
           draft="scaled", sigma=0.44 * 3.0, temperature=0.8, greedy="odd", seed=2),
    # 3: bf16, all rows sampled, noise tuned for mean alpha ~ 0.7.
    Config("b64_g5_v128256_bf16", B=64, gamma_max=5, V=128256, dtype="bf16", target_std=2.5,
           zipf=1.1, draft="additive", sigma=SIGMA_CFG3, temperature=1.0, seed=3),
    # 4: fp32, per-row noise U[0.2, 2.0] and per-row temperature U[0.5, 1.5].
    Config("b256_g7_v152064_f32", B=256, gamma_max=7, V=152064, dtype="f32", target_std=3.0,
           zipf=1.1, draft="additive", sigma=(0.2, 2.0), temperature=(0.5, 1.5), seed=4),
    # 5: bf16, ragged draft lengths 1..8, 10% greedy rows, noise 0.7.
    Config("b1024_g8ragged_v256000_bf16", B=1024, gamma_max=8, V=256000, dtype="bf16",
           target_std=2.0, zipf=1.1, draft="additive", sigma=0.7, temperature=1.0,
           greedy="frac:0.1", ragged=True, seed=5),
]


def get_config(key) -> Config:
    """By 1-based index (1..5) or by name."""
    if isinstance(key, int):
        return CONFIGS[key - 1]
    for c in CONFIGS:
        if c.name == key:
            return c
    raise KeyError(key)
