"""Finds the draft-noise sigma of the V=128256 bf16 workload that puts its mean acceptance rate
alpha = sum_x min(p, q) near 0.7, using the fp64 oracle on 16 seeded rows (bisection on sigma).

Test infrastructure; run by hand: ``python -m oracle.calibrate_sigma``. The value it prints is
recorded as ``SIGMA_CFG3`` in workloads/configs.py.
"""
from __future__ import annotations

import dataclasses

import numpy as np

from oracle.spec_verify_oracle import oracle_verify
from workloads import get_config, make_workload


def mean_alpha(sigma, rows=16):
    cfg = dataclasses.replace(get_config(3), B=rows, sigma=float(sigma))
    w = make_workload(cfg, backend="numpy")
    r = oracle_verify(w.target_logits, w.draft_logits, w.draft_tokens, w.draft_len,
                      w.temperature, w.uniforms)
    return float(np.mean(r.out_alpha))


def main(target=0.7, lo=0.1, hi=4.0, iters=14):
    for _ in range(iters):
        mid = 0.5 * (lo + hi)
        a = mean_alpha(mid)
        print(f"sigma={mid:.4f} mean_alpha={a:.4f}")
        if a > target:
            lo = mid
        else:
            hi = mid
    print(f"sigma ~ {0.5 * (lo + hi):.3f}")


if __name__ == "__main__":
    main()
