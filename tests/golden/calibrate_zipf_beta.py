"""Chooses the logit-bias scale beta of the Zipf-skewed routing workload.

The workload wants expert popularity following Zipf(s=1.2) with the busiest of the 64 experts
receiving about 4000 of the 16384 * 4 token assignments.  Logits are N(0,1) + beta * ln p_e; this
script bisects beta, routing every token with the oracle's router, and prints the result (stored
as synth.ZIPF_BETA together with the observed min / max expert loads).  It calls only the oracle.

    python tests/golden/calibrate_zipf_beta.py
"""
import os
import sys

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__)))))
import oracle  # noqa: E402
import synth  # noqa: E402


def loads(beta: float):
    cfg = synth.CONFIGS["skewed"]
    T = cfg.tokens[0]
    logits = synth.gen_logits(cfg, T, beta=beta).numpy()
    ids, _ = oracle.router(logits, cfg.top_k)
    return np.bincount(ids.reshape(-1), minlength=cfg.experts)


def main(target: int = 4000):
    lo, hi = 0.0, 8.0
    for _ in range(30):
        mid = 0.5 * (lo + hi)
        if loads(mid).max() < target:
            lo = mid
        else:
            hi = mid
    beta = round(0.5 * (lo + hi), 4)
    c = loads(beta)
    print(f"beta={beta} max_load={c.max()} min_load={c.min()} "
          f"loads_sorted={sorted(c.tolist(), reverse=True)}")


if __name__ == "__main__":
    main()
