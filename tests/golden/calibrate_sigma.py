"""Find the draft-logit noise sigma that puts the mean closed-form acceptance
sum_v min(p, q) of the accept workload near 0.945 (middle of the 92-97% median
acceptance band of the InvisibleLoRA abstract).  Uses only the oracle and the
input generators; the result is the ACCEPT_SIGMA constant in workloads.

    python tests/golden/calibrate_sigma.py
"""
import os
import sys

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__)))))
import workloads as WL  # noqa: E402
from oracle import accept as OA  # noqa: E402


def mean_rate(sigma, rows=16):
    p, q, _, _ = WL.accept_inputs(WL.LLAMA3_VOCAB, rows, 1, sigma=sigma, seed=0)
    return float(np.mean([OA.acceptance_rate(p[b, 0], q[b, 0]) for b in range(rows)]))


def main(target=0.945):
    lo, hi = 0.01, 1.0
    for _ in range(18):
        mid = 0.5 * (lo + hi)
        if mean_rate(mid) > target:
            lo = mid
        else:
            hi = mid
    s = 0.5 * (lo + hi)
    print(f"sigma={s:.4f} mean_acceptance={mean_rate(s):.4f}")


if __name__ == "__main__":
    main()
