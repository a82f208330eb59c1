"""Choose the d2t workload's support bias and per-position draft noise.

The target profile is the DSpark per-position acceptance quoted in
"speculative decoding for Omni models", section 3 (0.714, 0.619, 0.553,
0.508, 0.474, 0.446, 0.423), with a mean off-support p-mass near 0.10 (a
truncated draft vocabulary that keeps the frequent ids, section 4).  The
acceptance of a position is 1 - TV computed by the oracle; the bias is set
from the mean p-mass off the d2t support.  Prints D2T_DELTA and D2T_SIGMA
for workloads.py.  Run: python oracle/calibrate_d2t.py  (CPU, about a minute).
"""
import os
import sys

import numpy as np
import torch

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import oracle  # noqa: E402
import workloads  # noqa: E402

TARGET_ALPHA = [0.714, 0.619, 0.553, 0.508, 0.474, 0.446, 0.423]
R, V, VD, T = 48, workloads.V_QWEN, workloads.VD_DRAFT, 0.7


def off_support_mass(delta):
    w = workloads.sample_batch(R, 1, V, VD, torch.bfloat16, T=T, sigma_pos=1.0, delta=delta, seed=5, device="cpu")
    z = w["target"].float().numpy().astype(np.float64) / T
    p = np.exp(z - z.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    on = np.zeros(V, bool)
    on[w["d2t"].numpy()] = True
    return p[:, ~on].sum(1).mean()


def mean_alpha(delta, sigma, seed):
    w = workloads.sample_batch(R, 1, V, VD, torch.bfloat16, T=T, sigma_pos=sigma, delta=delta, seed=seed,
                               device="cpu")
    out = oracle.verify_sample(workloads.host_rows(w["target"]), workloads.host_rows(w["draft_logits"]),
                               w["d2t"].numpy(), R, 1, w["draft"].numpy(), w["seeds"].numpy().view(np.uint64),
                               w["temperature"].numpy())
    return 1.0 - out["tv"][:, 0].mean()


def bisect(f, lo, hi, target, increasing, iters=12):
    for _ in range(iters):
        mid = 0.5 * (lo + hi)
        v = f(mid)
        if (v < target) == increasing:
            lo = mid
        else:
            hi = mid
    return 0.5 * (lo + hi)


if __name__ == "__main__":
    delta = bisect(off_support_mass, 0.0, 12.0, 0.10, increasing=False)
    print(f"D2T_DELTA = {delta:.2f}  (mean off-support mass {off_support_mass(delta):.3f})")
    sig = []
    for i, a in enumerate(TARGET_ALPHA):
        s = bisect(lambda x: mean_alpha(delta, x, 100), 0.05, 12.0, a, increasing=False, iters=10)
        sig.append(round(s, 2))
        print(f"  position {i}: sigma {s:.2f} -> alpha {mean_alpha(delta, s, 200 + i):.3f} (target {a})")
    print(f"D2T_SIGMA = {sig}")
