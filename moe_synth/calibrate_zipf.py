"""Write ``zipf_sigma_v3.txt``: per-expert logit scales that skew the router
of the v3-shaped workload towards a Zipf(1.1) expert popularity.

With x ~ N(0, I) and centroids e_i = sigma_i q_i (q_i orthonormal), the
logits are independent N(0, sigma_i^2), so a calibration batch can draw the
logits directly.  The loads come from the CPU oracle's own routing (group
-limited top-k with zero bias); sigma is updated multiplicatively (damped) towards
the target load, renormalised to a geometric mean of 1 and clamped to
[0.05, 8] (without the clamp the hottest
experts' sigma runs away, their sigmoids saturate at 1.0f and exact ties
flood the routing).

Targets: rank r (1-based) gets T*K * r^-1.1 / H, capped at 0.45 T, because a
sign-symmetric x cannot send an expert more than about half of the tokens.
The rank -> expert map is a seeded permutation so hot experts spread over
groups.

Run from the repository root:  python -m moe_synth.calibrate_zipf
"""

from __future__ import annotations

import os
import sys

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

from oracle import sigmoid_affinity, select_experts, expert_load  # noqa: E402,F401

E, G, GTOP, K = 256, 8, 4, 8
T_CAL = 4096
ZIPF_S = 1.1
ITERS = 40
STEP = 0.3
SEED = 20241227


def targets():
    r = np.arange(1, E + 1, dtype=np.float64)
    p = r ** -ZIPF_S
    p /= p.sum()
    return np.minimum(p * T_CAL * K, 0.45 * T_CAL)


def main():
    rng = np.random.default_rng(SEED)
    rank_of_expert = rng.permutation(E)          # expert i has rank rank_of_expert[i]
    tgt = targets()[rank_of_expert]
    z = rng.standard_normal((T_CAL, E))
    sigma = np.ones(E)
    bias = np.zeros(E, dtype=np.float32)
    for it in range(ITERS):
        s = (1.0 / (1.0 + np.exp(-(z * sigma[None, :])))).astype(np.float32)
        idx = select_experts(s, bias, G, GTOP, K)
        load = expert_load(idx, E).astype(np.float64)
        ratio = (tgt + 1.0) / (load + 1.0)
        sigma = sigma * ratio ** STEP
        # Selection ranks the logits, so only the ratios of sigma matter:
        # pin their geometric mean to 1 before clamping.
        sigma = np.clip(sigma / np.exp(np.mean(np.log(sigma))), 0.05, 8.0)
        top = np.sort(load)[::-1][:6]
        print(f"iter {it}: top loads {top.astype(int).tolist()} "
              f"max/mean {load.max() / load.mean():.2f}", flush=True)
    out = os.path.join(os.path.dirname(os.path.abspath(__file__)), "zipf_sigma_v3.txt")
    with open(out, "w") as f:
        f.write(f"# per-expert logit scale, Zipf({ZIPF_S}) target, E={E}, "
                f"groups {G}/{GTOP}, K={K}; written by moe_synth/calibrate_zipf.py "
                f"(seed {SEED}, {ITERS} iterations on {T_CAL} tokens)\n")
        for v in sigma:
            f.write(f"{v:.9g}\n")
    print("wrote", out)


if __name__ == "__main__":
    main()
