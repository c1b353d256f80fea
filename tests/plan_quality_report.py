"""Plan quality of the planner variants against the brute-force optimum and
the lower bound on tiny instances (CPU, oracle only).  A report, not a test:

    python tests/plan_quality_report.py [--n 300] [--seed 1]

For n random tiny instances (R in {2,3,4}, H in {1,2}, S = 1, Zipf-like or
uniform counts) it prints, for the base rule and the two variants, the mean and
the worst of max_load / optimum and of max_load / LB, and how often the plan is
optimal.
"""
import argparse
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from oracle import bruteforce  # noqa: E402
from moe_expert_load_id_b300 import quality as Q  # noqa: E402


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--n", type=int, default=300)
    ap.add_argument("--seed", type=int, default=1)
    args = ap.parse_args()
    rng = np.random.default_rng(args.seed)
    variants = ("base", "skip", "skip+release")
    gap_opt = {v: [] for v in variants}
    gap_lb = {v: [] for v in variants}
    for _ in range(args.n):
        R = int(rng.integers(2, 5))
        H = int(rng.integers(1, 3))
        E = R * H
        if rng.random() < 0.5:
            c = (40.0 / (1 + rng.permutation(E)) ** rng.uniform(0.8, 1.6)).astype(np.int32)
        else:
            c = rng.integers(0, 16, size=E).astype(np.int32)
        if c.sum() == 0:
            continue
        opt = bruteforce.optimum(c, R, 1)
        lb = Q.lower_bound(c.astype(np.int64), R, 1)
        for v in variants:
            m = int(oracle.plan(c, R, E, 1, variant=v)["rank_load"].max())
            gap_opt[v].append(m / opt)
            gap_lb[v].append(m / lb)
    print(f"{len(gap_opt['base'])} tiny instances (R 2-4, H 1-2, S 1), seed {args.seed}")
    print("| rule | max/opt mean | max/opt worst | optimal | max/LB mean | max/LB worst |")
    print("|---|---|---|---|---|---|")
    for v in variants:
        g = np.array(gap_opt[v])
        b = np.array(gap_lb[v])
        print(f"| {v} | {g.mean():.4f} | {g.max():.4f} | {np.mean(g == 1.0):.1%} | "
              f"{b.mean():.4f} | {b.max():.4f} |")


if __name__ == "__main__":
    main()
