"""Brute-force optimal plan for tiny instances: a plan-quality reference (the
gap of a planning rule to the best possible maximum rank load), not a parity
target and not part of the balancing path.

For every replica placement (each spare slot empty or holding one expert its
rank does not hold yet) the smallest feasible integer maximum rank load is the
max-flow / min-cut value of the transportation network
    source -> expert e (capacity counts[e]) -> rank holding e -> sink (capacity M).
By max-flow / min-cut, all load fits under M exactly when every set X of
experts satisfies  sum_{e in X} counts[e] <= M * |ranks holding some e in X|,
so the optimum of one placement is  max over non-empty X of
ceil(sum_X counts / |holders(X)|).  Enumerating X is fine for E <= 8.
"""
import itertools

import numpy as np


def _placement_opt(tot, holders):
    """tot[X] = sum of counts over the expert set X (bit mask)."""
    E = len(holders)
    hold = [0] * (1 << E)
    best = 0
    for mask in range(1, 1 << E):
        low = (mask & -mask).bit_length() - 1
        hold[mask] = hold[mask & (mask - 1)] | holders[low]
        n = bin(hold[mask]).count("1")
        best = max(best, -(-tot[mask] // n))
    return best


def optimum(counts, R: int, S: int) -> int:
    """Smallest achievable max rank load over all placements (R <= 4, E <= 8, S <= 1)."""
    counts = [int(c) for c in counts]
    E = len(counts)
    H = E // R
    if R > 4 or E > 8 or S > 1:
        raise ValueError("brute force is for tiny instances only")
    home = [1 << (e // H) for e in range(E)]
    # per spare slot: empty (-1) or an expert not at home on that rank
    choices = []
    for r in range(R):
        for _ in range(S):
            choices.append([-1] + [e for e in range(E) if e // H != r])
    tot = [0] * (1 << E)
    for mask in range(1, 1 << E):
        low = (mask & -mask).bit_length() - 1
        tot[mask] = tot[mask & (mask - 1)] + counts[low]
    best = None
    for pick in itertools.product(*choices):
        holders = list(home)
        for slot, e in enumerate(pick):
            if e >= 0:
                holders[e] |= 1 << (slot // S)
        v = _placement_opt(tot, holders)
        best = v if best is None else min(best, v)
    return best
