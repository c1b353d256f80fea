"""Pins of the brute-force optimum (moe_expert_load_id_b300/bruteforce.py), the quality reference
the plan-quality report compares the planning rule with.  No GPU needed.

- hand-worked optima (tests/golden/bruteforce_optimum_examples.txt), including
  one below the base rule's maximum and one above the lower bound;
- an exhaustive search on tiny totals that tries every placement and every split
  of every unit of load over the ranks holding its expert, written from the
  definition of the optimum (not through max-flow / Hall's condition, which
  `optimum` relies on);
- planted mistakes in copies of bruteforce.py must each fail one of the pins.
"""
import itertools
import types

import numpy as np
import pytest

import oracle
from moe_expert_load_id_b300 import bruteforce
from golden_io import read_sections, as_array
from moe_expert_load_id_b300 import quality as Q

EX = read_sections("bruteforce_optimum_examples.txt")


def _splits(c, n):
    """Every way of giving c units to n holders (tuples of n non-negative ints)."""
    if n == 1:
        yield (c,)
        return
    for first in range(c + 1):
        for rest in _splits(c - first, n - 1):
            yield (first,) + rest


def exhaustive_optimum(counts, R, S):
    """The smallest maximum rank load over every replica placement (each spare
    slot empty or holding an expert its rank does not hold) and every split of
    every expert's units over the ranks holding it.  Tiny inputs only."""
    E = len(counts)
    H = E // R
    slots = [[-1] + [e for e in range(E) if e // H != r] for r in range(R) for _ in range(S)]
    best = None
    for pick in itertools.product(*slots):
        holders = [{e // H} for e in range(E)]
        for x, e in enumerate(pick):
            if e >= 0:
                holders[e].add(x // S)
        hl = [sorted(h) for h in holders]
        for split in itertools.product(*[list(_splits(int(counts[e]), len(hl[e])))
                                         for e in range(E)]):
            load = [0] * R
            for e in range(E):
                for r, u in zip(hl[e], split[e]):
                    load[r] += u
            m = max(load)
            if best is None or m < best:
                best = m
    return best


@pytest.mark.parametrize("name", sorted(EX))
def test_hand_worked_optimum(name, opt_fn=None):
    ex = EX[name]
    fn = opt_fn or bruteforce.optimum
    counts = as_array(ex["counts"])
    assert fn(counts, ex["R"], ex["S"]) == ex["opt"]


@pytest.mark.parametrize("name", sorted(n for n in EX if "base_max" in EX[n]))
def test_hand_worked_base_rule(name):
    ex = EX[name]
    pl = oracle.plan(as_array(ex["counts"]), ex["R"], ex["E"], ex["S"])
    assert int(pl["rank_load"].max()) == ex["base_max"]


def test_hand_worked_lower_bound_gap():
    # the one worked example where the optimum is strictly above the lower bound
    ex = EX["opt_ex4_above_the_lower_bound"]
    assert Q.lower_bound(as_array(ex["counts"]), ex["R"], ex["S"]) == ex["opt"] - 1


def _tiny_cases(seed, n):
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        R = int(rng.integers(2, 4))
        H = int(rng.integers(1, 3)) if R == 2 else 1
        E = R * H
        S = int(rng.integers(0, 2))
        counts = rng.multinomial(int(rng.integers(1, 8)), rng.dirichlet(np.ones(E) * 0.5))
        out.append((R, S, counts.astype(np.int64)))
    return out


@pytest.mark.parametrize("seed", range(6))
def test_against_exhaustive_search(seed, opt_fn=None):
    fn = opt_fn or bruteforce.optimum
    for R, S, counts in _tiny_cases(seed, 12):
        assert fn(counts, R, S) == exhaustive_optimum(counts, R, S), (R, S, counts.tolist())


def test_exhaustive_search_on_hand_examples():
    # the exhaustive search itself agrees with the hand-worked values it can reach
    for name in ("opt_ex1_two_ranks", "opt_ex3_below_the_base_rule", "opt_ex5_rounding_up",
                 "opt_ex6_no_spare_slots", "opt_ex7_replica_off_home_only"):
        ex = EX[name]
        assert exhaustive_optimum(as_array(ex["counts"]), ex["R"], ex["S"]) == ex["opt"], name


def test_optimum_between_bound_and_plan():
    rng = np.random.default_rng(11)
    for _ in range(30):
        R = int(rng.integers(2, 5))
        H = int(rng.integers(1, 3))
        counts = rng.integers(0, 20, size=R * H)
        opt = bruteforce.optimum(counts, R, 1)
        assert Q.lower_bound(counts, R, 1) <= opt
        assert opt <= int(oracle.plan(counts, R, R * H, 1)["rank_load"].max())


# ---------------------------------------------------------------- planted mistakes
MUTANTS = {
    "replica only on the home rank": ("if e // H != r", "if e // H == r"),
    "spare slots ignored": ("for _ in range(S):", "for _ in range(0):"),
    "rounding down": ("best = max(best, -(-tot[mask] // n))", "best = max(best, tot[mask] // n)"),
    "only the set of all experts": ("best = max(best, -(-tot[mask] // n))",
                                    "best = -(-tot[mask] // n)"),
    "first placement kept": ("best = v if best is None else min(best, v)",
                             "best = v if best is None else best"),
    "replica credited to the next rank": ("holders[e] |= 1 << (slot // S)",
                                          "holders[e] |= 1 << ((slot // S + 1) % R)"),
}


def _mutant(before, after):
    with open(bruteforce.__file__) as f:
        src = f.read()
    assert before in src, before
    mod = types.ModuleType("bruteforce_mutant")
    exec(compile(src.replace(before, after, 1), "bruteforce_mutant", "exec"), mod.__dict__)
    return mod.optimum


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name):
    fn = _mutant(*MUTANTS[name])
    failed = False
    for ex_name in sorted(EX):
        try:
            test_hand_worked_optimum(ex_name, opt_fn=fn)
        except AssertionError:
            failed = True
    if not failed:
        for seed in range(6):
            try:
                test_against_exhaustive_search(seed, opt_fn=fn)
            except AssertionError:
                failed = True
    assert failed, f"no pin fails for the planted mistake '{name}'"
