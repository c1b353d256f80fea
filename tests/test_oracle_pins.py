"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: library
routines (numpy bincount / stable argsort / fancy-index gather), hand-worked
examples of the rule (tests/golden), closed-form special cases, invariants of
the problem statement, the lower bound and the brute-force optimum.
"""
import numpy as np
import pytest

import oracle
from moe_expert_load_id_b300 import bruteforce
from moe_expert_load_id_b300 import quality as Q
from moe_expert_load_id_b300 import workload as W

from golden_io import read_sections, as_array
from plan_checks import check_plan, check_stopped, check_reroute

HAND = read_sections("plan_hand_examples.txt")


# ---------------------------------------------------------------- count
@pytest.mark.parametrize("T,k,R,E", [(0, 4, 8, 32), (1, 1, 4, 8), (37, 3, 4, 8),
                                     (1000, 8, 64, 128), (4096, 4, 8, 32), (5, 2, 8, 16)])
def test_count_is_a_histogram(T, k, R, E):
    rng = np.random.default_rng(T * 31 + k)
    ids = rng.integers(-2, E + 2, size=(T, k)).astype(np.int32)
    counts, counts_src, n_bad = oracle.count(ids, R, E)
    flat = ids.reshape(-1)
    ok = (flat >= 0) & (flat < E)
    assert n_bad == int((~ok).sum())
    assert (counts == np.bincount(flat[ok], minlength=E)).all()
    Tr = -(-T // R) if T else 1
    for r in range(R):
        part = ids[r * Tr:(r + 1) * Tr].reshape(-1)
        part = part[(part >= 0) & (part < E)]
        assert (counts_src[r] == np.bincount(part, minlength=E)).all()
    assert counts.sum() == ok.sum() == counts_src.sum()


# ---------------------------------------------------------------- plan: hand examples
@pytest.mark.parametrize("name", sorted(HAND))
def test_plan_hand_examples(name):
    ex = HAND[name]
    R, E, S = ex["R"], ex["E"], ex["S"]
    if "ids" in ex:
        ids = as_array(ex["ids"]).reshape(ex["T"], ex["k"])
        counts, counts_src, n_bad = oracle.count(ids, R, E)
        assert (counts == as_array(ex["counts"])).all()
        if "counts_src" in ex:
            assert (counts_src.reshape(-1) == as_array(ex["counts_src"])).all()
            assert n_bad == ex["n_invalid"]
    pl = oracle.plan(as_array(ex["counts"]), R, E, S, max_iters=ex["max_iters"])
    for key in ("quota", "rank_load", "inst_ptr"):
        assert (pl[key] == as_array(ex[key])).all(), key
    assert (pl["slot_expert"].reshape(-1) == as_array(ex["slot_expert"])).all()
    n_inst = pl["inst_ptr"][E]
    assert (pl["inst_id"][:n_inst] == as_array(ex["inst_id"])).all()
    assert (pl["inst_cum"][:n_inst] == as_array(ex["inst_cum"])).all()
    assert pl["n_iter"] == ex["n_iter"]
    assert pl["status"] == ex["status"]
    check_plan(as_array(ex["counts"]), R, E, S, pl, max_iters=ex["max_iters"])
    check_stopped(as_array(ex["counts"]), R, E, S, pl)


@pytest.mark.parametrize("name", [n for n in sorted(HAND) if "ids" in HAND[n]])
def test_reroute_hand_examples(name):
    ex = HAND[name]
    R, E, S = ex["R"], ex["E"], ex["S"]
    ids = as_array(ex["ids"]).reshape(ex["T"], ex["k"])
    pl = oracle.plan(as_array(ex["counts"]), R, E, S)
    dst_row, src_slot, inst_offset = oracle.reroute(ids, R, E, S, pl)
    assert (inst_offset == as_array(ex["inst_offset"])).all()
    assert (dst_row == as_array(ex["dst_row"])).all()
    assert (src_slot == as_array(ex["src_slot"])).all()


# ---------------------------------------------------------------- plan: properties
def _random_counts(rng, R, E, kind):
    if kind == "zipf":
        p = 1.0 / (rng.permutation(E) + 1.0) ** rng.uniform(0.5, 2.0)
        return rng.multinomial(int(rng.integers(0, 5000)), p / p.sum())
    if kind == "sparse":
        c = np.zeros(E, dtype=np.int64)
        c[rng.integers(0, E, size=3)] = rng.integers(0, 1000, size=3)
        return c
    return rng.integers(0, 200, size=E)


@pytest.mark.parametrize("seed", range(40))
def test_plan_invariants_random(seed):
    rng = np.random.default_rng(1000 + seed)
    R = int(rng.choice([1, 2, 3, 4, 8, 16, 40, 64]))
    H = int(rng.choice([1, 2, 3, 4]))
    S = int(rng.choice([0, 1, 2, 4]))
    E = R * H
    counts = _random_counts(rng, R, E, ["zipf", "sparse", "flat"][seed % 3])
    pl = oracle.plan(counts, R, E, S)
    assert pl["status"] == 0
    check_plan(counts, R, E, S, pl)
    check_stopped(counts, R, E, S, pl)
    assert pl["rank_load"].max() >= Q.lower_bound(counts, R, S)


def test_plan_no_spare_slots_is_identity():
    rng = np.random.default_rng(7)
    for R, H in [(4, 2), (8, 4), (64, 2)]:
        counts = rng.integers(0, 1000, size=R * H)
        pl = oracle.plan(counts, R, R * H, 0)
        assert pl["n_iter"] == 0
        home_p = np.arange(R * H)            # W = H when S = 0
        assert (pl["quota"][home_p] == counts).all()


def test_plan_balanced_input_does_not_move():
    # all rank loads within 1 of each other: q = floor(diff/2) = 0 at once
    for R, H, S in [(4, 2, 1), (8, 1, 2), (64, 2, 1)]:
        counts = np.full(R * H, 5)
        counts[0] += 1
        pl = oracle.plan(counts, R, R * H, S)
        assert pl["n_iter"] == 0


@pytest.mark.parametrize("R,S,total", [(2, 1, 11), (3, 1, 12), (8, 1, 1001), (8, 2, 77),
                                       (64, 1, 123457), (16, 4, 5)])
def test_plan_single_hot_expert_levels_ranks(R, S, total):
    # all load on one expert and a spare slot on every rank: the rule keeps
    # halving the gap between the hottest and the coldest rank, so the loads
    # end within 1 of each other, i.e. at ceil/floor(total / R).
    E = R
    counts = np.zeros(E, dtype=np.int64)
    counts[0] = total
    pl = oracle.plan(counts, R, E, S)
    load = pl["rank_load"]
    assert load.max() - load.min() <= 1
    assert load.max() == -(-total // R)


@pytest.mark.parametrize("seed", range(12))
def test_plan_against_bruteforce_optimum(seed):
    rng = np.random.default_rng(2000 + seed)
    R = int(rng.choice([2, 3, 4]))
    H = 2 if R == 4 else int(rng.choice([1, 2]))
    E, S = R * H, 1
    counts = rng.integers(0, 30, size=E)
    counts[rng.integers(0, E)] += int(rng.integers(0, 60))
    pl = oracle.plan(counts, R, E, S)
    opt = bruteforce.optimum(counts, R, S)
    lb = Q.lower_bound(counts, R, S)
    assert lb <= opt <= pl["rank_load"].max()


def test_plan_iteration_cap_random():
    rng = np.random.default_rng(5)
    counts = rng.multinomial(100000, np.ones(64) / 64 * np.linspace(0.1, 3, 64) / 1.55)
    full = oracle.plan(counts, 16, 64, 2)
    assert full["n_iter"] > 3
    for cap in (0, 1, full["n_iter"] // 2, full["n_iter"] - 1):
        pl = oracle.plan(counts, 16, 64, 2, max_iters=cap)
        assert pl["status"] == 2 and pl["n_iter"] == cap
        check_plan(counts, 16, 64, 2, pl, max_iters=cap)
    pl = oracle.plan(counts, 16, 64, 2, max_iters=full["n_iter"])
    assert pl["status"] == 0


def test_lower_bound_hand_values():
    # R=2, H=2, S=1: counts [9,1 | 1,1]: total 12 -> 6; LB_home: remove 9 -> ranks (1, 2) -> 2.
    assert Q.lower_bound([9, 1, 1, 1], 2, 1) == 6
    # S=0: LB_home = max home load
    assert Q.lower_bound([9, 1, 1, 1], 2, 0) == 10
    # R=2, H=2, S=1, counts [10,10 | 0,0]: one removal from rank 0 leaves 10 -> LB = 10
    assert Q.lower_bound([10, 10, 0, 0], 2, 1) == 10


# ---------------------------------------------------------------- reroute / permute
@pytest.mark.parametrize("seed", range(10))
def test_reroute_properties_random(seed):
    rng = np.random.default_rng(3000 + seed)
    R = int(rng.choice([2, 4, 8]))
    H = int(rng.choice([1, 2, 4]))
    S = int(rng.choice([0, 1, 2]))
    E = R * H
    T, k = int(rng.integers(0, 300)), int(rng.choice([1, 2, 4]))
    k = min(k, E)
    p = 1.0 / (rng.permutation(E) + 1.0) ** 1.2
    ids = W.gumbel_topk(p / p.sum(), T, k, seed).numpy()
    if T and seed % 3 == 0:
        ids[rng.integers(0, T), 0] = E + 3          # one invalid id
    counts, _, _ = oracle.count(ids, R, E)
    pl = oracle.plan(counts, R, E, S)
    dst_row, src_slot, inst_offset = oracle.reroute(ids, R, E, S, pl)
    check_reroute(ids, R, E, S, pl, dst_row, src_slot, inst_offset)
    # grouped order is a stable sort of the valid slots by their instance
    flat = ids.reshape(-1)
    valid = (flat >= 0) & (flat < E)
    p_of = np.searchsorted(inst_offset, dst_row, side="right") - 1
    key = np.where(valid, p_of, 1 << 30)
    order = np.argsort(key, kind="stable")[:int(valid.sum())]
    assert (src_slot[:order.size] == order).all()


@pytest.mark.parametrize("T,k,Hd", [(0, 2, 8), (1, 1, 8), (17, 3, 16), (64, 8, 24)])
def test_permute_unpermute_are_gathers(T, k, Hd):
    rng = np.random.default_rng(T + Hd)
    hidden = rng.integers(0, 1 << 16, size=(T, Hd), dtype=np.uint16)
    hidden[0:1, 0:2] = np.array([0x8000, 0x7FC1], dtype=np.uint16)[:Hd] if T else hidden[0:1, 0:2]
    N = T * k
    perm = rng.permutation(N).astype(np.int32)
    out = oracle.permute(hidden, k, perm, N)
    assert (out == hidden[perm // k]).all()           # numpy fancy-index gather
    dst_row = np.empty(N, np.int32)
    dst_row[perm] = np.arange(N, dtype=np.int32)
    if N:
        dst_row[0] = -1                               # one slot without a row
    y = oracle.unpermute(out, T, k, dst_row)
    flat = y.reshape(N, Hd)
    for i in range(N):
        if dst_row[i] < 0:
            assert (flat[i] == 0).all()
        else:
            assert (flat[i] == hidden[i // k]).all()  # round trip restores the token's row


def test_pipeline_round_trip_tiny_workload():
    w = W.WORKLOADS["tiny"]
    ids = W.topk_ids(w, 1, 0).numpy()
    hid = W.bf16_bits(W.hidden(w.T, w.Hd, 99))
    counts, _, _ = oracle.count(ids, w.R, w.E)
    pl = oracle.plan(counts, w.R, w.E, w.S)
    check_plan(counts, w.R, w.E, w.S, pl)
    dst_row, src_slot, inst_offset = oracle.reroute(ids, w.R, w.E, w.S, pl)
    check_reroute(ids, w.R, w.E, w.S, pl, dst_row, src_slot, inst_offset)
    grouped = oracle.permute(hid, w.k, src_slot, w.N)
    y = oracle.unpermute(grouped, w.T, w.k, dst_row)
    assert (y == hid[:, None, :]).all()
