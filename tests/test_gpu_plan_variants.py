"""ep_plan_ex (the planner's skip and release variants) against the CPU oracle,
bit for bit: the hand-worked examples, random count vectors up to R = 64 for
every flag combination, the iteration cap (including the prefix property: the
skip variant capped at the base rule's move count is in the base rule's state),
whole tiny-workload layers through reroute, and one full-size
Qwen3-235B-like layer."""
import numpy as np
import pytest
import torch

import oracle
from golden_io import read_sections, as_array
from moe_expert_load_id_b300 import workload as W

pytestmark = pytest.mark.gpu

FLAGS = {"skip": 1, "release": 2, "skip+release": 3}
EXAMPLES = read_sections("plan_skip_examples.txt")


def U():
    from moe_expert_load_id_b300 import ultraep
    return ultraep


def G():
    import gpu_common
    return gpu_common


def _gpu_plan(R, E, S, counts, flags, max_iters=0):
    counts = np.ascontiguousarray(counts, dtype=np.int32).reshape(-1, E)
    n = counts.shape[0]
    b = G().guarded_buffers(U().Domain(R, E, S, 1), 1, n)
    b.counts.copy_(torch.from_numpy(counts))
    b.plan(max_iters=max_iters, flags=flags)
    b.guard.check()
    return {key: getattr(b, key).cpu().numpy() for key in
            ("quota", "slot_expert", "rank_load", "inst_ptr", "inst_id", "inst_cum", "n_iter",
             "inst_status")}


def _same(got, g, want):
    for key in ("quota", "rank_load", "inst_ptr"):
        assert np.array_equal(got[key][g], want[key]), key
    assert np.array_equal(got["slot_expert"][g].reshape(-1), want["slot_expert"].reshape(-1))
    m = int(want["inst_ptr"][-1])
    assert np.array_equal(got["inst_id"][g][:m], want["inst_id"][:m])
    assert np.array_equal(got["inst_cum"][g][:m], want["inst_cum"][:m])
    assert int(got["n_iter"][g]) == want["n_iter"]
    assert int(got["inst_status"][g]) == want["status"]


@pytest.mark.parametrize("name", sorted(EXAMPLES))
def test_hand_examples(name):
    ex = EXAMPLES[name]
    variant = ("base" if name.endswith("_base_rule") else
               "skip+release" if name.endswith("_skip_release") else "skip")
    flags = 0 if variant == "base" else FLAGS[variant]
    got = _gpu_plan(ex["R"], ex["E"], ex["S"], as_array(ex["counts"]), flags, ex["max_iters"])
    want = dict(quota=as_array(ex["quota"]), slot_expert=as_array(ex["slot_expert"]),
                rank_load=as_array(ex["rank_load"]), inst_ptr=as_array(ex["inst_ptr"]),
                inst_id=as_array(ex["inst_id"]), inst_cum=as_array(ex["inst_cum"]),
                n_iter=ex["n_iter"], status=ex["status"])
    _same(got, 0, want)


def _random_batch(seed, n=24):
    rng = np.random.default_rng(seed)
    R = int(rng.choice([2, 3, 5, 8, 16, 33, 64]))
    H = int(rng.choice([1, 2, 4]))
    S = int(rng.choice([1, 2, 3]))
    while H + S > 32 or R * H > 1024:
        H = max(1, H // 2)
    E = R * H
    c = np.stack([(300.0 / (1 + rng.permutation(E)) ** rng.uniform(0.5, 1.6)).astype(np.int32)
                  if rng.random() < 0.7 else rng.integers(0, 60, size=E).astype(np.int32)
                  for _ in range(n)])
    return R, E, S, c


@pytest.mark.parametrize("variant", sorted(FLAGS))
@pytest.mark.parametrize("seed", range(6))
def test_random_counts(variant, seed):
    R, E, S, c = _random_batch(seed * 10 + len(variant))
    got = _gpu_plan(R, E, S, c, FLAGS[variant])
    for g in range(c.shape[0]):
        _same(got, g, oracle.plan(c[g], R, E, S, variant=variant))


def test_skip_cap_and_prefix():
    R, E, S, c = _random_batch(77, n=12)
    for g in range(c.shape[0]):
        base = oracle.plan(c[g], R, E, S)
        for cap in (1, max(1, base["n_iter"])):
            got = _gpu_plan(R, E, S, c[g], FLAGS["skip"], max_iters=cap)
            want = oracle.plan(c[g], R, E, S, max_iters=cap, variant="skip")
            _same(got, 0, want)
        capped = _gpu_plan(R, E, S, c[g], FLAGS["skip"], max_iters=max(1, base["n_iter"]))
        if base["n_iter"] > 0:
            assert np.array_equal(capped["quota"][0], base["quota"])


@pytest.mark.parametrize("variant", ["skip", "skip+release"])
def test_tiny_workload_through_reroute(variant):
    w = W.WORKLOADS["tiny"]
    ids = np.stack([W.topk_ids(w, l, 0).numpy() for l in range(w.layers)])
    out = G().gpu_run(G().dom_of(w.R, w.E, w.S, w.k), ids, flags=FLAGS[variant])
    orc = G().oracle_run(w.R, w.E, w.S, ids, variant=variant)
    G().compare(w.R, w.E, w.S, out, orc, check_rows=False)


def test_full_size_layer_skip():
    w = W.WORKLOADS["qwen3-235b"]
    ids = W.topk_ids(w, 11, 0, device="cuda")[None]
    b = G().guarded_buffers(U().Domain(w.R, w.E, w.S, w.k), w.T, 1)
    b.count(ids)
    b.plan(flags=FLAGS["skip+release"])
    b.guard.check()
    c = b.counts.cpu().numpy()[0]
    want = oracle.plan(c, w.R, w.E, w.S, variant="skip+release")
    got = {key: getattr(b, key).cpu().numpy() for key in
           ("quota", "slot_expert", "rank_load", "inst_ptr", "inst_id", "inst_cum", "n_iter",
            "inst_status")}
    _same(got, 0, want)
    base = oracle.plan(c, w.R, w.E, w.S)
    assert want["rank_load"].max() <= base["rank_load"].max()


# The flag-free rule with more than four instances per rank runs the planner's
# shared-memory table loop; these shapes (W = H + S from 5 to 12, one and two
# ranks per lane, both key widths) pin it to the oracle on random counts and
# under caps.
TABLE_SHAPES = [(3, 4, 1), (8, 4, 2), (33, 2, 3), (64, 4, 4), (64, 8, 4), (16, 4, 8)]


@pytest.mark.parametrize("shape", TABLE_SHAPES, ids=[f"R{r}H{h}S{s}" for r, h, s in TABLE_SHAPES])
def test_base_rule_table_loop(shape):
    R, H, S = shape
    E = R * H
    rng = np.random.default_rng(R * 100 + H * 10 + S)
    c = np.stack([(400.0 / (1 + rng.permutation(E)) ** rng.uniform(0.5, 1.6)).astype(np.int32)
                  for _ in range(16)])
    got = _gpu_plan(R, E, S, c, 0)
    for g in range(c.shape[0]):
        _same(got, g, oracle.plan(c[g], R, E, S))
    # caps: the state after exactly `cap` moves, flagged
    full = min(int(oracle.plan(c[g], R, E, S)["n_iter"]) for g in range(c.shape[0]))
    for cap in (1, max(1, full // 2)):
        got = _gpu_plan(R, E, S, c, 0, cap)
        for g in range(c.shape[0]):
            _same(got, g, oracle.plan(c[g], R, E, S, max_iters=cap))


def test_base_rule_table_loop_wide_keys():
    # totals of 2^25 and more take the planner's unpacked reductions
    R, H, S = 64, 4, 2
    E = R * H
    rng = np.random.default_rng(5)
    c = (rng.random((4, E)) ** 3 * 2.0e6).astype(np.int32)
    assert (c.sum(1) >= (1 << 25)).all()
    got = _gpu_plan(R, E, S, c, 0)
    for g in range(c.shape[0]):
        _same(got, g, oracle.plan(c[g], R, E, S))


# The skip variants keep each lane's ranks' instances in registers when a rank
# has at most 8 (W = H + S); wider ranks take the shared-memory table loop.
# These shapes pin both against the oracle: W = 1 (no spare slot), 8 (the
# widest cached), 9, 10 and 32 (the table loop), one and two ranks per lane,
# and totals past 2^25 (the unpacked reductions) on the cached loop.
SKIP_SHAPES = [(5, 1, 0), (16, 2, 6), (64, 4, 4), (8, 8, 1), (33, 4, 6), (20, 16, 16)]


@pytest.mark.parametrize("variant", ["skip", "skip+release"])
@pytest.mark.parametrize("shape", SKIP_SHAPES, ids=[f"R{r}H{h}S{s}" for r, h, s in SKIP_SHAPES])
def test_skip_instance_widths(shape, variant):
    R, H, S = shape
    E = R * H
    rng = np.random.default_rng(R * 1000 + H * 10 + S)
    c = np.stack([(500.0 / (1 + rng.permutation(E)) ** rng.uniform(0.5, 1.6)).astype(np.int32)
                  for _ in range(12)])
    got = _gpu_plan(R, E, S, c, FLAGS[variant])
    for g in range(c.shape[0]):
        _same(got, g, oracle.plan(c[g], R, E, S, variant=variant))
    cap = max(1, min(int(oracle.plan(c[g], R, E, S, variant=variant)["n_iter"])
                     for g in range(c.shape[0])) // 2)
    got = _gpu_plan(R, E, S, c, FLAGS[variant], cap)
    for g in range(c.shape[0]):
        _same(got, g, oracle.plan(c[g], R, E, S, max_iters=cap, variant=variant))


def test_skip_wide_keys():
    # totals of 2^25 and more: the cached skip loop's unpacked reductions
    R, H, S = 64, 2, 1
    E = R * H
    rng = np.random.default_rng(9)
    c = (rng.random((3, E)) ** 3 * 4.0e6).astype(np.int32)
    assert (c.sum(1) >= (1 << 25)).all()
    got = _gpu_plan(R, E, S, c, FLAGS["skip"], 3000)
    for g in range(c.shape[0]):
        _same(got, g, oracle.plan(c[g], R, E, S, max_iters=3000, variant="skip"))
