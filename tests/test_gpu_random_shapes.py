"""GPU parity on seeded random shapes: every output of count -> plan -> reroute
(-> permute -> unpermute), through the separate calls or the chained ep_balance,
bit-exact against the CPU oracle.

The hand-picked sweep in test_gpu_parity.py covers the edge cases one by one;
this file draws R, H, S, k, T, the number of instances, the hidden size and the
kind of ids at random (seeded), so that the launch choices (quad, mask-table or
clustered reroute; count chunks and clusters; one or two ranks per planner lane)
meet in combinations nobody wrote down.  Every output buffer carries a guard
tail that must be unchanged.
"""
import numpy as np
import pytest

from moe_expert_load_id_b300 import workload as W

from plan_checks import check_plan, check_reroute

pytestmark = pytest.mark.gpu

N_CASES = 64


def G():
    import gpu_common
    return gpu_common


def _case(i):
    rng = np.random.default_rng(20261203 + i)
    R = int(rng.choice([1, 2, 3, 5, 7, 8, 12, 16, 24, 31, 33, 40, 48, 63, 64]))
    H = int(rng.integers(1, 9))
    while R * H > 1024:
        H -= 1
    S = int(rng.integers(0, 5))
    S = min(S, 32 - H)
    E = R * H
    k = int(rng.integers(1, min(E, 12) + 1))
    if rng.random() < 0.4 and E >= 4:
        k = int(rng.choice([4, 8])) if E >= 8 else 4   # the quad kernel's layouts
    n_inst = int(rng.choice([1, 1, 1, 2, 3, 12, 40]))
    if k % 4 == 0 and rng.random() < 0.5:
        n_inst = max(n_inst, min(300, -(-300 // R)))     # enough ranks for the quad kernel
    T = int(rng.integers(0, 6001 if n_inst <= 3 else 2001))
    Hd = int(rng.choice([0, 8, 16, 520])) if n_inst <= 3 else 0
    kind = str(rng.choice(["zipf", "zipf", "bad", "uniform"]))
    fused = bool(rng.integers(0, 2))
    return R, H, S, k, T, n_inst, Hd, kind, fused


def _ids(R, E, k, T, n_inst, kind, seed):
    rng = np.random.default_rng(seed)
    out = []
    for g in range(n_inst):
        if kind == "uniform":
            ids = rng.integers(0, E, size=(T, k)).astype(np.int32)
        else:
            p = 1.0 / (rng.permutation(E) + 1.0) ** rng.uniform(0.6, 1.6)
            ids = W.gumbel_topk(p / p.sum(), T, k, seed * 131 + g).numpy()
            if kind == "bad" and T:
                ids[rng.integers(0, T, 4), 0] = E + 3
                ids[rng.integers(0, T, 4), k - 1] = -1
                if k > 2:
                    t2 = rng.integers(0, T, 4)
                    ids[t2, 1] = ids[t2, 2]            # an expert twice in one token
        out.append(ids)
    return np.stack(out) if n_inst else np.zeros((0, T, k), np.int32)


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_shape(i):
    R, H, S, k, T, n_inst, Hd, kind, fused = _case(i)
    E = R * H
    ids = _ids(R, E, k, T, n_inst, kind, seed=i + 7)
    hid = None
    if Hd:
        hid = np.random.default_rng(i).integers(0, 1 << 16, size=(n_inst, T, Hd), dtype=np.uint16)
    dom = G().dom_of(R, E, S, k)
    out = G().gpu_run(dom, ids, hid, fused=fused)
    orc = G().oracle_run(R, E, S, ids, hid)
    G().compare(R, E, S, out, orc)
    expect_flag = 1 if any(n > 0 for n in orc["n_bad"]) else 0
    assert int(out["dev_status"][0]) == expect_flag, (R, H, S, k, T, n_inst, kind, fused)
    for g in range(n_inst):
        pl = {key: out[key][g] for key in ("quota", "slot_expert", "rank_load", "inst_ptr",
                                          "inst_id", "inst_cum")}
        pl.update(n_iter=int(out["n_iter"][g]), status=int(out["inst_status"][g]))
        check_plan(out["counts"][g], R, E, S, pl)
        check_reroute(ids[g], R, E, S, pl, out["dst_row"][g], out["src_slot"][g],
                      out["inst_offset"][g])
