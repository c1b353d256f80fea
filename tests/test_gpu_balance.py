"""ep_balance (count -> plan -> reroute chained with programmatic dependent
launch) against the CPU oracle and against the three separate calls, bit for
bit, on seeded inputs; the workspace is left zero.  Plus back-to-back calls
that reuse every buffer on one stream, the way a forward pass calls it layer
after layer."""
import numpy as np
import pytest
import torch

from moe_expert_load_id_b300 import workload as W

pytestmark = pytest.mark.gpu


def G():
    import gpu_common
    return gpu_common


def _zipf_ids(R, E, k, T, n_inst, seed, bad=False):
    rng = np.random.default_rng(seed)
    out = []
    for g in range(n_inst):
        p = 1.0 / (rng.permutation(E) + 1.0) ** 1.1
        ids = W.gumbel_topk(p / p.sum(), T, k, seed * 100 + g).numpy()
        if bad and T:
            ids[rng.integers(0, T, 5), 0] = E + 7
            ids[rng.integers(0, T, 5), -1] = -3
        out.append(ids)
    return np.stack(out) if n_inst else np.zeros((0, T, k), np.int32)


CASES = [
    # name,            R,  H, S, k,  T,     n_inst, bad
    ("tiny_like",      8,  4, 1, 4,  4096,  4,      False),
    ("ragged_T",       8,  4, 1, 4,  1001,  3,      False),
    ("invalid_ids",    8,  4, 2, 4,  2000,  2,      True),
    ("R64",            64, 2, 1, 8,  8192,  1,      False),
    ("R64_full_rank",  64, 2, 1, 8,  131072, 1,     False),   # 16384 slots per source rank
    ("R64_E256_S2",    64, 4, 2, 8,  20000, 1,      False),
    ("R64_3_inst",     64, 2, 1, 8,  4096,  3,      False),   # more wide blocks than SMs
    ("R64_5_inst_quad", 64, 2, 1, 8, 4096,  5,      True),    # the quad reroute kernel
    ("many_chunks",    4,  4, 2, 8,  40000, 1,      False),   # 80000 slots per source rank
    ("max_E_and_k",    64, 16, 16, 32, 1024, 1,     False),
    ("no_spares",      8,  4, 0, 4,  3000,  2,      False),
    ("T_below_R",      8,  2, 1, 3,  5,     1,      False),
    ("R1",             1,  4, 1, 2,  500,   1,      False),
    ("W32",            8,  1, 31, 4, 3000,  2,      False),
    ("empty_T",        8,  4, 1, 4,  0,     2,      False),   # no slots: home placement
    ("k1",             8,  4, 1, 1,  777,   1,      False),
    ("glm_like_layer", 40, 4, 1, 8,  163840, 1,     False),   # 32768 slots per rank, clusters of 2
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_balance_matches_oracle_and_separate_calls(case):
    name, R, H, S, k, T, n_inst, bad = case
    E = R * H
    ids = _zipf_ids(R, E, k, T, n_inst, seed=len(name) * 131 + T, bad=bad)
    dom = G().dom_of(R, E, S, k)
    fused = G().gpu_run(dom, ids, src_slot=True, fused=True)
    assert not fused["workspace"].any()  # left zero for the next call
    assert int(fused["dev_status"][0]) == (1 if bad else 0)  # EP_DEV_BAD_ID only
    G().compare(R, E, S, fused, G().oracle_run(R, E, S, ids), check_rows=False)
    sep = G().gpu_run(dom, ids, src_slot=True, fused=False)
    for key in ("counts", "counts_src", "quota", "slot_expert", "rank_load", "inst_ptr",
                "n_iter", "inst_status", "dst_row", "inst_offset", "src_slot", "dev_status"):
        assert np.array_equal(fused[key], sep[key]), key


def test_balance_iteration_cap():
    R, H, S, k, T = 16, 4, 2, 8, 20000
    ids = _zipf_ids(R, R * H, k, T, 3, 99)
    dom = G().dom_of(R, R * H, S, k)
    out = G().gpu_run(dom, ids, max_iters=2, fused=True)
    G().compare(R, R * H, S, out, G().oracle_run(R, R * H, S, ids, max_iters=2), check_rows=False)
    assert (out["inst_status"] == 2).all()
    assert not out["workspace"].any()


def test_balance_cap_above_the_default():
    R, H, S, k, T = 8, 4, 1, 8, 3000
    ids = _zipf_ids(R, R * H, k, T, 2, 7)
    dom = G().dom_of(R, R * H, S, k)
    cap = (1 << 16) + 1
    out = G().gpu_run(dom, ids, max_iters=cap, fused=True)
    G().compare(R, R * H, S, out, G().oracle_run(R, R * H, S, ids, max_iters=cap),
                check_rows=False)


def test_balance_reuses_its_workspace():
    # the same buffers and workspace through five different instances: every
    # call must find the workspace zero, so a word left behind would show as a
    # wrong plan in a later call
    from moe_expert_load_id_b300 import ultraep as U
    R, H, S, k, T, n_inst = 16, 4, 1, 8, 6000, 2
    E = R * H
    dom = U.Domain(R, E, S, k)
    b = G().guarded_buffers(dom, T, n_inst)
    for it in range(5):
        ids = _zipf_ids(R, E, k, T, n_inst, seed=500 + it)
        b.balance_fused(torch.from_numpy(ids).cuda())
        torch.cuda.synchronize()
        ref = G().oracle_run(R, E, S, ids)
        assert np.array_equal(b.dst_row.cpu().numpy(), np.stack(ref["dst_row"]))
        assert np.array_equal(b.quota.cpu().numpy(), np.stack(ref["quota"]))
        assert not b.workspace.any().item()
    assert int(b.dev_status.item()) == 0
    b.guard.check()


def test_balance_layer_after_layer_reusing_buffers():
    # three Qwen3-235B-like layers through the same buffers on one stream:
    # balance, permute, next layer's balance ... (the benchmark's pattern)
    from moe_expert_load_id_b300 import ultraep as U
    w = W.WORKLOADS["qwen3-235b"]
    dom = U.Domain(w.R, w.E, w.S, w.k)
    b = G().guarded_buffers(dom, w.T, 1, Hd=w.Hd)
    hid = W.hidden(w.T, w.Hd, w.seed(1000, 2), device="cuda")[None]
    layers = [W.topk_ids(w, l, 2, device="cuda")[None] for l in range(3)]
    got = []
    for ids in layers:
        b.balance_fused(ids)
        b.permute(hid)
        got.append((b.counts.clone(), b.quota.clone(), b.dst_row.clone()))
    torch.cuda.synchronize()
    assert int(b.dev_status.item()) == 0
    ref = G().guarded_buffers(dom, w.T, 1, guard=b.guard)
    for ids, (c, q, d) in zip(layers, got):
        ref.count(ids)
        ref.plan()
        ref.reroute(ids)
        torch.cuda.synchronize()
        assert torch.equal(c, ref.counts) and torch.equal(q, ref.quota)
        assert torch.equal(d, ref.dst_row)
    # one layer fully against the oracle
    import oracle
    ids_h = layers[2][0].cpu().numpy()
    cnt, _, _ = oracle.count(ids_h, w.R, w.E)
    pl = oracle.plan(cnt, w.R, w.E, w.S)
    dst, _, _ = oracle.reroute(ids_h, w.R, w.E, w.S, pl)
    assert np.array_equal(got[2][2][0].cpu().numpy(), dst)
    b.guard.check()
