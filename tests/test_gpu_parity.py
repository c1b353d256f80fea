"""GPU parity: every C-ABI call against the CPU oracle, bit-exact, on seeded inputs.

Every case compares every output element.  At full size the bf16 rows are
compared on the device, in chunks: each permuted row against the hidden row
of the token the oracle's src_slot names, and each unpermuted slot against its
own token's row (what the oracle's unpermute of its permute gives).  Every
output buffer carries a guard tail that must be unchanged after the calls.
"""
import numpy as np
import pytest
import torch

import oracle
from moe_expert_load_id_b300 import workload as W

from golden_io import read_sections, as_array
from plan_checks import check_plan, check_reroute

pytestmark = pytest.mark.gpu

U = None


@pytest.fixture(scope="module", autouse=True)
def lib():
    """Load the C-ABI binding (an ImportError here means the library is not built)."""
    global U
    from moe_expert_load_id_b300 import ultraep
    U = ultraep
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    yield


def G():
    import gpu_common
    return gpu_common


def _ids_from_counts(counts, seed):
    rng = np.random.default_rng(seed)
    ids = np.repeat(np.arange(len(counts), dtype=np.int32), counts)
    rng.shuffle(ids)
    return ids.reshape(1, -1, 1)


# ------------------------------------------------------------------ hand examples
HAND = read_sections("plan_hand_examples.txt")


@pytest.mark.parametrize("name", sorted(HAND))
def test_hand_examples(name):
    ex = HAND[name]
    R, E, S = ex["R"], ex["E"], ex["S"]
    if "ids" in ex:
        ids = as_array(ex["ids"]).astype(np.int32).reshape(1, ex["T"], ex["k"])
    else:
        ids = _ids_from_counts(as_array(ex["counts"]), 5)
    k = ids.shape[2]
    dom = G().dom_of(R, E, S, k)
    out = G().gpu_run(dom, ids, max_iters=ex["max_iters"])
    for key in ("quota", "rank_load", "inst_ptr"):
        G().assert_equal(key, out[key][0], as_array(ex[key]))
    G().assert_equal("slot_expert", out["slot_expert"][0].reshape(-1), as_array(ex["slot_expert"]))
    m = int(as_array(ex["inst_ptr"])[-1])
    G().assert_equal("inst_id", out["inst_id"][0][:m], as_array(ex["inst_id"]))
    G().assert_equal("inst_cum", out["inst_cum"][0][:m], as_array(ex["inst_cum"]))
    assert int(out["n_iter"][0]) == ex["n_iter"]
    assert int(out["inst_status"][0]) == ex["status"]
    if "dst_row" in ex:
        G().assert_equal("dst_row", out["dst_row"][0], as_array(ex["dst_row"]))
        G().assert_equal("inst_offset", out["inst_offset"][0], as_array(ex["inst_offset"]))
        n = int(as_array(ex["inst_offset"])[-1])
        G().assert_equal("src_slot", out["src_slot"][0][:n], as_array(ex["src_slot"])[:n])
    orc = G().oracle_run(R, E, S, ids, max_iters=ex["max_iters"])
    G().compare(R, E, S, out, orc)


# ------------------------------------------------------------------ tiny workload
def _tiny_inputs(layers):
    w = W.WORKLOADS["tiny"]
    ids = np.stack([W.topk_ids(w, l, 0).numpy() for l in layers])
    hid = np.stack([W.bf16_bits(W.hidden(w.T, w.Hd, w.seed(l, 0))) for l in layers])
    return w, ids, hid


def test_tiny_workload_batched():
    w, ids, hid = _tiny_inputs(range(W.WORKLOADS["tiny"].layers))
    dom = G().dom_of(w.R, w.E, w.S, w.k)
    out = G().gpu_run(dom, ids, hid)
    orc = G().oracle_run(w.R, w.E, w.S, ids, hid)
    G().compare(w.R, w.E, w.S, out, orc)
    assert (out["dev_status"] == 0).all()
    assert (out["y"] == hid[:, :, None, :]).all()          # round trip is the identity


@pytest.mark.parametrize("layer", range(4))
def test_tiny_workload_per_layer(layer):
    w, ids, hid = _tiny_inputs([layer])
    dom = G().dom_of(w.R, w.E, w.S, w.k)
    out = G().gpu_run(dom, ids, hid)
    G().compare(w.R, w.E, w.S, out, G().oracle_run(w.R, w.E, w.S, ids, hid))


# ------------------------------------------------------------------ sweep of shapes and edge cases
CASES = [
    # name,                R,  H, S, k,  T,     n_inst, Hd,  kind
    ("empty_T",            8,  4, 1, 4,  0,     2,      16,  "zipf"),
    ("k1",                 8,  4, 1, 1,  777,   1,      16,  "zipf"),
    ("one_expert",         8,  1, 1, 1,  5000,  1,      8,   "one"),
    ("uniform",            16, 2, 2, 4,  4096,  1,      8,   "uniform"),
    ("no_spares",          8,  4, 0, 4,  3000,  2,      8,   "zipf"),
    ("H1",                 32, 1, 1, 2,  2048,  1,      8,   "zipf"),
    ("R64_mask_width",     64, 2, 1, 8,  8192,  1,      64,  "zipf"),
    ("R64_S4",             64, 4, 4, 8,  4096,  2,      8,   "zipf"),
    ("ragged_T",           8,  4, 1, 4,  1001,  3,      24,  "zipf"),
    ("T_below_R",          8,  2, 1, 3,  5,     1,      8,   "zipf"),
    ("invalid_and_dups",   8,  4, 1, 4,  2000,  2,      8,   "bad"),
    ("many_chunks",        4,  4, 2, 8,  40000, 1,      8,   "zipf"),
    ("max_E_and_k",        64, 16, 16, 32, 1024, 1,     8,   "zipf"),
    ("many_instances",     8,  4, 1, 4,  512,   33,     8,   "zipf"),
    ("hidden_264",         8,  4, 1, 4,  300,   1,      264, "zipf"),
    ("hidden_4096",        16, 4, 1, 8,  512,   1,      4096, "zipf"),
    # rows moved by TMA bulk copies: exactly the 1 KiB threshold, three
    # segments of 8192 + 8192 + 16 bytes, several instances with invalid ids
    ("bulk_row_1KiB",      8,  4, 1, 4,  333,   2,      512,  "zipf"),
    ("bulk_row_3_segments", 4, 2, 1, 3,  97,    1,      8200, "zipf"),
    ("bulk_rows_bad_ids",  8,  4, 2, 4,  250,   3,      1024, "bad"),
    # reroute kernels: E = 256 (ids held as bytes cannot mark an invalid id),
    # E in (256, 512] (the mask kernel, one wide block per rank), a rank in
    # several rounds of lane runs, many blocks (short runs, four warps) with
    # invalid ids, and with ranks that do not start on a 16-byte boundary
    ("E256_bad_ids",       8,  32, 0, 8, 3001,  2,      8,   "bad"),
    ("E320_mask_kernel",   16, 20, 2, 8, 3000,  1,      8,   "zipf"),
    ("E512_one_layer",     16, 32, 0, 8, 3000,  1,      8,   "zipf"),   # wide blocks do not fit
    ("runs_many_rounds",   2,  8, 1, 8,  20000, 1,      8,   "zipf"),
    ("runs_batched_bad",   8,  4, 1, 4,  3001,  40,     8,   "bad"),
    ("runs_batched_unaligned", 8, 4, 1, 3, 1001, 40,    8,   "zipf"),
    ("R1_single_rank",     1,  4, 1, 2,  500,   1,      8,   "zipf"),   # no other rank: no move
    ("R33_second_rank_per_lane", 33, 2, 1, 4, 3000, 1,  8,   "zipf"),   # ragged last rank
    ("R40_glm_like",       40, 4, 1, 8,  4000,  1,      8,   "zipf"),
    ("W32_max_instances",  8,  1, 31, 4, 3000,  1,      8,   "zipf"),   # H + S = 32
    # the quad reroute kernel (k a multiple of 4, 296 or more (instance, rank)
    # units): repeated ids in a lane's four slots, a ragged T, empty source
    # ranks, the largest E and k, a ragged last block of ranks (R = 36), every
    # slot on one expert (every step by slot, replica boundaries crossed all
    # the time)
    ("quad_dups_R64",      64, 2, 1, 8,  2000,  5,      8,   "bad"),
    ("quad_ragged_T",      16, 4, 2, 4,  3333,  19,     8,   "zipf"),
    ("quad_T_below_R",     64, 2, 1, 4,  50,    5,      8,   "zipf"),
    ("quad_max_E_and_k",   64, 16, 16, 32, 257, 5,      8,   "zipf"),
    ("quad_R36_uniform",   36, 4, 1, 4,  4000,  9,      8,   "uniform"),
    ("quad_one_expert",    8,  4, 2, 4,  5000,  40,     8,   "one"),
    # the quad kernel with many slots per rank and with E in (256, 512]
    ("quad_long_ranks",    8,  4, 1, 8,  20000, 37,     8,   "bad"),
    # one-layer launches with a rank split over a cluster of 4 or 2 blocks
    ("cluster4_ragged",    8,  4, 1, 8,  30001, 1,      8,   "bad"),
    ("cluster2_ragged",    16, 4, 2, 4,  50001, 1,      8,   "zipf"),
    ("quad_E320",          16, 20, 2, 8, 3000,  19,     8,   "bad"),
    # the quad kernel over many instances (several waves of blocks): even R,
    # an odd R (the last block of each instance holds one source rank),
    # invalid ids
    ("quad_tail_R64",      64, 2, 1, 8,  1500,  40,     8,   "bad"),
    ("quad_tail_R36",      36, 4, 1, 4,  999,   70,     8,   "zipf"),
    ("quad_tail_R37_odd",  37, 2, 1, 4,  500,   70,     8,   "zipf"),
]


def _make_ids(R, E, k, T, n_inst, kind, seed):
    rng = np.random.default_rng(seed)
    out = []
    for g in range(n_inst):
        if kind == "one":
            ids = np.zeros((T, k), np.int32)
        elif kind == "uniform":
            ids = (np.arange(T * k, dtype=np.int32) % E).reshape(T, k)
        else:
            p = 1.0 / (rng.permutation(E) + 1.0) ** 1.1
            ids = W.gumbel_topk(p / p.sum(), T, k, seed * 100 + g).numpy()
            if kind == "bad" and T:
                ids[rng.integers(0, T, 5), 0] = E + 7
                ids[rng.integers(0, T, 5), -1] = -3
                if k > 1:
                    ids[rng.integers(0, T, 5), 1] = ids[rng.integers(0, T, 5), 0] % E  # duplicates
                if k > 2:
                    t2 = rng.integers(0, T, 5)
                    ids[t2, 1] = ids[t2, 2]                # the same expert twice in one token
        out.append(ids)
    return np.stack(out) if n_inst else np.zeros((0, T, k), np.int32)


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_shape_sweep(case):
    name, R, H, S, k, T, n_inst, Hd, kind = case
    E = R * H
    ids = _make_ids(R, E, k, T, n_inst, kind, seed=len(name) * 7919 + T)
    rng = np.random.default_rng(T + Hd)
    hid = rng.integers(0, 1 << 16, size=(n_inst, T, Hd), dtype=np.uint16)
    dom = G().dom_of(R, E, S, k)
    out = G().gpu_run(dom, ids, hid)
    orc = G().oracle_run(R, E, S, ids, hid)
    G().compare(R, E, S, out, orc)
    expect_flag = 1 if any(n > 0 for n in orc["n_bad"]) else 0
    assert int(out["dev_status"][0]) == expect_flag
    for g in range(n_inst):
        pl = {key: out[key][g] for key in ("quota", "slot_expert", "rank_load", "inst_ptr",
                                          "inst_id", "inst_cum")}
        pl.update(n_iter=int(out["n_iter"][g]), status=int(out["inst_status"][g]))
        check_plan(out["counts"][g], R, E, S, pl)
        check_reroute(ids[g], R, E, S, pl, out["dst_row"][g], out["src_slot"][g],
                      out["inst_offset"][g])


def test_iteration_cap_matches_oracle():
    R, H, S, k, T = 16, 4, 2, 8, 20000
    ids = _make_ids(R, R * H, k, T, 3, "zipf", 99)
    dom = G().dom_of(R, R * H, S, k)
    full = G().oracle_run(R, R * H, S, ids)
    for cap in (1, 2, max(1, min(full["n_iter"]) // 2)):
        out = G().gpu_run(dom, ids, max_iters=cap)
        orc = G().oracle_run(R, R * H, S, ids, max_iters=cap)
        G().compare(R, R * H, S, out, orc)
        assert (out["inst_status"] == 2).any()


def test_plan_rejects_bad_counts():
    dom = G().dom_of(4, 8, 1, 2)
    b = G().guarded_buffers(dom, 16, 2)
    b.counts.copy_(torch.tensor([[5, -1, 0, 0, 0, 0, 0, 0],
                                 [2 ** 30, 2 ** 30, 0, 0, 0, 0, 0, 0]], dtype=torch.int32))
    b.plan()
    st = b.inst_status.cpu().numpy()
    assert st.tolist() == [U.EP_ERR_INVAL, U.EP_ERR_INVAL]
    assert (b.n_iter.cpu().numpy() == 0).all()
    b.guard.check()


def test_device_status_flags():
    R, E, S, k, T, Hd = 4, 8, 1, 2, 64, 8
    dom = G().dom_of(R, E, S, k)
    ids = _make_ids(R, E, k, T, 1, "zipf", 3)
    ids[0, 3, 1] = 99                                      # bad id
    out = G().gpu_run(dom, ids)
    assert int(out["dev_status"][0]) & U.EP_DEV_BAD_ID
    # a plan whose quotas do not cover the ids: overflowing slots get no row
    b = G().guarded_buffers(dom, T, 1)
    dids = torch.from_numpy(ids).cuda()
    b.count(dids)
    b.plan()
    b.quota.zero_()
    b.inst_cum.zero_()
    b.dev_status.zero_()
    b.reroute(dids)
    assert int(b.dev_status.item()) & U.EP_DEV_QUOTA_OVERFLOW
    assert (b.dst_row.cpu().numpy() == -1).all()
    # a dst_row past the last row: permute skips it, unpermute zeroes it
    hidden = torch.ones((T, Hd), dtype=torch.bfloat16, device="cuda")
    dst = torch.arange(T * k, dtype=torch.int32, device="cuda")
    dst[5] = T * k + 3
    out_rows = b.guard.alloc("out_rows", (T * k, Hd), torch.bfloat16, 0)
    st = b.guard.alloc("st", (1,), torch.int32, 0)
    U.ep_permute(hidden, k, dst, out_rows, st)
    assert int(st.item()) & U.EP_DEV_ROW_RANGE
    assert float(out_rows[5].float().abs().sum()) == 0.0
    y = b.guard.alloc("y", (T, k, Hd), torch.bfloat16, 7.0)
    st.zero_()
    U.ep_unpermute(out_rows, T, k, dst, y, st)
    assert int(st.item()) & U.EP_DEV_ROW_RANGE
    assert float(y.reshape(T * k, Hd)[5].float().abs().sum()) == 0.0
    b.guard.check()


@pytest.mark.parametrize("case", [(8, 4, 1, 4, 4096, 2), (64, 2, 1, 8, 131072, 1),
                                  (64, 2, 1, 8, 4096, 5), (64, 2, 1, 8, 2048, 40)])
def test_reroute_flags_counts_of_other_ids(case):
    # counts_src taken from other ids (another layer's buffer): every block
    # compares what it ranked with its own counts_src row and flags the
    # difference; the same call with the right counts_src raises nothing
    R, H, S, k, T, n_inst = case
    E = R * H
    dom = G().dom_of(R, E, S, k)
    ids_a = torch.from_numpy(_make_ids(R, E, k, T, n_inst, "zipf", 41)).cuda()
    ids_b = torch.from_numpy(_make_ids(R, E, k, T, n_inst, "zipf", 42)).cuda()
    b = G().guarded_buffers(dom, T, n_inst, src_slot=True)
    b.count(ids_a)
    b.plan()
    b.reroute(ids_a)
    torch.cuda.synchronize()
    assert int(b.dev_status.item()) == 0
    stale = b.counts_src.clone()
    b.count(ids_b)
    b.plan()
    b.counts_src.copy_(stale)              # the other ids' per-source-rank counts
    b.reroute(ids_b)
    torch.cuda.synchronize()
    assert int(b.dev_status.item()) & U.EP_DEV_COUNTS_MISMATCH
    # only the block of source rank 0 of an instance starts at prefix zero; a
    # counts_src differing in one entry still raises the flag
    for g in sorted({0, n_inst - 1}):     # the first and the last instance of the batch
        b.dev_status.zero_()
        b.count(ids_b)
        b.reroute(ids_b)
        torch.cuda.synchronize()
        assert int(b.dev_status.item()) == 0
        b.counts_src[g, R - 1, int(ids_b[g, -1, 0].item())] += 1
        b.reroute(ids_b)
        torch.cuda.synchronize()
        assert int(b.dev_status.item()) & U.EP_DEV_COUNTS_MISMATCH
    b.guard.check()


@pytest.mark.parametrize("case", [(64, 2, 1, 8, 8192, 5), (16, 4, 2, 4, 12000, 20),
                                  (64, 2, 1, 8, 4096, 40)])
def test_quad_reroute_past_the_quotas(case):
    # a plan whose last replicas hold less than their experts' counts (every
    # source rank walked by two warps, the backward one starting above the
    # quotas): the overflowing slots get no row and the flag, every other row
    # is the oracle's, bit for bit
    R, H, S, k, T, n_inst = case
    E = R * H
    dom = G().dom_of(R, E, S, k)
    ids_np = _make_ids(R, E, k, T, n_inst, "zipf", 77)
    ids = torch.from_numpy(ids_np).cuda()
    b = G().guarded_buffers(dom, T, n_inst, src_slot=True)
    b.count(ids)
    b.plan()
    quota = b.quota.cpu().numpy().copy()
    ptr = b.inst_ptr.cpu().numpy()
    iid = b.inst_id.cpu().numpy()
    cum = b.inst_cum.cpu().numpy().copy()
    short = 0
    for g in range(n_inst):
        for e in range(E):
            lo, hi = int(ptr[g, e]), int(ptr[g, e + 1])
            if hi - lo >= 2:                  # trim the last replica of a replicated expert
                p_last = int(iid[g, hi - 1])
                cut = (int(quota[g, p_last]) + 2) // 3
                quota[g, p_last] -= cut
                short += cut
                run = 0
                for m in range(lo, hi):
                    run += int(quota[g, int(iid[g, m])])
                    cum[g, m] = run
    assert short > 0
    b.quota.copy_(torch.from_numpy(quota))
    b.inst_cum.copy_(torch.from_numpy(cum))
    b.dev_status.zero_()
    b.reroute(ids)
    torch.cuda.synchronize()
    assert int(b.dev_status.item()) & U.EP_DEV_QUOTA_OVERFLOW
    dst = b.dst_row.cpu().numpy()
    src = b.src_slot.cpu().numpy()
    off = b.inst_offset.cpu().numpy()
    n_none = 0
    for g in range(n_inst):
        pl = dict(quota=quota[g], inst_ptr=ptr[g], inst_id=iid[g], inst_cum=cum[g])
        d_o, s_o, o_o = oracle.reroute(ids_np[g], R, E, S, pl)
        assert np.array_equal(dst[g], d_o), g
        assert np.array_equal(src[g], s_o), g
        assert np.array_equal(off[g], o_o), g
        n_none += int((d_o < 0).sum())
    assert n_none == short
    b.guard.check()


def test_workspace_reused_across_calls():
    w, ids, _ = _tiny_inputs([0, 1])
    dom = G().dom_of(w.R, w.E, w.S, w.k)
    b = G().guarded_buffers(dom, w.T, 2)
    d = torch.from_numpy(ids).cuda()
    outs = []
    for _ in range(3):
        b.count(d)
        outs.append((b.counts.cpu().numpy().copy(), b.counts_src.cpu().numpy().copy()))
        assert (b.workspace.cpu().numpy()[:2] == 0).all()          # the two instance tickets
    for c, cs in outs[1:]:
        assert (c == outs[0][0]).all() and (cs == outs[0][1]).all()
    b.guard.check()


def test_permute_preserves_bit_patterns():
    # NaN payloads, infinities and -0 pass through unchanged
    T, k, Hd = 7, 3, 16
    pat = np.array([0x7FC1, 0xFF80, 0x8000, 0x0001, 0x7F80, 0xFFFF, 0x1234, 0x8001], np.uint16)
    hid = np.tile(pat, (T, Hd // 8)).reshape(T, Hd)
    hid[:, 0] = np.arange(T, dtype=np.uint16)
    ids = np.stack([np.arange(T * k, dtype=np.int32).reshape(T, k) % 4])
    dom = G().dom_of(2, 4, 1, k)
    out = G().gpu_run(dom, ids, hid[None])
    G().compare(2, 4, 1, out, G().oracle_run(2, 4, 1, ids, hid[None]))


# ------------------------------------------------------------------ full-size workloads
ROW_CHUNK = 1 << 16


def check_all_rows(hid_d, grouped_d, y_d, src_slot_oracle, n_rows, k):
    """Every permuted row equals the hidden row of the token the oracle's
    src_slot names; every unpermuted slot equals its own token's row (the
    oracle's unpermute of its permute).  On the device, in chunks of rows."""
    src = torch.from_numpy(np.ascontiguousarray(src_slot_oracle[:n_rows])).cuda()
    for r0 in range(0, n_rows, ROW_CHUNK):
        r1 = min(n_rows, r0 + ROW_CHUNK)
        want = hid_d.index_select(0, (src[r0:r1] // k).long())
        got = grouped_d[r0:r1]
        if not torch.equal(got.view(torch.int16), want.view(torch.int16)):
            bad = (got.view(torch.int16) != want.view(torch.int16)).any(1).nonzero()[0].item()
            raise AssertionError(f"grouped row {r0 + bad} differs from the oracle's")
    if y_d is None:
        return
    N = y_d.shape[0] * y_d.shape[1] if y_d.dim() == 3 else y_d.shape[0]
    y2 = y_d.reshape(N, -1)
    for s0 in range(0, N, ROW_CHUNK):
        s1 = min(N, s0 + ROW_CHUNK)
        tok = torch.arange(s0, s1, device="cuda") // k
        if not torch.equal(y2[s0:s1].view(torch.int16), hid_d.index_select(0, tok).view(torch.int16)):
            raise AssertionError(f"unpermuted slots {s0}..{s1} differ from the oracle's")


def _full_size_layer(name, layer, microbatch):
    w = W.WORKLOADS[name]
    ids_d = W.topk_ids(w, layer, microbatch, device="cuda")
    hid_d = W.hidden(w.T, w.Hd, w.seed(layer, microbatch), device="cuda")
    ids = ids_d.cpu().numpy()[None]
    dom = U.Domain(w.R, w.E, w.S, w.k)
    b = G().guarded_buffers(dom, w.T, 1, Hd=w.Hd, src_slot=True)
    b.balance(ids_d[None], hid_d[None])                    # the per-layer launches the bench times
    y = b.guard.alloc("y", (1, w.T, w.k, w.Hd), torch.bfloat16)
    U.ep_unpermute(b.grouped, w.T, w.k, b.dst_row, y, b.dev_status)
    b.guard.check()
    orc = G().oracle_run(w.R, w.E, w.S, ids)
    out = {key: getattr(b, key).cpu().numpy() for key in
           ("counts", "counts_src", "quota", "slot_expert", "rank_load", "inst_ptr", "inst_id",
            "inst_cum", "n_iter", "inst_status", "dst_row", "inst_offset", "workspace",
            "src_slot", "dev_status")}
    G().compare(w.R, w.E, w.S, out, orc, check_rows=False)
    assert int(out["dev_status"][0]) == 0
    n_rows = int(orc["inst_offset"][0][-1])
    assert n_rows == w.N
    check_all_rows(hid_d, b.grouped[0], y[0], orc["src_slot"][0], n_rows, w.k)
    return out


@pytest.mark.parametrize("name,layer", [("qwen3-235b", 0), ("qwen3-235b", 93),
                                        ("deepseek-v3", 7), ("glm-4.5", 3)])
def test_full_size_layer(name, layer):
    out = _full_size_layer(name, layer, 0)
    w = W.WORKLOADS[name]
    assert out["rank_load"].max() <= out["counts"][0].reshape(w.R, -1).sum(1).max()


def test_full_size_batched_count_and_reroute():
    # all 94 layers of one Qwen3-235B-like microbatch in one launch per step
    w = W.WORKLOADS["qwen3-235b"]
    ids_d = torch.stack([W.topk_ids(w, l, 1, device="cuda") for l in range(w.layers)])
    ids = ids_d.cpu().numpy()
    out = G().gpu_run(U.Domain(w.R, w.E, w.S, w.k), ids, src_slot=False)
    orc = G().oracle_run(w.R, w.E, w.S, ids)
    G().compare(w.R, w.E, w.S, out, orc, check_rows=False)


def test_full_size_layer_without_src_slot():
    # one Qwen3-235B-like layer per launch, as the benchmark's step makes it
    # (no src_slot output)
    w = W.WORKLOADS["qwen3-235b"]
    ids = W.topk_ids(w, 7, 2, device="cuda").cpu().numpy()[None]
    out = G().gpu_run(U.Domain(w.R, w.E, w.S, w.k), ids, src_slot=False)
    orc = G().oracle_run(w.R, w.E, w.S, ids)
    G().compare(w.R, w.E, w.S, out, orc, check_rows=False)


# one point per (R, S) pair of the stress grid, its tokens per rank and Zipf
# skew cycling through the grid's values (the largest, 8192 tokens per rank at
# R = 64, included)
STRESS_POINTS = [(8, 1, 512, 0.6), (8, 2, 1024, 1.0), (8, 4, 8192, 1.6),
                 (16, 1, 2048, 1.0), (16, 2, 4096, 1.6), (16, 4, 512, 0.6),
                 (32, 1, 1024, 1.6), (32, 2, 2048, 1.0), (32, 4, 4096, 0.6),
                 (64, 1, 2048, 1.6), (64, 2, 1024, 0.6), (64, 4, 8192, 1.0)]


@pytest.mark.parametrize("R,S,tpr,s", STRESS_POINTS,
                         ids=[f"R{r}_S{s_}_T{t}_z{z}" for r, s_, t, z in STRESS_POINTS])
def test_stress_points(R, S, tpr, s):
    # two layers batched through the separate calls, every index output
    # against the oracle; then the first layer through the ep_balance and
    # ep_permute launches the benchmark makes, every row checked
    w = W.stress(R, S, tpr, s)
    ids_d = torch.stack([W.topk_ids(w, l, 0, device="cuda") for l in range(2)])
    ids = ids_d.cpu().numpy()
    dom = U.Domain(w.R, w.E, w.S, w.k)
    out = G().gpu_run(dom, ids, src_slot=True)
    orc = G().oracle_run(w.R, w.E, w.S, ids)
    G().compare(w.R, w.E, w.S, out, orc, check_rows=False)
    assert int(out["dev_status"][0]) == 0
    hid_d = W.hidden(w.T, w.Hd, w.seed(0, 0), device="cuda")
    b = G().guarded_buffers(dom, w.T, 1, Hd=w.Hd)
    b.balance_fused(ids_d[:1])
    b.permute(hid_d[None])
    b.guard.check()
    assert np.array_equal(b.dst_row[0].cpu().numpy(), orc["dst_row"][0])
    check_all_rows(hid_d, b.grouped[0], None, orc["src_slot"][0], int(orc["inst_offset"][0][-1]),
                   w.k)
    del b, hid_d
    torch.cuda.empty_cache()
