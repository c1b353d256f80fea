"""Properties every correct plan / reroute / permute result has.

Used to pin the oracle (against invariants the problem statement fixes) and,
in the GPU tests, as a second check of the library's outputs.  Nothing here
re-runs the rule: each check looks at a finished result.
"""
import numpy as np


def _inst_layout(R, E, S):
    H = E // R
    W = H + S
    return H, W, R * W


def instance_expert(E, R, S, slot_expert):
    """expert held by every physical instance p (-1 for an empty spare slot)."""
    H, W, P = _inst_layout(R, E, S)
    slot_expert = np.asarray(slot_expert).reshape(R, S)
    ex = np.full(P, -1, dtype=np.int64)
    for r in range(R):
        for j in range(W):
            ex[r * W + j] = r * H + j if j < H else slot_expert[r, j - H]
    return ex


def check_plan(counts, R, E, S, pl, max_iters=1 << 16):
    counts = np.asarray(counts, dtype=np.int64)
    H, W, P = _inst_layout(R, E, S)
    quota = np.asarray(pl["quota"], dtype=np.int64)
    slot = np.asarray(pl["slot_expert"], dtype=np.int64).reshape(R, S)
    load = np.asarray(pl["rank_load"], dtype=np.int64)
    ptr = np.asarray(pl["inst_ptr"], dtype=np.int64)
    iid = np.asarray(pl["inst_id"], dtype=np.int64)
    cum = np.asarray(pl["inst_cum"], dtype=np.int64)
    assert quota.shape == (P,)
    assert (quota >= 0).all(), "negative quota"
    # spare slots: filled lowest index first, expert ids valid, no copy on the
    # expert's home rank, at most one copy of an expert per rank
    for r in range(R):
        filled = slot[r] >= 0
        if S > 1:
            assert not np.any(~filled[:-1] & filled[1:]), "a free slot below a filled one"
        es = slot[r][filled]
        assert ((es >= 0) & (es < E)).all()
        assert len(set(es.tolist())) == len(es), "two copies of one expert on a rank"
        assert not any(e // H == r for e in es), "replica on its home rank"
    ex = instance_expert(E, R, S, slot)
    # an empty slot carries no load
    assert (quota[ex < 0] == 0).all(), "load on an empty slot"
    # per-expert conservation
    per_e = np.zeros(E, dtype=np.int64)
    np.add.at(per_e, ex[ex >= 0], quota[ex >= 0])
    assert (per_e == counts).all(), "quotas of an expert do not sum to its count"
    # rank loads
    assert (load == quota.reshape(R, W).sum(axis=1)).all(), "rank_load != sum of quotas"
    assert load.sum() == counts.sum()
    home = counts.reshape(R, H).sum(axis=1)
    assert load.max() <= home.max(), "max load grew"
    # CSR: home first, then the other holders by ascending p, inclusive cums
    assert ptr[0] == 0 and (np.diff(ptr) >= 1).all()
    assert ptr[E] == E + int((slot >= 0).sum())
    for e in range(E):
        lst = iid[ptr[e]:ptr[e + 1]]
        home_p = (e // H) * W + e % H
        assert lst[0] == home_p, "home instance not first"
        others = np.nonzero(ex == e)[0]
        others = others[others != home_p]
        assert (lst[1:] == others).all(), "replicas not listed by ascending p"
        assert (cum[ptr[e]:ptr[e + 1]] == np.cumsum(quota[lst])).all(), "bad cumulative quota"
    assert 0 <= pl["n_iter"] <= max_iters
    assert pl["status"] in (0, 2)
    if pl["status"] == 2:
        assert pl["n_iter"] == max_iters
    # each move lowers sum L^2 by at least 2, so the move count is bounded
    assert 2 * pl["n_iter"] <= int((home ** 2).sum() - (load ** 2).sum())


def check_stopped(counts, R, E, S, pl):
    """A plan that ended with status 0 satisfies the rule's stopping condition."""
    if pl["status"] != 0:
        return
    H, W, P = _inst_layout(R, E, S)
    quota = np.asarray(pl["quota"], dtype=np.int64)
    slot = np.asarray(pl["slot_expert"], dtype=np.int64).reshape(R, S)
    load = np.asarray(pl["rank_load"], dtype=np.int64)
    ex = instance_expert(E, R, S, slot)
    hot = int(np.argmax(load))                       # argmax returns the lowest index
    on_hot = [(-int(quota[p]), int(ex[p]), p) for p in range(hot * W, hot * W + W) if ex[p] >= 0]
    negq, e, p = min(on_hot)                        # largest quota, then lowest expert id
    elig = [c for c in range(R) if c != hot and (np.any(ex[c * W:(c + 1) * W] == e)
                                                 or np.any(slot[c] < 0))]
    if not elig:
        return
    cold = min(elig, key=lambda c: (load[c], c))
    assert min(-negq, (load[hot] - load[cold]) // 2) == 0, "plan stopped while a move was possible"


def check_reroute(ids, R, E, S, pl, dst_row, src_slot, inst_offset):
    """Rows form instance blocks in p order, each block holds exactly its quota of
    its own expert's slots in ascending slot order, and every expert fills its
    instances in list order (the quota prefix rule)."""
    ids = np.asarray(ids, dtype=np.int64).reshape(-1)
    N = ids.shape[0]
    H, W, P = _inst_layout(R, E, S)
    quota = np.asarray(pl["quota"], dtype=np.int64)
    ptr = np.asarray(pl["inst_ptr"], dtype=np.int64)
    iid = np.asarray(pl["inst_id"], dtype=np.int64)
    dst_row = np.asarray(dst_row, dtype=np.int64)
    inst_offset = np.asarray(inst_offset, dtype=np.int64)
    assert (inst_offset == np.concatenate([[0], np.cumsum(quota)])).all()
    valid = (ids >= 0) & (ids < E)
    assert (dst_row[~valid] == -1).all()
    n_rows = int(inst_offset[P])
    assert valid.sum() == n_rows
    rows = dst_row[valid]
    assert (np.sort(rows) == np.arange(n_rows)).all(), "rows are not a bijection"
    if src_slot is not None:
        src_slot = np.asarray(src_slot, dtype=np.int64)
        assert (src_slot[rows] == np.nonzero(valid)[0]).all(), "src_slot is not the inverse"
    ex = instance_expert(E, R, S, pl["slot_expert"])
    p_of = np.searchsorted(inst_offset, dst_row, side="right") - 1
    assert (ex[p_of[valid]] == ids[valid]).all(), "slot sent to an instance of another expert"
    # within a block, rows follow slot order (stable)
    order = np.argsort(np.where(valid, dst_row, n_rows + np.arange(N)), kind="stable")[:n_rows]
    for p in range(P):
        blk = order[inst_offset[p]:inst_offset[p + 1]]
        assert (np.diff(blk) > 0).all(), "rows of an instance not in slot order"
    # prefix rule: along each expert's slots, the list position never decreases
    pos_in_list = {int(iid[m]): m - ptr[e] for e in range(E) for m in range(ptr[e], ptr[e + 1])}
    for e in range(E):
        slots = np.nonzero(ids == e)[0]
        pos = np.array([pos_in_list[int(p_of[i])] for i in slots], dtype=np.int64)
        assert (np.diff(pos) >= 0).all(), "expert's slots do not fill its list in order"
