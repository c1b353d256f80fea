"""Plan-quality metrics and the history-based placement baseline (host side, not timed).

* ``imbalance``: max / mean rank load.  The UltraEP article (results
  paragraph) and the rack-scale summary ("Reported results": the most
  overloaded rank at 4.01x the average before, 1.04x after) quote imbalance
  this way; the EPLB tutorial's "balancedness" (mean / max, measured-speedup
  section) is its inverse.
* ``lower_bound``: no plan with at most R*S replica slots can beat
  max(ceil(total / R), LB_home), where LB_home is the smallest possible maximum
  over ranks of the home load of experts that get no replica (an expert with no
  replica cannot leave its home rank).
* ``eplb_global``: an EPLB-style Global placement built from HISTORICAL loads
  (EPLB tutorial: "Global: single-stage global packing" and "how are redundant
  experts allocated": extra slots go to heavy experts, every physical expert
  is packed onto all GPUs at once, hot and cold experts share a GPU).  It is
  written from that prose only; the EPLB source is not available, so its tie
  rules are this module's own.  Evaluated on the CURRENT microbatch's counts,
  an expert's tokens are split evenly over its copies (the tutorial: dispatch
  picks a copy "by load or by hash").
"""
import numpy as np


def imbalance(rank_load) -> float:
    rank_load = np.asarray(rank_load, dtype=np.float64)
    mean = rank_load.mean()
    return float(rank_load.max() / mean) if mean > 0 else 1.0


def home_load(counts, R: int) -> np.ndarray:
    counts = np.asarray(counts, dtype=np.int64)
    return counts.reshape(R, -1).sum(axis=1)


def lower_bound(counts, R: int, S: int) -> int:
    """max(ceil(total/R), LB_home) for one instance.

    LB_home: take away R*S experts, each time the largest remaining expert of
    the currently heaviest rank.  Greedy is exact here: while the maximum is
    above the optimum, the heaviest rank needs one more removal in every
    optimal choice, and removing a rank's largest expert is its best single
    removal.
    """
    counts = np.asarray(counts, dtype=np.int64)
    total = int(counts.sum())
    per_rank = [sorted(row.tolist(), reverse=True) for row in counts.reshape(R, -1)]
    removed = [0] * R
    resid = [sum(r) for r in per_rank]
    for _ in range(R * S):
        r = int(np.argmax(resid))
        if resid[r] == 0:
            break
        resid[r] -= per_rank[r][removed[r]]
        removed[r] += 1
    return max(-(-total // R), max(resid))


def eplb_global(hist_load, R: int, per_rank: int) -> np.ndarray:
    """phy2log [R, per_rank] from historical per-expert loads (float).

    R*per_rank physical slots hold the E logical experts and R*per_rank - E
    extra copies (per_rank = H + S in the UltraEP domain).
    Replication: each extra copy goes to the expert with the largest
    load-per-copy (ties: lowest id), at most R copies of one expert.
    Packing: all R*per_rank copies, heaviest load-per-copy first (ties: lowest
    id), each onto the least-loaded rank that has room and no copy of that
    expert yet (ties: lowest rank).
    """
    hist_load = np.asarray(hist_load, dtype=np.float64)
    E = hist_load.shape[0]
    n_extra = R * per_rank - E
    if n_extra < 0:
        raise ValueError("fewer physical slots than logical experts")
    n_copies = np.ones(E, dtype=np.int64)
    for _ in range(n_extra):
        per = np.where(n_copies < R, hist_load / n_copies, -np.inf)
        e = int(np.argmax(per))
        if per[e] == -np.inf:
            break
        n_copies[e] += 1
    items = []
    for e in range(E):
        items += [(-(hist_load[e] / n_copies[e]), e)] * int(n_copies[e])
    items.sort()
    cap = per_rank
    placed = [[] for _ in range(R)]
    load = np.zeros(R)
    for neg_w, e in items:
        best = -1
        for r in range(R):
            if len(placed[r]) >= cap or e in placed[r]:
                continue
            if best < 0 or load[r] < load[best]:
                best = r
        if best < 0:       # no rank without a copy of e has room: any rank with room
            best = min((r for r in range(R) if len(placed[r]) < cap), key=lambda r: load[r])
        placed[best].append(e)
        load[best] += -neg_w
    phy2log = np.full((R, cap), -1, dtype=np.int64)
    for r in range(R):
        phy2log[r, :len(placed[r])] = placed[r]
    return phy2log


def eval_placement(phy2log, counts) -> np.ndarray:
    """Rank loads when each expert's count is split evenly over its copies
    (remainder to the copies with the lowest physical index)."""
    phy2log = np.asarray(phy2log)
    counts = np.asarray(counts, dtype=np.int64)
    R, W = phy2log.shape
    flat = phy2log.reshape(-1)
    load = np.zeros(R, dtype=np.int64)
    for e in range(counts.shape[0]):
        where = np.nonzero(flat == e)[0]
        if where.size == 0:
            continue
        share, rem = divmod(int(counts[e]), where.size)
        for n, p in enumerate(where):
            load[p // W] += share + (1 if n < rem else 0)
    return load


def summarize(values):
    v = np.asarray(values, dtype=np.float64)
    return dict(median=float(np.median(v)), p95=float(np.percentile(v, 95)), max=float(v.max()))
