"""Host-side plan-quality helpers: imbalance, lower bound, EPLB-style baseline."""
import numpy as np

from moe_expert_load_id_b300 import quality as Q
from golden_io import read_sections, as_array

EPLB = read_sections("eplb_example.txt")[""]


def test_imbalance_definition():
    # the rack-scale summary quotes the hottest rank as a multiple of the average
    assert Q.imbalance([4, 1, 1, 2]) == 2.0
    assert Q.imbalance([3, 3, 3]) == 1.0
    assert Q.imbalance([0, 0]) == 1.0


def test_printed_eplb_example_structure():
    # the fixture itself is what the EPLB tutorial says it is
    for key in ("layer0", "layer1"):
        row = as_array(EPLB[key])
        assert row.size == EPLB["num_physical"] == EPLB["num_gpus"] * EPLB["per_gpu"]
        assert set(row.tolist()) == set(range(EPLB["num_logical"]))
    l0 = as_array(EPLB["layer0"])
    dup = sorted(e for e in range(12) if (l0 == e).sum() == 2)
    assert dup == sorted(as_array(EPLB["layer0_duplicated"]).tolist())
    assert not (l0 == as_array(EPLB["layer1"])).all()          # layers differ


def test_eplb_global_reproduces_the_example_structure():
    # 12 logical experts, 8 GPUs x 2 slots: the four heaviest historical experts
    # get the four extra copies, every logical expert keeps at least one copy,
    # no GPU holds two copies of one expert
    hist = np.ones(12)
    for e, w in zip(as_array(EPLB["layer0_duplicated"]), (9.0, 8.0, 7.0, 6.0)):
        hist[e] = w
    phy2log = Q.eplb_global(hist, 8, 2)
    assert phy2log.shape == (8, 2)
    flat = phy2log.reshape(-1)
    assert set(flat.tolist()) == set(range(12))
    dup = sorted(e for e in range(12) if (flat == e).sum() == 2)
    assert dup == sorted(as_array(EPLB["layer0_duplicated"]).tolist())
    for r in range(8):
        assert phy2log[r, 0] != phy2log[r, 1]


def test_eplb_global_balances_its_own_history():
    rng = np.random.default_rng(3)
    hist = rng.gamma(0.5, 1.0, size=128) * 1000
    phy2log = Q.eplb_global(hist, 64, 3)
    load = Q.eval_placement(phy2log, np.round(hist).astype(np.int64))
    home = Q.home_load(np.round(hist).astype(np.int64), 64)
    assert Q.imbalance(load) < Q.imbalance(home)


def test_eval_placement_splits_evenly():
    phy2log = np.array([[0, 1], [0, 2]])
    load = Q.eval_placement(phy2log, np.array([7, 4, 1]))
    assert load.tolist() == [4 + 4, 3 + 1]
