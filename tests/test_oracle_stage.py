"""Pins of the oracle's replica weight staging: it is a gather of expert rows
into spare-slot rows, checked against numpy fancy indexing, with empty slots
(-1), slots that already hold their expert, and invalid ids left untouched and
counted as the definition says.  No GPU needed."""
import numpy as np

import oracle


def _tables(E, nb, R, S, seed):
    rng = np.random.default_rng(seed)
    expert_w = rng.integers(0, 256, size=(E, nb), dtype=np.uint8)
    slot_w = rng.integers(0, 256, size=(R * S, nb), dtype=np.uint8)
    return rng, expert_w, slot_w


def test_stage_is_a_gather_of_expert_rows():
    rng, ew, sw = _tables(12, 48, 4, 2, 0)
    se = rng.integers(0, 12, size=8).astype(np.int32)
    out, n, bad = oracle.stage(ew, se, 4, 2, sw)
    assert np.array_equal(out, ew[se]) and n == 8 and bad == 0


def test_empty_invalid_and_unchanged_slots_are_left_alone():
    rng, ew, sw = _tables(6, 32, 3, 2, 1)
    se = np.array([2, -1, 7, 5, -4, 0], np.int32)     # slot 1 empty, 2 and 4 invalid
    prev = np.array([2, 3, 1, 1, 0, 0], np.int32)     # slots 0 and 5 already hold their expert
    out, n, bad = oracle.stage(ew, se, 3, 2, sw, prev=prev)
    assert n == 1 and bad == 2                         # only slot 3 (expert 5) is new
    assert np.array_equal(out[3], ew[5])
    for x in (0, 1, 2, 4, 5):
        assert np.array_equal(out[x], sw[x])
    # without prev, slots 0, 3 and 5 are copied
    out, n, bad = oracle.stage(ew, se, 3, 2, sw)
    assert n == 3 and bad == 2
    assert np.array_equal(out[[0, 3, 5]], ew[[2, 5, 0]])
    assert np.array_equal(out[[1, 2, 4]], sw[[1, 2, 4]])


def test_no_spare_slots():
    _, ew, _ = _tables(4, 16, 2, 1, 2)
    out, n, bad = oracle.stage(ew, np.zeros(0, np.int32), 2, 0, np.zeros((0, 16), np.uint8))
    assert out.shape == (0, 16) and n == 0 and bad == 0
