"""Pins of the oracle's weighted combine (the step after unpermute: each token's
k expert rows summed with its gate weights), against values the arithmetic
fixes by hand: exact binary fractions, the float32 order dependence of the
ascending-j sum, round-to-nearest-even ties of the bf16 conversion, NaN
canonicalisation, missing slots and the k = 1 identity.  No GPU needed."""
import numpy as np
import pytest

import oracle

ONE, TWO, FOUR, EIGHT = 0x3F80, 0x4000, 0x4080, 0x4100
P24, M24 = 0x4B80, 0xCB80                  # +2^24, -2^24 (exact in bf16)
EPS8 = 0x3B80                              # 2^-8
EPS20 = 0x3580                             # 2^-20


def _combine_one(values, weights, order=None):
    """One token, Hd = 1: rows are the given bf16 bit patterns, read in `order`."""
    g = np.array(values, np.uint16)[:, None]
    k = len(values)
    dst = np.arange(k, dtype=np.int32) if order is None else np.array(order, np.int32)
    w = np.array([weights], np.float32)
    return int(oracle.combine(g, 1, k, dst, w)[0, 0])


def test_exact_binary_fractions():
    # 0.5*2 + 0.25*4 + 0.25*8 = 4 exactly
    assert _combine_one([TWO, FOUR, EIGHT], [0.5, 0.25, 0.25]) == FOUR
    # 3 * 0.5 = 1.5 exactly (0x3FC0)
    assert _combine_one([ONE, ONE, ONE], [0.5, 0.5, 0.5]) == 0x3FC0


def test_float32_sum_in_ascending_j():
    # 2^24 + 1 rounds back to 2^24 in float32 (tie to even), so 2^24 + 1 - 2^24
    # is 0 in ascending j, although the exact sum is 1
    assert _combine_one([P24, ONE, M24], [1.0, 1.0, 1.0]) == 0x0000
    # the same three rows met in another slot order: -2^24 + 2^24 + 1 = 1
    assert _combine_one([P24, ONE, M24], [1.0, 1.0, 1.0], order=[2, 0, 1]) == ONE


def test_bf16_round_to_nearest_even():
    assert _combine_one([ONE, EPS8], [1.0, 1.0]) == 0x3F80          # 1+2^-8: tie, even is down
    assert _combine_one([0x3F81, EPS8], [1.0, 1.0]) == 0x3F82       # 1.0078125+2^-8: tie, even is up
    assert _combine_one([ONE, EPS8, EPS20], [1.0, 1.0, 1.0]) == 0x3F81  # just above the tie
    assert _combine_one([ONE, 0x3B00], [1.0, 1.0]) == 0x3F80        # 1+2^-9: below half


def test_nan_inf_and_signed_zero():
    assert _combine_one([0x7FC1], [1.0]) == 0x7FC0                  # NaN payload -> canonical
    assert _combine_one([0xFF81], [1.0]) == 0x7FC0                  # negative signalling NaN too
    assert _combine_one([0x7F80], [0.0]) == 0x7FC0                  # inf * 0
    assert _combine_one([0x7F80, 0xFF80], [1.0, 1.0]) == 0x7FC0     # inf - inf
    assert _combine_one([0x7F80], [1.0]) == 0x7F80                  # inf stays inf
    assert _combine_one([0x8000], [1.0]) == 0x0000                  # +0 + (-0) = +0


def test_missing_slots_add_nothing_and_zero_weights():
    g = np.array([[TWO], [FOUR]], np.uint16)
    w = np.array([[1.0, 1.0, 1.0]], np.float32)
    assert int(oracle.combine(g, 1, 3, np.array([0, -1, 1], np.int32), w)[0, 0]) == 0x40C0  # 6
    assert int(oracle.combine(g, 1, 3, np.array([-1, -1, -1], np.int32), w)[0, 0]) == 0
    assert _combine_one([TWO, FOUR], [0.0, 0.0]) == 0


@pytest.mark.parametrize("seed", [0, 1])
def test_k1_unit_weight_is_the_identity(seed):
    rng = np.random.default_rng(seed)
    bits = rng.integers(0, 1 << 16, size=(64, 32), dtype=np.uint16)
    finite = (bits & 0x7F80) != 0x7F80
    bits = np.where(finite, bits, np.uint16(ONE))
    bits[bits == 0x8000] = ONE                                         # -0 becomes +0 (see above)
    y = oracle.combine(bits, 64, 1, np.arange(64, dtype=np.int32), np.ones((64, 1), np.float32))
    assert np.array_equal(y, bits)


def test_rows_follow_dst_row_per_token():
    # two tokens, k = 2, rows permuted: token 0 takes rows 3, 1; token 1 rows 0, 2
    g = np.array([[ONE, TWO], [TWO, FOUR], [FOUR, EIGHT], [EIGHT, ONE]], np.uint16)
    dst = np.array([3, 1, 0, 2], np.int32)
    w = np.array([[0.5, 0.5], [0.25, 0.75]], np.float32)
    y = oracle.combine(g, 2, 2, dst, w)
    # token 0: 0.5*[8,1] + 0.5*[2,4] = [5, 2.5]; token 1: 0.25*[1,2] + 0.75*[4,8] = [3.25, 6.5]
    assert y.tolist() == [[0x40A0, 0x4020], [0x4050, 0x40D0]]
