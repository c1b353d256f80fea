"""The planner's quotient of a small index by a run-time size, floor(x / d) taken as
trunc((x + 1/2) * fl(1/d)) in float32 (round to nearest, as the GPU's multiply):
exact for every numerator below 2^21.  Checked here on the host, exhaustively over
the planner's range (numerators below 4096, divisors up to 2048) and over every
numerator below 2^21 for a few divisors, including the largest ones."""
import numpy as np


def _quotients(x, d):
    inv = np.float32(1.0) / np.float32(d)
    return ((x.astype(np.float32) + np.float32(0.5)) * inv).astype(np.int64)


def test_exact_over_the_planners_range():
    x = np.arange(4096, dtype=np.int64)
    for d in range(1, 2049):
        assert np.array_equal(_quotients(x, d), x // d), d


def test_exact_below_2_pow_21():
    x = np.arange(1 << 21, dtype=np.int64)
    for d in (1, 3, 7, 31, 32, 33, 1000, 1023, 1024, 2047, 2048, 4095, 65535, (1 << 21) - 1):
        assert np.array_equal(_quotients(x, d), x // d), d
