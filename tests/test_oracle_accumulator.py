"""Pins the oracle's exact sum-of-squares accumulator against Python's
correctly rounded math.fsum, and checks that its result does not depend on the
order of the terms.  The global norm is a sum of per-shard partial sums
(DeepSpeed ZeRO stages 1-2 walkthrough, 6 step 2), so an order-independent sum
is what makes the partitioned and unpartitioned steps agree bit for bit."""
import math

import numpy as np


def test_matches_fsum_wide_range(orc):
    rng = np.random.default_rng(7)
    for trial in range(20):
        n = int(rng.integers(1, 5000))
        mant = rng.random(n)
        exps = rng.integers(-300, 300, n)
        x = np.ldexp(mant, exps)
        assert orc.exact_sum(x) == math.fsum(x.tolist())


def test_matches_fsum_squares_of_16bit(orc):
    rng = np.random.default_rng(8)
    for dt, npdt in ((orc.F16, np.float16),):
        v = (rng.standard_normal(100000) * 10.0 ** rng.integers(-6, 4, 100000)).astype(npdt).astype(np.float64)
        sq = v * v
        assert orc.exact_sum(sq) == math.fsum(sq.tolist())


def test_subnormal_and_huge_terms(orc):
    x = np.array([5e-324, 1e308, 5e-324, 1e-310, 3.0, 1e300])
    assert orc.exact_sum(x) == math.fsum(x.tolist())
    assert orc.exact_sum(np.array([5e-324] * 7)) == 7 * 5e-324
    assert orc.exact_sum(np.array([1e308, 1e308])) == math.inf


def test_order_independent(orc):
    rng = np.random.default_rng(9)
    x = np.ldexp(rng.random(20000), rng.integers(-60, 60, 20000))
    ref = orc.exact_sum(x)
    for _ in range(5):
        assert orc.exact_sum(rng.permutation(x)) == ref
    # split into pieces, summed separately and merged
    acc = orc.ExactAccumulator()
    for piece in np.array_split(x, 7):
        a = orc.ExactAccumulator()
        for t in piece:
            a.add(t)
        acc.merge(a)
    assert acc.value() == ref


def test_ties_round_to_even(orc):
    # 2^53 + 1 is a tie between 2^53 and 2^53 + 2: even mantissa wins
    assert orc.exact_sum(np.array([2.0 ** 53, 1.0])) == 2.0 ** 53
    assert orc.exact_sum(np.array([2.0 ** 53, 3.0])) == 2.0 ** 53 + 4
    assert orc.exact_sum(np.array([2.0 ** 53, 1.0, 2.0 ** -60])) == 2.0 ** 53 + 2
