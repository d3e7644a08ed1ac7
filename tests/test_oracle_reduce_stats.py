"""Pins of the oracle's one-sweep reduce-and-statistics (orc_reduce_stats),
the checker of every full-size norm and overflow flag.

DeepSpeed ZeRO stages 1-2 walkthrough, 6 steps 1-2: the overflow check looks
for inf/NaN in the averaged gradient, and the global norm is the square root
of the sum over every element of its square.  What the sweep must give for a
window [off, off + numel) of N 16-bit slices is pinned here to values
computed without the oracle:
  * the averaged gradient by numpy (fp32 sum in rank order, one fp32
    division) and the 16-bit rounding by numpy (fp16) or torch (bf16);
  * the sum of squares by Python's correctly rounded math.fsum of the exact
    fp64 squares of the widened 16-bit values, which the oracle's exactly
    rounded accumulator must equal bit for bit;
  * the overflow flag from numpy's isfinite on the rounded values.
Random windows catch an offset applied twice or not at all; the 16-bit
rounding before the square catches statistics taken on the unrounded sum;
inf/NaN placed inside and just outside the window catch a window boundary
off by one; chunked sweeps merged with orc_acc_merge must give the one-sweep
value (what the full-size tests do); and the sweep must agree with orc_reduce
followed by orc_stats."""
import math

import numpy as np
import pytest
import torch

TORCH16 = {1: torch.float16, 2: torch.bfloat16}
NONFINITE = {1: (0x7C00, 0xFC00, 0x7E00), 2: (0x7F80, 0xFF80, 0x7FC0)}


def widen(h: np.ndarray, dt: int) -> np.ndarray:
    """16-bit patterns -> fp32 values, by torch."""
    return torch.from_numpy(h.view(np.int16).copy()).view(TORCH16[dt]).float().numpy()


def narrow(x: np.ndarray, dt: int) -> np.ndarray:
    """fp32 -> 16-bit patterns, round to nearest even (numpy for fp16, torch for bf16)."""
    if dt == 1:
        return x.astype(np.float16).view(np.uint16)
    return torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def independent(slices, dt, off, numel):
    """The averaged 16-bit gradient of the window, its exact sum of squares
    (rounded once, by math.fsum) and its overflow flag, without the oracle."""
    s = np.zeros(numel, np.float32)
    for g in slices:                                   # rank order, fp32 adds
        s = s + widen(g[off:off + numel], dt)
    a16 = narrow(s / np.float32(len(slices)), dt)
    a = widen(a16, dt).astype(np.float64)
    fin = np.isfinite(a)
    ovf = int(not fin.all())
    return a16, (math.fsum((a[fin] * a[fin]).tolist()) if not ovf else math.inf), ovf


def random_slices(rng, nd, P, dt, scale):
    out = []
    for _ in range(nd):
        x = (rng.standard_normal(P) * scale).astype(np.float32)
        out.append(narrow(x, dt))
    return out


@pytest.mark.parametrize("dt", [1, 2])
@pytest.mark.parametrize("nd", [1, 2, 3, 4, 8, 13])
def test_random_windows_equal_the_independent_sweep(orc, dt, nd):
    rng = np.random.default_rng(1000 + 10 * dt + nd)
    P = 6000
    scale = 4.0 if dt == 1 else 1e-3              # fp16: values far from the subnormal range
    slices = random_slices(rng, nd, P, dt, scale)
    for _ in range(12):
        off = int(rng.integers(0, P))
        numel = int(rng.integers(0, P - off + 1))
        _, want, want_ovf = independent(slices, dt, off, numel)
        acc = orc.ExactAccumulator()
        ovf = orc.reduce_stats(slices, dt, off, numel, acc)
        assert ovf == want_ovf == 0
        assert acc.value() == want                    # both exactly rounded: bit for bit


@pytest.mark.parametrize("dt", [1, 2])
def test_rounding_before_the_square_matters(orc, dt):
    """Inputs whose fp32 average is not a 16-bit value: the statistics of the
    rounded average differ from those of the unrounded one, and the sweep must
    give the former."""
    rng = np.random.default_rng(7 + dt)
    P = 4000
    slices = random_slices(rng, 3, P, dt, 2.0 if dt == 1 else 1e-2)
    a16, want, _ = independent(slices, dt, 0, P)
    s = sum(widen(g, dt).astype(np.float32) for g in slices) / np.float32(3)
    unrounded = math.fsum((s.astype(np.float64) ** 2).tolist())
    assert unrounded != want
    acc = orc.ExactAccumulator()
    orc.reduce_stats(slices, dt, 0, P, acc)
    assert acc.value() == want
    assert np.array_equal(orc.reduce(slices, dt, 0, P), a16)


@pytest.mark.parametrize("dt", [1, 2])
def test_nonfinite_inside_and_outside_the_window(orc, dt):
    rng = np.random.default_rng(21 + dt)
    P, nd = 3000, 4
    off, numel = 1000, 700
    for bad in NONFINITE[dt]:
        for pos, inside in ((off, True), (off + numel - 1, True), (off - 1, False), (off + numel, False),
                            (off + 333, True)):
            slices = random_slices(rng, nd, P, dt, 1.0 if dt == 1 else 1e-3)
            slices[int(rng.integers(0, nd))][pos] = bad
            _, want, want_ovf = independent(slices, dt, off, numel)
            acc = orc.ExactAccumulator()
            ovf = orc.reduce_stats(slices, dt, off, numel, acc)
            assert ovf == want_ovf == int(inside)
            if inside:
                assert math.isinf(acc.value())
            else:
                assert acc.value() == want


def test_finite_inputs_whose_sum_overflows(orc):
    """bf16 values near 3e38 in two slices: each is finite, their fp32 sum is
    +inf, so the average is an overflow; at a tenth of that size the same
    pair averages to a finite value with a finite (fp64) square."""
    big = np.full(6, 0x7F61, np.uint16)                  # ~2.99e38
    with np.errstate(over="ignore"):
        _, _, want_ovf = independent([big, big], 2, 0, 6)
    assert want_ovf == 1
    assert orc.reduce_stats([big, big], 2, 0, 6, orc.ExactAccumulator()) == 1
    small = narrow(np.full(6, 3e37, np.float32), 2)
    _, want, want_ovf = independent([small, small], 2, 0, 6)
    acc = orc.ExactAccumulator()
    assert orc.reduce_stats([small, small], 2, 0, 6, acc) == want_ovf == 0
    assert acc.value() == want and want > 1e75


@pytest.mark.parametrize("dt", [1, 2])
def test_chunked_sweeps_merged_equal_one_sweep(orc, dt):
    """What the full-size checks do: the window cut into chunks, each swept
    into an accumulator of its own, the accumulators merged."""
    rng = np.random.default_rng(31 + dt)
    P, nd = 20000, 5
    slices = random_slices(rng, nd, P, dt, 3.0 if dt == 1 else 5e-4)
    off, numel = 123, P - 500
    _, want, _ = independent(slices, dt, off, numel)
    for _ in range(4):
        cuts = np.sort(rng.integers(0, numel, int(rng.integers(1, 9))))
        bounds = [0] + [int(c) for c in cuts] + [numel]
        total = orc.ExactAccumulator()
        for lo, hi in zip(bounds[:-1], bounds[1:]):
            part = orc.ExactAccumulator()
            assert orc.reduce_stats(slices, dt, off + lo, hi - lo, part) == 0
            total.merge(part)
        assert total.value() == want


@pytest.mark.parametrize("dt", [1, 2])
def test_sweep_equals_reduce_then_stats(orc, dt):
    rng = np.random.default_rng(41 + dt)
    P, nd = 5000, 3
    slices = random_slices(rng, nd, P, dt, 1.0 if dt == 1 else 1e-3)
    slices[1][2500] = NONFINITE[dt][2]
    for off, numel in ((0, P), (17, 2000), (2400, 200), (4999, 1), (10, 0)):
        a = orc.reduce(slices, dt, off, numel)
        acc1, ovf1 = orc.stats(a, dt)
        acc2 = orc.ExactAccumulator()
        ovf2 = orc.reduce_stats(slices, dt, off, numel, acc2)
        assert ovf1 == ovf2
        v1, v2 = acc1.value(), acc2.value()
        assert v1 == v2 or (math.isinf(v1) and math.isinf(v2))
