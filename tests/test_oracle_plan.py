"""Pins the oracle's partition plan by brute force on small inputs.
Rules (DeepSpeed ZeRO stages 1-2 walkthrough, 4 (1), (2), (4) and 7):
flatten in declaration order; pad the flat length to a multiple of
2*world_size; base = total // dp with the remainder to the first ranks; rank r
owns contiguous segment r; a tensor may straddle two shards."""
import itertools

import numpy as np
import pytest


def _brute(numels, ws, mode):
    owner = []
    flat = []
    for t, n in enumerate(numels):
        flat += [(t, j) for j in range(n)]
    total = len(flat)
    if mode == 0:
        a = 2 * ws
        P = -(-total // a) * a
    else:
        P = total
    flat += [None] * (P - total)
    base, rem = divmod(P, ws)
    sizes = [base + (1 if r < rem else 0) for r in range(ws)]
    r = 0
    left = sizes[0]
    for i in range(P):
        while left == 0:
            r += 1
            left = sizes[r]
        owner.append(r)
        left -= 1
    return flat, owner, sizes, P


@pytest.mark.parametrize("mode", [0, 1])
def test_plan_brute_force(orc, mode):
    rng = np.random.default_rng(mode)
    cases = [([1], 1), ([0], 3), ([5], 8), ([3, 0, 4], 2), ([257 * 129, 129, 1000 * 37], 3)]
    for _ in range(150):
        n = int(rng.integers(1, 6))
        cases.append((list(rng.integers(0, 60, n)), int(rng.integers(1, 12))))
    for numels, ws in cases:
        if sum(numels) > 5000 and ws > 3:
            continue
        p = orc.plan(numels, ws, mode)
        flat, owner, sizes, P = _brute(numels, ws, mode)
        assert p["padded_total"] == P and p["padding"] == P - sum(numels)
        assert list(p["rank_numels"]) == sizes
        # every flat element covered exactly once, contiguous and in rank order
        cover = np.zeros(P, int)
        for r in range(ws):
            o, s = int(p["rank_offsets"][r]), int(p["rank_numels"][r])
            cover[o:o + s] += 1
            assert all(owner[i] == r for i in range(o, o + s))
        assert (cover == 1).all()
        # tensors in declaration order
        assert list(p["tensor_offsets"]) == list(np.concatenate([[0], np.cumsum(numels)[:-1]]).astype(int))
        # remainder to the first ranks: sizes never increase and differ by <= 1
        assert max(sizes) - min(sizes) <= 1 and sizes == sorted(sizes, reverse=True)
        if mode == 0:
            # padded shards are equal and start on a 4-byte boundary for 16-bit elements
            assert len(set(sizes)) == 1
            assert all((int(o) * 2) % 4 == 0 for o in p["rank_offsets"])
        # intersections reproduce the owner map
        for r in range(ws):
            rows = orc.plan_intersections(p["tensor_offsets"], numels, int(p["rank_offsets"][r]),
                                          int(p["rank_numels"][r]))
            seen = []
            for t, t0, s0, ln in rows:
                for q in range(ln):
                    assert flat[int(p["rank_offsets"][r]) + s0 + q] == (t, t0 + q)
                seen += list(range(s0, s0 + ln))
            real = [i for i in range(int(p["rank_numels"][r])) if flat[int(p["rank_offsets"][r]) + i] is not None]
            assert seen == real


def test_tiny_workload_both_readings(orc):
    numels = [257 * 129, 129, 1000 * 37]
    assert sum(numels) == 70282
    p0 = orc.plan(numels, 3, 0)
    assert p0["padded_total"] == 70284 and p0["padding"] == 2
    assert list(p0["rank_numels"]) == [23428] * 3
    p1 = orc.plan(numels, 3, 1)
    assert list(p1["rank_numels"]) == [23428, 23427, 23427]      # remainder 1 to rank 0
    assert list(p1["rank_offsets"]) == [0, 23428, 46855]


def test_invalid(orc):
    with pytest.raises(ValueError):
        orc.plan([1, 2], 0, 0)
    with pytest.raises(ValueError):
        orc.plan([1, -2], 2, 0)
