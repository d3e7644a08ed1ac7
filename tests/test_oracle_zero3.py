"""Pins the oracle's ZeRO-3 per-layer functions (ZeRO reading notes, 7 and 9:
a layer's parameter parts are gathered before its forward and its backward;
its gradients are reduced onto the owner of each part)."""
import numpy as np
import pytest
import torch

from helpers import t2u16, u16_to_t


@pytest.mark.parametrize("ws,part", [(1, 10), (2, 7), (4, 1000), (8, 33)])
def test_gather_inverts_the_partition(orc, ws, part):
    rng = np.random.default_rng(ws * part)
    layer = rng.integers(0, 1 << 16, ws * part, dtype=np.uint64).astype(np.uint16)
    parts = [layer[r * part:(r + 1) * part].copy() for r in range(ws)]
    assert np.array_equal(orc.zero3_gather(parts), layer)


@pytest.mark.parametrize("dt", [1, 2])
def test_bucket_reduce_is_the_owner_range_average(orc, dt):
    ws, part = 4, 5000
    g = torch.Generator().manual_seed(dt)
    tdt = {1: torch.float16, 2: torch.bfloat16}[dt]
    buckets = [t2u16((torch.randn(ws * part, generator=g) * 8).to(tdt)) for _ in range(ws)]
    acc = orc.ExactAccumulator()
    for owner in range(ws):
        a, ovf = orc.zero3_reduce(buckets, owner, part, dt, acc)
        sl = slice(owner * part, (owner + 1) * part)
        s = u16_to_t(buckets[0][sl], dt).float()
        for b in buckets[1:]:
            s = s + u16_to_t(b[sl], dt).float()
        assert np.array_equal(a, t2u16((s / ws).to(tdt)))            # torch's rank-ordered fp32 average
        assert ovf == 0
    # identical ranks give back their own values
    same = [buckets[0]] * ws
    a, _ = orc.zero3_reduce(same, 2, part, dt, orc.ExactAccumulator())
    assert np.array_equal(a, buckets[0][2 * part:3 * part])


def test_bucket_reduce_statistics(orc):
    ws, part, dt = 2, 3000, 2
    rng = np.random.default_rng(3)
    buckets = [orc.round_to_16(rng.standard_normal(ws * part).astype(np.float32), dt) for _ in range(ws)]
    acc = orc.ExactAccumulator()
    total = 0.0
    for owner in range(ws):
        a, _ = orc.zero3_reduce(buckets, owner, part, dt, acc)
        x = orc.widen_16(a, dt).astype(np.float64)
        total += float(np.sum(x * x))
    assert acc.value() == pytest.approx(total, rel=1e-12)
    bad = [b.copy() for b in buckets]
    bad[1][part + 3] = 0x7FC0                                        # NaN in owner 1's range only
    _, o0 = orc.zero3_reduce(bad, 0, part, dt, orc.ExactAccumulator())
    _, o1 = orc.zero3_reduce(bad, 1, part, dt, orc.ExactAccumulator())
    assert (o0, o1) == (0, 1)


def test_segment_gather_inverts_any_cut(orc):
    """Owner broadcast ([paper] 5.3): a layer rebuilt from the pieces of the
    owners' contiguous segments it spans is the layer."""
    rng = np.random.default_rng(4)
    for _ in range(50):
        layer = rng.integers(0, 1 << 16, int(rng.integers(0, 3000)), dtype=np.uint64).astype(np.uint16)
        cuts = np.sort(rng.integers(0, layer.size + 1, int(rng.integers(0, 5))))
        pieces = [layer[a:b].copy() for a, b in zip(np.concatenate([[0], cuts]), np.concatenate([cuts, [layer.size]]))]
        assert np.array_equal(orc.gather_segments(pieces), layer)


def test_broadcast_pieces_cover_each_unit_once(orc):
    """The pieces of a unit owned by each rank (the partition's intersections
    with the unit) cover the unit exactly once, in order."""
    units = [300, 1000, 48, 5000, 7]
    for nd in (1, 2, 4, 7):
        p = orc.plan(units, nd, 0)
        seen = {u: [] for u in range(len(units))}
        for r in range(nd):
            for u, u0, s0, ln in orc.plan_intersections(p["tensor_offsets"], units, int(p["rank_offsets"][r]),
                                                         int(p["rank_numels"][r])):
                seen[int(u)].append((int(u0), int(ln), r))
        for u, rows in seen.items():
            rows.sort()
            pos = 0
            for u0, ln, r in rows:
                assert u0 == pos
                pos += ln
            assert pos == units[u]
            assert [r for _, _, r in rows] == sorted(r for _, _, r in rows)     # owners in rank order
