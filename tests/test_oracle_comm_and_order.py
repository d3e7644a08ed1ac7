"""Pins the oracle's communication-volume model to the figures the pages
print (tests/golden/comm_volume.json), and its round-robin order to the
purpose the DeepSpeed ZeRO stages 1-2 walkthrough (4.1) gives it: tensors
adjacent in the original order land in different ranks' shards."""
import json
import os

import numpy as np
import pytest

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "comm_volume.json")))


@pytest.mark.parametrize("case", GOLD["cases"], ids=lambda c: f"stage{c['stage']}")
def test_printed_volumes(orc, case):
    psi = 7.5e9
    assert orc.comm_volume(psi, 64, case["stage"]) == case["psi_units"] * psi, case["cite"]


def test_stage3_is_one_and_a_half_times_dp(orc):
    for nd in (2, 8, 64):
        for ring in (False, True):
            assert orc.comm_volume(1e9, nd, 3, ring) == pytest.approx(1.5 * orc.comm_volume(1e9, nd, 0, ring))


def test_ring_factor(orc):
    psi = 1e9
    assert orc.comm_volume(psi, 1, 0, True) == 0.0                  # one rank sends nothing
    assert orc.comm_volume(psi, 2, 0, True) == pytest.approx(psi)    # each phase moves half
    for nd in (4, 64, 1024):
        v = orc.comm_volume(psi, nd, 0, True)
        assert v == pytest.approx(2 * psi * (nd - 1) / nd)
        assert v < 2 * psi and v > 2 * psi * 0.74
    assert orc.comm_volume(psi, 0, 0, False) == -1.0


def test_round_robin_rotates_owners(orc):
    for ws in (2, 3, 8):
        for per in (1, 2, 5):
            n = ws * per
            numels = [64] * n                                         # equal tensors
            order = orc.round_robin(n, ws)
            assert sorted(order.tolist()) == list(range(n))           # a permutation
            p = orc.plan([numels[i] for i in order], ws, 0)
            t_off = dict(zip(order.tolist(), p["tensor_offsets"].tolist()))
            owner = lambda i: int(np.searchsorted(p["rank_offsets"], t_off[i], side="right") - 1)
            for i in range(n - 1):
                assert owner(i) != owner(i + 1)                      # neighbours belong to different ranks
            assert [owner(i) for i in range(n)] == [i % ws for i in range(n)]


def test_round_robin_one_rank_keeps_the_order(orc):
    assert orc.round_robin(7, 1).tolist() == list(range(7))
    assert orc.round_robin(0, 3).tolist() == []
    with pytest.raises(ValueError):
        orc.round_robin(3, 0)
