"""Pins the oracle's memory model to the figures the pages print
(tests/golden/memory_model.json, each case with its citation)."""
import json
import os

import pytest

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "memory_model.json")))


@pytest.mark.parametrize("case", GOLD["cases"], ids=lambda c: f"{c['psi']:.3g}-K{c['K']}-N{c['nd']}-s{c['stage']}")
def test_printed_figures(orc, case):
    gb = orc.mem_model(case["psi"], case["K"], case["nd"], case["stage"]) / 1e9
    assert round(gb, case["digits"]) == pytest.approx(case["printed_gb"]), case["cite"]


def test_capacity_at_32gb(orc):
    for c in GOLD["capacity_32gb_nd64"]["cases"]:
        assert orc.mem_model(c["psi"], 12, 64, c["stage"]) <= 32e9 + 1


def test_closed_forms(orc):
    psi, K = 7.5e9, 12
    assert orc.mem_model(psi, K, 1, 0) == 16 * psi
    for nd in (1, 2, 7, 64, 1024):
        # every stage equals the DP figure at N_d = 1 and shrinks monotonically with the stage
        vals = [orc.mem_model(psi, K, nd, s) for s in range(4)]
        if nd == 1:
            assert all(v == pytest.approx(16 * psi) for v in vals)
        else:
            assert vals[0] > vals[1] > vals[2] > vals[3]
        assert vals[3] == pytest.approx(16 * psi / nd)
    # limits quoted on the pages: 4x, 8x, N_d x reduction for large N_d
    big = 1 << 30
    assert orc.mem_model(psi, K, big, 0) / orc.mem_model(psi, K, big, 1) == pytest.approx(4, rel=1e-6)
    assert orc.mem_model(psi, K, big, 0) / orc.mem_model(psi, K, big, 2) == pytest.approx(8, rel=1e-6)
    assert orc.mem_model(psi, K, 1, 5) == -1.0
