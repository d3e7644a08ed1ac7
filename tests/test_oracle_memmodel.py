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


# ------------------------------------------------------------------ plan-exact model
def _exact_share(psi, nd):
    return int(psi) // nd if int(psi) % nd == 0 else None


@pytest.mark.parametrize("case", [c for c in GOLD["cases"] if _exact_share(c["psi"], c["nd"]) is not None],
                         ids=lambda c: f"{c['psi']:.3g}-K{c['K']}-N{c['nd']}-s{c['stage']}")
def test_plan_exact_model_gives_the_printed_figures(orc, case):
    """With no padding (Psi divisible by N_d) the plan's sizes are Psi and
    Psi / N_d, and every printed figure must come out."""
    psi, nd = int(case["psi"]), case["nd"]
    got = orc.mem_model_plan(psi, psi // nd, case["K"], case["stage"])
    assert round(got["total"] / 1e9, case["digits"]) == pytest.approx(case["printed_gb"]), case["cite"]
    assert got["temp"] == 0.0


@pytest.mark.parametrize("case", GOLD["fused_fp32_buffer"]["cases"], ids=lambda c: f"{c['numel']:.3g}")
def test_fused_fp32_buffer_figures(orc, case):
    got = orc.mem_model_plan(1000, 1000, 12, 2, fp32_temp=int(case["numel"]))
    assert round(got["temp"] / 1e9, case["digits"]) == pytest.approx(case["printed_gb"]), case["cite"]
    base = orc.mem_model_plan(1000, 1000, 12, 2)
    assert got["total"] - base["total"] == got["temp"]


def test_sixteen_bit_temporaries_and_state_copies(orc):
    F = 1_557_611_200
    # a 16-bit temporary of F elements is as large as DP's 16-bit gradient buffer of F elements
    assert orc.mem_model_plan(F, F, 12, 0, b16_temp=F)["temp"] == orc.mem_model_plan(F, F, 12, 0)["grads"]
    # two copies of K-byte states hold what one copy of 2K-byte states holds, and nothing else changes
    for stage in range(4):
        two = orc.mem_model_plan(F, F // 8, 12, stage, sets=2)
        wide = orc.mem_model_plan(F, F // 8, 24, stage)
        one = orc.mem_model_plan(F, F // 8, 12, stage)
        assert two == wide
        assert (two["params"], two["grads"]) == (one["params"], one["grads"])
    for bad in (dict(sets=0), dict(fp32_temp=-1), dict(b16_temp=-1)):
        assert orc.mem_model_plan(F, F, 12, 1, **bad) is None
    assert orc.mem_model_plan(F, F, 12, 4) is None and orc.mem_model_plan(-1, 0, 12, 1) is None


def _plans(orc):
    import workloads as W
    out = [(W.numels(W.tiny_group()), 3, 0), (W.numels(W.tiny_group()), 3, 1), (W.numels(W.gpt2_group()), 8, 0),
           (W.numels(W.gpt2_group(52, 3456, 50257, 1024)), 64, 0), ([5, 1, 7], 4, 0), ([5, 1, 7], 4, 1)]
    return [(orc.plan(n, nd, mode), sum(n), nd) for n, nd, mode in out]


def test_ranks_together_hold_one_copy_of_what_is_partitioned(orc):
    """Summed over the plan's ranks: a partitioned term holds exactly one copy
    of the padded group; a term a stage keeps whole is held once per rank."""
    K = 12
    for p, psi, nd in _plans(orc):
        P = int(p["padded_total"])
        per = {s: [orc.mem_model_plan(P if s else psi, int(n), K, s, sets=2) for n in p["rank_numels"]]
               for s in range(4)}
        tot = lambda s, k: sum(x[k] for x in per[s])
        for s in (1, 2, 3):
            assert tot(s, "states") == 2 * K * P
        assert tot(0, "states") == 2 * K * psi * nd
        assert tot(0, "params") == tot(0, "grads") == 2 * psi * nd
        assert tot(1, "params") == tot(1, "grads") == tot(2, "params") == 2 * P * nd
        assert tot(2, "grads") == tot(3, "grads") == tot(3, "params") == 2 * P
        assert tot(3, "total") == (4 + 2 * K) * P
        # the largest rank holds at least the pages' Psi / N_d share
        assert max(x["total"] for x in per[3]) >= (4 + 2 * K) * psi / nd
