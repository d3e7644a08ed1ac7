"""Pins the oracle's whole partitioned step.

ZeRO-DP reaches exactly the data-parallel result: Adam is coordinate-wise
(ZeRO reading notes, 3) and all-reduce = reduce-scatter + all-gather (notes, 4),
so the partitioned step must equal the unpartitioned one bit for bit.  The
step order is the DeepSpeed ZeRO stages 1-2 walkthrough's 6: overflow check
(skip on overflow), global norm, unscale+clip, Adam on the shard, copy to 16 bit."""
import numpy as np
import pytest
import torch

from helpers import hyper32, make_problem, random_group, t2u16, u16_to_t


def _run_zero(orc, p, flat, grads, nd, dt, h, loss_scale, ranks=None, extra=(0.0, 0)):
    ranks = list(range(nd)) if ranks is None else ranks
    shards = []
    for r in ranks:
        o, n = int(p["rank_offsets"][r]), int(p["rank_numels"][r])
        master = orc.widen_16(flat[o:o + n], dt)
        shards.append(dict(numel=n, grad_off=o, param_off=o, master=master,
                           m=np.zeros(n, np.float32), v=np.zeros(n, np.float32)))
    flat = flat.copy()
    res_all = []
    t = 1
    for step_grads in grads:
        res, _ = orc.zero_step(step_grads, dt, shards, flat, dt, h, t, loss_scale, *extra)
        res_all.append(res.as_dict())
        if res.applied:
            t += 1
        else:
            loss_scale /= 2
    state = np.concatenate([np.concatenate([s["master"], s["m"], s["v"]]) for s in shards])
    return flat, state, res_all, shards


def _run_ddp(orc, flat, grads, nd, dt, h, loss_scale):
    master = orc.widen_16(flat, dt)
    m = np.zeros_like(master)
    v = np.zeros_like(master)
    flat = flat.copy()
    res_all = []
    t = 1
    for step_grads in grads:
        res = orc.ddp_step(step_grads, dt, master, m, v, flat, dt, h, t, loss_scale)
        res_all.append(res.as_dict())
        if res.applied:
            t += 1
        else:
            loss_scale /= 2
    return flat, master, m, v, res_all


@pytest.mark.parametrize("dt", [1, 2])
@pytest.mark.parametrize("mode", [0, 1])
def test_zero_equals_ddp_bitwise(orc, dt, mode):
    rng = np.random.default_rng(100 * dt + mode)
    for trial in range(12):
        numels = random_group(rng)
        nd = int(rng.choice([1, 2, 3, 4, 5, 8]))
        clip = float(rng.choice([0.0, 0.05, 1e3]))
        scale = float(rng.choice([1.0, 1024.0])) if dt == 1 else 1.0
        h = hyper32(max_grad_norm=clip)
        p, flat, grads = make_problem(numels, nd, dt, mode, seed=trial, loss_scale=scale)
        zf, zstate, zres, shards = _run_zero(orc, p, flat, grads, nd, dt, h, scale)
        df, dm, dmm, dv, dres = _run_ddp(orc, flat, grads, nd, dt, h, scale)
        assert np.array_equal(zf, df)
        for r, s in enumerate(shards):
            o, n = int(p["rank_offsets"][r]), int(p["rank_numels"][r])
            assert np.array_equal(s["master"], dm[o:o + n])
            assert np.array_equal(s["m"], dmm[o:o + n])
            assert np.array_equal(s["v"], dv[o:o + n])
        assert zres == dres


def test_clip_fires_and_bounds_the_norm(orc):
    numels = [4000, 123]
    p, flat, grads = make_problem(numels, 4, 2, 0, seed=3, grad_std=1e-2)
    h = hyper32(max_grad_norm=0.01)
    # the clipped, unscaled gradient has norm max_norm (up to the 1e-6 guard and fp32 rounding of k)
    res, red = orc.zero_step(grads[0], 2, [dict(numel=p["padded_total"], grad_off=0, param_off=0,
                                                master=orc.widen_16(flat, 2), m=np.zeros(p["padded_total"], np.float32),
                                                v=np.zeros(p["padded_total"], np.float32))],
                             flat.copy(), 2, h, 1, 1.0, want_grad=True)
    assert res.clip_coef < 1.0
    g = orc.widen_16(red[0], 2).astype(np.float64) * np.float64(res.grad_mult)
    assert np.linalg.norm(g) == pytest.approx(0.01, rel=1e-5)
    assert res.grad_norm == pytest.approx(np.linalg.norm(orc.widen_16(red[0], 2).astype(np.float64)), rel=1e-12)


@pytest.mark.parametrize("nd", [2, 4])
def test_reduce_and_norm_match_torch(orc, nd):
    # the average over ranks and its norm, computed by torch / numpy from the same inputs
    numels = [3000, 77]
    for dt in (1, 2):
        p, flat, grads = make_problem(numels, nd, dt, 0, seed=nd, loss_scale=8.0 if dt == 1 else 1.0)
        P = p["padded_total"]
        red = orc.reduce(grads[0], dt, 0, P)
        acc = sum((u16_to_t(g, dt).float() for g in grads[0][1:]), u16_to_t(grads[0][0], dt).float())
        ref = t2u16((acc / nd).to(u16_to_t(grads[0][0], dt).dtype))
        assert np.array_equal(red, ref)
        _, ovf = orc.stats(red, dt)
        res, _ = orc.zero_step(grads[0], dt, [], flat.copy(), dt, hyper32(), 1, 8.0 if dt == 1 else 1.0)
        full = orc.widen_16(red, dt).astype(np.float64)
        acc_o, _ = orc.stats(red, dt)
        assert acc_o.value() == pytest.approx(float(np.sum(full * full)), rel=1e-12)
        assert ovf == 0


def test_identical_ranks_average_to_the_same_value(orc):
    rng = np.random.default_rng(1)
    for dt in (1, 2):
        g = orc.round_to_16((rng.standard_normal(5000) * 3).astype(np.float32), dt)
        for nd in (1, 2, 3, 7, 64):
            assert np.array_equal(orc.reduce([g] * nd, dt, 0, g.size), g)


@pytest.mark.parametrize("bad", [np.inf, -np.inf, np.nan])
def test_overflow_skips_and_changes_nothing(orc, bad):
    numels = [500, 33]
    nd, dt = 3, 1
    p, flat, grads = make_problem(numels, nd, dt, 0, seed=9, loss_scale=1024.0, steps=1)
    g = grads[0]
    g[2] = g[2].copy()
    g[2][17] = orc.round_to_16(np.array([bad], np.float32), dt)[0]   # owned by rank 0
    h = hyper32()
    shards = []
    for r in range(nd):
        o, n = int(p["rank_offsets"][r]), int(p["rank_numels"][r])
        shards.append(dict(numel=n, grad_off=o, param_off=o, master=orc.widen_16(flat[o:o + n], dt),
                           m=np.full(n, 0.5, np.float32), v=np.full(n, 0.25, np.float32)))
    before = [{k: s[k].copy() for k in ("master", "m", "v")} for s in shards]
    f = flat.copy()
    res, _ = orc.zero_step(g, dt, shards, f, dt, h, 1, 1024.0)
    assert res.overflow == 1 and res.applied == 0
    assert np.array_equal(f, flat)
    for s, b in zip(shards, before):
        for k in b:
            assert np.array_equal(s[k], b[k])


def test_finite_inputs_whose_sum_overflows_are_an_overflow(orc):
    big = orc.round_to_16(np.array([3.0e38], np.float32), 2)
    res, _ = orc.zero_step([big, big], 2, [dict(numel=1, grad_off=0, param_off=0, master=np.zeros(1, np.float32),
                                                m=np.zeros(1, np.float32), v=np.zeros(1, np.float32))],
                           np.zeros(1, np.uint16), 2, hyper32(), 1, 1.0)
    assert res.overflow == 1 and res.applied == 0


def test_extra_overflow_and_sumsq_from_other_ranks(orc):
    numels = [100]
    p, flat, grads = make_problem(numels, 2, 2, 0, seed=4, steps=1)
    sh = lambda: [dict(numel=50, grad_off=0, param_off=0, master=np.zeros(50, np.float32),
                       m=np.zeros(50, np.float32), v=np.zeros(50, np.float32))]
    r0, _ = orc.zero_step(grads[0], 2, sh(), flat.copy(), 2, hyper32(), 1, 1.0)
    r1, _ = orc.zero_step(grads[0], 2, sh(), flat.copy(), 2, hyper32(), 1, 1.0, extra_sumsq=2.5)
    assert r1.sumsq == r0.sumsq + 2.5
    r2, _ = orc.zero_step(grads[0], 2, sh(), flat.copy(), 2, hyper32(), 1, 1.0, extra_overflow=1)
    assert r2.overflow == 1 and r2.applied == 0


def test_padding_stays_zero(orc):
    numels = [7, 5]   # 12 elements, nd = 5 -> padded to 20
    p, flat, grads = make_problem(numels, 5, 1, 0, seed=2, loss_scale=1024.0)
    assert p["padding"] == 8
    zf, *_ = _run_zero(orc, p, flat, grads, 5, 1, hyper32(), 1024.0)
    assert not zf[12:].any()


@pytest.mark.parametrize("mode", [0, 1])
def test_tiny_workload_three_steps_with_skip(orc, mode):
    """The tiny fp16 workload: N_d = 3, loss scale 1024, +inf at flat index
    30000 of rank 0's gradient at step 2 (owned by rank 1 in both readings):
    step 2 is skipped, the scale halves to 512, and step 3 runs with t = 2."""
    import workloads as W
    numels = [s.numel for s in W.tiny_group()]
    p, flat, grads = make_problem(numels, 3, 1, mode, seed=0, loss_scale=1024.0)
    grads[1][0] = grads[1][0].copy()
    grads[1][0][30000] = 0x7C00
    assert p["rank_offsets"][1] <= 30000 < p["rank_offsets"][1] + p["rank_numels"][1]
    h = hyper32()
    zf, zstate, zres, shards = _run_zero(orc, p, flat, grads, 3, 1, h, 1024.0)
    assert [r["applied"] for r in zres] == [1, 0, 1]
    assert [r["overflow"] for r in zres] == [0, 1, 0]
    df, dm, dmm, dv, dres = _run_ddp(orc, flat, grads, 3, 1, h, 1024.0)
    assert np.array_equal(zf, df) and zres == dres
