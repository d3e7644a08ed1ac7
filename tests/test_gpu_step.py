"""GPU parity of the partitioned step against the CPU oracle, at sizes the
oracle finishes in seconds (several tiles per shard, ragged tails), through
the C ABI.

Tolerances: plan, overflow flag, reduced gradients bit-exact; without
clipping every state and parameter is bit-exact too (both sides do the same
rounded fp32 operations, and the multiplier 1/S is exact).  With clipping the
multiplier k = fp32(c / S) comes from the fp64 norm: the device sums the
squares with compensation in fp32 and fp64, the oracle exactly, so the two
norms agree to ~1e-13 relative and k is in practice the same fp32 value --
then every state and parameter must be bit-exact as well.  Only if k came out
one ulp apart (c / S on an fp32 rounding boundary) are fp32 states held to
rel 2e-6 of the operands each update combines and 16-bit parameters to 1 ulp.
The norm is compared within rel 1e-5."""
import numpy as np
import pytest
import torch

import oracle as orc
import workloads as W
from helpers import hyper32, make_problem, random_group, t2u16

pytestmark = pytest.mark.gpu

DEV = "cuda"
TDT = {1: torch.float16, 2: torch.bfloat16}


@pytest.fixture(scope="module")
def Z():
    import zero_dp_partitioned_gb300 as Z
    return Z


def dev16(a: np.ndarray, dt):
    return torch.from_numpy(a.view(np.int16).copy()).view(TDT[dt]).to(DEV)


def dev32(a: np.ndarray):
    return torch.from_numpy(a.copy()).to(DEV)


class DeviceRun:
    """Device copy of a problem: per-rank grads, flat params, per-shard state (A and optionally B)."""

    def __init__(self, Z, p, flat, dt, ranks, pingpong, want_grad=True, state_pad=0, param_pad=0):
        self.Z, self.p, self.dt, self.ranks, self.pingpong = Z, p, dt, ranks, pingpong
        self.param_pad = param_pad
        base = torch.zeros(flat.size + param_pad, dtype=TDT[dt], device=DEV)
        base[param_pad:] = dev16(flat, dt)
        self.flat_base = base
        self.flat = base[param_pad:]
        self.state = []
        # state_pad: floats each state array starts into its buffer (one for all
        # six, or one per array: master, m, v in, then out)
        pads = tuple(state_pad) if isinstance(state_pad, (tuple, list)) else (state_pad,) * 6
        for r in ranks:
            o, n = int(p["rank_offsets"][r]), int(p["rank_numels"][r])
            mk = lambda v, q: torch.cat([torch.zeros(q, device=DEV), v])[q:]
            A = [mk(torch.empty(n, device=DEV), pads[i]) for i in range(3)]
            B = [mk(torch.empty(n, device=DEV), pads[3 + i]) for i in range(3)] if pingpong else A
            g = torch.empty(n, dtype=TDT[dt], device=DEV) if want_grad else None
            self.state.append(dict(o=o, n=n, A=A, B=B, g=g))
        Z.zero_shard_init(self.shards(), self.flat, dt)       # master = fp32(parameters), m = v = 0
        self.ws = torch.zeros(Z.zero_workspace_bytes(), dtype=torch.uint8, device=DEV)
        self.res = torch.zeros(48, dtype=torch.uint8, device=DEV)

    def shards(self):
        return [self.Z.shard(s["n"], s["o"], s["o"], *s["A"], *s["B"], s["g"]) for s in self.state]

    def step(self, grads_u16, h, t, S, extra=(0.0, 0), grad_offsets=None):
        Z = self.Z
        slices = [dev16(g, self.dt) for g in grads_u16]
        sh = self.shards()
        if grad_offsets is not None:
            for x, go in zip(sh, grad_offsets):
                x.grad_offset = go
        hy = Z.hyper(h["lr"], h["beta1"], h["beta2"], h["eps"], h["weight_decay"], h["max_grad_norm"], t)
        Z.zero_shard_step(slices, self.dt, sh, self.flat, self.dt, hy, S, extra[0], extra[1], self.ws,
                          self.ws.numel(), self.res)
        torch.cuda.synchronize()
        r = Z.read_result(self.res)
        if r.applied and self.pingpong:
            for s in self.state:
                s["A"], s["B"] = s["B"], s["A"]
        return r

    def master(self):
        return [[x.cpu().numpy() for x in s["A"]] for s in self.state]


def oracle_shards(p, flat, dt, ranks):
    out = []
    for r in ranks:
        o, n = int(p["rank_offsets"][r]), int(p["rank_numels"][r])
        out.append(dict(numel=n, grad_off=o, param_off=o, master=orc.widen_16(flat[o:o + n], dt),
                        m=np.zeros(n, np.float32), v=np.zeros(n, np.float32)))
    return out


def compare(run, osh, oflat, r_gpu, r_or, exact, prev=None, red=None):
    """Bit-exact without clipping, and with clipping whenever the device's
    multiplier k equals the oracle's (the AdamW arithmetic is the same
    sequence of rounded fp32 operations on both sides).  If k differs (one
    fp32 ulp, from the last bits of the fp64 norm), fp32 state is held to rel
    2e-6 of the operands each update combines (theta_new = theta wdf - update
    and m_new = b1 m + (1-b1) g can be far smaller than their terms), v to rel
    2e-6 of itself, parameters to 1 ulp."""
    assert (r_gpu.overflow, r_gpu.applied) == (r_or.overflow, r_or.applied)
    gflat = t2u16(run.flat)
    if r_or.applied:
        assert r_gpu.grad_norm == pytest.approx(r_or.grad_norm, rel=1e-5)
        exact = exact or r_gpu.grad_mult == r_or.grad_mult
    else:
        exact = True
    if exact:
        assert np.array_equal(gflat, oflat)
    else:
        d = np.abs(gflat.astype(np.int32) - oflat.astype(np.int32))
        assert d.max() <= 1
    for i, ((th, m, v), o) in enumerate(zip(run.master(), osh)):
        if exact:
            for got, ref in ((th, o["master"]), (m, o["m"]), (v, o["v"])):
                assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))
            continue
        th_prev, m_prev = (np.abs(x.astype(np.float64)) for x in prev[i])
        g = np.abs(orc.widen_16(red[i], run.dt).astype(np.float64)) * r_or.grad_mult
        sc_th = np.maximum(th_prev + np.abs(th_prev - o["master"]), np.abs(o["master"]))
        sc_m = np.maximum(0.9 * m_prev + 0.1 * g, np.abs(o["m"]))
        for got, ref, sc in ((th, o["master"], sc_th), (m, o["m"], sc_m), (v, o["v"], np.abs(o["v"]))):
            assert np.all(np.abs(got.astype(np.float64) - ref) <= 2e-6 * np.maximum(sc, 1e-30))


def run_both(Z, numels, nd, dt, mode, seed, h, S, pingpong, steps=3, inject=None, extra=(0.0, 0), ranks=None,
             state_pad=0, param_pad=0, grad_std=1e-3, t0=1):
    p, flat, grads = make_problem(numels, nd, dt, mode, seed, loss_scale=S, grad_std=grad_std, steps=steps)
    if inject:
        inject(grads)
    ranks = list(range(nd)) if ranks is None else ranks
    run = DeviceRun(Z, p, flat, dt, ranks, pingpong, state_pad=state_pad, param_pad=param_pad)
    osh = oracle_shards(p, flat, dt, ranks)
    oflat = flat.copy()
    t, Sg, So = t0, S, S
    exact = h["max_grad_norm"] <= 0
    results = []
    for k in range(steps):
        r_gpu = run.step(grads[k], h, t, Sg, extra)
        prev = [(o["master"].copy(), o["m"].copy()) for o in osh]
        r_or, red = orc.zero_step(grads[k], dt, osh, oflat, dt, h, t, So, *extra, want_grad=True)
        compare(run, osh, oflat, r_gpu, r_or, exact, prev, red)
        results.append((r_gpu.as_dict(), r_or.as_dict()))
        if r_or.applied:
            t += 1
        else:
            Sg /= 2
            So /= 2
    return results


@pytest.mark.parametrize("dt", [1, 2])
@pytest.mark.parametrize("pingpong", [True, False])
def test_random_groups_match_oracle(Z, dt, pingpong):
    rng = np.random.default_rng(40 + dt + 2 * pingpong)
    for trial in range(6):
        nd = int(rng.choice([1, 2, 3, 4, 5, 8, 13]))
        numels = random_group(rng, 6, 40000)
        mode = int(rng.integers(0, 2))
        h = hyper32()
        S = 1024.0 if dt == 1 else 1.0
        run_both(Z, numels, nd, dt, mode, trial, h, S, pingpong)


@pytest.mark.parametrize("dt", [1, 2])
def test_clipped_two_pass_matches_oracle(Z, dt):
    rng = np.random.default_rng(7 + dt)
    for trial in range(4):
        nd = int(rng.choice([2, 3, 4, 8]))
        numels = random_group(rng, 5, 30000)
        h = hyper32(max_grad_norm=0.01)
        res = run_both(Z, numels, nd, dt, 0, 100 + trial, h, 8.0 if dt == 1 else 1.0, pingpong=bool(trial % 2),
                       grad_std=1e-2)
        assert all(g["clip_coef"] < 1.0 for g, _ in res)


def stats_tensor(Z, sumsq, overflow=0):
    """A device zero_stats holding the given sum of squares and flag."""
    return torch.frombuffer(bytearray(bytes(Z.zero_stats(sumsq, overflow, 0))), dtype=torch.uint8).to(DEV)


@pytest.mark.parametrize("dt", [1, 2])
@pytest.mark.parametrize("pingpong", [False, True])
def test_clipped_update_is_exact_given_the_oracle_norm(Z, dt, pingpong):
    """The clipped update's arithmetic alone: the reduce pass writes the
    reduced gradients and its statistics, then the statistics the apply pass
    reads are overwritten with the oracle's exactly rounded sum of squares, so
    both sides derive the multiplier k from the same fp64 number.  Every
    reduced gradient, fp32 state and 16-bit parameter must then equal the
    oracle's bit for bit, every step, with the clip firing (and the other
    ranks' share of the norm added on both sides in two of the groups)."""
    rng = np.random.default_rng(300 + dt + 2 * pingpong)
    for trial in range(3):
        nd = int(rng.choice([2, 3, 4, 8]))
        numels = random_group(rng, 5, 30000)
        S = 8.0 if dt == 1 else 1.0
        p, flat, grads = make_problem(numels, nd, dt, 0, 200 + trial, loss_scale=S, grad_std=1e-2, steps=3)
        ranks = list(range(nd))
        run = DeviceRun(Z, p, flat, dt, ranks, pingpong)
        osh = oracle_shards(p, flat, dt, ranks)
        oflat = flat.copy()
        h = hyper32(max_grad_norm=0.01)
        extra = 0.0 if trial == 0 else 0.25 * trial
        stats = torch.zeros(16, dtype=torch.uint8, device=DEV)
        for t in (1, 2, 3):
            sh = run.shards()
            Z.zero_shard_reduce([dev16(g, dt) for g in grads[t - 1]], dt, sh, 0, stats, run.ws, run.ws.numel())
            ro, red = orc.zero_step(grads[t - 1], dt, osh, oflat, dt, h, t, S, extra, 0, want_grad=True)
            acc = orc.ExactAccumulator()
            for rr in red:
                orc.stats(rr, dt, acc)
            own = acc.value()
            torch.cuda.synchronize()
            dev = Z.read_stats(stats)
            assert dev.overflow == 0 and dev.sumsq == pytest.approx(own, rel=1e-9)
            stats.copy_(stats_tensor(Z, own))
            Z.zero_shard_apply(sh, dt, run.flat, dt, Z.hyper(h["lr"], h["beta1"], h["beta2"], h["eps"],
                                                             h["weight_decay"], h["max_grad_norm"], t),
                               S, stats, extra, 0, run.ws, run.ws.numel(), run.res)
            torch.cuda.synchronize()
            rg = Z.read_result(run.res)
            assert ro.applied == 1 and ro.clip_coef < 1.0
            assert rg.grad_mult == ro.grad_mult and rg.sumsq == ro.sumsq and rg.clip_coef == ro.clip_coef
            for s_, rr in zip(run.state, red):
                assert np.array_equal(t2u16(s_["g"]), rr)
            if pingpong:
                for s_ in run.state:
                    s_["A"], s_["B"] = s_["B"], s_["A"]
            compare(run, osh, oflat, rg, ro, True)


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("pingpong", [True, False])
def test_tiny_workload_with_skip(Z, mode, pingpong):
    """Tiny fp16 workload: N_d = 3, S = 1024, +inf at flat index 30000 of rank
    0's gradient at step 2 -> step 2 skipped everywhere, S halves, t stays."""
    def inject(grads):
        grads[1][0] = grads[1][0].copy()
        grads[1][0][30000] = 0x7C00
    res = run_both(Z, W.numels(W.tiny_group()), 3, 1, mode, 0, hyper32(), 1024.0, pingpong, inject=inject)
    assert [g["applied"] for g, _ in res] == [1, 0, 1]


@pytest.mark.parametrize("bad", [0x7E00, 0xFC00])
def test_nan_and_negative_inf_skip(Z, bad):
    def inject(grads):
        grads[0][2] = grads[0][2].copy()
        grads[0][2][5] = bad
    res = run_both(Z, [3000, 5000], 4, 1, 0, 3, hyper32(), 256.0, True, steps=2, inject=inject)
    assert res[0][0]["overflow"] == 1 and res[0][0]["applied"] == 0


def test_finite_inputs_whose_sum_overflows(Z):
    big = np.uint16(0x7F61)   # bf16 ~2.99e38
    def inject(grads):
        for r in range(2):
            grads[0][r] = grads[0][r].copy()
            grads[0][r][1234] = big
    res = run_both(Z, [4096], 2, 2, 0, 5, hyper32(), 1.0, True, steps=2, inject=inject)
    assert res[0][0]["overflow"] == 1 and res[1][0]["applied"] == 1


def test_huge_finite_squares_use_fp64(Z):
    # bf16 values near 1e20: their squares exceed the fp32 range but the norm is finite
    def inject(grads):
        for r in range(2):
            grads[0][r] = grads[0][r].copy()
            grads[0][r][100:108] = 0x60AD   # ~1e20
    res = run_both(Z, [20000], 2, 2, 0, 6, hyper32(), 1.0, True, steps=1, inject=inject)
    g, o = res[0]
    assert np.isfinite(g["grad_norm"]) and g["grad_norm"] == pytest.approx(o["grad_norm"], rel=1e-6)


@pytest.mark.parametrize("nd", [1, 7, 8, 13, 64])
def test_slice_counts(Z, nd):
    # the loss scale crosses the C ABI as fp32: give the oracle that same value
    run_both(Z, [9000, 1234], nd, 1, 0, nd, hyper32(), float(np.float32(4096.0 / nd)), True, steps=2)


@pytest.mark.parametrize("dt", [1, 2])
@pytest.mark.parametrize("case", ["lr 0", "wd 0", "betas 0", "t from 1e6", "eps 1", "S 2^14", "S 2^-8"])
def test_hyperparameters_at_their_edges(Z, dt, case):
    """Bit-exact steps with the hyper-parameters at the edges of their range:
    lr = 0 (only the moments move), no weight decay, beta1 = beta2 = 0 (m = g,
    v = g^2), t starting at 10^6 (both bias corrections round to 1 in fp32),
    eps = 1, and loss scales of 2^14 and 2^-8 (gradients drawn scaled by S:
    fp16 gradients of 2^-8 are mostly subnormal)."""
    kw, S, t0 = {}, 1.0, 1
    if case == "lr 0":
        kw = dict(lr=0.0)
    elif case == "wd 0":
        kw = dict(weight_decay=0.0)
    elif case == "betas 0":
        kw = dict(beta1=0.0, beta2=0.0)
    elif case == "t from 1e6":
        t0 = 1_000_000
    elif case == "eps 1":
        kw = dict(eps=1.0)
    elif case == "S 2^14":
        S = 2.0 ** 14
    else:
        S = 2.0 ** -8
    res = run_both(Z, [20000, 4096, 333], 4, dt, 0, 70, hyper32(**kw), S, True, steps=2, t0=t0)
    assert all(g["applied"] == 1 for g, _ in res)


@pytest.mark.parametrize("dt", [1, 2])
@pytest.mark.parametrize("state_pad", [0, 1])
def test_shard_init_widens_the_parameters(Z, dt, state_pad):
    """zero_shard_init: every rank's master_in = fp32(its 16-bit parameters),
    bit for bit the oracle's widening, and m_in = v_in = 0, over a group with
    odd shard offsets (the unpadded plan), an empty rank, state pointers on
    and off 16-byte alignment, and parameters holding infinities, zeros of
    both signs and subnormals (NaN patterns need only widen to NaN)."""
    numels, nd = [20000, 4096, 7, 333], 5
    p, flat, _ = make_problem(numels, nd, dt, 1, 90, steps=1)
    flat = flat.copy()
    specials = ([0x7C00, 0xFC00, 0x7E00, 0x0001, 0x8001, 0x03FF, 0x0000, 0x8000] if dt == 1 else
                [0x7F80, 0xFF80, 0x7FC0, 0x0001, 0x8001, 0x007F, 0x0000, 0x8000])
    flat[100:108] = specials
    flat[int(p["rank_offsets"][3]):int(p["rank_offsets"][3]) + 8] = specials
    fdev = dev16(flat, dt)
    ranks = list(range(nd)) + [nd]       # plus an empty shard
    shards, state = [], []
    for r in ranks:
        o = int(p["rank_offsets"][r]) if r < nd else 0
        n = int(p["rank_numels"][r]) if r < nd else 0
        bufs = [torch.full((n + state_pad,), float("nan"), device=DEV)[state_pad:] for _ in range(3)]
        shards.append(Z.shard(n, o, o, *bufs, *bufs))
        state.append((o, n, bufs))
    Z.zero_shard_init(shards, fdev, dt)
    torch.cuda.synchronize()
    for o, n, (m0, m1, m2) in state:
        want = orc.widen_16(flat[o:o + n], dt)
        got = m0.cpu().numpy()
        nan = np.isnan(want)
        assert np.array_equal(np.isnan(got), nan)
        assert np.array_equal(got[~nan].view(np.uint32), want[~nan].view(np.uint32))
        for z in (m1, m2):
            assert np.array_equal(z.cpu().numpy().view(np.uint32), np.zeros(n, np.uint32))
    assert torch.equal(fdev.view(torch.int16), dev16(flat, dt).view(torch.int16))     # parameters untouched


def test_unaligned_pointers_take_the_scalar_path(Z):
    # state views 1 float into their buffers and a flat parameter buffer 1 element in: not 16-byte aligned
    run_both(Z, [5000, 77], 3, 2, 0, 8, hyper32(), 1.0, True, state_pad=1, param_pad=1, steps=2)
    run_both(Z, [5000, 77], 3, 1, 1, 9, hyper32(), 512.0, False, state_pad=1, param_pad=3, steps=2)


@pytest.mark.parametrize("dt", [1, 2])
@pytest.mark.parametrize("pads", [(4, 4, 4, 4, 4, 4), (0, 0, 4, 0, 0, 0), (0, 0, 0, 0, 0, 12), (8, 8, 8, 8, 8, 8),
                                  (32, 8, 24, 16, 8, 0)])
def test_state_on_16_and_32_byte_boundaries(Z, dt, pads):
    """The apply pass moves a vector's 8 values of each state array in one
    256-bit access when, in every shard, all six arrays are 32-byte aligned
    and the gradient stream starts on a 128-byte line (the last case: master
    128 bytes into its buffer, the others at other multiples of 32), else in
    two 128-bit accesses (arrays 16 bytes past a 32-byte boundary, all six or
    only one; all six 32 bytes in, which puts the gradient stream off its
    line).
    Neither may change a bit, on the reduce + apply passes with the state in
    place (clipping on); the fused pass (ping-pong state) runs on the same
    layouts."""
    S = 512.0 if dt == 1 else 1.0
    numels = [5000, 77, 40000]
    run_both(Z, numels, 3, dt, 0, 60 + sum(pads) + dt, hyper32(), S, True, steps=2, state_pad=pads)
    run_both(Z, numels, 3, dt, 0, 61 + sum(pads) + dt, hyper32(max_grad_norm=0.01), S, False, steps=2,
             state_pad=pads[:3] * 2, grad_std=1e-2)


def test_empty_shards_and_no_shards(Z):
    run_both(Z, [3], 8, 2, 1, 11, hyper32(), 1.0, True, steps=2)      # ranks 3..7 own nothing
    ws = torch.zeros(Z.zero_workspace_bytes(), dtype=torch.uint8, device=DEV)
    res = torch.zeros(48, dtype=torch.uint8, device=DEV)
    g = torch.zeros(16, dtype=torch.bfloat16, device=DEV)
    Z.zero_shard_step([g], Z.ZERO_BF16, [], None, Z.ZERO_BF16, Z.hyper(), 1.0, 2.25, 0, ws, ws.numel(), res)
    torch.cuda.synchronize()
    r = Z.read_result(res)
    assert r.applied == 1 and r.sumsq == 2.25 and r.grad_norm == 1.5


def test_rank_local_view_with_other_ranks_statistics(Z):
    numels = [30000, 999]
    nd, dt = 4, 2
    p, flat, grads = make_problem(numels, nd, dt, 0, 12, steps=3)
    r = 1
    o, n = int(p["rank_offsets"][r]), int(p["rank_numels"][r])
    staged = [[g[o:o + n].copy() for g in step] for step in grads]   # the 4 slices staged for rank 1
    h = hyper32(max_grad_norm=0.02)
    run = DeviceRun(Z, p, flat, dt, [r], pingpong=False)
    osh = oracle_shards(p, flat, dt, [r])
    osh[0]["grad_off"] = 0
    oflat = flat.copy()
    extra = (0.37, 0)
    for t in (1, 2, 3):
        rg = run.step(staged[t - 1], h, t, 1.0, extra, grad_offsets=[0])
        prev = [(o["master"].copy(), o["m"].copy()) for o in osh]
        ro, red = orc.zero_step(staged[t - 1], dt, osh, oflat, dt, h, t, 1.0, *extra, want_grad=True)
        compare(run, osh, oflat, rg, ro, False, prev, red)
        outside = np.concatenate([t2u16(run.flat)[:o], t2u16(run.flat)[o + n:]])
        assert np.array_equal(outside, np.concatenate([flat[:o], flat[o + n:]]))   # other ranks' slots untouched
    rg = run.step(staged[0], h, 4, 1.0, (0.0, 1))
    assert rg.overflow == 1 and rg.applied == 0


def test_reduce_and_apply_separately_accumulate(Z):
    """Two reduce calls (accumulate 0 then 1) over two halves of the shards,
    then one apply: same as the oracle's single step."""
    numels = [40000, 333]
    nd, dt = 3, 1
    p, flat, grads = make_problem(numels, nd, dt, 0, 13, loss_scale=64.0, steps=1)
    run = DeviceRun(Z, p, flat, dt, list(range(nd)), pingpong=False)
    slices = [dev16(g, dt) for g in grads[0]]
    sh = run.shards()
    stats = torch.zeros(16, dtype=torch.uint8, device=DEV)
    Z.zero_shard_reduce(slices, dt, sh[:1], 0, stats, run.ws, run.ws.numel())
    Z.zero_shard_reduce(slices, dt, sh[1:], 1, stats, run.ws, run.ws.numel())
    h = hyper32(max_grad_norm=5.0)
    Z.zero_shard_apply(sh, dt, run.flat, dt, Z.hyper(h["lr"], h["beta1"], h["beta2"], h["eps"], h["weight_decay"],
                                                     h["max_grad_norm"], 1), 64.0, stats, 0.0, 0, run.ws, run.ws.numel(),
                       run.res)
    torch.cuda.synchronize()
    osh = oracle_shards(p, flat, dt, list(range(nd)))
    oflat = flat.copy()
    prev = [(o["master"].copy(), o["m"].copy()) for o in osh]
    ro, red = orc.zero_step(grads[0], dt, osh, oflat, dt, h, 1, 64.0, want_grad=True)
    for s, rr in zip(run.state, red):
        assert np.array_equal(t2u16(s["g"]), rr)            # reduced gradients bit-exact
    st = Z.read_stats(stats)
    assert st.overflow == 0 and st.sumsq == pytest.approx(ro.sumsq, rel=1e-6)
    compare(run, osh, oflat, Z.read_result(run.res), ro, False, prev, red)


def test_deterministic(Z):
    numels = [200000]
    p, flat, grads = make_problem(numels, 8, 2, 0, 14, steps=1)
    outs = []
    for _ in range(2):
        run = DeviceRun(Z, p, flat, 2, list(range(8)), pingpong=True)
        r = run.step(grads[0], hyper32(), 1, 1.0)
        outs.append((r.sumsq, t2u16(run.flat)))
    assert outs[0][0] == outs[1][0] and np.array_equal(outs[0][1], outs[1][1])


def _staged_rank_local(Z, numel, nd, dt, param_off, clip, steps=3, seed=21, S=1.0):
    """Rank-local view (staged slices, gradient offset 0): slices and state
    16-byte aligned, so the vector passes run; param_off sets the parameter
    slot's alignment (16-, 4- or 2-byte stores)."""
    total = param_off + numel + 5
    p = {"rank_offsets": np.array([param_off]), "rank_numels": np.array([numel])}
    flat = np.zeros(total, np.uint16)
    g = W.generator(seed, "cpu")
    ft = torch.zeros(total, dtype=TDT[dt])
    W.fill_normal_(ft, 0.02, g)
    flat[:] = t2u16(ft)
    gens = [W.generator(seed + 1 + j, "cpu") for j in range(nd)]
    h = hyper32(max_grad_norm=clip)
    run = DeviceRun(Z, p, flat, dt, [0], pingpong=(clip == 0.0))
    osh = oracle_shards(p, flat, dt, [0])
    osh[0]["grad_off"] = 0
    oflat = flat.copy()
    paths = []
    for t in range(1, steps + 1):
        staged = []
        for j in range(nd):
            x = torch.zeros(numel, dtype=TDT[dt])
            W.fill_normal_(x, 1e-2, gens[j], S)
            staged.append(t2u16(x))
        rg = run.step(staged, h, t, S, grad_offsets=[0])
        prev = [(o["master"].copy(), o["m"].copy()) for o in osh]
        ro, red = orc.zero_step(staged, dt, osh, oflat, dt, h, t, S, want_grad=True)
        compare(run, osh, oflat, rg, ro, clip <= 0.0, prev, red)
        paths.append(rg.path)
    return paths


@pytest.mark.parametrize("dt", [1, 2])
@pytest.mark.parametrize("numel,param_off,nd", [(1024, 0, 4), (123457, 8, 4), (123457, 3, 8), (5000, 6, 1),
                                               (7, 0, 2), (2049, 2, 8), (1792 * 7 + 5, 8, 8), (300001, 0, 3),
                                               (2048 * 3, 4, 12)])
def test_rank_local_ragged_and_unaligned_params(Z, dt, numel, param_off, nd):
    """Rank-local shards of exact tile multiples, ragged tails, shards shorter
    than one vector, parameter slots at every alignment, 1-12 slices: the
    fused pass (path 1) bit-exact against the oracle, and the reduce + apply
    passes (path 2, clipping on) within the step's tolerances."""
    S = 256.0 if dt == 1 else 1.0
    assert set(_staged_rank_local(Z, numel, nd, dt, param_off, 0.0, S=S)) == {1}
    assert set(_staged_rank_local(Z, numel, nd, dt, param_off, 0.05, S=S)) == {2}


def test_stage1_full_allreduce_then_shard_update(Z):
    """Stage 1 without reduce-scatter: the reduce pass writes the whole
    averaged gradient into one buffer (every rank's copy of the all-reduce),
    then each shard is updated from its slice of it."""
    numels = [33333, 2222, 4444]
    nd, dt = 4, 2
    p, flat, grads = make_problem(numels, nd, dt, 0, 41, steps=2)
    P = p["padded_total"]
    run = DeviceRun(Z, p, flat, dt, list(range(nd)), pingpong=False, want_grad=False)
    avg = torch.empty(P, dtype=torch.bfloat16, device=DEV)
    for s_, o, n in zip(run.state, p["rank_offsets"], p["rank_numels"]):
        s_["g"] = avg[int(o):int(o) + int(n)]
    osh = oracle_shards(p, flat, dt, list(range(nd)))
    oflat = flat.copy()
    stats = torch.zeros(16, dtype=torch.uint8, device=DEV)
    h = hyper32()
    for t in (1, 2):
        slices = [dev16(g, dt) for g in grads[t - 1]]
        sh = run.shards()
        Z.zero_shard_reduce(slices, dt, sh, 0, stats, run.ws, run.ws.numel())
        Z.zero_shard_apply(sh, dt, run.flat, dt, Z.hyper(h["lr"], h["beta1"], h["beta2"], h["eps"],
                                                         h["weight_decay"], 0.0, t), 1.0, stats, 0.0, 0, run.ws,
                           run.ws.numel(), run.res)
        torch.cuda.synchronize()
        assert np.array_equal(t2u16(avg), orc.reduce(grads[t - 1], dt, 0, P))     # the full all-reduce
        ro, _ = orc.zero_step(grads[t - 1], dt, osh, oflat, dt, h, t, 1.0)
        compare(run, osh, oflat, Z.read_result(run.res), ro, True)


@pytest.mark.parametrize("dt", [1, 2])
@pytest.mark.parametrize("total,nd", [(48, 2), (80, 2), (4096 + 48, 2), (3 * 8 * 1000 + 24, 3), (64 * 1024 + 16, 4)])
def test_unaligned_shard_heads(Z, dt, total, nd):
    """Shards that start 16 bytes past a 128-byte line: the passes take a head
    of up to 63 elements one by one so the vector loop starts aligned; heads
    shorter than, equal to and longer than the shard, on the fused and the
    two-pass path, must not change a bit."""
    S = 512.0 if dt == 1 else 1.0
    run_both(Z, [total], nd, dt, 0, total + nd, hyper32(), S, True, steps=2)
    run_both(Z, [total], nd, dt, 0, total + nd, hyper32(max_grad_norm=0.01), S, False, steps=2, grad_std=1e-2)


@pytest.mark.parametrize("gdt,pdt", [(2, 1), (1, 2)])
@pytest.mark.parametrize("clip", [0.0, 0.05])
def test_mixed_gradient_and_parameter_dtypes(Z, gdt, pdt, clip):
    """bf16 gradients with fp16 parameters and the reverse: the reduce rounds
    to the gradient dtype, the store to the parameter dtype."""
    numels = [20000, 555]
    nd = 4
    p = orc.plan(numels, nd, 0)
    P = p["padded_total"]
    specs = [W.ParamSpec(f"t{i}", n) for i, n in enumerate(numels)]
    ft = torch.zeros(P, dtype=TDT[pdt])
    W.init_params_(ft, specs, W.generator(7, "cpu"))
    flat = t2u16(ft)
    gens = [W.generator(8 + r, "cpu") for r in range(nd)]
    S = 64.0 if gdt == 1 else 1.0
    grads = [[t2u16(W.fill_grad_(torch.zeros(P, dtype=TDT[gdt]), specs, gens[r], lambda s: 1e-2, S))
              for r in range(nd)] for _ in range(2)]
    h = hyper32(max_grad_norm=clip)
    dflat = dev16(flat, pdt)
    st = []
    for o, n in zip(p["rank_offsets"], p["rank_numels"]):
        o, n = int(o), int(n)
        A = [dflat[o:o + n].float(), torch.zeros(n, device=DEV), torch.zeros(n, device=DEV)]
        B = [torch.empty(n, device=DEV) for _ in range(3)] if clip == 0.0 else A
        st.append(dict(o=o, n=n, A=A, B=B, g=torch.empty(n, dtype=TDT[gdt], device=DEV)))
    osh = [dict(numel=s_["n"], grad_off=s_["o"], param_off=s_["o"], master=orc.widen_16(flat[s_["o"]:s_["o"] + s_["n"]], pdt),
                m=np.zeros(s_["n"], np.float32), v=np.zeros(s_["n"], np.float32)) for s_ in st]
    oflat = flat.copy()
    ws = torch.zeros(Z.zero_workspace_bytes(), dtype=torch.uint8, device=DEV)
    res = torch.zeros(48, dtype=torch.uint8, device=DEV)
    for t in (1, 2):
        sh = [Z.shard(s_["n"], s_["o"], s_["o"], *s_["A"], *s_["B"], s_["g"]) for s_ in st]
        Z.zero_shard_step([dev16(g, gdt) for g in grads[t - 1]], gdt, sh, dflat, pdt,
                          Z.hyper(h["lr"], h["beta1"], h["beta2"], h["eps"], h["weight_decay"], h["max_grad_norm"], t),
                          S, 0.0, 0, ws, ws.numel(), res)
        torch.cuda.synchronize()
        rg = Z.read_result(res)
        prev = [(o["master"].copy(), o["m"].copy()) for o in osh]
        ro, red = orc.zero_step(grads[t - 1], gdt, osh, oflat, pdt, h, t, S, want_grad=True)
        assert (rg.overflow, rg.applied) == (ro.overflow, ro.applied) == (0, 1)
        if clip == 0.0:
            for s_ in st:
                s_["A"], s_["B"] = s_["B"], s_["A"]
        got_flat = t2u16(dflat)
        exact = clip == 0.0 or rg.grad_mult == ro.grad_mult       # the same k: the same rounded operations
        if exact:
            assert np.array_equal(got_flat, oflat)
        else:
            assert np.abs(got_flat.astype(np.int32) - oflat.astype(np.int32)).max() <= 1
        for s_, o, pv, rd in zip(st, osh, prev, red):
            if clip != 0.0:
                assert np.array_equal(t2u16(s_["g"]), rd)
            if exact:
                for x, ref in zip(s_["A"], (o["master"], o["m"], o["v"])):
                    assert np.array_equal(x.cpu().numpy().view(np.uint32), ref.view(np.uint32))
            else:
                th_prev = np.abs(pv[0].astype(np.float64))
                sc = np.maximum(th_prev + np.abs(th_prev - o["master"]), np.abs(o["master"]))
                assert np.all(np.abs(s_["A"][0].cpu().numpy().astype(np.float64) - o["master"]) <= 2e-6 * np.maximum(sc, 1e-30))


@pytest.mark.parametrize("clip", [0.0, 0.05])
def test_step_captured_in_a_cuda_graph(Z, clip):
    """The step enqueues only kernels on the caller's stream (no allocation,
    no synchronisation), so a call can be captured into a CUDA graph and
    replayed: the replay must equal the same call made eagerly."""
    numels = [70000, 123]
    nd, dt = 3, 2
    p, flat, grads = make_problem(numels, nd, dt, 0, 51, steps=1)
    h = hyper32(max_grad_norm=clip)
    outs = []
    for mode in ("eager", "graph"):
        run = DeviceRun(Z, p, flat, dt, list(range(nd)), pingpong=(clip == 0.0))
        slices = [dev16(g, dt) for g in grads[0]]
        hy = Z.hyper(h["lr"], h["beta1"], h["beta2"], h["eps"], h["weight_decay"], h["max_grad_norm"], 1)
        sh = run.shards()
        if mode == "eager":
            Z.zero_shard_step(slices, dt, sh, run.flat, dt, hy, 1.0, 0.0, 0, run.ws, run.ws.numel(), run.res)
        else:
            # one eager call on scratch copies first, so the library's one-time per-kernel set-up is done
            warm = DeviceRun(Z, p, flat, dt, list(range(nd)), pingpong=(clip == 0.0))
            Z.zero_shard_step(slices, dt, warm.shards(), warm.flat, dt, hy, 1.0, 0.0, 0, warm.ws, warm.ws.numel(),
                              warm.res)
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            s = torch.cuda.Stream()
            with torch.cuda.graph(g, stream=s):
                Z.zero_shard_step(slices, dt, sh, run.flat, dt, hy, 1.0, 0.0, 0, run.ws, run.ws.numel(), run.res)
            g.replay()
        torch.cuda.synchronize()
        r = Z.read_result(run.res)
        state = run.state[0]["B"] if clip == 0.0 else run.state[0]["A"]
        outs.append((t2u16(run.flat), [x.cpu().numpy() for x in state], r.as_dict()))
    assert np.array_equal(outs[0][0], outs[1][0])
    for a, b in zip(outs[0][1], outs[1][1]):
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    assert outs[0][2] == outs[1][2]
