"""GPU parity of chained steps: the step's bookkeeping (t, the loss scale, the
state set in use) kept on the device by zero_shard_step_chained, against the
CPU oracle driven with the same bookkeeping on the host (an overflowing step
is skipped: t is not advanced and S halves), eagerly and replayed from a
CUDA graph.  Unclipped steps are bit-exact; clipped ones too whenever every
step's multiplier k equals the oracle's (k comes from an fp64 norm whose
last bits may differ), else they follow the step's tolerances."""
import numpy as np
import pytest
import torch

import oracle as orc
from helpers import hyper32, make_problem, t2u16

pytestmark = pytest.mark.gpu

DEV = "cuda"
TDT = {1: torch.float16, 2: torch.bfloat16}


@pytest.fixture(scope="module")
def Z():
    import zero_dp_partitioned_gb300 as Z
    return Z


def dev16(a, dt):
    return torch.from_numpy(a.view(np.int16).copy()).view(TDT[dt]).to(DEV)


def chain_tensor(Z, step, S, min_loss_scale=0.0):
    c = Z.chain(step=step, loss_scale=S, min_loss_scale=min_loss_scale)
    return torch.frombuffer(bytearray(bytes(c)), dtype=torch.uint8).to(DEV)


class ChainRun:
    """Device copy of a problem with two state sets and a device chain."""

    def __init__(self, Z, p, flat, dt, h, S, n_table=16, min_loss_scale=0.0):
        self.Z, self.p, self.dt, self.h = Z, p, dt, h
        P = flat.size
        self.flat = dev16(flat, dt)
        self.sets = [[torch.empty(P, device=DEV) for _ in range(3)] for _ in range(2)]
        self.gshard = torch.empty(P, dtype=TDT[dt], device=DEV)
        self.chain = chain_tensor(Z, 1, S, min_loss_scale)
        self.hyper = Z.hyper(h["lr"], h["beta1"], h["beta2"], h["eps"], h["weight_decay"], h["max_grad_norm"], 1)
        self.table = torch.from_numpy(Z.zero_adam_scalar_table(self.hyper, 1, n_table)).to(DEV)
        self.n_table = n_table
        self.ws = torch.zeros(Z.zero_workspace_bytes(), dtype=torch.uint8, device=DEV)
        self.res = torch.zeros(48, dtype=torch.uint8, device=DEV)
        A, B = self.sets
        self.shards = [Z.shard(int(n), int(o), int(o), *(x[int(o):int(o) + int(n)] for x in A),
                               *(x[int(o):int(o) + int(n)] for x in B), self.gshard[int(o):int(o) + int(n)])
                       for o, n in zip(p["rank_offsets"], p["rank_numels"])]
        Z.zero_shard_init(self.shards, self.flat, dt)     # master = fp32(parameters), m = v = 0

    def step(self, slices_dev, stream=None, res=None):
        self.Z.zero_shard_step_chained(slices_dev, self.dt, self.shards, self.flat, self.dt, self.hyper, self.table, 1,
                                       self.n_table, self.chain, 0.0, 0, self.ws, self.ws.numel(),
                                       self.res if res is None else res, stream=stream)

    def state(self):
        c = self.Z.read_chain(self.chain)
        return c, [x.cpu().numpy() for x in self.sets[c.cur]]


def oracle_run(p, flat, dt, h, S, grads):
    """The oracle over the same steps with the host bookkeeping."""
    osh = [dict(numel=int(n), grad_off=int(o), param_off=int(o), master=orc.widen_16(flat[int(o):int(o) + int(n)], dt),
                m=np.zeros(int(n), np.float32), v=np.zeros(int(n), np.float32))
           for o, n in zip(p["rank_offsets"], p["rank_numels"])]
    oflat = flat.copy()
    t, results = 1, []
    for g in grads:
        r, _ = orc.zero_step(g, dt, osh, oflat, dt, h, t, np.float32(S))
        results.append(r)
        if r.applied:
            t += 1
        else:
            S /= 2
    return osh, oflat, t, S, results


def check(run, p, osh, oflat, exact):
    c, (th, m, v) = run.state()
    got_flat = t2u16(run.flat)
    if exact:
        assert np.array_equal(got_flat, oflat)
    else:
        assert np.abs(got_flat.astype(np.int32) - oflat.astype(np.int32)).max() <= 1
    for o, n, os_ in zip(p["rank_offsets"], p["rank_numels"], osh):
        o, n = int(o), int(n)
        for got, ref in ((th[o:o + n], os_["master"]), (m[o:o + n], os_["m"]), (v[o:o + n], os_["v"])):
            if exact:
                assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))
            else:
                # the clipped multiplier may differ by an ulp in a step (fp64 norm, summed in another order):
                # 1e-5 relative, with a floor of 1e-3 of the array's largest value where the update cancels
                ref64 = ref.astype(np.float64)
                floor = 1e-3 * np.abs(ref64).max()
                assert np.all(np.abs(got.astype(np.float64) - ref64) <= 1e-5 * np.maximum(np.abs(ref64), floor))
    return c


# aligned: 16-byte vectors; misaligned: one element at a time; 12 slices: the many-slice loop
@pytest.mark.parametrize("numels,nd,dt", [([20000, 4096, 992], 4, 2), ([20000, 555], 3, 1), ([3000, 5000], 8, 2),
                                          ([24000, 576], 12, 2)])
@pytest.mark.parametrize("clip", [0.0, 0.05])
def test_chained_steps_match_the_oracle(Z, numels, nd, dt, clip):
    """Five chained steps, the second with a NaN in one slice (skipped: t stays,
    S halves), no host synchronisation in between; each step writes its own
    result slot, read after the last."""
    S = 256.0 if dt == 1 else 1.0
    p, flat, grads = make_problem(numels, nd, dt, 0, 61, loss_scale=S, grad_std=1e-2, steps=5)
    grads[1][0] = grads[1][0].copy()
    grads[1][0][7] = 0x7E00 if dt == 1 else 0x7FC0
    h = hyper32(max_grad_norm=clip)
    run = ChainRun(Z, p, flat, dt, h, S)
    slices = [[dev16(g, dt) for g in step] for step in grads]
    res = torch.zeros(5, 48, dtype=torch.uint8, device=DEV)
    for k in range(5):
        run.step(slices[k], res=res[k])
    torch.cuda.synchronize()
    osh, oflat, t, So, results = oracle_run(p, flat, dt, h, S, grads)
    assert [r.applied for r in results] == [1, 0, 1, 1, 1]
    rg = [Z.read_result(res[k]) for k in range(5)]
    assert [r.applied for r in rg] == [1, 0, 1, 1, 1]
    same_k = all(a.grad_mult == b.grad_mult for a, b in zip(rg, results) if b.applied)
    c = check(run, p, osh, oflat, clip <= 0.0 or same_k)
    assert (c.step, c.loss_scale, c.applied, c.skipped, c.failed) == (t, So, 4, 1, 0)
    r = rg[-1]
    assert r.applied == 1 and r.status == 0 and r.path == (1 if clip <= 0.0 else 2)


@pytest.mark.parametrize("floor", [0.5, 0.0])
def test_chained_loss_scale_stops_at_its_floor(Z, floor):
    """Overflow after overflow: S halves while S / 2 stays at or above the
    chain's floor (0.5 here; 2^-126 when none is given), then stays, and the
    skipped steps at the floor count as failed; the state and parameters never
    change, and the next finite step is applied at the floor's S."""
    numels, nd, dt = [4096, 100], 2, 2
    S0 = 1.0 if floor > 0 else 2.0 ** -124
    p, flat, grads = make_problem(numels, nd, dt, 0, 65, loss_scale=S0, steps=5)
    for k in range(4):
        grads[k][1] = grads[k][1].copy()
        grads[k][1][3] = 0x7F80                         # +inf in rank 1's slice: steps 1-4 overflow
    run = ChainRun(Z, p, flat, dt, hyper32(), S0, min_loss_scale=floor)
    before = t2u16(run.flat)
    slices = [[dev16(g, dt) for g in step] for step in grads]
    for k in range(4):
        run.step(slices[k])
    torch.cuda.synchronize()
    c, _ = run.state()
    S_floor = 0.5 if floor > 0 else 2.0 ** -126
    assert c.loss_scale == S_floor and c.step == 1 and c.applied == 0
    assert (c.skipped, c.failed) == ((1, 3) if floor > 0 else (2, 2))
    assert np.array_equal(t2u16(run.flat), before)
    run.step(slices[4])
    torch.cuda.synchronize()
    c, _ = run.state()
    r = Z.read_result(run.res)
    assert r.applied == 1 and c.applied == 1 and c.step == 2 and c.loss_scale == S_floor
    assert np.isfinite(r.grad_norm)


@pytest.mark.parametrize("clip", [0.0, 0.05])
def test_chained_steps_replayed_from_a_cuda_graph(Z, clip):
    """Three chained steps captured in one CUDA graph and replayed twice equal
    six eager chained steps from the same start, bit for bit."""
    numels, nd, dt = [20000, 4096, 992], 4, 2
    p, flat, grads = make_problem(numels, nd, dt, 0, 62, grad_std=1e-2, steps=3)
    h = hyper32(max_grad_norm=clip)
    slices = [[dev16(g, dt) for g in step] for step in grads]
    eager = ChainRun(Z, p, flat, dt, h, 1.0)
    for _ in range(2):
        for k in range(3):
            eager.step(slices[k])
    graphed = ChainRun(Z, p, flat, dt, h, 1.0)
    warm = ChainRun(Z, p, flat, dt, h, 1.0)          # the library's one-time set-up, outside the capture
    warm.step(slices[0])
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.graph(g, stream=s):
        for k in range(3):
            graphed.step(slices[k])
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    ce, se = eager.state()
    cg, sg = graphed.state()
    assert ce.as_dict() == cg.as_dict() and ce.step == 7
    assert torch.equal(eager.flat.view(torch.int16), graphed.flat.view(torch.int16))
    for a, b in zip(se, sg):
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_chained_step_outside_its_table_changes_nothing(Z):
    numels, nd, dt = [20000, 4096, 992], 4, 2
    p, flat, grads = make_problem(numels, nd, dt, 0, 63, grad_std=1e-2, steps=3)
    h = hyper32()
    run = ChainRun(Z, p, flat, dt, h, 1.0, n_table=2)
    slices = [[dev16(g, dt) for g in step] for step in grads]
    run.step(slices[0])
    run.step(slices[1])
    torch.cuda.synchronize()
    c2, s2 = run.state()
    f2 = t2u16(run.flat)
    run.step(slices[2])
    torch.cuda.synchronize()
    c3, s3 = run.state()
    r = Z.read_result(run.res)
    assert r.applied == 0 and r.status == Z.ZERO_ELIMIT
    assert (c3.step, c3.cur, c3.applied, c3.failed) == (3, c2.cur, 2, 1)
    assert np.array_equal(t2u16(run.flat), f2)
    for a, b in zip(s2, s3):
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_chained_step_argument_errors(Z):
    numels, nd, dt = [4096], 2, 2
    p, flat, grads = make_problem(numels, nd, dt, 0, 64, steps=1)
    run = ChainRun(Z, p, flat, dt, hyper32(), 1.0)
    slices = [dev16(g, dt) for g in grads[0]]
    inplace = [Z.shard(s.numel, s.grad_offset, s.param_offset, s.master_in, s.m_in, s.v_in, s.master_in, s.m_in,
                       s.v_in) for s in run.shards]
    for kw, code in ((dict(shards=inplace), Z.ZERO_EINVAL), (dict(chain_dev=0), Z.ZERO_EINVAL),
                     (dict(n_table=0), Z.ZERO_EINVAL), (dict(table=0), Z.ZERO_EINVAL)):
        args = dict(shards=run.shards, chain_dev=run.chain, n_table=run.n_table, table=run.table)
        args.update(kw)
        with pytest.raises(Z.ZeroError) as e:
            Z.zero_shard_step_chained(slices, dt, args["shards"], run.flat, dt, run.hyper, args["table"], 1,
                                      args["n_table"], args["chain_dev"], 0.0, 0, run.ws, run.ws.numel(), run.res)
        assert e.value.code == code


@pytest.mark.parametrize("inplace", [True, False])
@pytest.mark.parametrize("clip", [0.0, 0.05])
def test_chained_apply_after_reduce_matches_the_oracle(Z, inplace, clip):
    """zero_shard_reduce, then zero_shard_apply_chained: five steps, the second
    with a NaN in one slice, no host synchronisation in between, each step's
    result in its own slot.  The chain advances t, halves S on the skipped
    step and flips its current set; the state is updated in place (the apply
    pass writes nothing on a skipped step) or between two sets.  Bit-exact
    against the oracle driven with the same bookkeeping on the host whenever
    every step's multiplier k equals the oracle's."""
    numels, nd, dt = [20000, 4096, 992], 4, 2
    S = 1.0
    p, flat, grads = make_problem(numels, nd, dt, 0, 66, loss_scale=S, grad_std=1e-2, steps=5)
    grads[1][2] = grads[1][2].copy()
    grads[1][2][11] = 0x7FC0
    h = hyper32(max_grad_norm=clip)
    run = ChainRun(Z, p, flat, dt, h, S)
    A, B = run.sets
    shards = [Z.shard(int(n), int(o), int(o), *(x[int(o):int(o) + int(n)] for x in A),
                      *(x[int(o):int(o) + int(n)] for x in (A if inplace else B)),
                      run.gshard[int(o):int(o) + int(n)])
              for o, n in zip(p["rank_offsets"], p["rank_numels"])]
    slices = [[dev16(g, dt) for g in step] for step in grads]
    stats = torch.zeros(16, dtype=torch.uint8, device=DEV)
    res = torch.zeros(5, 48, dtype=torch.uint8, device=DEV)
    for k in range(5):
        Z.zero_shard_reduce(slices[k], dt, shards, 0, stats, run.ws, run.ws.numel())
        Z.zero_shard_apply_chained(shards, dt, run.flat, dt, run.hyper, run.table, 1, run.n_table, run.chain, stats,
                                   0.0, 0, run.ws, run.ws.numel(), res[k])
    torch.cuda.synchronize()
    osh, oflat, t, So, results = oracle_run(p, flat, dt, h, S, grads)
    rg = [Z.read_result(res[k]) for k in range(5)]
    assert [r.applied for r in rg] == [r.applied for r in results] == [1, 0, 1, 1, 1]
    assert all(r.path == 2 and r.status == 0 for r in rg)
    c = Z.read_chain(run.chain)
    assert (c.step, c.loss_scale, c.applied, c.skipped, c.failed, c.cur) == (t, So, 4, 1, 0, 0)
    exact = all(a.grad_mult == b.grad_mult for a, b in zip(rg, results) if b.applied)
    got_flat = t2u16(run.flat)
    state = A if inplace else run.sets[c.cur]           # four applied steps: the set read first is current again
    if exact:
        assert np.array_equal(got_flat, oflat)
    else:
        assert np.abs(got_flat.astype(np.int32) - oflat.astype(np.int32)).max() <= 1
    for o, n, os_ in zip(p["rank_offsets"], p["rank_numels"], osh):
        o, n = int(o), int(n)
        for x, ref in zip(state, (os_["master"], os_["m"], os_["v"])):
            got = x[o:o + n].cpu().numpy()
            if exact:
                assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))
            else:
                assert np.allclose(got, ref, rtol=1e-5, atol=1e-3 * np.abs(ref).max())


def test_chained_apply_argument_errors(Z):
    numels, nd, dt = [4096], 2, 2
    p, flat, grads = make_problem(numels, nd, dt, 0, 67, steps=1)
    run = ChainRun(Z, p, flat, dt, hyper32(), 1.0)
    stats = torch.zeros(16, dtype=torch.uint8, device=DEV)
    for kw in (dict(chain=0), dict(table=0), dict(n_table=0), dict(stats=0), dict(res=run.res[4:])):
        args = dict(chain=run.chain, table=run.table, n_table=run.n_table, stats=stats, res=run.res)
        args.update(kw)
        with pytest.raises(Z.ZeroError) as e:
            Z.zero_shard_apply_chained(run.shards, dt, run.flat, dt, run.hyper, args["table"], 1, args["n_table"],
                                       args["chain"], args["stats"], 0.0, 0, run.ws, run.ws.numel(), args["res"])
        assert e.value.code == Z.ZERO_EINVAL


def test_chained_zero3_step_replayed_from_a_cuda_graph(Z):
    """A chained ZeRO-3 step -- every unit gathered forward and backward by the
    TMA gather, every unit's bucket reduced onto rank 1's part, then the
    chained apply -- has no host round trip, so steps can be captured into a
    CUDA graph: two steps captured and the graph replayed twice equal four
    eager steps from the same start, bit for bit (parameters, state, chain,
    the last gathered unit, the gathers' status word)."""
    import workloads as W
    nd, dt, me = 4, 2, 1
    units = [8192 * 4, 30000 * 4, 4096 * 4 + 64]
    parts = [u // nd for u in units]
    uoff = [sum(parts[:i]) for i in range(len(parts))]
    L = sum(parts)
    h = hyper32()

    def make():
        gen = W.generator(91, DEV)
        rsh = [W.fill_normal_(torch.empty(L, dtype=torch.bfloat16, device=DEV), 0.02, gen) for _ in range(nd)]
        bk = [[W.fill_normal_(torch.empty(u, dtype=torch.bfloat16, device=DEV), 1e-2, gen) for _ in range(nd)]
              for u in units]
        st = [torch.empty(L, device=DEV) for _ in range(3)]
        g = torch.empty(L, dtype=torch.bfloat16, device=DEV)
        sh = [Z.shard(L, 0, 0, *st, grad_shard=g)]
        Z.zero_shard_init(sh, rsh[me], dt)
        hy = Z.hyper(h["lr"], h["beta1"], h["beta2"], h["eps"], h["weight_decay"], 0.0, 1)
        return dict(rsh=rsh, bk=bk, st=st, g=g, sh=sh, hy=hy,
                    table=torch.from_numpy(Z.zero_adam_scalar_table(hy, 1, 16)).to(DEV),
                    chain=chain_tensor(Z, 1, 1.0), layer=torch.empty(max(units), dtype=torch.bfloat16, device=DEV),
                    status=torch.zeros(1, dtype=torch.int32, device=DEV),
                    ws=torch.zeros(Z.zero_workspace_bytes(), dtype=torch.uint8, device=DEV),
                    stats=torch.zeros(16, dtype=torch.uint8, device=DEV),
                    res=torch.zeros(48, dtype=torch.uint8, device=DEV))

    def step(x):
        for u in list(range(len(units))) + list(reversed(range(len(units)))):
            Z.zero3_gather_bulk([x["rsh"][r][uoff[u]:uoff[u] + parts[u]] for r in range(nd)], [parts[u]] * nd, dt,
                                x["layer"], 0, x["status"])
        for k, u in enumerate(reversed(range(len(units)))):
            Z.zero3_reduce_bucket(x["bk"][u], me, units[u], dt, x["g"][uoff[u]:uoff[u] + parts[u]], k > 0, x["stats"],
                                  x["ws"], x["ws"].numel())
        Z.zero_shard_apply_chained(x["sh"], dt, x["rsh"][me], dt, x["hy"], x["table"], 1, 16, x["chain"], x["stats"],
                                   0.0, 0, x["ws"], x["ws"].numel(), x["res"])

    eager = make()
    for _ in range(4):
        step(eager)
    warm = make()
    step(warm)                                   # the library's one-time set-up, outside the capture
    torch.cuda.synchronize()
    graphed = make()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=torch.cuda.Stream(), capture_error_mode="relaxed"):
        step(graphed)
        step(graphed)
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    ce, cg = Z.read_chain(eager["chain"]), Z.read_chain(graphed["chain"])
    assert ce.as_dict() == cg.as_dict() and ce.step == 5 and ce.applied == 4
    for a, b in zip(eager["st"] + [eager["rsh"][me], eager["layer"], eager["status"]],
                    graphed["st"] + [graphed["rsh"][me], graphed["layer"], graphed["status"]]):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))
    assert int(graphed["status"].item()) == 0


@pytest.mark.parametrize("numels,nd,dt", [([20000, 4096, 992], 4, 2), ([20000, 555], 3, 1)])
def test_chained_partial_passes_then_commit_match_the_oracle(Z, numels, nd, dt):
    """A step split into partial fused passes -- one per shard, each adding its
    statistics -- and a commit, chained: five steps, the second with a NaN in
    one slice, no host synchronisation, each step's result in its own slot.
    Equal to the oracle's whole steps with the same bookkeeping, bit for bit.
    Then a step outside the scalar table: reported ZERO_ELIMIT by the commit,
    nothing updated, the chain's t and set kept."""
    S = 256.0 if dt == 1 else 1.0
    p, flat, grads = make_problem(numels, nd, dt, 0, 68, loss_scale=S, grad_std=1e-2, steps=6)
    grads[1][0] = grads[1][0].copy()
    grads[1][0][7] = 0x7E00 if dt == 1 else 0x7FC0
    h = hyper32()
    run = ChainRun(Z, p, flat, dt, h, S, n_table=6)
    slices = [[dev16(g, dt) for g in step] for step in grads]
    stats = torch.zeros(16, dtype=torch.uint8, device=DEV)
    res = torch.zeros(6, 48, dtype=torch.uint8, device=DEV)

    def step(k):
        for i, sh in enumerate(run.shards):
            Z.zero_shard_step_partial(slices[k], dt, [sh], run.flat, dt, run.hyper, 0.0, i > 0, stats, run.ws,
                                      run.ws.numel(), scalar_table=run.table, table_t0=1, n_table=run.n_table,
                                      chain_dev=run.chain)
        Z.zero_shard_step_commit(run.shards, run.flat, dt, 0.0, stats, 0.0, 0, res[k], table_t0=1,
                                 n_table=run.n_table, chain_dev=run.chain)

    for k in range(5):
        step(k)
    torch.cuda.synchronize()
    osh, oflat, t, So, results = oracle_run(p, flat, dt, h, S, grads[:5])
    rg = [Z.read_result(res[k]) for k in range(5)]
    assert [r.applied for r in rg] == [r.applied for r in results] == [1, 0, 1, 1, 1]
    assert all(r.path == 3 and r.status == 0 for r in rg)
    assert all(a.grad_mult == b.grad_mult for a, b in zip(rg, results))
    c = check(run, p, osh, oflat, True)
    assert (c.step, c.loss_scale, c.applied, c.skipped, c.failed) == (t, So, 4, 1, 0)
    # four steps applied: t = 5; a table of steps 1..4 does not cover it
    assert c.step == 5
    run.n_table = 4
    before_flat = t2u16(run.flat)
    c5, s5 = run.state()
    step(5)
    torch.cuda.synchronize()
    r = Z.read_result(res[5])
    c6, s6 = run.state()
    assert r.applied == 0 and r.status == Z.ZERO_ELIMIT
    assert (c6.step, c6.cur, c6.applied, c6.failed) == (c5.step, c5.cur, c5.applied, 1)
    assert np.array_equal(t2u16(run.flat), before_flat)
    for a, b in zip(s5, s6):
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
