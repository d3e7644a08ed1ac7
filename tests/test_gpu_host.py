"""GPU parity of the step from host memory (zero_shard_step_host) against the
CPU oracle: gradients in page-locked host buffers, copied up chunk by chunk
into a small device ring while the chunks already up are reduced and
updated, and the updated parameters copied back to page-locked host memory.

Every chunk is an independent piece of a shard, so the results are those of
zero_shard_step: bit-exact state and parameters without clipping (path 3:
partial passes and a commit), and with clipping whenever the multiplier k
equals the oracle's (path 2: a reduce per chunk, then the apply), held to
the same comparison as the device-buffer step.  The host copy of the
parameters must equal the device's bit for bit after every step, a skipped
step included."""
import numpy as np
import pytest
import torch

import oracle as orc
import workloads as W
from helpers import hyper32, make_problem, random_group, t2u16
from test_gpu_step import DeviceRun, compare, oracle_shards

pytestmark = pytest.mark.gpu

DEV = "cuda"
TDT = {1: torch.float16, 2: torch.bfloat16}
RING = 4          # chunk slots of the library's ring


@pytest.fixture(scope="module")
def Z():
    import zero_dp_partitioned_gb300 as Z
    return Z


def pinned16(a: np.ndarray, dt):
    return torch.from_numpy(a.view(np.int16).copy()).view(TDT[dt]).pin_memory()


class HostRun(DeviceRun):
    """A DeviceRun whose steps take their gradients from page-locked host
    memory and return the parameters to it."""

    def __init__(self, Z, p, flat, dt, ranks, pingpong, chunk, download=True, **kw):
        super().__init__(Z, p, flat, dt, ranks, pingpong, **kw)
        nd = len(p["rank_offsets"])
        self.staging_bytes = RING * nd * 2 * chunk
        self.staging = torch.zeros(self.staging_bytes // 2 + 64, dtype=torch.int16, device=DEV)
        self.host_param = self.flat.cpu().pin_memory() if download else None

    def step(self, grads_u16, h, t, S, extra=(0.0, 0), grad_offsets=None):
        Z = self.Z
        slices = [pinned16(g, self.dt) for g in grads_u16]
        hy = Z.hyper(h["lr"], h["beta1"], h["beta2"], h["eps"], h["weight_decay"], h["max_grad_norm"], t)
        Z.zero_shard_step_host(slices, self.dt, self.shards(), self.flat, self.dt, self.host_param, hy, S,
                               extra[0], extra[1], self.staging, self.staging_bytes, self.ws, self.ws.numel(),
                               self.res)
        torch.cuda.synchronize()
        r = Z.read_result(self.res)
        if self.host_param is not None:
            assert np.array_equal(t2u16(self.host_param), t2u16(self.flat))
        if r.applied and self.pingpong:
            for s in self.state:
                s["A"], s["B"] = s["B"], s["A"]
        return r


def run_host(Z, numels, nd, dt, seed, h, S, pingpong, chunk, steps=3, inject=None, mode=0, download=True,
             ranks=None, extra=(0.0, 0)):
    p, flat, grads = make_problem(numels, nd, dt, mode, seed, loss_scale=S, grad_std=1e-2 if
                                  h["max_grad_norm"] > 0 else 1e-3, steps=steps)
    if inject:
        inject(grads)
    ranks = list(range(nd)) if ranks is None else ranks
    run = HostRun(Z, p, flat, dt, ranks, pingpong, chunk, download=download)
    osh = oracle_shards(p, flat, dt, ranks)
    oflat = flat.copy()
    t, Sg, So = 1, S, S
    exact = h["max_grad_norm"] <= 0
    out = []
    for k in range(steps):
        r_gpu = run.step(grads[k], h, t, Sg, extra)
        prev = [(o["master"].copy(), o["m"].copy()) for o in osh]
        r_or, red = orc.zero_step(grads[k], dt, osh, oflat, dt, h, t, So, *extra, want_grad=True)
        compare(run, osh, oflat, r_gpu, r_or, exact, prev, red)
        out.append(r_gpu.as_dict())
        if r_or.applied:
            t += 1
        else:
            Sg /= 2
            So /= 2
    return out


@pytest.mark.parametrize("dt", [1, 2])
@pytest.mark.parametrize("chunk", [64, 448, 4096])
def test_host_step_matches_oracle(Z, dt, chunk):
    """Unclipped, two state sets: partial passes per chunk and a commit."""
    rng = np.random.default_rng(500 + dt + chunk)
    for trial in range(3):
        nd = int(rng.choice([1, 3, 4, 8]))
        numels = random_group(rng, 5, 20000)
        res = run_host(Z, numels, nd, dt, 600 + trial, hyper32(), 1024.0 if dt == 1 else 1.0, True, chunk)
        assert all(r["path"] == 3 and r["applied"] == 1 for r in res)


@pytest.mark.parametrize("dt", [1, 2])
@pytest.mark.parametrize("pingpong", [False, True])
def test_host_step_two_pass(Z, dt, pingpong):
    """Clipped (either state layout) and unclipped in place: a reduce pass per
    chunk into the gradient shard, then the apply pass."""
    rng = np.random.default_rng(700 + dt + 2 * pingpong)
    for trial, clip in enumerate((0.01, 0.0 if not pingpong else 0.02)):
        nd = int(rng.choice([2, 3, 4]))
        numels = random_group(rng, 4, 15000)
        res = run_host(Z, numels, nd, dt, 800 + trial, hyper32(max_grad_norm=clip), 8.0 if dt == 1 else 1.0,
                       pingpong, 256)
        assert all(r["path"] == 2 for r in res)


@pytest.mark.parametrize("pingpong", [True, False])
def test_host_step_skip_restores_host_parameters(Z, pingpong):
    """+inf in rank 0's gradient at step 2: the step is skipped, and the
    parameters -- already copied down chunk by chunk on the fused path --
    are restored in host memory as on the device (checked after every step)."""
    def inject(grads):
        grads[1][0] = grads[1][0].copy()
        grads[1][0][30000] = 0x7C00
    res = run_host(Z, W.numels(W.tiny_group()), 3, 1, 0, hyper32(), 1024.0, pingpong, 1024, inject=inject)
    assert [r["applied"] for r in res] == [1, 0, 1]
    assert res[1]["overflow"] == 1


@pytest.mark.parametrize("clip", [0.0, 0.01])
def test_host_step_rank_local_with_other_ranks_statistics(Z, clip):
    """One rank's shard of an N_d = 4 group, the other ranks' share of the
    sum of squares given as extra_sumsq (and their overflow flag clear): the
    norm, the clip and every update as the oracle's over the same view."""
    res = run_host(Z, [9000, 13000, 2500], 4, 2, 21, hyper32(max_grad_norm=clip), 1.0, True, 512, ranks=[1],
                   extra=(0.75, 0))
    assert all(r["applied"] == 1 and r["path"] == (2 if clip else 3) for r in res)
    assert all(r["sumsq"] > 0.75 for r in res)


def test_host_step_without_download(Z):
    res = run_host(Z, [5000, 7000], 4, 2, 11, hyper32(), 1.0, True, 512, download=False)
    assert [r["applied"] for r in res] == [1, 1, 1]


def test_host_step_argument_errors(Z):
    """Pageable or device gradient buffers, a pageable parameter destination,
    a ring too small for one 64-element chunk per slot and slice, and a
    misaligned ring are refused before anything is enqueued."""
    p, flat, grads = make_problem([3000], 2, 2, 0, 3)
    run = HostRun(Z, p, flat, 2, [0, 1], True, 128)
    hy = Z.hyper()
    before = t2u16(run.flat)
    pinned = [pinned16(g, 2) for g in grads[0]]
    pageable = [torch.from_numpy(g.view(np.int16).copy()).view(torch.bfloat16) for g in grads[0]]
    on_device = [x.to(DEV) for x in pinned]
    args = lambda sl, hp, stg, nbytes: (sl, 2, run.shards(), run.flat, 2, hp, hy, 1.0, 0.0, 0, stg, nbytes, run.ws,
                                        run.ws.numel(), run.res)
    cases = [
        (args(pageable, run.host_param, run.staging, run.staging_bytes), Z.ZERO_EINVAL),
        (args(on_device, run.host_param, run.staging, run.staging_bytes), Z.ZERO_EINVAL),
        (args(pinned, run.flat.cpu(), run.staging, run.staging_bytes), Z.ZERO_EINVAL),
        (args(pinned, run.host_param, run.staging, RING * 2 * 2 * 63), Z.ZERO_EWORKSPACE),
        (args(pinned, run.host_param, run.staging[1:], run.staging_bytes - 64), Z.ZERO_EALIGN),
    ]
    for a, code in cases:
        with pytest.raises(Z.ZeroError) as e:
            Z.zero_shard_step_host(*a)
        assert e.value.code == code, e.value
    torch.cuda.synchronize()
    assert np.array_equal(t2u16(run.flat), before)
    assert not run.res.any()
    Z.zero_shard_step_host(*args(pinned, run.host_param, run.staging, run.staging_bytes))
    torch.cuda.synchronize()
    assert Z.read_result(run.res).applied == 1
