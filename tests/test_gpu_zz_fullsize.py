"""GPU parity at the full workload sizes, through the same C-ABI calls and
launch configuration the benchmark times.

The oracle cannot redo billions of elements one by one in a test, so:
  * the global statistics (sum of squares, overflow) are computed by the
    oracle over every element, chunk by chunk (the oracle stays
    single-threaded; chunks run in a thread pool);
  * the per-element outputs (reduced gradient, master/m/v, 16-bit parameter)
    are checked on a sample of indices -- shard starts and ends, tile
    boundaries, the ragged tail, and random positions -- the oracle carrying
    its own copy of the sampled state through the three steps;
  * properties that hold at any size are checked on all elements: the slots of
    the flat buffer that belong to other ranks are untouched, a gathered layer
    is the concatenation of its parts.
Tolerances are those of the small-size tests: bit-exact without clipping,
and with clipping whenever the device's multiplier k equals the oracle's
(else rel 2e-6 of the operands for fp32 state and 1 ulp for 16-bit
parameters); bit-exact always when the apply pass is given the oracle's
exact sum of squares; the norm within rel 1e-5; the plan and the overflow
flag bit-exact."""
import concurrent.futures as cf
import os

import numpy as np
import pytest
import torch

import oracle as orc
import workloads as W
from helpers import hyper32

pytestmark = pytest.mark.gpu
DEV = "cuda"
TDT = {1: torch.float16, 2: torch.bfloat16}
TILE = 2048


@pytest.fixture(scope="module")
def Z():
    import zero_dp_partitioned_gb300 as Z
    return Z


@pytest.fixture(autouse=True)
def _free():
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def u16(t):
    return t.contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def sample_idx(numel, seed, n_random=40000):
    rng = np.random.default_rng(seed)
    ks = [k * TILE + d for k in (1, 2, 1000, numel // TILE - 1) for d in (-1, 0, 1, 7, 8)]
    idx = np.concatenate([np.arange(min(16, numel)), np.arange(max(0, numel - 16), numel), ks,
                          rng.integers(0, numel, n_random)])
    return np.unique(idx[(idx >= 0) & (idx < numel)]).astype(np.int64)


def oracle_stats(slices, gdt, grad_off, numel):
    """Exact sum of squares and overflow flag of the averaged gradient over
    [grad_off, grad_off + numel) of every slice, by the oracle."""
    chunk = max(1 << 20, (1 << 27) // len(slices))

    def work(c0):
        n = min(chunk, numel - c0)
        host = [u16(s[grad_off + c0: grad_off + c0 + n]) for s in slices]
        acc = orc.ExactAccumulator()
        return acc, orc.reduce_stats(host, gdt, 0, n, acc)

    with cf.ThreadPoolExecutor(min(16, os.cpu_count() or 4)) as ex:
        parts = list(ex.map(work, range(0, numel, chunk)))
    total = orc.ExactAccumulator()
    ovf = 0
    for a, o in parts:
        total.merge(a)
        ovf |= o
    return total, ovf


class Sampled:
    """The oracle's copy of one shard's state at sampled indices."""

    def __init__(self, idx, params16, dt):
        self.idx = idx
        self.master = orc.widen_16(params16, dt)
        self.m = np.zeros(idx.size, np.float32)
        self.v = np.zeros(idx.size, np.float32)
        self.param = params16.copy()

    def step(self, slices_at_idx, dt, k, sc):
        a = orc.reduce(slices_at_idx, dt, 0, self.idx.size)
        orc.apply(a, dt, self.master, self.m, self.v, self.param, dt, k, sc)
        return a


def check_state(samp, master, m, v, param16, exact, prev=None, g=None):
    """Bit-exact, or (clipped steps, where the multiplier k comes from an fp64
    norm whose last bits differ between the two sides) rel 2e-6 measured
    against the operands each update combines: theta_new = theta wdf - update
    and m_new = b1 m + (1-b1) g are differences whose result can be far
    smaller than their terms, where a relative bound on the result alone is
    not meaningful; v sums non-negative terms and is compared to itself."""
    idx = torch.from_numpy(samp.idx).to(DEV)
    got = [x[idx].cpu().numpy() for x in (master, m, v)]
    gp = u16(param16[idx])
    if exact:
        for gg, r in zip(got, (samp.master, samp.m, samp.v)):
            assert np.array_equal(gg.view(np.uint32), r.view(np.uint32))
        assert np.array_equal(gp, samp.param)
        return
    th_prev, m_prev = (np.abs(x.astype(np.float64)) for x in prev)
    upd = np.abs(th_prev - samp.master.astype(np.float64))
    scale_th = np.maximum(th_prev + upd, np.abs(samp.master))
    scale_m = np.maximum(0.9 * m_prev + 0.1 * np.abs(g), np.abs(samp.m))
    for gg, r, sc in ((got[0], samp.master, scale_th), (got[1], samp.m, scale_m), (got[2], samp.v, np.abs(samp.v))):
        assert np.all(np.abs(gg.astype(np.float64) - r) <= 2e-6 * np.maximum(sc, 1e-30))
    assert np.abs(gp.astype(np.int32) - samp.param.astype(np.int32)).max() <= 1


def scalars(h, t):
    return orc.make_scalars(h["lr"], h["beta1"], h["beta2"], h["eps"], h["weight_decay"], t)


@pytest.mark.parametrize("chained", [False, True])
def test_gpt2_1p5b_all_ranks(Z, chained):
    """GPT-2 1.5B-shaped group, N_d = 8, all ranks, bf16, fused single pass, 3
    steps: host-driven (the caller swaps the state sets and advances t), and
    chained as the benchmark runs it (t, S and the current set on the device)."""
    wl = W.workload("gpt2-1.5b-nd8")
    nd, dt = 8, 2
    numels = W.numels(wl.specs)
    plan = Z.zero_plan(numels, nd)
    op = orc.plan(numels, nd, 0)
    assert plan["rank_offsets"] == list(op["rank_offsets"]) and plan["padded_total"] == op["padded_total"]
    P = plan["padded_total"]
    flat = W.flat_params(wl.specs, P, torch.bfloat16, wl.param_seed, DEV)
    grads = [torch.empty(P, dtype=torch.bfloat16, device=DEV) for _ in range(nd)]
    gs = W.GradStream([1 + r for r in range(nd)], DEV)
    sets = [[flat.float(), torch.zeros(P, device=DEV), torch.zeros(P, device=DEV)],
            [torch.empty(P, device=DEV) for _ in range(3)]]
    ws = torch.zeros(Z.zero_workspace_bytes(), dtype=torch.uint8, device=DEV)
    res = torch.zeros(48, dtype=torch.uint8, device=DEV)
    samp = []
    for r in range(nd):
        o, n = plan["rank_offsets"][r], plan["rank_numels"][r]
        idx = o + sample_idx(n, r, 8000)
        samp.append(Sampled(idx, u16(flat[torch.from_numpy(idx).to(DEV)]), dt))
    h = hyper32()
    hz = {k: h[k] for k in ("lr", "beta1", "beta2", "eps", "weight_decay", "max_grad_norm")}
    if chained:
        hy = Z.hyper(step=1, **hz)
        table = torch.from_numpy(Z.zero_adam_scalar_table(hy, 1, 16)).to(DEV)
        chain = torch.frombuffer(bytearray(bytes(Z.chain(step=1, loss_scale=1.0))), dtype=torch.uint8).to(DEV)
    cur = 0
    for t in (1, 2, 3):
        gs.draw_flat(grads, wl.specs, W.gpt2_grad_std())
        A, B = sets[0 if chained else cur], sets[1 if chained else 1 - cur]
        sh = [Z.shard(n, o, o, A[0][o:o + n], A[1][o:o + n], A[2][o:o + n], B[0][o:o + n], B[1][o:o + n],
                      B[2][o:o + n]) for o, n in zip(plan["rank_offsets"], plan["rank_numels"])]
        if chained:
            Z.zero_shard_step_chained(grads, dt, sh, flat, dt, hy, table, 1, 16, chain, 0.0, 0, ws, ws.numel(), res)
        else:
            Z.zero_shard_step(grads, dt, sh, flat, dt, Z.hyper(step=t, **hz), 1.0, 0.0, 0, ws, ws.numel(), res)
        acc, ovf = oracle_stats(grads, dt, 0, P)
        r_gpu = Z.read_result(res)
        k, norm, _ = orc.grad_multiplier(acc.value(), 1.0, 0.0)
        assert r_gpu.overflow == ovf == 0 and r_gpu.applied == 1 and r_gpu.path == 1
        assert r_gpu.grad_norm == pytest.approx(norm, rel=1e-5)
        cur ^= 1
        if chained:
            c = Z.read_chain(chain)
            assert (c.step, c.cur, c.applied, c.skipped, c.failed) == (t + 1, cur, t, 0, 0)
        for s in samp:
            ti = torch.from_numpy(s.idx).to(DEV)
            s.step([u16(g[ti]) for g in grads], dt, k, scalars(h, t))
            check_state(s, *sets[cur], flat, exact=True)


def test_gpt2_1p5b_from_host_buffers(Z):
    """The end-to-end call at full size: the GPT-2 1.5B-shaped group's 8
    gradient buffers (24.9 GB) in page-locked host memory, zero_shard_step_host
    with the benchmark's 512 MiB device ring (8 Mi-element chunks), the
    updated 16-bit parameters returned to page-locked host memory; 2 steps,
    the host keeping t and the state set.  The statistics against the
    oracle's over every element, state and parameters at sampled indices bit
    for bit, and the host copy of the parameters equal to the device's."""
    wl = W.workload("gpt2-1.5b-nd8")
    nd, dt = 8, 2
    plan = Z.zero_plan(W.numels(wl.specs), nd)
    P = plan["padded_total"]
    flat = W.flat_params(wl.specs, P, torch.bfloat16, wl.param_seed, DEV)
    grads = [torch.empty(P, dtype=torch.bfloat16, device=DEV) for _ in range(nd)]
    host_grads = [torch.empty(P, dtype=torch.bfloat16, pin_memory=True) for _ in range(nd)]
    host_params = torch.empty(P, dtype=torch.bfloat16, pin_memory=True)
    gs = W.GradStream([1 + r for r in range(nd)], DEV)
    sets = [[flat.float(), torch.zeros(P, device=DEV), torch.zeros(P, device=DEV)],
            [torch.empty(P, device=DEV) for _ in range(3)]]
    ring_bytes = 512 << 20
    ring = torch.empty(ring_bytes // 2, dtype=torch.int16, device=DEV)
    ws = torch.zeros(Z.zero_workspace_bytes(), dtype=torch.uint8, device=DEV)
    res = torch.zeros(48, dtype=torch.uint8, device=DEV)
    samp = []
    for r in range(nd):
        o, n = plan["rank_offsets"][r], plan["rank_numels"][r]
        idx = o + sample_idx(n, 20 + r, 8000)
        samp.append(Sampled(idx, u16(flat[torch.from_numpy(idx).to(DEV)]), dt))
    h = hyper32()
    hz = {k: h[k] for k in ("lr", "beta1", "beta2", "eps", "weight_decay", "max_grad_norm")}
    cur = 0
    for t in (1, 2):
        gs.draw_flat(grads, wl.specs, W.gpt2_grad_std())
        for g, hg in zip(grads, host_grads):
            hg.copy_(g)
        A, B = sets[cur], sets[1 - cur]
        sh = [Z.shard(n, o, o, A[0][o:o + n], A[1][o:o + n], A[2][o:o + n], B[0][o:o + n], B[1][o:o + n],
                      B[2][o:o + n]) for o, n in zip(plan["rank_offsets"], plan["rank_numels"])]
        Z.zero_shard_step_host(host_grads, dt, sh, flat, dt, host_params, Z.hyper(step=t, **hz), 1.0, 0.0, 0, ring,
                               ring_bytes, ws, ws.numel(), res)
        torch.cuda.synchronize()
        acc, ovf = oracle_stats(host_grads, dt, 0, P)
        r_gpu = Z.read_result(res)
        k, norm, _ = orc.grad_multiplier(acc.value(), 1.0, 0.0)
        assert r_gpu.overflow == ovf == 0 and r_gpu.applied == 1 and r_gpu.path == 3
        assert r_gpu.grad_norm == pytest.approx(norm, rel=1e-5)
        assert torch.equal(host_params.view(torch.int16), flat.cpu().view(torch.int16))
        cur ^= 1
        for s in samp:
            s.step([u16(g[torch.from_numpy(s.idx)]) for g in host_grads], dt, k, scalars(h, t))
            check_state(s, *sets[cur], flat, exact=True)


def stats_tensor(Z, sumsq, overflow=0):
    """A device zero_stats holding the given sum of squares and flag."""
    return torch.frombuffer(bytearray(bytes(Z.zero_stats(sumsq, overflow, 0))), dtype=torch.uint8).to(DEV)


def test_llama3_8b_rank1_clipped(Z):
    """Llama-3-8B-shaped group, N_d = 4, rank 1's shard (2.0B elements) with 4
    staged slices, global-norm clip 1.0 (the other ranks' share of the norm
    generated from their own seeded slices), 3 steps, two routes on two state
    sets from the same start:
      A  zero_shard_step (the in-place two-pass path, the device's own norm):
         bit-exact whenever its multiplier k equals the oracle's;
      B  zero_shard_reduce, then the statistics overwritten with the oracle's
         exactly rounded sum of squares, then zero_shard_apply: k is derived
         from the same fp64 number on both sides, so every sampled state and
         parameter must be bit-exact -- the clipped arithmetic itself."""
    wl = W.workload("llama3-8b-nd4-r1")
    nd, dt, me = 4, 2, 1
    numels = W.numels(wl.specs)
    plan = Z.zero_plan(numels, nd)
    P = plan["padded_total"]
    o, n = plan["rank_offsets"][me], plan["rank_numels"][me]
    assert (o, n) == (2_007_565_312, 2_007_565_312)
    flat = W.flat_params(wl.specs, P, torch.bfloat16, wl.param_seed, DEV)
    before = flat.clone()
    flat_b = flat[o:o + n].clone()                       # route B's parameter slot
    slices = [torch.empty(n, dtype=torch.bfloat16, device=DEV) for _ in range(nd)]
    gs = W.GradStream([2 + j for j in range(nd)], DEV)
    state_a = [flat[o:o + n].float(), torch.zeros(n, device=DEV), torch.zeros(n, device=DEV)]
    state_b = [x.clone() for x in state_a]
    gshard = torch.empty(n, dtype=torch.bfloat16, device=DEV)
    ws = torch.zeros(Z.zero_workspace_bytes(), dtype=torch.uint8, device=DEV)
    res = torch.zeros(48, dtype=torch.uint8, device=DEV)
    res_b = torch.zeros(48, dtype=torch.uint8, device=DEV)
    stats_b = torch.zeros(16, dtype=torch.uint8, device=DEV)
    extra = W.other_ranks_sumsq(wl)
    assert extra > 0.0
    idx = sample_idx(n, 3)
    ti = torch.from_numpy(idx).to(DEV)
    samp = Sampled(idx, u16(flat[o + ti]), dt)
    h = hyper32(max_grad_norm=wl.max_grad_norm)
    hz = {k: h[k] for k in ("lr", "beta1", "beta2", "eps", "weight_decay", "max_grad_norm")}
    a_exact = True                                       # route A has followed the oracle bit for bit so far
    for t in (1, 2, 3):
        gs.draw_plain(slices, wl.grad_std)
        Z.zero_shard_step(slices, dt, [Z.shard(n, 0, o, *state_a, grad_shard=gshard)], flat, dt,
                          Z.hyper(step=t, **hz), 1.0, extra, 0, ws, ws.numel(), res)
        acc, ovf = oracle_stats(slices, dt, 0, n)
        own = acc.value()
        total = own + extra
        k, norm, clip = orc.grad_multiplier(total, 1.0, wl.max_grad_norm)
        r_gpu = Z.read_result(res)
        assert r_gpu.overflow == ovf == 0 and r_gpu.applied == 1 and r_gpu.path == 2
        assert r_gpu.grad_norm == pytest.approx(norm, rel=1e-5) and clip < 1.0
        assert r_gpu.clip_coef == pytest.approx(clip, rel=1e-5)
        prev = (samp.master.copy(), samp.m.copy())
        a = samp.step([u16(s[ti]) for s in slices], dt, k, scalars(h, t))
        assert np.array_equal(u16(gshard[ti]), a)                       # reduced gradient: bit-exact
        kg = np.float32(r_gpu.grad_mult)
        print(f"step {t}: k gpu {kg!r} oracle {np.float32(k)!r}, sumsq rel diff {(r_gpu.sumsq - total) / total:.3e}")
        a_exact = a_exact and kg == np.float32(k)
        check_state(samp, *state_a, flat[o:o + n], exact=a_exact, prev=prev, g=orc.widen_16(a, dt) * k)

        sh_b = [Z.shard(n, 0, 0, *state_b, grad_shard=gshard)]
        Z.zero_shard_reduce(slices, dt, sh_b, 0, stats_b, ws, ws.numel())
        torch.cuda.synchronize()
        dev = Z.read_stats(stats_b)
        assert dev.overflow == 0 and dev.sumsq == pytest.approx(own, rel=1e-9)
        stats_b.copy_(stats_tensor(Z, own))
        Z.zero_shard_apply(sh_b, dt, flat_b, dt, Z.hyper(step=t, **hz), 1.0, stats_b, extra, 0, ws, ws.numel(),
                           res_b)
        rb = Z.read_result(res_b)
        assert rb.applied == 1 and np.float32(rb.grad_mult) == np.float32(k) and rb.sumsq == total
        assert np.array_equal(u16(gshard[ti]), a)
        check_state(samp, *state_b, flat_b, exact=True)
    for lo, hi in ((0, o), (o + n, P)):                                  # other ranks' slots untouched
        for c in range(lo, hi, 1 << 30):
            e = min(hi, c + (1 << 30))
            assert torch.equal(flat[c:e], before[c:e])


def test_gpt_7p5b_rank63_nd64(Z):
    """The 7.5B GPT-like group, N_d = 64, rank 63's shard (119,259,162
    elements, flat offset = 6 mod 8), fp16, loss scale 65536, exact zeros in
    slice 0 at every 100th element, fused single pass, 3 steps."""
    wl = W.workload("gpt-7.5b-nd64-r63")
    nd, dt, me = 64, 1, 63
    plan = Z.zero_plan(W.numels(wl.specs), nd)
    P = plan["padded_total"]
    o, n = plan["rank_offsets"][me], plan["rank_numels"][me]
    assert n == 119_259_162 and o % 8 == 6
    flat = W.flat_params(wl.specs, P, torch.float16, wl.param_seed, DEV)
    head = flat[:o].clone()
    slices = [torch.empty(n, dtype=torch.float16, device=DEV) for _ in range(nd)]
    gs = W.GradStream([4 + j for j in range(nd)], DEV)
    sets = [[flat[o:o + n].float(), torch.zeros(n, device=DEV), torch.zeros(n, device=DEV)],
            [torch.empty(n, device=DEV) for _ in range(3)]]
    ws = torch.zeros(Z.zero_workspace_bytes(), dtype=torch.uint8, device=DEV)
    res = torch.zeros(48, dtype=torch.uint8, device=DEV)
    idx = sample_idx(n, 4)
    ti = torch.from_numpy(idx).to(DEV)
    samp = Sampled(idx, u16(flat[o + ti]), dt)
    h = hyper32()
    cur, S = 0, wl.loss_scale
    for t in (1, 2, 3):
        gs.draw_plain(slices, wl.grad_std, S)
        W.zero_every_100th_(slices[0])
        A, B = sets[cur], sets[1 - cur]
        sh = [Z.shard(n, 0, o, *A, *B)]
        Z.zero_shard_step(slices, dt, sh, flat, dt, Z.hyper(step=t, **{k: h[k] for k in
                          ("lr", "beta1", "beta2", "eps", "weight_decay", "max_grad_norm")}), S, 0.0, 0, ws,
                          ws.numel(), res)
        acc, ovf = oracle_stats(slices, dt, 0, n)
        k, norm, _ = orc.grad_multiplier(acc.value(), S, 0.0)
        r_gpu = Z.read_result(res)
        assert r_gpu.overflow == ovf == 0 and r_gpu.applied == 1
        assert r_gpu.grad_norm == pytest.approx(norm, rel=1e-5)
        cur ^= 1
        samp.step([u16(s[ti]) for s in slices], dt, k, scalars(h, t))
        check_state(samp, *sets[cur], flat[o:o + n], exact=True)
    assert torch.equal(flat[:o], head)


def test_zero3_llama3_8b_rank1(Z):
    """ZeRO-3 per-layer path on the Llama-3-8B group, N_d = 4, rank 1: for each
    of the 34 units a forward gather, a backward gather (reverse order) and the
    bucket reduce onto rank 1's part; then the shard update; 3 steps."""
    wl = W.workload("zero3-llama3-8b")
    nd, dt, me = 4, 2, 1
    units = W.llama_units(wl.specs)
    parts = [u // nd for u in units]
    uoff = np.concatenate([[0], np.cumsum(parts)[:-1]]).astype(np.int64)
    L = int(sum(parts))
    flat = W.flat_params(wl.specs, sum(units), torch.bfloat16, wl.param_seed, DEV)
    # rank r's persistent parameter shard: its part of every unit
    starts = np.concatenate([[0], np.cumsum(units)[:-1]])
    rshards = [torch.cat([flat[s + r * p: s + (r + 1) * p] for s, p in zip(starts, parts)]) for r in range(nd)]
    del flat
    torch.cuda.empty_cache()
    layer = torch.empty(max(units), dtype=torch.bfloat16, device=DEV)
    layer2 = torch.empty(max(units), dtype=torch.bfloat16, device=DEV)
    gstatus = torch.zeros(1, dtype=torch.int32, device=DEV)
    buckets = [torch.empty(max(units), dtype=torch.bfloat16, device=DEV) for _ in range(nd)]
    gs = W.GradStream([5 + r for r in range(nd)], DEV)
    master = rshards[me].float()
    m = torch.zeros(L, device=DEV)
    v = torch.zeros(L, device=DEV)
    gshard = torch.empty(L, dtype=torch.bfloat16, device=DEV)
    ws = torch.zeros(Z.zero_workspace_bytes(), dtype=torch.uint8, device=DEV)
    stats = torch.zeros(16, dtype=torch.uint8, device=DEV)
    res = torch.zeros(48, dtype=torch.uint8, device=DEV)
    idx = sample_idx(L, 5)
    ti = torch.from_numpy(idx).to(DEV)
    samp = Sampled(idx, u16(rshards[me][ti]), dt)
    h = hyper32()
    for t in (1, 2, 3):
        for u in list(range(len(units))) + list(reversed(range(len(units)))):
            ptrs = [rshards[r][uoff[u]:uoff[u] + parts[u]] for r in range(nd)]
            Z.zero3_gather_layer(ptrs, units[u], dt, layer)
            if u in (0, 1, len(units) - 1):
                assert torch.equal(layer[:units[u]], torch.cat(ptrs))     # gather = inverse of the partition
            if t == 1:      # the TMA gather, on every SM and on 32 CTAs, equals it unit by unit
                for n_ctas in (0, 32):
                    Z.zero3_gather_bulk(ptrs, [parts[u]] * nd, dt, layer2, n_ctas, gstatus)
                    assert torch.equal(layer2[:units[u]].view(torch.int16), layer[:units[u]].view(torch.int16))
        acc = orc.ExactAccumulator()
        a_samp = np.empty(idx.size, np.uint16)
        for k_u, u in enumerate(reversed(range(len(units)))):
            bu = [b[:units[u]] for b in buckets]
            gs.draw_plain(bu, wl.grad_std)
            Z.zero3_reduce_bucket(bu, me, units[u], dt, gshard[uoff[u]:uoff[u] + parts[u]], k_u > 0, stats, ws,
                                  ws.numel())
            a_u, o_u = oracle_stats(bu, dt, me * parts[u], parts[u])
            acc.merge(a_u)
            assert o_u == 0
            sel = (idx >= uoff[u]) & (idx < uoff[u] + parts[u])
            if sel.any():
                loc = torch.from_numpy(idx[sel] - uoff[u] + me * parts[u]).to(DEV)
                a_samp[sel] = orc.reduce([u16(b[loc]) for b in bu], dt, 0, int(sel.sum()))
        sh = [Z.shard(L, 0, 0, master, m, v, grad_shard=gshard)]
        Z.zero_shard_apply(sh, dt, rshards[me], dt, Z.hyper(step=t, **{k: h[k] for k in
                           ("lr", "beta1", "beta2", "eps", "weight_decay", "max_grad_norm")}), 1.0, stats, 0.0, 0,
                           ws, ws.numel(), res)
        k, norm, _ = orc.grad_multiplier(acc.value(), 1.0, 0.0)
        r_gpu = Z.read_result(res)
        assert r_gpu.applied == 1 and r_gpu.grad_norm == pytest.approx(norm, rel=1e-5)
        assert np.array_equal(u16(gshard[ti]), a_samp)
        orc.apply(a_samp, dt, samp.master, samp.m, samp.v, samp.param, dt, k, scalars(h, t))
        check_state(samp, master, m, v, rshards[me], exact=True)
    assert int(gstatus.item()) == 0


def test_zero3_llama3_8b_rank1_fused_units(Z):
    """The ZeRO-3 update as the benchmark runs it, at full size: per unit, in
    reverse order, the 4 full-unit buckets reduced onto rank 1's part and
    that part updated in one partial fused pass (chained: t, S and the state
    set from the device; the result into the other state set), then one
    commit deciding the step; 3 steps.  The statistics against the oracle's
    over every element, the state and parameters at sampled indices of the
    2.0B-element shard bit for bit."""
    wl = W.workload("zero3-llama3-8b")
    nd, dt, me = 4, 2, 1
    units = W.llama_units(wl.specs)
    parts = [u // nd for u in units]
    uoff = np.concatenate([[0], np.cumsum(parts)[:-1]]).astype(np.int64)
    L = int(sum(parts))
    flat = W.flat_params(wl.specs, sum(units), torch.bfloat16, wl.param_seed, DEV)
    starts = np.concatenate([[0], np.cumsum(units)[:-1]])
    rshard = torch.cat([flat[s + me * p: s + (me + 1) * p] for s, p in zip(starts, parts)])
    del flat
    torch.cuda.empty_cache()
    buckets = [torch.empty(max(units), dtype=torch.bfloat16, device=DEV) for _ in range(nd)]
    gs = W.GradStream([5 + r for r in range(nd)], DEV)
    sets = [[rshard.float(), torch.zeros(L, device=DEV), torch.zeros(L, device=DEV)],
            [torch.empty(L, device=DEV) for _ in range(3)]]
    A, B = sets
    part_sh = [Z.shard(parts[u], me * parts[u], int(uoff[u]), *(x[uoff[u]:uoff[u] + parts[u]] for x in A),
                       *(x[uoff[u]:uoff[u] + parts[u]] for x in B)) for u in range(len(units))]
    whole = [Z.shard(L, 0, 0, *A, *B)]
    ws = torch.zeros(Z.zero_workspace_bytes(), dtype=torch.uint8, device=DEV)
    stats = torch.zeros(16, dtype=torch.uint8, device=DEV)
    res = torch.zeros(48, dtype=torch.uint8, device=DEV)
    h = hyper32()
    hy = Z.hyper(step=1, **{k: h[k] for k in ("lr", "beta1", "beta2", "eps", "weight_decay", "max_grad_norm")})
    table = torch.from_numpy(Z.zero_adam_scalar_table(hy, 1, 16)).to(DEV)
    chain = torch.frombuffer(bytearray(bytes(Z.chain(step=1, loss_scale=1.0))), dtype=torch.uint8).to(DEV)
    idx = sample_idx(L, 6)
    ti = torch.from_numpy(idx).to(DEV)
    samp = Sampled(idx, u16(rshard[ti]), dt)
    cur = 0
    for t in (1, 2, 3):
        acc = orc.ExactAccumulator()
        a_samp = np.empty(idx.size, np.uint16)
        for k_u, u in enumerate(reversed(range(len(units)))):
            bu = [b[:units[u]] for b in buckets]
            gs.draw_plain(bu, wl.grad_std)
            Z.zero_shard_step_partial(bu, dt, [part_sh[u]], rshard, dt, hy, 0.0, k_u > 0, stats, ws, ws.numel(),
                                      scalar_table=table, table_t0=1, n_table=16, chain_dev=chain)
            a_u, o_u = oracle_stats(bu, dt, me * parts[u], parts[u])
            acc.merge(a_u)
            assert o_u == 0
            sel = (idx >= uoff[u]) & (idx < uoff[u] + parts[u])
            if sel.any():
                loc = torch.from_numpy(idx[sel] - uoff[u] + me * parts[u]).to(DEV)
                a_samp[sel] = orc.reduce([u16(b[loc]) for b in bu], dt, 0, int(sel.sum()))
        Z.zero_shard_step_commit(whole, rshard, dt, 0.0, stats, 0.0, 0, res, table_t0=1, n_table=16,
                                 chain_dev=chain)
        k, norm, _ = orc.grad_multiplier(acc.value(), 1.0, 0.0)
        r_gpu = Z.read_result(res)
        assert r_gpu.applied == 1 and r_gpu.overflow == 0 and r_gpu.path == 3
        assert r_gpu.grad_norm == pytest.approx(norm, rel=1e-5)
        cur ^= 1
        c = Z.read_chain(chain)
        assert (c.step, c.cur, c.applied, c.skipped, c.failed) == (t + 1, cur, t, 0, 0)
        orc.apply(a_samp, dt, samp.master, samp.m, samp.v, samp.param, dt, k, scalars(h, t))
        check_state(samp, *sets[cur], rshard, exact=True)


@pytest.mark.parametrize("clip", [0.0, 1.0])
def test_shard_past_the_int32_index_range(Z, clip):
    """One shard of 2^31 + 4099 elements, so that element, gradient and
    parameter indices run past 2^31 and the shard ends 3 elements after its
    last full vector; N_d = 2 staged bf16 slices; parameter offset 8 inside a
    flat buffer whose other slots must stay untouched.  Without clipping: the
    fused pass out of place, 2 steps (both state-set directions); with a
    clip that fires: the in-place two-pass path, 1 step."""
    nd, dt, o = 2, 2, 8
    n = (1 << 31) + 4099
    flat = torch.empty(o + n + 8, dtype=torch.bfloat16, device=DEV)
    W.fill_normal_(flat, 0.02, W.generator(71, DEV))
    head, tail = flat[:o].clone(), flat[o + n:].clone()
    slices = [torch.empty(n, dtype=torch.bfloat16, device=DEV) for _ in range(nd)]
    gs = W.GradStream([72 + r for r in range(nd)], DEV)
    idx = np.unique(np.concatenate([sample_idx(n, 7, 20000), np.arange((1 << 31) - 24, (1 << 31) + 24),
                                    np.arange((1 << 31) - TILE - 8, (1 << 31) - TILE + 8)])).astype(np.int64)
    ti = torch.from_numpy(idx).to(DEV)
    samp = Sampled(idx, u16(flat[o + ti]), dt)
    ws = torch.zeros(Z.zero_workspace_bytes(), dtype=torch.uint8, device=DEV)
    res = torch.zeros(48, dtype=torch.uint8, device=DEV)
    h = hyper32(max_grad_norm=clip)
    hz = {k: h[k] for k in ("lr", "beta1", "beta2", "eps", "weight_decay", "max_grad_norm")}
    if clip <= 0.0:
        sets = [[flat[o:o + n].float(), torch.zeros(n, device=DEV), torch.zeros(n, device=DEV)],
                [torch.empty(n, device=DEV) for _ in range(3)]]
        cur = 0
        for t in (1, 2):
            gs.draw_plain(slices, 1e-3)
            sh = [Z.shard(n, 0, o, *sets[cur], *sets[1 - cur])]
            Z.zero_shard_step(slices, dt, sh, flat, dt, Z.hyper(step=t, **hz), 1.0, 0.0, 0, ws, ws.numel(), res)
            acc, ovf = oracle_stats(slices, dt, 0, n)
            k, norm, _ = orc.grad_multiplier(acc.value(), 1.0, 0.0)
            r_gpu = Z.read_result(res)
            assert r_gpu.overflow == ovf == 0 and r_gpu.applied == 1 and r_gpu.path == 1
            assert r_gpu.grad_norm == pytest.approx(norm, rel=1e-5)
            cur ^= 1
            samp.step([u16(s[ti]) for s in slices], dt, k, scalars(h, t))
            check_state(samp, *sets[cur], flat[o:o + n], exact=True)
        del sets
    else:
        master = flat[o:o + n].float()
        m = torch.zeros(n, device=DEV)
        v = torch.zeros(n, device=DEV)
        gshard = torch.empty(n, dtype=torch.bfloat16, device=DEV)
        gs.draw_plain(slices, 1e-3)
        sh = [Z.shard(n, 0, o, master, m, v, grad_shard=gshard)]
        Z.zero_shard_step(slices, dt, sh, flat, dt, Z.hyper(step=1, **hz), 1.0, 0.0, 0, ws, ws.numel(), res)
        acc, ovf = oracle_stats(slices, dt, 0, n)
        k, norm, c = orc.grad_multiplier(acc.value(), 1.0, clip)
        r_gpu = Z.read_result(res)
        assert r_gpu.overflow == ovf == 0 and r_gpu.applied == 1 and r_gpu.path == 2
        assert r_gpu.grad_norm == pytest.approx(norm, rel=1e-5) and c < 1.0
        prev = (samp.master.copy(), samp.m.copy())
        a = samp.step([u16(s[ti]) for s in slices], dt, k, scalars(h, 1))
        assert np.array_equal(u16(gshard[ti]), a)                       # reduced gradient: bit-exact
        check_state(samp, master, m, v, flat[o:o + n], exact=np.float32(r_gpu.grad_mult) == np.float32(k),
                    prev=prev, g=orc.widen_16(a, dt) * k)
    assert torch.equal(flat[:o], head) and torch.equal(flat[o + n:], tail)


def test_gather_past_the_int32_index_range(Z):
    """A 16-bit unit of 2^31 + 32 elements (4.3 GB) gathered from 4 equal
    parts by the register gather and by the TMA gather on every SM and on 32
    CTAs, then from 4 ragged segments (the TMA gather's fallback to register
    copies): each equals the concatenation of its parts."""
    nd = 4
    p = (1 << 29) + 8
    parts = [torch.empty(p, dtype=torch.bfloat16, device=DEV) for _ in range(nd)]
    gs = W.GradStream([81 + r for r in range(nd)], DEV)
    gs.draw_plain(parts, 0.02)
    want = torch.cat(parts).view(torch.int16)
    out = torch.empty(nd * p, dtype=torch.bfloat16, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out.zero_()
    Z.zero3_gather_layer(parts, nd * p, 2, out)
    assert torch.equal(out.view(torch.int16), want)
    for n_ctas in (0, 32):
        out.zero_()
        Z.zero3_gather_bulk(parts, [p] * nd, 2, out, n_ctas, status)
        assert torch.equal(out.view(torch.int16), want)
    lens = [p - 3, p, p - 1, p - 5]
    segs = [x[:n] for x, n in zip(parts, lens)]
    out.zero_()
    Z.zero3_gather_bulk(segs, lens, 2, out, 32, status)
    assert torch.equal(out[:sum(lens)].view(torch.int16), torch.cat(segs).view(torch.int16))
    assert int(status.item()) == 0
