"""GPU parity of the ZeRO-3 per-layer steps against the CPU oracle.

Stage 3 (ZeRO reading notes, 7 and 9): before a layer's forward, and again
before its backward, the layer's parameter parts are gathered from every rank
into one contiguous buffer; after its backward the layer's gradients are
reduced onto the owner of each part; the owner then runs the shard update.
Gather and reduce are bit-exact; the update follows the step's tolerances."""
import numpy as np
import pytest
import torch

import oracle as orc
import workloads as W
from helpers import hyper32, t2u16

pytestmark = pytest.mark.gpu
DEV = "cuda"
TDT = {1: torch.float16, 2: torch.bfloat16}


@pytest.fixture(scope="module")
def Z():
    import zero_dp_partitioned_gb300 as Z
    return Z


def dev16(a, dt):
    return torch.from_numpy(a.view(np.int16).copy()).view(TDT[dt]).to(DEV)


@pytest.mark.parametrize("ws,part", [(1, 5000), (2, 4096), (4, 54528), (4, 1001), (8, 2049), (3, 7)])
def test_gather_is_exact(Z, ws, part):
    rng = np.random.default_rng(ws * 1000 + part)
    parts = [rng.integers(0, 1 << 16, part, dtype=np.uint64).astype(np.uint16) for _ in range(ws)]
    dparts = [dev16(p, 2) for p in parts]
    out = torch.full((ws * part,), float("nan"), dtype=torch.bfloat16, device=DEV)
    Z.zero3_gather_layer(dparts, ws * part, Z.ZERO_BF16, out)
    torch.cuda.synchronize()
    assert np.array_equal(t2u16(out), orc.zero3_gather(parts))


@pytest.mark.parametrize("dt", [1, 2])
@pytest.mark.parametrize("ws,part", [(4, 54528), (4, 999), (2, 8), (8, 10000)])
def test_reduce_bucket_is_exact(Z, dt, ws, part):
    g = W.generator(ws + part, "cpu")
    buckets = []
    for r in range(ws):
        b = torch.zeros(ws * part, dtype=TDT[dt])
        W.fill_normal_(b, 5e-4, g, 256.0 if dt == 1 else 1.0)
        buckets.append(t2u16(b))
    ws_buf = torch.zeros(Z.zero_workspace_bytes(), dtype=torch.uint8, device=DEV)
    stats = torch.zeros(16, dtype=torch.uint8, device=DEV)
    acc = orc.ExactAccumulator()
    for owner in range(ws):
        out = torch.empty(part, dtype=TDT[dt], device=DEV)
        Z.zero3_reduce_bucket([dev16(b, dt) for b in buckets], owner, ws * part, dt, out, owner > 0, stats, ws_buf,
                              ws_buf.numel())
        torch.cuda.synchronize()
        ref, ovf = orc.zero3_reduce(buckets, owner, part, dt, acc)
        assert np.array_equal(t2u16(out), ref) and ovf == 0
    st = Z.read_stats(stats)
    assert st.overflow == 0 and st.sumsq == pytest.approx(acc.value(), rel=1e-6)


def test_layer_pipeline_three_steps(Z):
    """A small Llama-shaped group as ZeRO-3 units, rank 1 of 4: each step
    gathers every unit forward and backward, reduces every unit's gradients
    onto rank 1's part, and updates rank 1's parameter shard."""
    specs = W.llama_group(L=3, d=64, hq=4, hkv=2, hd=16, ff=160, V=300)
    units = W.llama_units(specs, L=3)
    nd, me, dt = 4, 1, 2
    assert all(u % nd == 0 for u in units)
    parts = [u // nd for u in units]
    uoff = np.concatenate([[0], np.cumsum(parts)[:-1]]).astype(int)
    shard_len = int(sum(parts))
    # the full model's parameters, cut into units and parts: rank r's persistent shard is its parts of every unit
    flat = torch.zeros(sum(units), dtype=torch.bfloat16)
    W.init_params_(flat, specs, W.generator(3, "cpu"))
    flat = t2u16(flat)
    shards = [np.concatenate([flat[sum(units[:u]) + r * parts[u]: sum(units[:u]) + (r + 1) * parts[u]]
                              for u in range(len(units))]) for r in range(nd)]
    gens = [W.generator(5 + r, "cpu") for r in range(nd)]
    h = hyper32()

    d_shards = [dev16(s, dt) for s in shards]
    master = torch.from_numpy(orc.widen_16(shards[me], dt)).to(DEV)
    m = torch.zeros(shard_len, device=DEV)
    v = torch.zeros(shard_len, device=DEV)
    gshard = torch.empty(shard_len, dtype=torch.bfloat16, device=DEV)
    layer = torch.empty(max(units), dtype=torch.bfloat16, device=DEV)
    wsb = torch.zeros(Z.zero_workspace_bytes(), dtype=torch.uint8, device=DEV)
    stats = torch.zeros(16, dtype=torch.uint8, device=DEV)
    res = torch.zeros(48, dtype=torch.uint8, device=DEV)

    o_master = orc.widen_16(shards[me], dt)
    o_m = np.zeros(shard_len, np.float32)
    o_v = np.zeros(shard_len, np.float32)
    o_param = shards[me].copy()
    for t in (1, 2, 3):
        buckets = []
        for u, U in enumerate(units):
            row = []
            for r in range(nd):
                b = torch.zeros(U, dtype=torch.bfloat16)
                W.fill_normal_(b, 5e-4, gens[r])
                row.append(t2u16(b))
            buckets.append(row)
        order = list(range(len(units))) + list(reversed(range(len(units))))   # forward, then backward
        for u in order:
            ptrs = [d_shards[r][uoff[u]:uoff[u] + parts[u]] for r in range(nd)]
            Z.zero3_gather_layer(ptrs, units[u], dt, layer)
            torch.cuda.synchronize()
            host_parts = [s[uoff[u]:uoff[u] + parts[u]] for s in shards]
            host_parts[me] = t2u16(d_shards[me][uoff[u]:uoff[u] + parts[u]])
            assert np.array_equal(t2u16(layer[:units[u]]), orc.zero3_gather(host_parts))
        acc = orc.ExactAccumulator()
        o_g = np.empty(shard_len, np.uint16)
        for k, u in enumerate(reversed(range(len(units)))):
            Z.zero3_reduce_bucket([dev16(b, dt) for b in buckets[u]], me, units[u], dt,
                                  gshard[uoff[u]:uoff[u] + parts[u]], k > 0, stats, wsb, wsb.numel())
            o_g[uoff[u]:uoff[u] + parts[u]], _ = orc.zero3_reduce(buckets[u], me, parts[u], dt, acc)
        sh = [Z.shard(shard_len, 0, 0, master, m, v, grad_shard=gshard)]
        Z.zero_shard_apply(sh, dt, d_shards[me], dt, Z.hyper(step=t, **{k: h[k] for k in
                           ("lr", "beta1", "beta2", "eps", "weight_decay", "max_grad_norm")}), 1.0, stats, 0.0, 0, wsb,
                           wsb.numel(), res)
        torch.cuda.synchronize()
        # the oracle, in the same order: reduce every unit, then the shard update
        k_mult, norm, _ = orc.grad_multiplier(acc.value(), 1.0, 0.0)
        sc = orc.make_scalars(h["lr"], h["beta1"], h["beta2"], h["eps"], h["weight_decay"], t)
        orc.apply(o_g, dt, o_master, o_m, o_v, o_param, dt, k_mult, sc)
        assert np.array_equal(t2u16(gshard), o_g)
        r = Z.read_result(res)
        assert r.applied == 1 and r.grad_norm == pytest.approx(norm, rel=1e-5)
        assert np.array_equal(t2u16(d_shards[me]), o_param)
        assert np.array_equal(master.cpu().numpy().view(np.uint32), o_master.view(np.uint32))
        assert np.array_equal(v.cpu().numpy().view(np.uint32), o_v.view(np.uint32))


def test_gather_segments_is_exact(Z):
    rng = np.random.default_rng(12)
    for trial in range(12):
        n = int(rng.integers(1, 6))
        lens = [int(x) for x in rng.choice([0, 1, 7, 8, 1000, 4097, 54528], n)]
        host = [rng.integers(0, 1 << 16, L + 3, dtype=np.uint64).astype(np.uint16) for L in lens]
        shift = int(rng.integers(0, 2))                  # 2-byte offset: the unaligned path
        dev = [dev16(h, 2)[shift:shift + L] for h, L in zip(host, lens)]
        out = torch.zeros(max(1, sum(lens)), dtype=torch.bfloat16, device=DEV)
        Z.zero3_gather_segments(dev, lens, Z.ZERO_BF16, out)
        torch.cuda.synchronize()
        ref = orc.gather_segments([h[shift:shift + L].copy() for h, L in zip(host, lens)])
        assert np.array_equal(t2u16(out)[:sum(lens)], ref)


def _pieces(plan_fn, inter_fn, units, nd):
    """pieces[u] = [(rank, first element in the unit, first element in the rank's segment, length)]."""
    p = plan_fn(units, nd)
    offs, rnum = list(p["tensor_offsets"]), list(p["rank_numels"])
    out = {u: [] for u in range(len(units))}
    for r in range(nd):
        for u, u0, s0, ln in inter_fn(offs, units, int(p["rank_offsets"][r]), int(rnum[r])):
            out[int(u)].append((r, int(u0), int(s0), int(ln)))
    return p, out


def test_owner_broadcast_pipeline_three_steps(Z):
    """ZeRO-3 with owner broadcast, rank 1 of 4 on a small Llama-shaped group:
    each rank keeps one contiguous segment of the flat vector; every unit is
    rebuilt forward and backward from the pieces of its owners' segments;
    rank 1 reduces every rank's gradient over the pieces it owns and updates
    its segment.  Bit-exact against the oracle."""
    specs = W.llama_group(L=3, d=64, hq=4, hkv=2, hd=16, ff=160, V=300)
    units = W.llama_units(specs, L=3)
    nd, me, dt = 4, 1, 2
    p, pieces = _pieces(Z.zero_plan, Z.zero_plan_intersections, units, nd)
    po, pieces_o = _pieces(lambda u, n: orc.plan(u, n, 0), orc.plan_intersections, units, nd)
    assert pieces == pieces_o and list(p["rank_offsets"]) == list(po["rank_offsets"])
    P = p["padded_total"]
    flat = torch.zeros(P, dtype=torch.bfloat16)
    W.init_params_(flat, specs, W.generator(3, "cpu"))
    flat = t2u16(flat)
    segs_h = [flat[int(o):int(o) + int(n)].copy() for o, n in zip(p["rank_offsets"], p["rank_numels"])]
    segs = [dev16(s, dt) for s in segs_h]
    L = int(p["rank_numels"][me])
    master = torch.from_numpy(orc.widen_16(segs_h[me], dt)).to(DEV)
    m, v = torch.zeros(L, device=DEV), torch.zeros(L, device=DEV)
    gseg = torch.zeros(L, dtype=torch.bfloat16, device=DEV)
    layer = torch.empty(max(units), dtype=torch.bfloat16, device=DEV)
    wsb = torch.zeros(Z.zero_workspace_bytes(), dtype=torch.uint8, device=DEV)
    stats = torch.zeros(16, dtype=torch.uint8, device=DEV)
    res = torch.zeros(48, dtype=torch.uint8, device=DEV)
    o_master, o_m, o_v = orc.widen_16(segs_h[me], dt), np.zeros(L, np.float32), np.zeros(L, np.float32)
    o_param = segs_h[me].copy()
    gens = [W.generator(5 + r, "cpu") for r in range(nd)]
    h = hyper32()
    for t in (1, 2, 3):
        buckets = {}
        for u, U in enumerate(units):
            buckets[u] = [t2u16(W.fill_normal_(torch.zeros(U, dtype=torch.bfloat16), 5e-4, gens[r])) for r in range(nd)]
        host_segs = list(segs_h)
        host_segs[me] = t2u16(segs[me])
        for u in list(range(len(units))) + list(reversed(range(len(units)))):
            Z.zero3_gather_segments([segs[r][s0:s0 + ln] for r, u0, s0, ln in pieces[u]],
                                    [ln for *_, ln in pieces[u]], dt, layer)
            torch.cuda.synchronize()
            ref = orc.gather_segments([host_segs[r][s0:s0 + ln] for r, u0, s0, ln in pieces[u]])
            assert np.array_equal(t2u16(layer[:units[u]]), ref)
        acc = orc.ExactAccumulator()
        o_g = np.zeros(L, np.uint16)
        first = True
        for u in reversed(range(len(units))):
            for r, u0, s0, ln in pieces[u]:
                if r != me:
                    continue
                sh = [Z.shard(ln, u0, 0, None, None, None, grad_shard=gseg[s0:s0 + ln])]
                Z.zero_shard_reduce([dev16(b, dt) for b in buckets[u]], dt, sh, not first, stats, wsb, wsb.numel())
                first = False
                o_g[s0:s0 + ln] = orc.reduce(buckets[u], dt, u0, ln)
                orc.stats(o_g[s0:s0 + ln], dt, acc)
        Z.zero_shard_apply([Z.shard(L, 0, 0, master, m, v, grad_shard=gseg)], dt, segs[me], dt,
                           Z.hyper(step=t, **{k: h[k] for k in ("lr", "beta1", "beta2", "eps", "weight_decay",
                                                                  "max_grad_norm")}),
                           1.0, stats, 0.0, 0, wsb, wsb.numel(), res)
        torch.cuda.synchronize()
        k_mult, norm, _ = orc.grad_multiplier(acc.value(), 1.0, 0.0)
        orc.apply(o_g, dt, o_master, o_m, o_v, o_param, dt, k_mult,
                  orc.make_scalars(h["lr"], h["beta1"], h["beta2"], h["eps"], h["weight_decay"], t))
        r_ = Z.read_result(res)
        assert r_.applied == 1 and r_.grad_norm == pytest.approx(norm, rel=1e-5)
        assert np.array_equal(t2u16(gseg), o_g)
        assert np.array_equal(t2u16(segs[me]), o_param)
        assert np.array_equal(master.cpu().numpy().view(np.uint32), o_master.view(np.uint32))
        assert np.array_equal(m.cpu().numpy().view(np.uint32), o_m.view(np.uint32))


def _aligned_view(host_u16, shift, L):
    """A device view of L elements starting `shift` elements past a 256-byte aligned allocation."""
    base = dev16(host_u16, 2)
    assert base.data_ptr() % 256 == 0
    return base[shift:shift + L]


@pytest.mark.parametrize("n_ctas", [0, 1, 3, 32])
def test_gather_bulk_is_exact(Z, n_ctas):
    """Segments that agree with their slot modulo 16 bytes (the TMA path, with
    unaligned heads and ragged tails) and segments that do not (the
    register-staged fallback), on a bounded CTA count."""
    rng = np.random.default_rng(40 + n_ctas)
    for trial in range(10):
        n = int(rng.integers(1, 7))
        lens = [int(x) for x in rng.choice([0, 1, 7, 8, 9, 1000, 4097, 54528, 300001], n)]
        out_shift = int(rng.integers(0, 8))
        congruent = trial % 3 != 2
        offs = np.concatenate([[0], np.cumsum(lens)[:-1]]).astype(int)
        shifts = [((out_shift + int(o)) % 8) if congruent else int(rng.integers(0, 8)) for o in offs]
        host = [rng.integers(0, 1 << 16, L + 8, dtype=np.uint64).astype(np.uint16) for L in lens]
        dev = [_aligned_view(h, s, L) for h, s, L in zip(host, shifts, lens)]
        out_base = torch.zeros(sum(lens) + 16, dtype=torch.bfloat16, device=DEV)
        out = out_base[out_shift:out_shift + max(1, sum(lens))]
        status = torch.zeros(1, dtype=torch.int32, device=DEV)
        Z.zero3_gather_bulk(dev, lens, Z.ZERO_BF16, out, n_ctas, status)
        torch.cuda.synchronize()
        ref = orc.gather_segments([h[s:s + L].copy() for h, s, L in zip(host, shifts, lens)])
        got = t2u16(out_base)
        assert np.array_equal(got[out_shift:out_shift + sum(lens)], ref), (lens, shifts, out_shift)
        assert not got[:out_shift].any() and not got[out_shift + sum(lens):].any()     # nothing outside the slot
        assert int(status.item()) == 0


def test_gather_bulk_equals_gather_layer_on_llama_parts(Z):
    """One Llama-3-8B block unit (218,112,000 elements, world-size-4 parts of
    54,528,000; 436 MB, larger than L2): the TMA gather on every SM and on 32
    CTAs equals zero3_gather_layer."""
    U, nd = 218_112_000, 4
    rng = np.random.default_rng(3)
    parts = [dev16(rng.integers(0, 1 << 16, U // nd, dtype=np.uint16), 2) for _ in range(nd)]
    a = torch.empty(U, dtype=torch.bfloat16, device=DEV)
    b = torch.empty(U, dtype=torch.bfloat16, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    Z.zero3_gather_layer(parts, U, Z.ZERO_BF16, a)
    for n_ctas in (0, 32):
        b.zero_()
        Z.zero3_gather_bulk(parts, [U // nd] * nd, Z.ZERO_BF16, b, n_ctas, status)
        torch.cuda.synchronize()
        assert torch.equal(a.view(torch.int16), b.view(torch.int16)) and int(status.item()) == 0


def test_gather_bulk_wait_timeout_is_reported_and_harmless(Z, monkeypatch):
    """With the wait limit at zero tries every CTA gives up on its first load:
    status bit 0 is set, the CTAs drain what they started and return, and the
    next call (default limit) is exact."""
    L = 200_000
    rng = np.random.default_rng(5)
    host = rng.integers(0, 1 << 16, L, dtype=np.uint64).astype(np.uint16)
    src = dev16(host, 2)
    out = torch.zeros(L, dtype=torch.bfloat16, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    monkeypatch.setenv("ZERO_GB300_SPIN_LIMIT", "0")
    Z.zero3_gather_bulk([src], [L], Z.ZERO_BF16, out, 4, status)
    torch.cuda.synchronize()
    assert int(status.item()) & 1
    monkeypatch.delenv("ZERO_GB300_SPIN_LIMIT")
    status.zero_()
    Z.zero3_gather_bulk([src], [L], Z.ZERO_BF16, out, 4, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0 and np.array_equal(t2u16(out), host)


def test_gather_bulk_argument_errors(Z):
    src = torch.zeros(64, dtype=torch.bfloat16, device=DEV)
    out = torch.zeros(64, dtype=torch.bfloat16, device=DEV)
    status = torch.zeros(2, dtype=torch.int32, device=DEV)
    for args, code in (((([src], [64], 7, out, 0, status)), Z.ZERO_EINVAL),
                       ((([src], [64], Z.ZERO_BF16, out, -1, status)), Z.ZERO_EINVAL),
                       ((([src], [-1], Z.ZERO_BF16, out, 0, status)), Z.ZERO_EINVAL),
                       ((([src] * 65, [1] * 65, Z.ZERO_BF16, out, 0, status)), Z.ZERO_ELIMIT),
                       ((([src], [64], Z.ZERO_BF16, out, 0, status.view(torch.uint8)[1:])), Z.ZERO_EINVAL),
                       ((([src.view(torch.uint8)[1:]], [8], Z.ZERO_BF16, out, 0, status)), Z.ZERO_EALIGN)):
        with pytest.raises(Z.ZeroError) as e:
            Z.zero3_gather_bulk(*args)
        assert e.value.code == code


def test_prefetch_schedule_gives_every_consumer_its_own_unit(Z):
    """The pipelined schedule: unit u+1 is gathered on a side stream (TMA, 8
    CTAs) into the other of two layer buffers while the consumer of unit u
    runs on the main stream; forward then backward (reverse order).  Each
    consumer snapshots the buffer it was given; every snapshot equals the
    oracle's gather of its unit, so no gather overwrote a buffer in use and no
    consumer ran ahead of its gather."""
    rng = np.random.default_rng(9)
    nd = 4
    units = [int(x) * 8 * nd for x in rng.integers(2000, 40000, 7)]
    host = [[rng.integers(0, 1 << 16, u // nd, dtype=np.uint64).astype(np.uint16) for _ in range(nd)] for u in units]
    parts = [[dev16(h, 2) for h in hu] for hu in host]
    bufs = [torch.empty(max(units), dtype=torch.bfloat16, device=DEV) for _ in range(2)]
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    main, side = torch.cuda.current_stream(), torch.cuda.Stream()
    order = list(range(len(units))) + list(reversed(range(len(units))))
    gathered = [torch.cuda.Event() for _ in order]
    consumed = [torch.cuda.Event() for _ in order]
    snaps = []
    x = torch.randn(256, 256, device=DEV)

    def gather(i):
        if i >= 2:
            side.wait_event(consumed[i - 2])          # its buffer's previous consumer is done
        u = order[i]
        Z.zero3_gather_bulk(parts[u], [units[u] // nd] * nd, Z.ZERO_BF16, bufs[i % 2], 8, status, stream=side)
        gathered[i].record(side)

    side.wait_stream(main)
    gather(0)
    for i, u in enumerate(order):
        if i + 1 < len(order):
            gather(i + 1)                             # prefetch the next unit
        main.wait_event(gathered[i])
        for _ in range(3):                            # a stand-in consumer that takes some time
            x = torch.tanh(x @ x)
        snaps.append(bufs[i % 2][:units[u]].clone())
        consumed[i].record(main)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for i, u in enumerate(order):
        assert np.array_equal(t2u16(snaps[i]), orc.gather_segments([h.copy() for h in host[u]])), (i, u)


def _fused_pipeline_problem(seed, units, nd, dt, steps, S):
    """Rank shards of a ZeRO-3 group (every rank's part of every unit) and, per
    step, every rank's full-unit gradient buckets, as host bit patterns."""
    parts = [u // nd for u in units]
    g = W.generator(seed, "cpu")
    shards = []
    for r in range(nd):
        x = torch.zeros(sum(parts), dtype=TDT[dt])
        W.fill_normal_(x, 0.02, g)
        shards.append(t2u16(x))
    gens = [W.generator(seed + 1 + r, "cpu") for r in range(nd)]
    buckets = []
    for _ in range(steps):
        step = []
        for U in units:
            row = []
            for r in range(nd):
                b = torch.zeros(U, dtype=TDT[dt])
                W.fill_normal_(b, 1e-2, gens[r], S)
                row.append(t2u16(b))
            step.append(row)
        buckets.append(step)
    return parts, shards, buckets


def _owner_slices(buckets_step, parts, nd, me):
    """Rank r's gradient over the owner's concatenated shard: its bucket of
    every unit, cut to the owner's part -- what the oracle reduces."""
    return [np.concatenate([buckets_step[u][r][me * p:(me + 1) * p] for u, p in enumerate(parts)]) for r in range(nd)]


@pytest.mark.parametrize("dt", [1, 2])
def test_fused_unit_passes_then_commit_match_the_oracle(Z, dt):
    """ZeRO-3 without clipping, fused per unit: after each unit's backward its
    buckets are reduced onto rank 1's part and that part is updated in the
    same pass (zero_shard_step_partial, speculatively, into the second state
    set), and the step is decided after the last unit (zero_shard_step_commit).
    Three steps, the second with +inf in one rank's bucket of the middle unit:
    skipped everywhere, the parameters restored, t kept, S halved.  Bit-exact
    against the oracle's step over the concatenated shard."""
    nd, me, steps = 4, 1, 3
    units = [4096 * 4, 10001 * 4, 333 * 4, 7 * 4]
    S = 256.0 if dt == 1 else 1.0
    parts, shards, buckets = _fused_pipeline_problem(40 + dt, units, nd, dt, steps, S)
    buckets[1][1][2] = buckets[1][1][2].copy()
    buckets[1][1][2][me * parts[1] + 17] = 0x7C00 if dt == 1 else 0x7F80
    uoff = [sum(parts[:i]) for i in range(len(parts))]
    L = sum(parts)
    param = dev16(shards[me], dt)
    sets = [[torch.from_numpy(orc.widen_16(shards[me], dt)).to(DEV), torch.zeros(L, device=DEV),
             torch.zeros(L, device=DEV)], [torch.empty(L, device=DEV) for _ in range(3)]]
    wsb = torch.zeros(Z.zero_workspace_bytes(), dtype=torch.uint8, device=DEV)
    stats = torch.zeros(16, dtype=torch.uint8, device=DEV)
    res = torch.zeros(48, dtype=torch.uint8, device=DEV)
    h = hyper32()
    o = dict(numel=L, grad_off=0, param_off=0, master=orc.widen_16(shards[me], dt), m=np.zeros(L, np.float32),
             v=np.zeros(L, np.float32))
    o_param = shards[me].copy()
    cur, t, So = 0, 1, S
    applied = []
    for k in range(steps):
        A, B = sets[cur], sets[1 - cur]
        hy = Z.hyper(h["lr"], h["beta1"], h["beta2"], h["eps"], h["weight_decay"], 0.0, t)
        for i, u in enumerate(reversed(range(len(units)))):
            part = Z.shard(parts[u], me * parts[u], uoff[u], *(x[uoff[u]:uoff[u] + parts[u]] for x in A),
                           *(x[uoff[u]:uoff[u] + parts[u]] for x in B))
            Z.zero_shard_step_partial([dev16(b, dt) for b in buckets[k][u]], dt, [part], param, dt, hy, So, i > 0,
                                      stats, wsb, wsb.numel())
        whole = [Z.shard(L, 0, 0, *A, *B)]
        Z.zero_shard_step_commit(whole, param, dt, So, stats, 0.0, 0, res)
        torch.cuda.synchronize()
        rg = Z.read_result(res)
        ro, _ = orc.zero_step(_owner_slices(buckets[k], parts, nd, me), dt, [o], o_param, dt, h, t, np.float32(So))
        assert (rg.overflow, rg.applied, rg.path, rg.status) == (ro.overflow, ro.applied, 3, 0)
        assert rg.grad_mult == ro.grad_mult
        if ro.applied:
            assert rg.sumsq == pytest.approx(ro.sumsq, rel=1e-9)
            cur ^= 1
            t += 1
        else:
            So /= 2
        applied.append(rg.applied)
        assert np.array_equal(t2u16(param), o_param)
        for x, ref in zip(sets[cur], (o["master"], o["m"], o["v"])):
            assert np.array_equal(x.cpu().numpy().view(np.uint32), ref.view(np.uint32))
    assert applied == [1, 0, 1]


def test_partial_pass_argument_errors(Z):
    n = 4096
    g = torch.zeros(n, dtype=torch.bfloat16, device=DEV)
    st = [torch.zeros(n, device=DEV) for _ in range(6)]
    flat = torch.zeros(n, dtype=torch.bfloat16, device=DEV)
    wsb = torch.zeros(Z.zero_workspace_bytes(), dtype=torch.uint8, device=DEV)
    stats = torch.zeros(16, dtype=torch.uint8, device=DEV)
    res = torch.zeros(48, dtype=torch.uint8, device=DEV)
    two = [Z.shard(n, 0, 0, *st)]
    for sh, hy, s_, code in (([Z.shard(n, 0, 0, *st[:3])], Z.hyper(), stats, Z.ZERO_EINVAL),     # in place
                             (two, Z.hyper(max_grad_norm=1.0), stats, Z.ZERO_EINVAL),            # clipping
                             (two, Z.hyper(), 0, Z.ZERO_EINVAL),                                  # no stats
                             (two, Z.hyper(step=0), stats, Z.ZERO_EINVAL)):
        with pytest.raises(Z.ZeroError) as e:
            Z.zero_shard_step_partial([g], Z.ZERO_BF16, sh, flat, Z.ZERO_BF16, hy, 1.0, 0, s_, wsb, wsb.numel())
        assert e.value.code == code
    with pytest.raises(Z.ZeroError) as e:
        Z.zero_shard_step_commit(two, flat, Z.ZERO_BF16, 1.0, stats, 0.0, 0, res[4:])
    assert e.value.code == Z.ZERO_EINVAL
