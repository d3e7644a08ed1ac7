#!/usr/bin/env python
"""Benchmark of the partitioned mixed-precision optimizer step on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--no-e2e] [--no-cpu-baseline]

One step = one pass of the per-step hot path over one batch of synthetic
gradients: reduce the N_d ranks' gradient slices, overflow check, norm,
unscale/clip, AdamW on the fp32 shards, cast-store of the 16-bit parameters
into the flat buffer (and, for the ZeRO-3 workload, the per-layer gathers and
bucket reduces).  The default workload is the GPT-2 1.5B-shaped group with all
8 ranks simulated on one GPU.  Rank 0 prints one JSON line.

Metric: shard AdamW-step elements per second (shard elements updated per
step / step time), with the dominant kernel's achieved HBM bandwidth against
the measured copy bandwidth of this GPU.  Under torchrun each rank runs an
independent replica (the simulated ranks already live on one GPU; there is no
cross-GPU exchange), so scaling is weak and the value is the sum over ranks.

--impl reference times the CPU oracle on the host cores on a bounded sample of
the same workload (the oracle is the only reference this method has).
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "shard AdamW-step elements/s; achieved HBM GB/s vs GB300 roofline"
NOMINAL_HBM_GBS = 8000.0      # HBM3e, nominal


def log(*a):
    print(*a, file=sys.stderr, flush=True)


# ------------------------------------------------------------------ environment
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, ws, local


def mem_available_bytes():
    try:
        for line in open("/proc/meminfo"):
            if line.startswith("MemAvailable:"):
                return int(line.split()[1]) * 1024
    except OSError:
        pass
    return 0


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def kernel_source_hash():
    """Hash of the kernel sources' code: comments and blank lines are left
    out, so that a capture stays valid across edits that change no code."""
    import re
    h = hashlib.sha256()
    d = os.path.join(ROOT, "zero_dp_partitioned_gb300", "csrc")
    for f in sorted(os.listdir(d)):
        text = open(os.path.join(d, f)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        code = "\n".join(line.rstrip() for line in text.splitlines() if line.strip())
        h.update(f.encode() + b"\0" + code.encode() + b"\0")
    return h.hexdigest()[:16]


def ncu_traffic(workload, kernel):
    """DRAM bytes per launch from a committed ncu capture of this kernel, if it
    was taken on the current kernel sources (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        d = json.load(open(p))
        e = d[workload][kernel]
        if e.get("source_hash") == kernel_source_hash():
            return float(e["bytes_per_launch"])
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.f = None

    def start(self):
        try:
            self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                                          "-i", str(self.index), "-lms", "100"], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if not self.proc:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.flush()
        rows = [r.split(",") for r in open(self.f.name).read().strip().splitlines() if r.strip()]
        os.unlink(self.f.name)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        sm, mx, reasons = [], [], set()
        for r in rows:
            try:
                sm.append(float(r[0]))
                mx.append(float(r[1]))
                for n, v in zip(names, r[3:7]):
                    if v.strip().lower().startswith("active"):
                        reasons.add(n)
            except (ValueError, IndexError):
                continue
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ kernel timing
class KernelTimer:
    """CUDA events on the launching (current) stream around library calls,
    grouped by kernel kind.  One pair of events may enclose several
    back-to-back launches of the same kernel (`launches`): consecutive
    launches then run with no event between them, and the kind's time per
    launch is the enclosed time divided by the launch count."""

    def __init__(self, torch):
        self.torch = torch
        self.events = []          # (kind, launches, start, end)
        self.on = False

    def _event(self):
        return self.torch.cuda.Event(enable_timing=True)

    def __call__(self, kind, launches=1):
        timer = self

        class _Ctx:
            def __enter__(self):
                if timer.on:
                    self.a = timer._event()
                    self.a.record()

            def __exit__(self, *exc):
                if timer.on:
                    b = timer._event()
                    b.record()
                    timer.events.append((kind, launches, self.a, b))
        return _Ctx()

    def per_kind(self, steps):
        out, each = {}, {}
        for kind, n, a, b in self.events:
            d = out.setdefault(kind, {"ms_total": 0.0, "launches": 0, "event_pairs": 0})
            ms = a.elapsed_time(b)
            d["ms_total"] += ms
            d["launches"] += n
            d["event_pairs"] += 1
            each.setdefault(kind, []).append(ms / n)
        for kind, d in out.items():
            d["ms_per_launch"] = d["ms_total"] / d["launches"]
            d["ms_median"] = statistics.median(each[kind])
            d["ms_per_step"] = d["ms_total"] / steps
        return out


def _hyper(Z, h, t, clip=0.0):
    return Z.hyper(h["lr"], h["beta1"], h["beta2"], h["eps"], h["weight_decay"], clip, t)


PATH_NAMES = {1: "k_step_fused (fused single pass)", 2: "k_apply (apply pass after k_reduce)",
              3: "k_step_fused partial passes, decided by k_commit"}


def _finish_step(Z, torch, res, res_h, st):
    res_h.copy_(res, non_blocking=True)
    torch.cuda.current_stream().synchronize()
    r = Z.read_result(res_h)
    st["path"] = r.path
    if r.applied:
        st["cur"] ^= 1
        st["t"] += 1
    else:
        st["S"] /= 2
    return r


E2E_SOURCE = {"mode": None}
HOST_RING_BYTES = 512 << 20      # device ring of zero_shard_step_host in the end-to-end runs


def _device_chain(Z, torch, dev, wl, n_table=1 << 16):
    """A device zero_chain starting at t = 1 with the workload's loss scale, and
    the AdamW scalar table of steps 1 .. n_table: the chained calls read t, S
    and the current state set from it, so steps follow one another with no
    host round trip."""
    hy = _hyper(Z, wl.hyper, 1, wl.max_grad_norm)
    table = torch.from_numpy(Z.zero_adam_scalar_table(hy, 1, n_table)).to(dev)
    chain = torch.frombuffer(bytearray(bytes(Z.chain(step=1, loss_scale=wl.loss_scale))), dtype=torch.uint8).to(dev)
    return hy, table, n_table, chain


def _check_chain(Z, chain):
    """After the timed steps: no chained step may have failed."""
    def check(steps):
        c = Z.read_chain(chain)
        if c.failed:
            raise RuntimeError(f"{c.failed} chained steps failed (status != 0)")
        return {"chain_after_timing": {"step": c.step, "applied": c.applied, "skipped": c.skipped}}
    return check


def _pin_copies(torch, bufs, e2e):
    """Pinned host copies of a step's input buffers for the end-to-end run.
    Every rank of the job pins at the same time, so the check is on the job's
    whole footprint: with room for all ranks' distinct buffers (and margin),
    each buffer gets its own pinned copy; otherwise one pinned buffer of the
    largest size is the host source of every device buffer -- the same bytes
    cross the link each step -- and the JSON line says so."""
    if not e2e:
        return None
    world = dist_env()[1]
    need = sum(b.numel() * b.element_size() for b in bufs)
    one = max(b.numel() * b.element_size() for b in bufs)
    avail = mem_available_bytes()
    if avail > 1.25 * world * need + (32 << 30):
        log(f"[bench] pinning {need / 1e9:.1f} GB of host gradients for the end-to-end run")
        E2E_SOURCE["mode"] = "a pinned host copy of every input buffer"
        return [torch.empty(b.shape, dtype=b.dtype, pin_memory=True).copy_(b) for b in bufs]
    if avail > 1.25 * world * one + (32 << 30):
        log(f"[bench] pinning one {one / 1e9:.1f} GB host buffer as the source of every input buffer")
        E2E_SOURCE["mode"] = "one pinned host buffer copied into every input buffer (host memory too small for all)"
        src = torch.empty(max(b.numel() for b in bufs), dtype=bufs[0].dtype, pin_memory=True)
        src[:bufs[0].numel()].copy_(bufs[0])
        return [src[:b.numel()] for b in bufs]
    log("[bench] not enough host memory for the end-to-end run")
    return None


# ------------------------------------------------------------------ workloads (our path)
def _small(layers, vocab):
    """Name suffix of a reduced case (fewer layers and/or a smaller vocabulary)
    of a workload's group: the same kernels on a few GB, for profiler captures."""
    return (f"-{layers}layers" if layers else "") + (f"-v{vocab}" if vocab else "")


def gpt2_desc(name, layers=48):
    """The GPT-2 workload's description, shared by both arms' `config`."""
    return (f"{name}: GPT-2-shaped group ({layers} layers, d=1600, vocab 50257, ctx 1024), "
            "N_d=8, all 8 ranks simulated on one GPU")


def gpt2_all_ranks(Z, W, torch, dev, e2e, timer, layers=None, vocab=None):
    """GPT-2 1.5B-shaped group, N_d = 8, all ranks on this GPU, bf16, ping-pong state (fused single pass)."""
    wl = W.workload("gpt2-1.5b-nd8")
    small = layers or vocab
    layers = layers or 48
    specs = W.gpt2_group(L=layers, V=vocab or 50257) if small else wl.specs
    nd = wl.nd
    plan = Z.zero_plan(W.numels(specs), nd)
    P = plan["padded_total"]
    name = f"gpt2{_small(layers, vocab)}-nd8" if small else "gpt2-1.5b-nd8"
    log(f"[bench] {name}: Psi={P} N_d={nd}; generating inputs")
    flat = W.flat_params(specs, P, torch.bfloat16, wl.param_seed, dev)
    grads = W.GradStream([1 + r for r in range(nd)], dev).draw_flat(
        [torch.empty(P, dtype=torch.bfloat16, device=dev) for _ in range(nd)], specs, W.gpt2_grad_std())
    sets = [[torch.empty(P, device=dev) for _ in range(3)] for _ in range(2)]

    def shards(cur):
        i, o = sets[cur], sets[1 - cur]
        return [Z.shard(n, off, off, i[0][off:off + n], i[1][off:off + n], i[2][off:off + n],
                        o[0][off:off + n], o[1][off:off + n], o[2][off:off + n])
                for off, n in zip(plan["rank_offsets"], plan["rank_numels"])]

    variants = [shards(0), shards(1)]
    Z.zero_shard_init(variants[0], flat, Z.ZERO_BF16)
    ws = torch.zeros(Z.zero_workspace_bytes(), dtype=torch.uint8, device=dev)
    res = torch.zeros(48, dtype=torch.uint8, device=dev)
    res_h = torch.zeros(48, dtype=torch.uint8).pin_memory()
    st = dict(cur=0, t=1, S=wl.loss_scale, chained=True)
    pinned = _pin_copies(torch, grads, e2e)
    # Device-timed steps are chained: t, S and the state set in use stay on the
    # device, so steps follow one another with no host round trip.
    hy = _hyper(Z, wl.hyper, 1)
    n_table = 1 << 16
    table = torch.from_numpy(Z.zero_adam_scalar_table(hy, 1, n_table)).to(dev)
    chain_dev = torch.frombuffer(bytearray(bytes(Z.chain(step=1, loss_scale=wl.loss_scale))),
                                 dtype=torch.uint8).to(dev)

    def host_from_chain():
        """The end-to-end steps keep the bookkeeping on the host: take it over."""
        if st["chained"]:
            c = Z.read_chain(chain_dev)
            if c.failed:
                raise RuntimeError(f"{c.failed} chained steps failed (status != 0)")
            st.update(cur=c.cur, t=c.step, S=c.loss_scale, chained=False)
    # End to end, the step takes its gradients from pinned host memory and
    # returns its product -- the updated 16-bit flat parameters, the
    # all-gather destination -- there: zero_shard_step_host copies the slices
    # up chunk by chunk into a device ring while the chunks already up are
    # reduced and updated, and copies each chunk's parameters down beside the
    # uploads (the link carries both directions at once).
    host = dict(params=None, staging=None)
    if pinned is not None:
        host["staging"] = torch.empty(HOST_RING_BYTES // 2, dtype=torch.int16, device=dev)
        if mem_available_bytes() > flat.numel() * flat.element_size() + (16 << 30):
            host["params"] = torch.empty(flat.shape, dtype=flat.dtype, pin_memory=True)
        else:
            log("[bench] not enough host memory for the parameter download of the end-to-end run")

    def step(from_host=False):
        if not from_host and st["chained"]:
            with timer("fused pass+k_recover"):
                Z.zero_shard_step_chained(grads, Z.ZERO_BF16, variants[0], flat, Z.ZERO_BF16, hy, table, 1, n_table,
                                          chain_dev, 0.0, 0, ws, ws.numel(), res)
            return
        host_from_chain()
        h = _hyper(Z, wl.hyper, st["t"])
        if from_host:
            Z.zero_shard_step_host(pinned, Z.ZERO_BF16, variants[st["cur"]], flat, Z.ZERO_BF16, host["params"], h,
                                   st["S"], 0.0, 0, host["staging"], HOST_RING_BYTES, ws, ws.numel(), res)
        else:
            with timer("fused pass+k_recover"):
                Z.zero_shard_step(grads, Z.ZERO_BF16, variants[st["cur"]], flat, Z.ZERO_BF16, h, st["S"], 0.0, 0,
                                  ws, ws.numel(), res)
        _finish_step(Z, torch, res, res_h, st)

    def path_of_last_step():
        return Z.read_result(res).path

    def e2e_parts():
        """The host link alone, timed like the end-to-end steps: one step's
        gradient upload, one parameter download, and both at once on two
        streams (what the end-to-end steps overlap)."""
        out = {}
        if host["params"] is None:
            return out
        main = torch.cuda.current_stream()
        lanes = {"up": torch.cuda.Stream(device=dev), "down": torch.cuda.Stream(device=dev)}

        def up():
            with torch.cuda.stream(lanes["up"]):
                for g, hp in zip(grads, pinned):
                    g.copy_(hp, non_blocking=True)

        def down():
            with torch.cuda.stream(lanes["down"]):
                host["params"].copy_(flat, non_blocking=True)

        times = {"upload_ms": [], "download_ms": [], "both_ms": []}
        for _ in range(3):                       # interleaved, so that each leg sees the link's moods
            for key, fns in (("upload_ms", (up,)), ("download_ms", (down,)), ("both_ms", (up, down))):
                torch.cuda.synchronize()
                a = torch.cuda.Event(enable_timing=True)
                a.record(main)
                for st_ in lanes.values():
                    st_.wait_event(a)
                for f in fns:
                    f()
                for st_ in lanes.values():
                    main.wait_stream(st_)
                b = torch.cuda.Event(enable_timing=True)
                b.record(main)
                torch.cuda.synchronize()
                times[key].append(a.elapsed_time(b))
        for key, x in times.items():
            out[key] = statistics.median(x)
            out[key + "_all"] = x
        out["upload_gbs"] = sum(g.numel() * 2 for g in grads) / (out["upload_ms"] / 1e3) / 1e9
        out["download_gbs"] = flat.numel() * 2 / (out["download_ms"] / 1e3) / 1e9
        return out

    bytes_step = (2 * nd + 26) * P
    return dict(name=name, step=step, state=st, elements=P, nd=nd, launches_per_step=3,
                path_of_last_step=path_of_last_step,
                kernel_bytes={"fused pass+k_recover": bytes_step},
                dominant_label=None,
                h2d=sum(g.numel() * 2 for g in grads) if pinned else None,
                d2h=(flat.numel() * flat.element_size() if host["params"] is not None else 0) + 48,
                e2e_ok=pinned is not None,
                e2e_parts=e2e_parts,
                e2e_note="zero_shard_step_host: each step's gradients are copied from pinned host memory in chunks "
                         f"into a {HOST_RING_BYTES >> 20} MiB device ring while the chunks already up are reduced and "
                         "updated (partial fused passes, one commit), and each chunk's updated 16-bit parameters are "
                         "copied to pinned host memory beside the uploads; the timed region holds one upload, one "
                         "parameter download and one result read per step",
                config={"workload": gpt2_desc(name, layers),
                        "psi": P, "n_d": nd, "shard_elements": plan["rank_numels"][0], "grad_dtype": "bf16",
                        "param_dtype": "bf16", "state": "f32 master/m/v, ping-pong", "path": "fused single pass",
                        "steps": "zero_shard_step_chained: t, S and the state set in use stay on the device "
                                 "(3 launches a step: the pass, the parameter restore check, the bookkeeping)",
                        "bytes_per_step": bytes_step,
                        "l2": f"inputs larger than L2 ({bytes_step / 1e9:.1f} GB per step), no flush"},
                formula_bytes=bytes_step, sample_for_cpu=lambda n: cpu_sample_gpt2(W, n))


def tiny_nd3(Z, W, torch, dev, e2e, timer, layers=None, vocab=None):
    """The small fp16 group (Psi = 70,282, N_d = 3, all ranks, S = 1024): a
    launch-bound step.  Its 2.3 MB of inputs fit in L2, so every step first
    writes a 256 MB buffer (an L2 flush); the flush is inside the step time,
    and the library call alone is timed by events around it."""
    wl = W.workload("tiny-nd3")
    nd = wl.nd
    numels = W.numels(wl.specs)
    plan = Z.zero_plan(numels, nd)
    P = plan["padded_total"]
    flat = W.flat_params(wl.specs, P, torch.float16, wl.param_seed, dev)
    grads = W.GradStream([1 + r for r in range(nd)], dev).draw_flat(
        [torch.empty(P, dtype=torch.float16, device=dev) for _ in range(nd)], wl.specs, lambda s: wl.grad_std,
        wl.loss_scale)
    sets = [[torch.empty(P, device=dev) for _ in range(3)] for _ in range(2)]

    def shards(cur):
        i, o = sets[cur], sets[1 - cur]
        return [Z.shard(n, off, off, i[0][off:off + n], i[1][off:off + n], i[2][off:off + n],
                        o[0][off:off + n], o[1][off:off + n], o[2][off:off + n])
                for off, n in zip(plan["rank_offsets"], plan["rank_numels"])]

    variants = [shards(0), shards(1)]
    Z.zero_shard_init(variants[0], flat, Z.ZERO_F16)
    ws = torch.zeros(Z.zero_workspace_bytes(), dtype=torch.uint8, device=dev)
    res = torch.zeros(48, dtype=torch.uint8, device=dev)
    res_h = torch.zeros(48, dtype=torch.uint8).pin_memory()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    st = dict(cur=0, t=1, S=wl.loss_scale)

    def step(from_host=False):
        flush.fill_(st["t"] & 0xFF)
        with timer("fused pass+k_recover"):
            Z.zero_shard_step(grads, Z.ZERO_F16, variants[st["cur"]], flat, Z.ZERO_F16, _hyper(Z, wl.hyper, st["t"]),
                              st["S"], 0.0, 0, ws, ws.numel(), res)
        _finish_step(Z, torch, res, res_h, st)

    hy = _hyper(Z, wl.hyper, 1)
    table = torch.from_numpy(Z.zero_adam_scalar_table(hy, 1, 1 << 12)).to(dev)

    def extra(steps):
        """The same steps chained on the device and replayed from one CUDA graph
        (20 steps, each with its L2 flush), against the host-driven steps above."""
        chain_dev = torch.frombuffer(bytearray(bytes(Z.chain(step=1, loss_scale=wl.loss_scale))),
                                     dtype=torch.uint8).to(dev)

        def chained():
            flush.fill_(7)
            Z.zero_shard_step_chained(grads, Z.ZERO_F16, variants[0], flat, Z.ZERO_F16, hy, table, 1, 1 << 12,
                                      chain_dev, 0.0, 0, ws, ws.numel(), res)

        chained()                               # one-time set-up outside the capture
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=torch.cuda.Stream()):
            for _ in range(20):
                chained()
        g.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = 10
        a.record()
        for _ in range(reps):
            g.replay()
        b.record()
        torch.cuda.synchronize()
        c = Z.read_chain(chain_dev)
        if c.failed:
            raise RuntimeError("chained tiny steps failed")
        return {"graph_of_chained_steps_ms_per_step": a.elapsed_time(b) / (20 * reps),
                "graph_steps_applied": c.applied}

    bytes_step = (2 * nd + 26) * P
    return dict(name="tiny-nd3", step=step, state=st, elements=P, nd=nd, launches_per_step=2,
                kernel_bytes={"fused pass+k_recover": bytes_step}, dominant_label=None, h2d=None, d2h=48,
                e2e_ok=False, formula_bytes=bytes_step, sample_for_cpu=None, extra=extra,
                config={"workload": "tiny-nd3: three tensors [257,129], [129], [1000,37] (Psi = 70,282), N_d=3, "
                                    "all ranks, fp16, S = 1024",
                        "psi": sum(numels), "padded": P, "n_d": nd, "path": "fused single pass",
                        "l2": "inputs fit in L2: a 256 MB write before every step flushes it (inside the step "
                              "time); the kernels' own time is in kernels.*.ms_per_launch"})


def gpt2_allreduce(Z, W, torch, dev, e2e, timer, layers=None, vocab=None):
    """The GPT-2 1.5B group with stage 1's full all-reduce: the reduce pass
    writes the whole averaged gradient (the all-reduce result every rank
    holds), then each rank's shard is updated from its slice of it."""
    wl = W.workload("gpt2-1.5b-nd8")
    layers = layers or 48
    specs = wl.specs if layers == 48 else W.gpt2_group(L=layers)
    nd = wl.nd
    plan = Z.zero_plan(W.numels(specs), nd)
    P = plan["padded_total"]
    name = "gpt2-1.5b-nd8-allreduce" if layers == 48 else f"gpt2-{layers}layers-nd8-allreduce"
    log(f"[bench] {name}: Psi={P} N_d={nd}; generating inputs")
    flat = W.flat_params(specs, P, torch.bfloat16, wl.param_seed, dev)
    grads = W.GradStream([1 + r for r in range(nd)], dev).draw_flat(
        [torch.empty(P, dtype=torch.bfloat16, device=dev) for _ in range(nd)], specs, W.gpt2_grad_std())
    state = [torch.empty(P, device=dev) for _ in range(3)]
    avg = torch.empty(P, dtype=torch.bfloat16, device=dev)          # the all-reduced gradient
    sh = [Z.shard(n, off, off, *(x[off:off + n] for x in state), grad_shard=avg[off:off + n])
          for off, n in zip(plan["rank_offsets"], plan["rank_numels"])]
    Z.zero_shard_init(sh, flat, Z.ZERO_BF16)
    ws = torch.zeros(Z.zero_workspace_bytes(), dtype=torch.uint8, device=dev)
    stats = torch.zeros(16, dtype=torch.uint8, device=dev)
    res = torch.zeros(48, dtype=torch.uint8, device=dev)
    res_h = torch.zeros(48, dtype=torch.uint8).pin_memory()
    st = dict(cur=0, t=1, S=wl.loss_scale)
    hy, table, n_table, chain = _device_chain(Z, torch, dev, wl)

    def step(from_host=False):
        with timer("k_reduce"):
            Z.zero_shard_reduce(grads, Z.ZERO_BF16, sh, 0, stats, ws, ws.numel())
        with timer("k_apply"):
            Z.zero_shard_apply_chained(sh, Z.ZERO_BF16, flat, Z.ZERO_BF16, hy, table, 1, n_table, chain, stats, 0.0, 0,
                                       ws, ws.numel(), res)

    def path_of_last_step():
        return Z.read_result(res).path

    return dict(name=name, step=step, state=st, elements=P, nd=nd, launches_per_step=3,
                path_of_last_step=path_of_last_step, extra=_check_chain(Z, chain),
                kernel_bytes={"k_reduce": (2 * nd + 2) * P, "k_apply": 28 * P}, dominant_label=None,
                h2d=None, d2h=48, e2e_ok=False, formula_bytes=(2 * nd + 26) * P,
                config={"workload": f"{name}: GPT-2-shaped group, N_d=8, all ranks, stage 1 with a full "
                                    "all-reduce of the gradient then a per-shard update",
                        "psi": P, "n_d": nd, "path": "reduce into a full averaged-gradient buffer, then apply",
                        "bytes_per_step_actual": (2 * nd + 30) * P, "bytes_per_step_formula": (2 * nd + 26) * P,
                        "l2": "inputs larger than L2, no flush"},
                sample_for_cpu=None)


def llama_rank_local(Z, W, torch, dev, e2e, timer, layers=None, vocab=None):
    """Llama-3-8B-shaped group, N_d = 4, rank 1's shard with 4 staged slices,
    clip 1.0: two passes (reduce + statistics, then apply), state in place."""
    wl = W.workload("llama3-8b-nd4-r1")
    extra = W.other_ranks_sumsq(wl)
    if layers or vocab:
        wl.specs = W.llama_group(L=layers or 32, V=vocab or 128256)
        wl.name = f"llama3{_small(layers, vocab)}-nd4-r1"
    nd, me = wl.nd, 1
    plan = Z.zero_plan(W.numels(wl.specs), nd)
    P = plan["padded_total"]
    o, n = plan["rank_offsets"][me], plan["rank_numels"][me]
    log(f"[bench] llama3-8b-nd4-r1: Psi={P}, shard {n} at {o}; generating inputs")
    flat = W.flat_params(wl.specs, P, torch.bfloat16, wl.param_seed, dev)
    slices = W.GradStream([2 + j for j in range(nd)], dev).draw_plain(
        [torch.empty(n, dtype=torch.bfloat16, device=dev) for _ in range(nd)], wl.grad_std)
    master, m, v = (torch.empty(n, device=dev) for _ in range(3))
    gshard = torch.empty(n, dtype=torch.bfloat16, device=dev)
    sh = [Z.shard(n, 0, o, master, m, v, grad_shard=gshard)]
    Z.zero_shard_init(sh, flat, Z.ZERO_BF16)
    ws = torch.zeros(Z.zero_workspace_bytes(), dtype=torch.uint8, device=dev)
    stats = torch.zeros(16, dtype=torch.uint8, device=dev)
    res = torch.zeros(48, dtype=torch.uint8, device=dev)
    res_h = torch.zeros(48, dtype=torch.uint8).pin_memory()
    st = dict(cur=0, t=1, S=wl.loss_scale)
    pinned = _pin_copies(torch, slices, e2e)
    staging = torch.empty(HOST_RING_BYTES // 2, dtype=torch.int16, device=dev) if pinned else None
    hy, table, n_table, chain = _device_chain(Z, torch, dev, wl)

    def step(from_host=False):
        # chained: t, S and the bookkeeping on the device (the apply pass, then
        # a one-thread update of the chain); end to end, zero_shard_step_host
        # from the pinned slices, its result read back every step (the host
        # takes the bookkeeping over from the chain)
        if from_host:
            if "host" not in st:
                c = Z.read_chain(chain)
                st.update(host=True, t=c.step, S=c.loss_scale)
            Z.zero_shard_step_host(pinned, Z.ZERO_BF16, sh, flat, Z.ZERO_BF16, None,
                                   _hyper(Z, wl.hyper, st["t"], wl.max_grad_norm), st["S"], extra, 0, staging,
                                   HOST_RING_BYTES, ws, ws.numel(), res)
            _finish_step(Z, torch, res, res_h, st)
            return
        with timer("k_reduce"):
            Z.zero_shard_reduce(slices, Z.ZERO_BF16, sh, 0, stats, ws, ws.numel())
        with timer("k_apply"):
            Z.zero_shard_apply_chained(sh, Z.ZERO_BF16, flat, Z.ZERO_BF16, hy, table, 1, n_table, chain, stats,
                                       extra, 0, ws, ws.numel(), res)

    def path_of_last_step():
        return Z.read_result(res).path

    return dict(name=wl.name, step=step, state=st, elements=n, nd=nd, launches_per_step=3,
                path_of_last_step=path_of_last_step, extra=_check_chain(Z, chain),
                kernel_bytes={"k_reduce": (2 * nd + 2) * n, "k_apply": 28 * n},
                dominant_label=None, h2d=nd * n * 2 if pinned else None, d2h=48, e2e_ok=pinned is not None,
                formula_bytes=(2 * nd + 26) * n,
                config={"workload": f"{wl.name}: Llama-3-8B-shaped group, N_d=4, rank 1's shard, 4 staged "
                                    "bf16 slices, global-norm clip 1.0", "psi": P, "n_d": nd, "shard_elements": n,
                        "other_ranks_sumsq": extra,
                        "path": "two passes (reduce+stats, apply), state in place",
                        "steps": "zero_shard_reduce + zero_shard_apply_chained: t, S and the state set in use stay "
                                 "on the device (3 launches a step: reduce, apply, the bookkeeping)",
                        "bytes_per_step_actual": (2 * nd + 30) * n, "bytes_per_step_formula": (2 * nd + 26) * n,
                        "l2": "inputs larger than L2, no flush"},
                sample_for_cpu=None)


def gpt75_rank63(Z, W, torch, dev, e2e, timer, layers=None, vocab=None):
    """The 7.5B GPT-like group, N_d = 64, rank 63's shard, fp16, S = 65536: fused single pass."""
    wl = W.workload("gpt-7.5b-nd64-r63")
    if layers or vocab:
        wl.specs = W.gpt2_group(layers or 52, 3456, vocab or 50257, 1024)
        wl.name = f"gpt{_small(layers, vocab)}-nd64-r63"
    nd, me = wl.nd, 63
    plan = Z.zero_plan(W.numels(wl.specs), nd)
    P = plan["padded_total"]
    o, n = plan["rank_offsets"][me], plan["rank_numels"][me]
    log(f"[bench] gpt-7.5b-nd64-r63: Psi={P}, shard {n} at {o}; generating inputs")
    flat = W.flat_params(wl.specs, P, torch.float16, wl.param_seed, dev)
    slices = W.GradStream([4 + j for j in range(nd)], dev).draw_plain(
        [torch.empty(n, dtype=torch.float16, device=dev) for _ in range(nd)], wl.grad_std, wl.loss_scale)
    W.zero_every_100th_(slices[0])
    sets = [[torch.empty(n, device=dev) for _ in range(3)] for _ in range(2)]
    variants = [[Z.shard(n, 0, o, *sets[c], *sets[1 - c])] for c in (0, 1)]
    Z.zero_shard_init(variants[0], flat, Z.ZERO_F16)
    ws = torch.zeros(Z.zero_workspace_bytes(), dtype=torch.uint8, device=dev)
    res = torch.zeros(48, dtype=torch.uint8, device=dev)
    res_h = torch.zeros(48, dtype=torch.uint8).pin_memory()
    st = dict(cur=0, t=1, S=wl.loss_scale)
    pinned = _pin_copies(torch, slices, e2e)
    staging = torch.empty(HOST_RING_BYTES // 2, dtype=torch.int16, device=dev) if pinned else None

    def step(from_host=False):
        # host-driven (the caller reads zero_result and swaps the state sets):
        # the chained fused pass for 64 slices needs more registers than 4
        # blocks per SM leave it (3 per SM: 2.77 ms a step, against 2.69-2.74
        # host-driven at 4 per SM); end to end, zero_shard_step_host from the
        # pinned slices
        if from_host:
            Z.zero_shard_step_host(pinned, Z.ZERO_F16, variants[st["cur"]], flat, Z.ZERO_F16, None,
                                   _hyper(Z, wl.hyper, st["t"]), st["S"], 0.0, 0, staging, HOST_RING_BYTES, ws,
                                   ws.numel(), res)
            _finish_step(Z, torch, res, res_h, st)
            return
        with timer("fused pass+k_recover"):
            Z.zero_shard_step(slices, Z.ZERO_F16, variants[st["cur"]], flat, Z.ZERO_F16, _hyper(Z, wl.hyper, st["t"]),
                              st["S"], 0.0, 0, ws, ws.numel(), res)
        _finish_step(Z, torch, res, res_h, st)

    return dict(name=wl.name, step=step, state=st, elements=n, nd=nd, launches_per_step=2,
                kernel_bytes={"fused pass+k_recover": (2 * nd + 26) * n}, dominant_label=None,
                h2d=nd * n * 2 if pinned else None, d2h=48, e2e_ok=pinned is not None,
                formula_bytes=(2 * nd + 26) * n,
                config={"workload": f"{wl.name}: GPT-like 7.5B-shaped group, N_d=64, rank 63's shard "
                                    "(flat offset = 6 mod 8), fp16, loss scale 65536", "psi": P, "n_d": nd,
                        "shard_elements": n, "path": "fused single pass, ping-pong state",
                        "steps": "zero_shard_step, host-driven (2 launches a step: the pass, the parameter restore "
                                 "check; the result read back every step)",
                        "l2": "inputs larger than L2, no flush"},
                sample_for_cpu=None)


def _gather_status_check(gstatus):
    """After the timed steps: the bulk gathers' sticky status word must be clear."""
    def check(steps):
        if int(gstatus.item()) != 0:
            raise RuntimeError("zero3_gather_bulk reported a timed-out wait")
        return {}
    return check


def zero3_llama(Z, W, torch, dev, e2e, timer, layers=None, vocab=None, fused=True):
    """ZeRO-3 per-layer path, Llama-3-8B group as 34 units, N_d = 4, rank 1:
    per step 34 forward gathers and 34 backward gathers (reverse order); then,
    fused (the default: this workload does not clip), each unit's buckets
    reduced onto rank 1's part and that part updated in one partial pass
    (speculatively, into the second state set) and the step decided by one
    commit; or, two-pass, 34 bucket reduces and one apply of the whole shard
    (in place)."""
    wl = W.workload("zero3-llama3-8b")
    base = "zero3-llama3" if fused else "zero3-twopass-llama3"
    wl.name = f"{base}-8b"
    if layers or vocab:
        wl.specs = W.llama_group(L=layers or 32, V=vocab or 128256)
        wl.name = f"{base}{_small(layers, vocab)}"
    nd, me = wl.nd, 1
    units = W.llama_units(wl.specs, L=layers or 32)
    parts = [u // nd for u in units]
    starts = [sum(units[:i]) for i in range(len(units))]
    uoff = [sum(parts[:i]) for i in range(len(parts))]
    L = sum(parts)
    log(f"[bench] {wl.name}: {len(units)} units, rank shard {L}; generating inputs")
    flat = W.flat_params(wl.specs, sum(units), torch.bfloat16, wl.param_seed, dev)
    rshards = [torch.cat([flat[s + r * p: s + (r + 1) * p] for s, p in zip(starts, parts)]) for r in range(nd)]
    del flat
    torch.cuda.empty_cache()
    gs = W.GradStream([5 + r for r in range(nd)], dev)
    buckets = []          # buckets[u][r]: rank r's full gradient of unit u
    for u in reversed(range(len(units))):
        row = [torch.empty(units[u], dtype=torch.bfloat16, device=dev) for _ in range(nd)]
        gs.draw_plain(row, wl.grad_std)
        buckets.append((u, row))
    layer = torch.empty(max(units), dtype=torch.bfloat16, device=dev)
    A = [torch.empty(L, device=dev) for _ in range(3)]
    B = [torch.empty(L, device=dev) for _ in range(3)] if fused else A
    gshard = None if fused else torch.empty(L, dtype=torch.bfloat16, device=dev)
    sh = [Z.shard(L, 0, 0, *A, *B, grad_shard=gshard)]
    Z.zero_shard_init(sh, rshards[me], Z.ZERO_BF16)
    part_sh = [Z.shard(parts[u], me * parts[u], uoff[u], *(x[uoff[u]:uoff[u] + parts[u]] for x in A),
                       *(x[uoff[u]:uoff[u] + parts[u]] for x in B)) for u in range(len(units))]
    ws = torch.zeros(Z.zero_workspace_bytes(), dtype=torch.uint8, device=dev)
    stats = torch.zeros(16, dtype=torch.uint8, device=dev)
    res = torch.zeros(48, dtype=torch.uint8, device=dev)
    st = dict(cur=0, t=1, S=wl.loss_scale)
    hy, table, n_table, chain = _device_chain(Z, torch, dev, wl)
    part_ptrs = [[rshards[r][uoff[u]:uoff[u] + parts[u]] for r in range(nd)] for u in range(len(units))]

    gstatus = torch.zeros(1, dtype=torch.int32, device=dev)

    order = list(range(len(units))) + list(reversed(range(len(units))))

    def step(from_host=False):
        # one event pair per group of back-to-back launches of a kernel
        with timer("k_gather_bulk", len(order)):
            for u in order:
                Z.zero3_gather_bulk(part_ptrs[u], [parts[u]] * nd, Z.ZERO_BF16, layer, 0, gstatus)
        if fused:
            with timer("k_step_fused", len(buckets)):
                for k, (u, row) in enumerate(buckets):
                    Z.zero_shard_step_partial(row, Z.ZERO_BF16, [part_sh[u]], rshards[me], Z.ZERO_BF16, hy, 0.0,
                                              k > 0, stats, ws, ws.numel(), scalar_table=table, table_t0=1,
                                              n_table=n_table, chain_dev=chain)
            with timer("k_commit+k_recover"):
                Z.zero_shard_step_commit(sh, rshards[me], Z.ZERO_BF16, 0.0, stats, 0.0, 0, res, table_t0=1,
                                         n_table=n_table, chain_dev=chain)
            return
        with timer("k_reduce", len(buckets)):
            for k, (u, row) in enumerate(buckets):
                Z.zero3_reduce_bucket(row, me, units[u], Z.ZERO_BF16, gshard[uoff[u]:uoff[u] + parts[u]], k > 0,
                                      stats, ws, ws.numel())
        with timer("k_apply"):
            Z.zero_shard_apply_chained(sh, Z.ZERO_BF16, rshards[me], Z.ZERO_BF16, hy, table, 1, n_table, chain,
                                       stats, 0.0, 0, ws, ws.numel(), res)

    def path_of_last_step():
        return Z.read_result(res).path

    def checks(steps):
        out = _gather_status_check(gstatus)(steps)
        out.update(_check_chain(Z, chain)(steps))
        return out

    total_units = sum(units)
    gather_bytes = 2 * 4 * total_units
    if fused:
        kernel_bytes = {"k_gather_bulk": gather_bytes, "k_step_fused": (2 * nd + 26) * L, "k_commit+k_recover": 0}
        launches = 3 * len(units) + 3
        path = ("per unit: gather x2 (zero3_gather_bulk on every SM); then per unit the bucket reduce fused with the "
                "part's AdamW (zero_shard_step_partial, speculative, ping-pong state), and one commit "
                "(zero_shard_step_commit: the decision, the parameter restore check, the bookkeeping); t, S and the "
                "state set on the device, no host round trip between steps")
    else:
        kernel_bytes = {"k_gather_bulk": gather_bytes, "k_reduce": (2 * nd + 2) * L, "k_apply": 28 * L}
        launches = 3 * len(units) + 2
        path = ("per unit: gather x2 (zero3_gather_bulk on every SM), bucket reduce; then zero_shard_apply_chained "
                "(in place; t, S and the bookkeeping on the device, no host round trip between steps)")
    return dict(name=wl.name, step=step, state=st, elements=L, nd=nd, launches_per_step=launches,
                path_of_last_step=path_of_last_step, kernel_bytes=kernel_bytes,
                dominant_label=None, h2d=None, d2h=48, e2e_ok=False, extra=checks,
                formula_bytes=gather_bytes + (2 * nd + 2) * L + 28 * L,
                config={"workload": f"{wl.name}: Llama-3-8B group as {len(units)} ZeRO-3 units, N_d=4, rank 1",
                        "units": len(units), "shard_elements": L, "psi": total_units, "path": path,
                        "state": "f32 master/m/v, ping-pong" if fused else "f32 master/m/v, in place",
                        "formula_bytes_are": "the two-pass accounting: gathers 8 psi + reduce (2 N_d + 2) + apply 28 "
                                             "per shard element; the fused path moves (2 N_d + 26) per shard element "
                                             "instead of (2 N_d + 30)",
                        "l2": "inputs larger than L2, no flush"},
                sample_for_cpu=None)


def zero3_twopass(Z, W, torch, dev, e2e, timer, layers=None, vocab=None):
    """The ZeRO-3 step with the two-pass update (bucket reduces, then one apply
    of the whole shard in place): the path a clipped ZeRO-3 step takes."""
    return zero3_llama(Z, W, torch, dev, e2e, timer, layers, vocab, fused=False)


def zero3_broadcast(Z, W, torch, dev, e2e, timer, layers=None, vocab=None):
    """ZeRO-3 with owner broadcast on the Llama-3-8B group, N_d = 4, rank 1:
    each rank keeps one contiguous segment of the flat vector (the plan's
    partition); per step every one of the 34 units is rebuilt forward and
    backward from the pieces of its owners' segments, rank 1 reduces every
    rank's gradient over the pieces it owns, and updates its segment."""
    wl = W.workload("zero3-llama3-8b")
    if layers:
        wl.specs = W.llama_group(L=layers)
    name = "zero3-bcast-llama3-8b" if not layers else f"zero3-bcast-llama3-{layers}layers"
    nd, me = wl.nd, 1
    units = W.llama_units(wl.specs, L=layers or 32)
    plan = Z.zero_plan(units, nd)
    P = plan["padded_total"]
    pieces = {u: [] for u in range(len(units))}
    for r in range(nd):
        for u, u0, s0, ln in Z.zero_plan_intersections(plan["tensor_offsets"], units, plan["rank_offsets"][r],
                                                       plan["rank_numels"][r]):
            pieces[u].append((r, u0, s0, ln))
    log(f"[bench] {name}: {len(units)} units, segment of rank 1 {plan['rank_numels'][me]}; generating inputs")
    flat = W.flat_params(wl.specs, P, torch.bfloat16, wl.param_seed, dev)
    segs = [flat[o:o + n].clone() for o, n in zip(plan["rank_offsets"], plan["rank_numels"])]
    del flat
    torch.cuda.empty_cache()
    L = plan["rank_numels"][me]
    gs = W.GradStream([5 + r for r in range(nd)], dev)
    mine = [u for u in reversed(range(len(units))) if any(r == me for r, *_ in pieces[u])]
    buckets = {}
    for u in mine:          # only the units whose gradient rank 1 reduces are read by it
        buckets[u] = gs.draw_plain([torch.empty(units[u], dtype=torch.bfloat16, device=dev) for _ in range(nd)],
                                   wl.grad_std)
    layer = torch.empty(max(units), dtype=torch.bfloat16, device=dev)
    master, m, v = (torch.empty(L, device=dev) for _ in range(3))
    gseg = torch.empty(L, dtype=torch.bfloat16, device=dev)
    sh_apply = [Z.shard(L, 0, 0, master, m, v, grad_shard=gseg)]
    Z.zero_shard_init(sh_apply, segs[me], Z.ZERO_BF16)
    ws = torch.zeros(Z.zero_workspace_bytes(), dtype=torch.uint8, device=dev)
    stats = torch.zeros(16, dtype=torch.uint8, device=dev)
    res = torch.zeros(48, dtype=torch.uint8, device=dev)
    res_h = torch.zeros(48, dtype=torch.uint8).pin_memory()
    st = dict(cur=0, t=1, S=wl.loss_scale)
    hy, table, n_table, chain = _device_chain(Z, torch, dev, wl)
    gathers = [([segs[r][s0:s0 + ln] for r, u0, s0, ln in pieces[u]], [ln for *_, ln in pieces[u]])
               for u in range(len(units))]
    reduces = [(buckets[u], [Z.shard(ln, u0, 0, None, None, None, grad_shard=gseg[s0:s0 + ln])])
               for u in mine for r, u0, s0, ln in pieces[u] if r == me]

    gstatus = torch.zeros(1, dtype=torch.int32, device=dev)

    order = list(range(len(units))) + list(reversed(range(len(units))))

    def step(from_host=False):
        with timer("k_gather_bulk", len(order)):
            for u in order:
                Z.zero3_gather_bulk(gathers[u][0], gathers[u][1], Z.ZERO_BF16, layer, 0, gstatus)
        with timer("k_reduce", len(reduces)):
            for k, (bk, sh) in enumerate(reduces):
                Z.zero_shard_reduce(bk, Z.ZERO_BF16, sh, k > 0, stats, ws, ws.numel())
        with timer("k_apply"):
            Z.zero_shard_apply_chained(sh_apply, Z.ZERO_BF16, segs[me], Z.ZERO_BF16, hy, table, 1, n_table, chain,
                                       stats, 0.0, 0, ws, ws.numel(), res)

    def path_of_last_step():
        return Z.read_result(res).path

    def checks(steps):
        out = _gather_status_check(gstatus)(steps)
        out.update(_check_chain(Z, chain)(steps))
        return out

    total = sum(units)
    return dict(name=name, step=step, state=st, elements=L, nd=nd,
                launches_per_step=2 * len(units) + len(reduces) + 2, path_of_last_step=path_of_last_step,
                kernel_bytes={"k_gather_bulk": 2 * 4 * total, "k_reduce": (2 * nd + 2) * L, "k_apply": 28 * L},
                dominant_label=None, h2d=None, d2h=48, e2e_ok=False, extra=checks,
                formula_bytes=2 * 4 * total + (2 * nd + 2) * L + 28 * L,
                config={"workload": f"{name}: Llama-3-8B group as {len(units)} ZeRO-3 units, owner broadcast "
                                    "from contiguous rank segments, N_d=4, rank 1",
                        "units": len(units), "segment_elements": L, "psi": total,
                        "path": "per unit: gather of the owners' pieces x2 (zero3_gather_bulk on every SM), reduce "
                                "of rank 1's pieces; then apply",
                        "l2": "inputs larger than L2, no flush"},
                sample_for_cpu=None)


def zero3_prefetch(Z, W, torch, dev, e2e, timer, layers=None, vocab=None, tokens=1024, gather_ctas=32):
    """ZeRO-3 on the Llama-3-8B group (N_d = 4, rank 1) with the parameter
    gather of the next unit prefetched on a side stream while the current unit
    computes.  The units' computation is a stand-in: per unit a bf16 GEMM of
    the gathered parameters, viewed as [unit/4096, 4096], with `tokens`
    activations (twice in the backward).  The gathers go to two alternating
    layer buffers through zero3_gather_bulk on `gather_ctas` CTAs; each
    backward unit's bucket reduce and the final shard update run on the main
    stream.  The same step is also timed in order on one stream (each gather
    by zero3_gather_bulk on every SM) and with the stand-in GEMMs alone."""
    wl = W.workload("zero3-llama3-8b")
    if layers:
        wl.specs = W.llama_group(L=layers)
    name = "zero3-prefetch-llama3-8b" if not layers else f"zero3-prefetch-llama3-{layers}layers"
    nd, me, cols = wl.nd, 1, 4096
    units = W.llama_units(wl.specs, L=layers or 32)
    assert all(u % cols == 0 for u in units)
    parts = [u // nd for u in units]
    starts = [sum(units[:i]) for i in range(len(units))]
    uoff = [sum(parts[:i]) for i in range(len(parts))]
    L = sum(parts)
    log(f"[bench] {name}: {len(units)} units, rank shard {L}, stand-in GEMMs with {tokens} tokens; generating inputs")
    flat = W.flat_params(wl.specs, sum(units), torch.bfloat16, wl.param_seed, dev)
    rshards = [torch.cat([flat[s + r * p: s + (r + 1) * p] for s, p in zip(starts, parts)]) for r in range(nd)]
    del flat
    torch.cuda.empty_cache()
    gs = W.GradStream([5 + r for r in range(nd)], dev)
    buckets = {}
    for u in reversed(range(len(units))):
        buckets[u] = gs.draw_plain([torch.empty(units[u], dtype=torch.bfloat16, device=dev) for _ in range(nd)],
                                   wl.grad_std)
    bufs = [torch.empty(max(units), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    X = W.fill_normal_(torch.empty(tokens * cols, dtype=torch.bfloat16, device=dev), 1.0,
                       W.generator(77, dev)).view(tokens, cols)
    Y = torch.empty(max(units) // cols, tokens, dtype=torch.bfloat16, device=dev)
    master, m, v = (torch.empty(L, device=dev) for _ in range(3))
    gshard = torch.empty(L, dtype=torch.bfloat16, device=dev)
    sh = [Z.shard(L, 0, 0, master, m, v, grad_shard=gshard)]
    Z.zero_shard_init(sh, rshards[me], Z.ZERO_BF16)
    ws = torch.zeros(Z.zero_workspace_bytes(), dtype=torch.uint8, device=dev)
    stats = torch.zeros(16, dtype=torch.uint8, device=dev)
    res = torch.zeros(48, dtype=torch.uint8, device=dev)
    res_h = torch.zeros(48, dtype=torch.uint8).pin_memory()
    gstatus = torch.zeros(1, dtype=torch.int32, device=dev)
    st = dict(cur=0, t=1, S=wl.loss_scale)
    hy, table, n_table, chain = _device_chain(Z, torch, dev, wl)
    part_ptrs = [[rshards[r][uoff[u]:uoff[u] + parts[u]] for r in range(nd)] for u in range(len(units))]
    n_units = len(units)
    order = [(u, 1) for u in range(n_units)] + [(u, 2) for u in reversed(range(n_units))]   # (unit, GEMMs)
    side = torch.cuda.Stream(device=dev)
    gathered = [torch.cuda.Event() for _ in order]
    consumed = [torch.cuda.Event() for _ in order]

    def consume(buf, u, k):
        w = buf[:units[u]].view(-1, cols)
        for _ in range(k):
            torch.matmul(w, X.t(), out=Y[:w.shape[0]])

    def backward_reduce(i, u):
        if i >= n_units:
            with timer("k_reduce"):
                Z.zero3_reduce_bucket(buckets[u], me, units[u], Z.ZERO_BF16, gshard[uoff[u]:uoff[u] + parts[u]],
                                      i > n_units, stats, ws, ws.numel())

    def finish():
        with timer("k_apply"):
            Z.zero_shard_apply_chained(sh, Z.ZERO_BF16, rshards[me], Z.ZERO_BF16, hy, table, 1, n_table, chain, stats,
                                       0.0, 0, ws, ws.numel(), res)

    def step(from_host=False):
        main = torch.cuda.current_stream()

        def gather(i):
            if i >= 2:
                side.wait_event(consumed[i - 2])
            u = order[i][0]
            Z.zero3_gather_bulk(part_ptrs[u], [parts[u]] * nd, Z.ZERO_BF16, bufs[i % 2], gather_ctas, gstatus,
                                stream=side)
            gathered[i].record(side)

        side.wait_stream(main)          # the last step's update of rank 1's parameters comes first
        gather(0)
        for i, (u, k) in enumerate(order):
            if i + 1 < len(order):
                gather(i + 1)
            main.wait_event(gathered[i])
            consume(bufs[i % 2], u, k)
            consumed[i].record(main)
            backward_reduce(i, u)
        finish()

    def step_serial():
        for i, (u, k) in enumerate(order):
            Z.zero3_gather_bulk(part_ptrs[u], [parts[u]] * nd, Z.ZERO_BF16, bufs[0], 0, gstatus)
            consume(bufs[0], u, k)
            backward_reduce(i, u)
        finish()

    def step_consumers_only():
        for u, k in order:
            consume(bufs[0], u, k)

    def extra(steps):
        """The serial schedule and the stand-in GEMMs alone, timed like the step."""
        out = {}
        for key, fn in (("serial_ms_per_step", step_serial), ("consumer_ms_per_step", step_consumers_only)):
            for _ in range(2):
                fn()
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            for _ in range(steps):
                fn()
            b.record()
            torch.cuda.synchronize()
            out[key] = a.elapsed_time(b) / steps
        if int(gstatus.item()) != 0:
            raise RuntimeError("zero3_gather_bulk reported a timed-out wait")
        out.update(_check_chain(Z, chain)(steps))
        return out

    total = sum(units)
    return dict(name=name, step=step, state=st, elements=L, nd=nd,
                path_of_last_step=lambda: Z.read_result(res).path,
                launches_per_step=len(order) + n_units + 2,
                kernel_bytes={"k_reduce": (2 * nd + 2) * L, "k_apply": 28 * L},
                dominant_label=None, h2d=None, d2h=48, e2e_ok=False, extra=extra,
                formula_bytes=2 * 4 * total + (2 * nd + 2) * L + 28 * L,
                config={"workload": f"{name}: Llama-3-8B group as {n_units} ZeRO-3 units, N_d=4, rank 1; the next "
                                    "unit's gather prefetched on a side stream beside a stand-in compute",
                        "units": n_units, "shard_elements": L, "psi": total, "tokens": tokens,
                        "gather_ctas": gather_ctas,
                        "consumer": f"stand-in per unit: bf16 GEMM [unit/{cols}, {cols}] x [{cols}, {tokens}] "
                                    "(torch.matmul), once forward and twice backward",
                        "path": "side stream: zero3_gather_bulk into two alternating layer buffers; main stream: "
                                "stand-in GEMMs, bucket reduce after each backward unit, then apply",
                        "l2": "inputs larger than L2, no flush"},
                sample_for_cpu=None)


def cpu_sample_gpt2(W, n_per_shard):
    """The first n_per_shard elements of each of the 8 shards of the GPT-2 1.5B
    group, with seeded inputs drawn for that sample (CPU generators)."""
    import numpy as np
    import torch
    wl = W.workload("gpt2-1.5b-nd8")
    nd = wl.nd
    g = W.generator(0, "cpu")
    flat = torch.empty(nd * n_per_shard, dtype=torch.bfloat16)
    W.fill_normal_(flat, 0.02, g)
    grads = []
    for r in range(nd):
        x = torch.empty(nd * n_per_shard, dtype=torch.bfloat16)
        W.fill_normal_(x, 1e-3, W.generator(1 + r, "cpu"))
        grads.append(x.view(torch.int16).numpy().view(np.uint16).copy())
    return nd, grads, flat.view(torch.int16).numpy().view(np.uint16).copy(), wl.hyper


WORKLOADS = {"gpt2-1.5b-nd8": gpt2_all_ranks, "gpt2-1.5b-nd8-allreduce": gpt2_allreduce, "tiny-nd3": tiny_nd3,
             "llama3-8b-nd4-r1": llama_rank_local, "gpt-7.5b-nd64-r63": gpt75_rank63,
             "zero3-llama3-8b": zero3_llama, "zero3-twopass-llama3-8b": zero3_twopass,
             "zero3-bcast-llama3-8b": zero3_broadcast, "zero3-prefetch-llama3-8b": zero3_prefetch}


# ------------------------------------------------------------------ CPU oracle timing
def time_oracle(sample, n_per_shard, steps):
    """The oracle as it stands, in this process: each step's wall time."""
    import numpy as np
    import oracle
    nd, grads, flat, h = sample
    flat = flat.copy()
    shards = [dict(numel=n_per_shard, grad_off=r * n_per_shard, param_off=r * n_per_shard,
                   master=oracle.widen_16(flat[r * n_per_shard:(r + 1) * n_per_shard], 2),
                   m=np.zeros(n_per_shard, np.float32), v=np.zeros(n_per_shard, np.float32)) for r in range(nd)]
    hh = dict(h, max_grad_norm=0.0)
    times = []
    for t in range(1, steps + 1):
        t0 = time.perf_counter()
        oracle.zero_step(grads, 2, shards, flat, 2, hh, t, 1.0)
        times.append(time.perf_counter() - t0)
    return nd * n_per_shard, times


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_model():
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    import platform
    return platform.processor() or platform.machine()


_BARRIER = None


def _oracle_worker_init(barrier):
    global _BARRIER
    _BARRIER = barrier


def _oracle_chunk(task):
    """One process's share of the all-cores oracle timing: the oracle's step on
    elements [lo, hi) of every shard, repacked as a problem of its own (the
    elements' updates are independent without clipping).  Every step starts
    behind a barrier across the processes; returns each step's (start, end)
    and, if asked, the parameters after the last step."""
    import numpy as np
    import oracle
    nd, c, grads, flat, hyper, steps, want_params = task
    shards = [dict(numel=c, grad_off=r * c, param_off=r * c, master=oracle.widen_16(flat[r * c:(r + 1) * c], 2),
                   m=np.zeros(c, np.float32), v=np.zeros(c, np.float32)) for r in range(nd)]
    hh = dict(hyper, max_grad_norm=0.0)
    marks = []
    for t in range(1, steps + 1):
        _BARRIER.wait(timeout=600)
        t0 = time.perf_counter()
        oracle.zero_step(grads, 2, shards, flat, 2, hh, t, 1.0)
        marks.append((t0, time.perf_counter()))
    return marks, (flat if want_params else None)


def time_oracle_parallel(sample, n_per_shard, steps, procs, want_params=False):
    """The oracle as it stands, run by `procs` spawned processes at once, each
    on an equal share of every shard's elements.  Returns the elements per step,
    each step's wall time (last end minus first start over the processes) and,
    if asked, the parameters after the last step reassembled in flat order."""
    import multiprocessing as mp
    import numpy as np
    nd, grads, flat, h = sample
    n = n_per_shard
    bounds = [n * w // procs for w in range(procs + 1)]
    tasks = []
    for w in range(procs):
        lo, hi = bounds[w], bounds[w + 1]
        pick = lambda a: np.concatenate([a[r * n + lo:r * n + hi] for r in range(nd)])
        tasks.append((nd, hi - lo, [pick(g) for g in grads], pick(flat), h, steps, want_params))
    ctx = mp.get_context("spawn")
    barrier = ctx.Barrier(procs)
    with ctx.Pool(procs, initializer=_oracle_worker_init, initargs=(barrier,)) as pool:
        res = pool.map(_oracle_chunk, tasks, chunksize=1)
    walls = [max(r[0][s][1] for r in res) - min(r[0][s][0] for r in res) for s in range(steps)]
    params = None
    if want_params:
        params = np.empty_like(flat)
        for w, (_, fw) in enumerate(res):
            lo, hi = bounds[w], bounds[w + 1]
            c = hi - lo
            for r in range(nd):
                params[r * n + lo:r * n + hi] = fw[r * c:(r + 1) * c]
    return nd * n, walls, params


# ------------------------------------------------------------------ multi-rank timing and the output line
def max_over_ranks(x: float, world: int, device) -> float:
    """The largest of every rank's x (the step time the job is charged)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.item()


# Timer labels of the update pass, whose kernel the path choice names.
UPDATE_KINDS = ("fused pass+k_recover", "k_apply", "k_step_fused")


def build_line(world, steps, warmup, ms, elements, nd, config, roofline, kernels, cpu, e2e, clocks, launches,
               formula_bytes=None, actual_bytes=None, peak=None):
    """The JSON line rank 0 prints: value is the whole job's shard elements per
    second (every rank runs its own copy of the workload, so scaling is weak).
    The step's bandwidth is given twice: by the formula's bytes ((2 N_d + 26)
    per element, or the ZeRO-3 sum) and by the bytes the kernels of the step
    move by design, each as a fraction of the measured and the nominal peak."""
    fb = formula_bytes if formula_bytes is not None else elements * (2 * nd + 26)
    step_bw = None
    if actual_bytes is not None and peak:
        f, a = fb / (ms / 1e3) / 1e9, actual_bytes / (ms / 1e3) / 1e9
        step_bw = {"formula_bytes": fb, "formula_gbs": f, "formula_frac": f / peak,
                   "formula_frac_of_nominal": f / NOMINAL_HBM_GBS, "actual_bytes": actual_bytes, "actual_gbs": a,
                   "actual_frac": a / peak, "actual_frac_of_nominal": a / NOMINAL_HBM_GBS}
    return {"metric": METRIC, "value": world * elements / (ms / 1e3), "unit": "elements/s",
            "n_gpus": world, "steps": steps, "warmup": warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded torch generators; no data set or weights)",
            "config": config, "achieved_gbs_formula": fb / (ms / 1e3) / 1e9, "step_bandwidth": step_bw,
            "roofline": roofline, "kernels": kernels, "cpu_baseline": cpu, "e2e": e2e, "clocks": clocks,
            "gpu_launches": launches, "impl": "ours"}


# ------------------------------------------------------------------ main
# Workloads measured after the headline one in the default run, each on its
# own (the previous one's buffers freed first): the clipped rank-local
# Llama-3-8B step and the ZeRO-3 Llama-3-8B step (the 8B-shaped
# configurations), and the 7.5B-shaped rank-local step with 64 slices.
ALSO = ("llama3-8b-nd4-r1", "zero3-llama3-8b", "gpt-7.5b-nd64-r63")


def measure(wl, args, world, local, dev, torch, timer, barrier, e2e_on):
    """W untimed steps, then K steps between barriers and synchronisations,
    timed by CUDA events on the launching stream, with the SM clocks sampled
    during the timed region; then, if the workload has one, the end-to-end
    leg.  Returns the step time (max over ranks), the per-kernel times, the
    clock record and the end-to-end record."""
    step = wl["step"]
    sampler = ClockSampler(local)
    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    barrier()
    sampler.start()
    time.sleep(0.3)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    timer.events.clear()
    timer.on = True
    start.record()
    for _ in range(args.steps):
        step()
    end.record()
    torch.cuda.synchronize()
    timer.on = False
    barrier()
    clocks = sampler.stop()
    ms = max_over_ranks(start.elapsed_time(end) / args.steps, world, dev)
    kinds = timer.per_kind(args.steps)
    if wl.get("path_of_last_step"):
        wl["state"]["path"] = wl["path_of_last_step"]()
    if wl.get("extra"):
        wl["config"].update(wl["extra"](args.steps))

    e2e = None
    timed_path = wl["state"].get("path")
    if e2e_on and wl["e2e_ok"]:
        for _ in range(2):
            step(from_host=True)
        torch.cuda.synchronize()
        barrier()
        s2, e2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s2.record()
        for _ in range(args.e2e_steps):
            step(from_host=True)
        e2.record()
        torch.cuda.synchronize()
        barrier()
        ms_e2e = max_over_ranks(s2.elapsed_time(e2) / args.e2e_steps, world, dev)
        e2e = {"value": world * wl["elements"] / (ms_e2e / 1e3), "unit": "elements/s",
               "h2d_bytes_per_step": wl["h2d"], "d2h_bytes_per_step": wl["d2h"], "ms_per_step": ms_e2e,
               "steps": args.e2e_steps, "source": E2E_SOURCE["mode"],
               "note": "bound by the host link: ~211 GB/s at best on this host, shared with other tenants"}
        if wl.get("e2e_note"):
            e2e["overlap"] = wl["e2e_note"]
        if wl.get("e2e_parts"):
            e2e["link_alone"] = wl["e2e_parts"]()
        e2e["update_kernel"] = PATH_NAMES.get(wl["state"].get("path"), "?")
        wl["state"]["path"] = timed_path          # the line's kernel figures are the device-timed steps'
    return ms, kinds, clocks, e2e


def kernel_figures(wl, kinds, steps):
    """Per-kernel algorithmic bytes and bandwidth, and the roofline entry of the
    dominant kernel (the one with the most time per step)."""
    peak, peak_src = measured_peaks()
    per_kernel = {}
    for kind, d in kinds.items():
        per_launch_bytes = wl["kernel_bytes"][kind] / (d["launches"] / steps)
        gbs = per_launch_bytes / (d["ms_per_launch"] / 1e3) / 1e9
        per_kernel[kind] = dict(d, algorithmic_bytes_per_launch=per_launch_bytes, achieved_gbs=gbs,
                                frac=gbs / peak)
    dom = max(per_kernel, key=lambda k: per_kernel[k]["ms_total"])
    dk = per_kernel[dom]
    wl["config"]["update_kernel"] = PATH_NAMES.get(wl["state"].get("path"), "?")
    roofline = {"bound": "hbm", "achieved": dk["achieved_gbs"], "peak": peak, "unit": "GB/s",
                "frac": dk["achieved_gbs"] / peak, "traffic": ncu_traffic(wl["name"], dom),
                "peak_source": peak_src,
                "kernel": f"{dom} [{wl['config']['update_kernel']}]" if dom in UPDATE_KINDS else dom,
                "kernel_ms_per_launch": dk["ms_per_launch"], "kernel_ms_median": dk["ms_median"],
                "algorithmic_bytes_per_launch": dk["algorithmic_bytes_per_launch"],
                "nominal_peak": NOMINAL_HBM_GBS, "frac_of_nominal": dk["achieved_gbs"] / NOMINAL_HBM_GBS}
    if roofline["traffic"] is not None:
        dram = roofline["traffic"] / (dk["ms_per_launch"] / 1e3) / 1e9
        roofline.update(dram_gbs=dram, dram_frac=dram / peak, dram_frac_of_nominal=dram / NOMINAL_HBM_GBS,
                        traffic_over_algorithmic=roofline["traffic"] / dk["algorithmic_bytes_per_launch"])
    return roofline, per_kernel, peak


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="gpt2-1.5b-nd8", choices=sorted(WORKLOADS))
    ap.add_argument("--layers", type=int, default=None,
                    help="layer count of the workload's group (default: the full model); fewer gives a small case "
                         "of the same kernels, e.g. for profiler captures")
    ap.add_argument("--vocab", type=int, default=None,
                    help="vocabulary of the workload's group (default: the model's); smaller gives a small case")
    ap.add_argument("--no-also", action="store_true",
                    help="measure only --workload (the default run also measures " + ", ".join(ALSO) + ")")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--tokens", type=int, default=1024,
                    help="zero3-prefetch-llama3-8b: activations of the stand-in GEMM per unit")
    ap.add_argument("--gather-ctas", type=int, default=32,
                    help="zero3-prefetch-llama3-8b: CTAs the prefetched gather may use")
    args = ap.parse_args()
    rank, world, local = dist_env()
    import workloads as W

    if args.impl == "reference":
        return reference_arm(args, rank, world, W)

    import gc

    import torch
    import torch.distributed as dist
    import zero_dp_partitioned_gb300 as Z
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if world > 1:
            dist.barrier()

    timer = KernelTimer(torch)
    kw = dict(tokens=args.tokens, gather_ctas=args.gather_ctas) if args.workload == "zero3-prefetch-llama3-8b" else {}
    wl = WORKLOADS[args.workload](Z, W, torch, dev, not args.no_e2e, timer, layers=args.layers, vocab=args.vocab,
                                  **kw)
    ms, kinds, clocks, e2e = measure(wl, args, world, local, dev, torch, timer, barrier, not args.no_e2e)
    roofline, per_kernel, peak = kernel_figures(wl, kinds, args.steps)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and wl["sample_for_cpu"]:
        cpu = cpu_baseline(wl)
    line = None
    if rank == 0:
        line = build_line(world, args.steps, max(3, args.warmup), ms, wl["elements"], wl["nd"], wl["config"],
                          roofline, per_kernel, cpu, e2e, clocks, wl["launches_per_step"] * args.steps,
                          wl["formula_bytes"] if wl["name"].startswith("zero3") else None,
                          actual_bytes=sum(wl["kernel_bytes"].values()), peak=peak)
    also = [] if (args.no_also or args.workload != "gpt2-1.5b-nd8" or args.layers or args.vocab) else ALSO
    if also:
        del wl
        gc.collect()
        torch.cuda.empty_cache()
        entries = []
        for name in also:
            w2 = WORKLOADS[name](Z, W, torch, dev, False, timer)
            ms2, kinds2, clocks2, _ = measure(w2, args, world, local, dev, torch, timer, barrier, False)
            roof2, per2, _ = kernel_figures(w2, kinds2, args.steps)
            if rank == 0:
                sub = build_line(world, args.steps, max(3, args.warmup), ms2, w2["elements"], w2["nd"],
                                 w2["config"], roof2, per2, None, None, clocks2, w2["launches_per_step"] * args.steps,
                                 w2["formula_bytes"] if w2["name"].startswith("zero3") else None,
                                 actual_bytes=sum(w2["kernel_bytes"].values()), peak=peak)
                for k in ("vs_baseline", "cpu_baseline", "e2e", "impl", "data", "dtype", "higher_is_better",
                          "scaling", "n_gpus"):
                    sub.pop(k, None)
                entries.append(sub)
            del w2
            gc.collect()
            torch.cuda.empty_cache()
        if rank == 0:
            line["also"] = entries
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def cpu_baseline(wl):
    """The oracle timed on the host cores on a bounded sample of the workload:
    the first 2^22 elements of each shard, 3 steps, run by one process per
    host core (each on an equal share of every shard's elements); the value is
    the mean of steps 2 and 3.  The single-threaded figure on the same sample
    (2 steps) is given beside it."""
    n_per = 1 << 22
    sample = wl["sample_for_cpu"](n_per)
    n, times = time_oracle(sample, n_per, 2)
    procs = host_cores()
    n, walls, _ = time_oracle_parallel(sample, n_per, 3, procs)
    return {"value": n / statistics.mean(walls[1:]), "unit": "elements/s", "cores": procs, "kind": "oracle",
            "sample": f"the first {n_per} elements of each of the {wl['nd']} shards ({n} elements), 3 steps, "
                      f"{procs} processes each on an equal share of every shard; mean of steps 2-3",
            "cpu_model": cpu_model(),
            "single_thread": {"value": n / statistics.mean(times), "cores": 1,
                              "sample": "the same elements, 2 steps, one process"}}


def reference_arm(args, rank, world, W):
    """The CPU oracle on the host cores: one process per core, each on an equal
    share of a bounded sample of the workload (the first 2^22 elements of each
    of the GPT-2 group's 8 shards); every step starts behind a barrier and its
    time is the last process's end minus the first one's start."""
    if rank != 0:
        return
    n_per = 1 << 22
    procs = host_cores()
    n, walls, _ = time_oracle_parallel(cpu_sample_gpt2(W, n_per), n_per, args.steps + args.warmup, procs)
    walls = walls[args.warmup:]
    ms = 1e3 * statistics.mean(walls)
    value = n / (ms / 1e3)
    line = {"metric": METRIC, "value": value, "unit": "elements/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic", "impl": "reference",
            "config": {"workload": gpt2_desc("gpt2-1.5b-nd8"), "sample_elements_per_step": n},
            "cpu_baseline": {"value": value, "unit": "elements/s", "cores": procs, "kind": "oracle",
                             "sample": f"the first {n_per} elements of each of the 8 shards per step, "
                                       f"{procs} processes each on an equal share",
                             "cpu_model": cpu_model()},
            "e2e": {"value": value, "unit": "elements/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
