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
    h = hashlib.sha256()
    d = os.path.join(ROOT, "zero_dp_partitioned_gb300", "csrc")
    for f in sorted(os.listdir(d)):
        h.update(open(os.path.join(d, f), "rb").read())
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


# ------------------------------------------------------------------ workloads (our path)
def gpt2_all_ranks(Z, W, torch, dev, e2e):
    """GPT-2 1.5B-shaped group, N_d = 8, all ranks on this GPU, bf16, ping-pong state (fused single pass)."""
    wl = W.workload("gpt2-1.5b-nd8")
    nd = wl.nd
    plan = Z.zero_plan(W.numels(wl.specs), nd)
    P = plan["padded_total"]
    log(f"[bench] gpt2-1.5b-nd8: Psi={P} N_d={nd}; generating inputs")
    flat = torch.zeros(P, dtype=torch.bfloat16, device=dev)
    W.init_params_(flat, wl.specs, W.generator(wl.param_seed, dev))
    grads = [W.fill_grad_(torch.empty(P, dtype=torch.bfloat16, device=dev), wl.specs, W.generator(1 + r, dev),
                          W.gpt2_grad_std()) for r in range(nd)]
    A = [flat.float(), torch.zeros(P, device=dev), torch.zeros(P, device=dev)]
    B = [torch.empty(P, device=dev) for _ in range(3)]
    sets = [A, B]

    def shards(cur):
        i, o = sets[cur], sets[1 - cur]
        return [Z.shard(n, off, off, i[0][off:off + n], i[1][off:off + n], i[2][off:off + n],
                        o[0][off:off + n], o[1][off:off + n], o[2][off:off + n])
                for off, n in zip(plan["rank_offsets"], plan["rank_numels"])]

    variants = [shards(0), shards(1)]
    ws = torch.zeros(Z.zero_workspace_bytes(), dtype=torch.uint8, device=dev)
    res = torch.zeros(48, dtype=torch.uint8, device=dev)
    res_h = torch.zeros(48, dtype=torch.uint8).pin_memory()
    st = dict(cur=0, t=1, S=wl.loss_scale)
    h = wl.hyper
    pinned = None
    if e2e:
        need = nd * P * 2
        if mem_available_bytes() > 2 * need + (16 << 30):
            log(f"[bench] pinning {need / 1e9:.1f} GB of host gradients for the end-to-end run")
            pinned = [torch.empty(P, dtype=torch.bfloat16, pin_memory=True).copy_(g) for g in grads]
        else:
            log("[bench] not enough host memory for the end-to-end run")

    def step(kernel_events=None, from_host=False):
        if from_host:
            for g, hp in zip(grads, pinned):
                g.copy_(hp, non_blocking=True)
        if kernel_events is not None:
            kernel_events[0].record()
        Z.zero_shard_step(grads, Z.ZERO_BF16, variants[st["cur"]], flat, Z.ZERO_BF16,
                          Z.hyper(h["lr"], h["beta1"], h["beta2"], h["eps"], h["weight_decay"], 0.0, st["t"]),
                          st["S"], 0.0, 0, ws, ws.numel(), res)
        if kernel_events is not None:
            kernel_events[1].record()
        res_h.copy_(res, non_blocking=True)
        torch.cuda.current_stream().synchronize()
        r = Z.read_result(res_h)
        if r.applied:
            st["cur"] ^= 1
            st["t"] += 1
        else:
            st["S"] /= 2

    return dict(name="gpt2-1.5b-nd8", step=step, elements=P, nd=nd,
                bytes_per_elem=2 * nd + 26, launches_per_step=2,
                dominant="k_step_fused<bf16,bf16,8,8> (+ k_recover, a no-op without overflow)",
                dominant_key="k_step_fused", dominant_bytes=(2 * nd + 26) * P,
                h2d=nd * P * 2 if pinned else None, d2h=48, e2e_ok=pinned is not None,
                config={"workload": "gpt2-1.5b-nd8: GPT-2 1.5B-shaped group (48 layers, d=1600, vocab 50257, "
                                    "ctx 1024), N_d=8, all 8 ranks simulated on one GPU",
                        "psi": P, "n_d": nd, "shard_elements": plan["rank_numels"][0],
                        "grad_dtype": "bf16", "param_dtype": "bf16", "state": "f32 master/m/v, ping-pong",
                        "path": "fused single pass", "bytes_per_step": (2 * nd + 26) * P,
                        "l2": f"inputs larger than L2 ({(2 * nd + 26) * P / 1e9:.1f} GB per step), no flush"},
                sample_for_cpu=lambda n: cpu_sample_gpt2(W, n))


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


WORKLOADS = {"gpt2-1.5b-nd8": gpt2_all_ranks}


# ------------------------------------------------------------------ CPU oracle timing
def time_oracle(W, wl_fn, n_per_shard, steps):
    import numpy as np
    import oracle
    nd, grads, flat, h = wl_fn(n_per_shard)
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


# ------------------------------------------------------------------ main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="gpt2-1.5b-nd8", choices=sorted(WORKLOADS))
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=5)
    args = ap.parse_args()
    rank, world, local = dist_env()
    import workloads as W

    if args.impl == "reference":
        return reference_arm(args, rank, world, W)

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

    wl = WORKLOADS[args.workload](Z, W, torch, dev, e2e=not args.no_e2e)
    step = wl["step"]
    sampler = ClockSampler(local)
    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    barrier()
    sampler.start()
    time.sleep(0.3)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    start.record()
    for k in range(args.steps):
        step(kernel_events=evs[k])
    end.record()
    torch.cuda.synchronize()
    barrier()
    clocks = sampler.stop()
    ms = start.elapsed_time(end) / args.steps
    k_ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
    if world > 1:
        t = torch.tensor([ms, k_ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms, k_ms = t.tolist()

    e2e = None
    if wl["e2e_ok"]:
        for _ in range(1):
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
        ms_e2e = s2.elapsed_time(e2) / args.e2e_steps
        if world > 1:
            t = torch.tensor([ms_e2e], device=dev)
            dist.all_reduce(t, op=dist.ReduceOp.MAX)
            ms_e2e = t.item()
        e2e = {"value": world * wl["elements"] / (ms_e2e / 1e3), "unit": "elements/s",
               "h2d_bytes_per_step": wl["h2d"], "d2h_bytes_per_step": wl["d2h"], "ms_per_step": ms_e2e,
               "steps": args.e2e_steps}

    peak, peak_src = measured_peaks()
    achieved = wl["dominant_bytes"] / (k_ms / 1e3) / 1e9
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "traffic": ncu_traffic(wl["name"], wl["dominant_key"]), "peak_source": peak_src,
                "kernel": wl["dominant"], "kernel_ms": k_ms,
                "algorithmic_bytes_per_launch": wl["dominant_bytes"]}
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        n, times = time_oracle(W, wl["sample_for_cpu"], 1 << 22, 2)
        cpu = {"value": n / statistics.mean(times), "unit": "elements/s", "cores": 1, "kind": "oracle",
               "sample": f"the first {1 << 22} elements of each of the {wl['nd']} shards "
                         f"({n} elements), 2 steps, single-threaded plain C oracle"}
    if rank == 0:
        line = {"metric": METRIC, "value": world * wl["elements"] / (ms / 1e3), "unit": "elements/s",
                "n_gpus": world, "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": ms,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
                "data": "synthetic (seeded torch generators; no data set or weights)",
                "config": wl["config"], "achieved_gbs_formula": wl["elements"] * wl["bytes_per_elem"] / (ms / 1e3) / 1e9,
                "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "clocks": clocks,
                "gpu_launches": wl["launches_per_step"] * args.steps, "impl": "ours"}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def reference_arm(args, rank, world, W):
    """The CPU oracle on the host cores: each step one oracle step over a
    bounded sample of the workload (the first 2^20 elements of each shard)."""
    if rank != 0:
        return
    n_per = 1 << 20
    wl_fn = cpu_sample_gpt2
    _, times = time_oracle(W, lambda n: wl_fn(W, n), n_per, args.steps + args.warmup)
    times = times[args.warmup:]
    n = 8 * n_per
    ms = 1e3 * statistics.mean(times)
    value = n / (ms / 1e3)
    line = {"metric": METRIC, "value": value, "unit": "elements/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic", "impl": "reference",
            "config": {"workload": "gpt2-1.5b-nd8: GPT-2 1.5B-shaped group, N_d=8, all ranks",
                       "sample_elements_per_step": n},
            "cpu_baseline": {"value": value, "unit": "elements/s", "cores": 1, "kind": "oracle",
                             "sample": f"the first {n_per} elements of each of the 8 shards per step"},
            "e2e": {"value": value, "unit": "elements/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
