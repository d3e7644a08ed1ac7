"""Two real processes (torch.distributed, gloo, CPU) run the partitioned step
with real collectives, and the result must equal the single-process
data-parallel step bit for bit.

* all-reduce = all-gather(reduce-scatter) (ZeRO reading notes, 4; the CMU
  11-868 notes suggest exactly this two-process check).
* The reduce-scatter is done as one reduce per owner segment, as the CMU
  11-868 notes describe for ZeRO-2 (ncclReduce of segment M_i to GPU i); the
  norm partials and overflow flags are all-reduced; the updated 16-bit
  shards are all-gathered (DeepSpeed ZeRO stages 1-2 walkthrough, 6)."""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, ws, port, out_path):
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    import oracle as orc
    from helpers import hyper32, make_problem, t2u16, u16_to_t

    dt, S = 1, 1024.0
    h = hyper32()
    numels = [1500, 37, 211]
    p, flat, grads = make_problem(numels, ws, dt, 0, seed=21, loss_scale=S, steps=3)
    P = p["padded_total"]
    o, n = int(p["rank_offsets"][rank]), int(p["rank_numels"][rank])
    my = dict(numel=n, grad_off=0, param_off=o, master=orc.widen_16(flat[o:o + n], dt),
              m=np.zeros(n, np.float32), v=np.zeros(n, np.float32))
    ddp = dict(master=orc.widen_16(flat, dt), m=np.zeros(P, np.float32), v=np.zeros(P, np.float32))
    zflat, dflat = flat.copy(), flat.copy()
    ok = True
    t = 1
    for step in range(3):
        local = grads[step][rank]                       # this rank's own gradient (full flat vector)
        g32 = u16_to_t(local, dt).float()
        # all-reduce = reduce-scatter + all-gather, on the fp32 widening (2 ranks: a + b is exact-rounded
        # and commutative, so the order inside the library does not matter)
        ar = g32.clone()
        dist.all_reduce(ar)
        chunks = [g32[int(p["rank_offsets"][k]):int(p["rank_offsets"][k] + p["rank_numels"][k])].clone()
                  for k in range(ws)]
        for k in range(ws):
            dist.reduce(chunks[k], dst=k)                 # segment k reduced onto its owner
        gathered = [torch.empty_like(chunks[k]) for k in range(ws)]
        dist.all_gather(gathered, chunks[rank])
        ok &= torch.equal(torch.cat(gathered), ar)
        # the owner's averaged 16-bit shard, from the reduced segment
        avg16 = t2u16((chunks[rank] / ws).to(torch.float16))
        # partitioned step on the own shard, with the scalar all-reduce of the statistics
        acc, ovf = orc.stats(avg16, dt)
        stat = torch.tensor([acc.value(), float(ovf)], dtype=torch.float64)
        dist.all_reduce(stat)
        ovf_all = stat[1].item() > 0
        if not ovf_all:
            k_mult, _, _ = orc.grad_multiplier(stat[0].item(), S, 0.0)
            sc = orc.make_scalars(h["lr"], h["beta1"], h["beta2"], h["eps"], h["weight_decay"], t)
            shard16 = np.empty(n, np.uint16)
            orc.apply(avg16, dt, my["master"], my["m"], my["v"], shard16, dt, k_mult, sc)
            # gloo gathers no 16-bit integers: carry the bit patterns as int32
            parts = [torch.empty(int(p["rank_numels"][k]), dtype=torch.int32) for k in range(ws)]
            dist.all_gather(parts, torch.from_numpy(shard16.astype(np.int32)))
            zflat = torch.cat(parts).numpy().astype(np.uint16)
        # the single-process data-parallel reference over the full vector
        res = orc.ddp_step(grads[step], dt, ddp["master"], ddp["m"], ddp["v"], dflat, dt, h, t, S)
        ok &= bool(res.applied) == (not ovf_all)
        ok &= np.array_equal(zflat, dflat)
        ok &= np.array_equal(my["master"], ddp["master"][o:o + n]) and np.array_equal(my["v"], ddp["v"][o:o + n])
        if res.applied:
            t += 1
    with open(f"{out_path}.{rank}", "w") as f:
        f.write("ok" if ok else "mismatch")
    dist.destroy_process_group()


@pytest.mark.timeout(300)
def test_two_process_partitioned_step_equals_ddp(tmp_path):
    out = str(tmp_path / "res")
    mp.start_processes(_worker, args=(2, _free_port(), out), nprocs=2, start_method="spawn", join=True)
    for r in range(2):
        assert open(f"{out}.{r}").read() == "ok"
