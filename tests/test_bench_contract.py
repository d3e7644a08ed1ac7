"""CPU tests of bench.py's host logic: the max-over-ranks step time across
two real processes (torch.distributed, gloo), and the fields of the JSON line
the driver reads."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, port, out):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE="2",
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=2)
    import bench
    r, w, local = bench.dist_env()
    got = bench.max_over_ranks(10.0 + 3.5 * rank, w, "cpu")          # rank 1 is the slower one
    line = bench.build_line(w, 100, 5, got, 1000, 8, {"workload": "w"}, {}, {}, None, None, {}, 300)
    dist.barrier()
    open(f"{out}.{rank}", "w").write(f"{r} {w} {local} {got!r} {line['value']!r} {line['n_gpus']}")
    dist.destroy_process_group()


@pytest.mark.timeout(300)
def test_two_ranks_charge_the_slowest_and_sum_the_work(tmp_path):
    """The N > 1 timing path over two gloo processes: each rank reads its rank
    from the environment, both are charged the slowest rank's time, and the
    job's value counts both ranks' elements over that time (weak scaling)."""
    out = str(tmp_path / "r")
    mp.start_processes(_worker, args=(_port(), out), nprocs=2, start_method="spawn", join=True)
    for rank in range(2):
        r, w, local, got, value, n = open(f"{out}.{rank}").read().split()
        assert (int(r), int(w), int(local), int(n)) == (rank, 2, rank, 2)
        assert float(got) == 13.5 and float(value) == pytest.approx(2 * 1000 / 0.0135)


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(4.25, 1, "cpu") == 4.25


def test_line_fields():
    import bench
    roof = {"bound": "hbm", "achieved": 6500.0, "peak": 6792.1, "unit": "GB/s", "frac": 6500.0 / 6792.1,
            "traffic": None}
    cpu = {"value": 1.2e7, "unit": "elements/s", "cores": 1, "kind": "oracle", "sample": "x"}
    e2e = {"value": 1e10, "unit": "elements/s", "h2d_bytes_per_step": 1, "d2h_bytes_per_step": 48}
    clocks = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": []}
    line = bench.build_line(4, 100, 5, 10.0, 1_557_611_200, 8, {"workload": "w"}, roof, {}, cpu, e2e, clocks, 200)
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "e2e", "clocks", "gpu_launches"):
        assert k in line, k
    assert line["value"] == pytest.approx(4 * 1_557_611_200 / 0.010)            # whole job: all ranks
    assert line["scaling"] == "weak" and line["higher_is_better"] is True and line["n_gpus"] == 4
    assert set(line["roofline"]) >= {"bound", "achieved", "peak", "unit", "frac", "traffic"}
    assert line["achieved_gbs_formula"] == pytest.approx(1_557_611_200 * 42 / 0.010 / 1e9)
    assert line["config"]["workload"] == "w" and "model" not in line["config"]
    assert line["step_bandwidth"] is None
    two_pass = bench.build_line(1, 100, 5, 10.0, 1000, 4, {"workload": "w"}, roof, {}, cpu, e2e, clocks, 200,
                                actual_bytes=38 * 1000, peak=6792.1)
    bw = two_pass["step_bandwidth"]
    assert bw["formula_bytes"] == 34 * 1000 and bw["actual_gbs"] == pytest.approx(38 * 1000 / 0.010 / 1e9)
    assert bw["actual_frac"] == pytest.approx(bw["actual_gbs"] / 6792.1)
    assert bw["formula_frac_of_nominal"] == pytest.approx(bw["formula_gbs"] / bench.NOMINAL_HBM_GBS)


def test_every_input_helper_bench_and_tests_use_exists():
    """bench.py and the GPU tests build their inputs from workloads.py; a
    helper they name but the module lacks would only fail on a GPU."""
    import ast
    sys.path.insert(0, ROOT)
    import workloads as W
    files = [os.path.join(ROOT, "bench.py")] + [os.path.join(ROOT, "tests", f)
                                                for f in os.listdir(os.path.join(ROOT, "tests")) if f.endswith(".py")]
    missing = set()
    for f in files:
        for node in ast.walk(ast.parse(open(f).read())):
            if isinstance(node, ast.Attribute) and isinstance(node.value, ast.Name) and node.value.id == "W":
                if not hasattr(W, node.attr):
                    missing.add(f"{os.path.basename(f)}: W.{node.attr}")
    assert not missing, sorted(missing)


@pytest.mark.timeout(300)
def test_all_cores_oracle_timing_splits_the_work_exactly():
    """The all-cores CPU baseline runs the oracle on an equal share of every
    shard in each process; reassembled, the parameters after three steps equal
    one process's run over the whole sample."""
    import numpy as np
    import bench
    import oracle
    import workloads as W
    n = 1001
    sample = bench.cpu_sample_gpt2(W, n)
    nd, grads, flat, h = sample
    ne, walls, got = bench.time_oracle_parallel(sample, n, 3, 3, want_params=True)
    assert ne == nd * n and len(walls) == 3 and all(w > 0 for w in walls)
    ref = flat.copy()
    shards = [dict(numel=n, grad_off=r * n, param_off=r * n, master=oracle.widen_16(ref[r * n:(r + 1) * n], 2),
                   m=np.zeros(n, np.float32), v=np.zeros(n, np.float32)) for r in range(nd)]
    for t in (1, 2, 3):
        oracle.zero_step(grads, 2, shards, ref, 2, dict(h, max_grad_norm=0.0), t, 1.0)
    assert not np.array_equal(ref, flat)
    assert np.array_equal(got, ref)



class _FakeEvent:
    def __init__(self, t):
        self.t = t

    def elapsed_time(self, other):
        return other.t - self.t


def test_grouped_kernel_timing_and_the_dominant_kernel():
    """One event pair may enclose several back-to-back launches of a kernel
    (the ZeRO-3 step's 68 gathers, 34 reduces): the time per launch is the
    enclosed time over the launch count, and the roofline entry names the
    kernel with the most time per step, with its algorithmic bytes per launch
    (the workload's bytes per step over its launches per step)."""
    import bench
    timer = bench.KernelTimer(None)
    steps = 2
    for s in range(steps):
        timer.events.append(("k_gather_bulk", 68, _FakeEvent(0.0), _FakeEvent(9.92)))
        timer.events.append(("k_reduce", 34, _FakeEvent(0.0), _FakeEvent(3.06)))
        timer.events.append(("k_apply", 1, _FakeEvent(0.0), _FakeEvent(8.6)))
    kinds = timer.per_kind(steps)
    assert kinds["k_gather_bulk"]["launches"] == 136 and kinds["k_gather_bulk"]["event_pairs"] == 2
    assert kinds["k_gather_bulk"]["ms_per_launch"] == pytest.approx(9.92 / 68)
    assert kinds["k_reduce"]["ms_per_step"] == pytest.approx(3.06)
    wl = {"name": "w", "state": {"path": 2}, "config": {},
          "kernel_bytes": {"k_gather_bulk": 64_242_089_984, "k_reduce": 20_075_653_120, "k_apply": 56_211_828_736}}
    roof, per, peak = bench.kernel_figures(wl, kinds, steps)
    assert roof["kernel"] == "k_gather_bulk" and roof["bound"] == "hbm"
    assert roof["algorithmic_bytes_per_launch"] == pytest.approx(64_242_089_984 / 68)
    assert roof["achieved"] == pytest.approx(64_242_089_984 / 68 / (9.92 / 68 / 1e3) / 1e9)
    assert roof["frac"] == pytest.approx(roof["achieved"] / peak)
    assert per["k_apply"]["achieved_gbs"] == pytest.approx(56_211_828_736 / 8.6e-3 / 1e9)
