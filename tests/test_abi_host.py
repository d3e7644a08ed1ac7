"""CPU tests of the C-ABI library: it loads, exports every function
include/zero.h declares, its host-only calls (plan, intersections, memory
model) equal the oracle bit for bit, and argument errors are reported before
any device work (no GPU is touched here)."""
import ctypes
import os
import re
import subprocess
import sys

import numpy as np
import pytest

import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def Z():
    import __graft_entry__
    __graft_entry__.build()
    import zero_dp_partitioned_gb300 as Z
    return Z


def _declared():
    src = open(os.path.join(ROOT, "include", "zero.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w]+\s*\**\s*(zero\w*)\s*\(", src, flags=re.M)))


def test_exports_every_declared_symbol(Z):
    names = _declared()
    assert len(names) >= 10
    for n in names:
        assert hasattr(Z.lib, n), n
    assert set(names) == set(Z.EXPORTS)
    nm = subprocess.run(["nm", "-D", "--defined-only", Z.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r" T (\w+)$", nm, flags=re.M))
    assert set(names) <= exported


def test_struct_sizes_match_header(Z):
    assert ctypes.sizeof(Z.zero_result) == 48 and ctypes.sizeof(Z.zero_shard) == 80
    assert Z.zero_workspace_bytes() >= 128 + 12 * 2048


@pytest.mark.parametrize("mode", [0, 1])
def test_plan_equals_oracle(Z, orc, mode):
    rng = np.random.default_rng(3 + mode)
    cases = [(W.numels(W.tiny_group()), 3), (W.numels(W.gpt2_group()), 8), (W.numels(W.llama_group()), 4),
             (W.numels(W.gpt2_group(52, 3456, 50257, 1024)), 64), ([0], 5), ([1, 2, 3], 1)]
    for _ in range(200):
        cases.append(([int(x) for x in rng.integers(0, 1000, int(rng.integers(1, 8)))], int(rng.integers(1, 70))))
    for numels, ws in cases:
        a = Z.zero_plan(numels, ws, mode)
        b = orc.plan(numels, ws, mode)
        assert a["tensor_offsets"] == list(b["tensor_offsets"])
        assert a["rank_offsets"] == list(b["rank_offsets"]) and a["rank_numels"] == list(b["rank_numels"])
        assert (a["padded_total"], a["padding"]) == (b["padded_total"], b["padding"])
        for r in {0, ws // 2, ws - 1}:
            x = Z.zero_plan_intersections(a["tensor_offsets"], numels, a["rank_offsets"][r], a["rank_numels"][r])
            y = orc.plan_intersections(b["tensor_offsets"], numels, int(b["rank_offsets"][r]), int(b["rank_numels"][r]))
            assert [list(t) for t in x] == y.tolist()


def test_workload_shapes(Z):
    # derived sizes of the benchmark workloads (flat lengths, shard sizes and offsets)
    g2 = Z.zero_plan(W.numels(W.gpt2_group()), 8)
    assert g2["padded_total"] == 1_557_611_200 and g2["padding"] == 0 and g2["rank_numels"][0] == 194_701_400
    l3 = Z.zero_plan(W.numels(W.llama_group()), 4)
    assert l3["padded_total"] == 8_030_261_248 and l3["rank_numels"][1] == 2_007_565_312
    assert l3["rank_offsets"][1] == 2_007_565_312
    g75 = Z.zero_plan(W.numels(W.gpt2_group(52, 3456, 50257, 1024)), 64)
    assert g75["padded_total"] == 7_632_586_368 and g75["rank_numels"][63] == 119_259_162
    assert g75["rank_offsets"][63] == 7_513_327_206 and g75["rank_offsets"][63] % 8 == 6
    units = W.llama_units(W.llama_group())
    assert len(units) == 34 and sum(units) == 8_030_261_248 and all(u % 8 == 0 for u in units)


def test_mem_model_equals_oracle(Z, orc):
    for psi in (7.5e9, 1e12, 8e9, 1.5e9, 123.0):
        for K in (12, 16, 8):
            for nd in (1, 4, 64, 1024):
                for st in range(4):
                    assert Z.zero_mem_model(psi, K, nd, st) == orc.mem_model(psi, K, nd, st)
    with pytest.raises(Z.ZeroError):
        Z.zero_mem_model(1e9, 12, 64, 4)
    with pytest.raises(Z.ZeroError):
        Z.zero_mem_model(1e9, 12, 0, 1)


def test_mem_model_plan_equals_oracle(Z, orc):
    units = W.llama_units(W.llama_group())
    cases = []
    for numels, nd, mode in ((W.numels(W.tiny_group()), 3, 0), (W.numels(W.tiny_group()), 3, 1),
                             (W.numels(W.gpt2_group()), 8, 0), (W.numels(W.llama_group()), 4, 0),
                             (W.numels(W.gpt2_group(52, 3456, 50257, 1024)), 64, 0)):
        p = Z.zero_plan(numels, nd, mode)
        cases += [(p["padded_total"], n) for n in set(p["rank_numels"])]
    cases.append((sum(units), sum(u // 4 for u in units)))          # ZeRO-3 rank: its part of every unit
    for F, n in cases:
        for st in range(4):
            for sets, f32, b16 in ((1, 0, 0), (2, 0, 0), (1, F, 0), (2, 0, max(units))):
                assert Z.zero_mem_model_plan(F, n, 12, st, sets, f32, b16) == \
                    orc.mem_model_plan(F, n, 12, st, sets, f32, b16)
    for bad in ((-1, 0, 12, 1, 1, 0, 0), (8, 2, 12, 4, 1, 0, 0), (8, 2, 12, 1, 0, 0, 0), (8, 2, -1.0, 1, 1, 0, 0),
                (8, 2, 12, 1, 1, -5, 0), (8, -2, 12, 1, 1, 0, 0)):
        with pytest.raises(Z.ZeroError):
            Z.zero_mem_model_plan(*bad)


def test_adam_scalar_table_equals_oracle(Z, orc):
    for lr, b1, b2, wd in ((1e-3, 0.9, 0.999, 0.01), (3e-4, 0.95, 0.98, 0.1), (1.0, 0.5, 0.5, 0.0)):
        h = Z.hyper(lr=lr, beta1=b1, beta2=b2, weight_decay=wd, step=1)
        tab = Z.zero_adam_scalar_table(h, 7, 50)
        for i in range(50):
            sc = orc.make_scalars(np.float32(lr), np.float32(b1), np.float32(b2), np.float32(1e-8), np.float32(wd),
                                  7 + i)
            assert tab[2 * i] == np.float32(sc.ss) and tab[2 * i + 1] == np.float32(sc.rb2)
    with pytest.raises(Z.ZeroError):
        Z.zero_adam_scalar_table(Z.hyper(), 0, 4)


def test_argument_errors_before_any_device_work(Z):
    fake = 0x10000   # never dereferenced: every case below fails validation first
    ws = Z.zero_workspace_bytes()
    sh = [Z.shard(8, 0, 0, fake, fake, fake, fake + 64, fake + 128, fake + 192)]
    h = Z.hyper()
    cases = [
        (dict(grad_slices=[], n_err=Z.ZERO_EINVAL)),
        (dict(grad_slices=[fake] * 65, n_err=Z.ZERO_ELIMIT)),
        (dict(grad_slices=[fake + 1], n_err=Z.ZERO_EALIGN)),
        (dict(grad_slices=[fake], workspace=None, n_err=Z.ZERO_EWORKSPACE)),
        (dict(grad_slices=[fake], ws_bytes=ws - 1, n_err=Z.ZERO_EWORKSPACE)),
        (dict(grad_slices=[fake], gdt=3, n_err=Z.ZERO_EINVAL)),
        (dict(grad_slices=[fake], loss_scale=0.0, n_err=Z.ZERO_EINVAL)),
        (dict(grad_slices=[fake], step=0, n_err=Z.ZERO_EINVAL)),
        (dict(grad_slices=[fake], shards=[Z.shard(-1, 0, 0, fake, fake, fake)], n_err=Z.ZERO_EINVAL)),
        (dict(grad_slices=[fake], shards=[Z.shard(8, 0, 0, fake + 2, fake, fake, fake + 64, fake + 128, fake + 192)],
              n_err=Z.ZERO_EALIGN)),
        # clipping needs the two-pass path, which needs grad_shard
        (dict(grad_slices=[fake], clip=1.0, n_err=Z.ZERO_EINVAL)),
        (dict(grad_slices=[fake], shards=sh * 65, n_err=Z.ZERO_ELIMIT)),
    ]
    for c in cases:
        hh = Z.hyper(max_grad_norm=c.get("clip", 0.0), step=c.get("step", 1))
        with pytest.raises(Z.ZeroError) as e:
            Z.zero_shard_step(c["grad_slices"], c.get("gdt", Z.ZERO_BF16), c.get("shards", sh), fake, Z.ZERO_BF16,
                              hh, c.get("loss_scale", 1.0), 0.0, 0, c.get("workspace", fake),
                              c.get("ws_bytes", ws), fake, stream=0)
        assert e.value.code == c["n_err"], (c, str(e.value))
    with pytest.raises(Z.ZeroError) as e:
        Z.zero3_gather_layer([fake] * 3, 10, Z.ZERO_BF16, fake, stream=0)      # 10 does not divide by 3
    assert e.value.code == Z.ZERO_EINVAL
    with pytest.raises(Z.ZeroError) as e:
        Z.zero3_reduce_bucket([fake] * 4, 4, 16, Z.ZERO_BF16, fake, 0, fake, fake, ws, stream=0)  # owner 4 of 4
    assert e.value.code == Z.ZERO_EINVAL
    with pytest.raises(Z.ZeroError):
        Z.zero_plan([1, 2], 0)
    for shards, flat, pdt, code in ((sh, fake, 3, Z.ZERO_EINVAL),                              # unknown dtype
                                    (sh, fake + 1, Z.ZERO_BF16, Z.ZERO_EINVAL),                # odd parameter buffer
                                    (sh, 0, Z.ZERO_BF16, Z.ZERO_EINVAL),                       # no parameter buffer
                                    ([Z.shard(8, 0, 0, fake + 2, fake, fake, fake, fake, fake)], fake, Z.ZERO_BF16,
                                     Z.ZERO_EALIGN),
                                    ([Z.shard(8, 0, 0, 0, fake, fake, fake, fake, fake)], fake, Z.ZERO_BF16,
                                     Z.ZERO_EINVAL),
                                    (sh * 65, fake, Z.ZERO_BF16, Z.ZERO_ELIMIT)):
        with pytest.raises(Z.ZeroError) as e:
            Z.zero_shard_init(shards, flat, pdt, stream=0)
        assert e.value.code == code
    Z.zero_shard_init([Z.shard(0, 0, 0, 0, 0, 0, 0, 0, 0)], 0, Z.ZERO_BF16, stream=0)   # nothing to do: no launch
    # the step from host buffers: the checks that come before it asks the
    # driver about any pointer
    for c in (dict(gdt=3, code=Z.ZERO_EINVAL), dict(loss_scale=float("inf"), code=Z.ZERO_EINVAL),
              dict(step=0, code=Z.ZERO_EINVAL), dict(result=0, code=Z.ZERO_EINVAL),
              dict(result=fake + 4, code=Z.ZERO_EINVAL), dict(slices=[], code=Z.ZERO_EINVAL),
              dict(slices=[fake] * 65, code=Z.ZERO_ELIMIT), dict(slices=[fake + 1], code=Z.ZERO_EALIGN)):
        with pytest.raises(Z.ZeroError) as e:
            Z.zero_shard_step_host(c.get("slices", [fake]), c.get("gdt", Z.ZERO_BF16), sh, fake, Z.ZERO_BF16, fake,
                                   Z.hyper(step=c.get("step", 1)), c.get("loss_scale", 1.0), 0.0, 0, fake, 1 << 20,
                                   fake, ws, c.get("result", fake), stream=0)
        assert e.value.code == c["code"], (c, str(e.value))


def test_comm_volume_equals_oracle(Z, orc):
    for psi in (7.5e9, 1e12, 123.0):
        for nd in (1, 2, 8, 64, 1024):
            for st in range(4):
                for ring in (False, True):
                    assert Z.zero_comm_volume(psi, nd, st, ring) == orc.comm_volume(psi, nd, st, ring)
    with pytest.raises(Z.ZeroError):
        Z.zero_comm_volume(1e9, 8, 4)


def test_round_robin_equals_oracle(Z, orc):
    for n in (0, 1, 5, 17, 580):
        for ws in (1, 2, 3, 8, 64):
            assert Z.zero_plan_round_robin(n, ws) == orc.round_robin(n, ws).tolist()
    with pytest.raises(Z.ZeroError):
        Z.zero_plan_round_robin(4, 0)


def test_import_without_the_library_fails_loudly(tmp_path):
    """The package has no fallback: without its built library the import
    raises, and nothing in it reaches for the oracle."""
    pkg = tmp_path / "zero_dp_partitioned_gb300"
    pkg.mkdir()
    src = open(os.path.join(ROOT, "zero_dp_partitioned_gb300", "__init__.py")).read()
    assert "oracle" not in src
    (pkg / "__init__.py").write_text(src)
    r = subprocess.run([sys.executable, "-c", "import zero_dp_partitioned_gb300"], cwd=tmp_path,
                       capture_output=True, text=True)
    assert r.returncode != 0 and "ImportError" in r.stderr and "libzero_gb300.so is missing" in r.stderr
