"""zero_shard_step_noalloc: the step for callers that cannot allocate device
memory (for instance code that must not call cudaMalloc because it can stall
the device, or callers whose host program owns all device memory).  It must
give what zero_shard_step gives: two calls in a row on each path (the fused
single pass, and the two-pass path that clipping selects), compared with the
same calls made through zero_shard_step with caller-provided scratch.  The
comparison is exact: both entry points run the same kernels with the same
launch shape.  This file is collected last on purpose."""
import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def Z():
    import zero_dp_partitioned_gb300 as Z
    return Z


def _setup(Z, numels, nd, seed):
    specs = [W.ParamSpec(f"t{i}", n) for i, n in enumerate(numels)]
    plan = Z.zero_plan(numels, nd)
    P = plan["padded_total"]
    flat = W.flat_params(specs, P, torch.bfloat16, seed, DEV)
    gs = W.GradStream([seed + 1 + r for r in range(nd)], DEV)
    grads = [[torch.empty(P, dtype=torch.bfloat16, device=DEV) for _ in range(nd)] for _ in range(2)]
    for g in grads:
        gs.draw_flat(g, specs, lambda s: 1e-2)
    return plan, flat, grads


def _state(plan, flat, pingpong):
    out = []
    for o, n in zip(plan["rank_offsets"], plan["rank_numels"]):
        A = [flat[o:o + n].float(), torch.zeros(n, device=DEV), torch.zeros(n, device=DEV)]
        B = [torch.empty(n, device=DEV) for _ in range(3)] if pingpong else A
        out.append(dict(o=o, n=n, A=A, B=B, g=torch.empty(n, dtype=torch.bfloat16, device=DEV)))
    return out


@pytest.mark.parametrize("clip", [0.0, 0.05])
def test_noalloc_matches_the_step_with_caller_scratch(Z, clip):
    nd = 4
    plan, flat0, grads = _setup(Z, [300001, 4097, 77777], nd, seed=31)
    runs = {}
    for entry in ("step", "noalloc"):
        flat = flat0.clone()
        st = _state(plan, flat, pingpong=(clip == 0.0))
        ws = torch.zeros(Z.zero_workspace_bytes(), dtype=torch.uint8, device=DEV)
        res = torch.zeros(48, dtype=torch.uint8, device=DEV)
        results = []
        for t in (1, 2):                                   # two calls in a row, state carried over
            sh = [Z.shard(s["n"], s["o"], s["o"], *s["A"], *s["B"], s["g"]) for s in st]
            h = Z.hyper(max_grad_norm=clip, step=t)
            if entry == "step":
                Z.zero_shard_step(grads[t - 1], Z.ZERO_BF16, sh, flat, Z.ZERO_BF16, h, 1.0, 0.0, 0, ws, ws.numel(), res)
            else:
                Z.zero_shard_step_noalloc(grads[t - 1], Z.ZERO_BF16, sh, flat, Z.ZERO_BF16, h, 1.0, 0.0, 0, res)
            torch.cuda.synchronize()
            r = Z.read_result(res)
            assert r.applied == 1 and r.status == 0
            results.append(r.as_dict())
            if clip == 0.0:
                for s in st:
                    s["A"], s["B"] = s["B"], s["A"]
            runs[(entry, t)] = (flat.clone(), [[x.clone() for x in s["A"]] for s in st], r.as_dict())
    for t in (1, 2):
        fa, sa, ra = runs[("step", t)]
        fb, sb, rb = runs[("noalloc", t)]
        assert torch.equal(fa, fb)
        for xa, xb in zip(sa, sb):
            for a, b in zip(xa, xb):
                assert torch.equal(a, b)
        assert ra == rb
        if clip > 0.0:
            assert ra["clip_coef"] < 1.0 and ra["path"] in (2, 4, 6)


def test_noalloc_rejects_two_pass_calls_beyond_its_scratch(Z):
    n = (1 << 21) + 1          # one element more than the built-in reduced-gradient scratch holds
    g = torch.zeros(n, dtype=torch.bfloat16, device=DEV)
    st = [torch.zeros(n, device=DEV) for _ in range(3)]
    res = torch.zeros(48, dtype=torch.uint8, device=DEV)
    flat = torch.zeros(n, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(Z.ZeroError) as e:
        Z.zero_shard_step_noalloc([g], Z.ZERO_BF16, [Z.shard(n, 0, 0, *st)], flat, Z.ZERO_BF16,
                                  Z.hyper(max_grad_norm=1.0), 1.0, 0.0, 0, res)
    assert e.value.code == Z.ZERO_ELIMIT and "scratch" in str(e.value)
