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
            assert ra["clip_coef"] < 1.0 and ra["path"] == 2


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


def _cudart():
    """The CUDA runtime this process has loaded (for the stream-capture calls)."""
    import ctypes
    paths = sorted({line.split()[-1] for line in open("/proc/self/maps") if "libcudart.so" in line})
    assert paths, "no CUDA runtime mapped"
    rt = ctypes.CDLL(paths[0])
    rt.cudaStreamBeginCapture.argtypes = [ctypes.c_void_p, ctypes.c_int]
    rt.cudaStreamEndCapture.argtypes = [ctypes.c_void_p, ctypes.POINTER(ctypes.c_void_p)]
    rt.cudaGraphGetNodes.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.POINTER(ctypes.c_size_t)]
    rt.cudaGraphDestroy.argtypes = [ctypes.c_void_p]
    return rt


def test_noalloc_argument_errors_enqueue_nothing(Z):
    """A call rejected for its arguments must return before it clears the
    shared scratch or launches anything: calls with a bad dtype, step 0, a NaN
    loss scale, a misaligned result and a NULL slice are made on a stream
    under capture, and the captured graph must be empty -- while a valid
    gather captured after them adds exactly its one kernel."""
    import ctypes
    nd = 2
    plan, flat, grads = _setup(Z, [5000, 333], nd, seed=41)
    st = _state(plan, flat, pingpong=True)
    sh = [Z.shard(s["n"], s["o"], s["o"], *s["A"], *s["B"], s["g"]) for s in st]
    res = torch.zeros(64, dtype=torch.uint8, device=DEV)
    Z.zero_shard_step_noalloc(grads[0], Z.ZERO_BF16, sh, flat, Z.ZERO_BF16, Z.hyper(step=1), 1.0, 0.0, 0, res)
    torch.cuda.synchronize()                   # a valid call first: the library's device code is loaded
    layer = torch.empty(2 * 4096, dtype=torch.bfloat16, device=DEV)
    parts = [flat[:4096], flat[4096:8192]]
    Z.zero3_gather_layer(parts, 2 * 4096, Z.ZERO_BF16, layer)    # and the gather's launch set-up done eagerly
    torch.cuda.synchronize()
    bad = [dict(gdt=7), dict(h=Z.hyper(step=0)), dict(S=float("nan")), dict(r=res[4:]),
           dict(g=[grads[0][0], 0])]
    rt = _cudart()
    s = torch.cuda.Stream()
    for with_gather in (False, True):
        assert rt.cudaStreamBeginCapture(s.cuda_stream, 2) == 0           # relaxed mode
        for b in bad:
            with pytest.raises(Z.ZeroError) as e:
                Z.zero_shard_step_noalloc(b.get("g", grads[0]), b.get("gdt", Z.ZERO_BF16), sh, flat, Z.ZERO_BF16,
                                          b.get("h", Z.hyper(step=1)), b.get("S", 1.0), 0.0, 0, b.get("r", res),
                                          stream=s)
            assert e.value.code in (Z.ZERO_EINVAL, Z.ZERO_EALIGN)
        if with_gather:
            Z.zero3_gather_layer(parts, 2 * 4096, Z.ZERO_BF16, layer, stream=s)
        graph = ctypes.c_void_p()
        assert rt.cudaStreamEndCapture(s.cuda_stream, ctypes.byref(graph)) == 0
        nodes = ctypes.c_size_t(0)
        assert rt.cudaGraphGetNodes(graph, None, ctypes.byref(nodes)) == 0
        rt.cudaGraphDestroy(graph)
        assert nodes.value == (1 if with_gather else 0)
