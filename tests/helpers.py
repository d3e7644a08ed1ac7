"""Small shared helpers for the tests: building seeded all-ranks problems as
numpy arrays for the oracle, and bit-level comparisons."""
import numpy as np
import torch

import workloads as W

HYPER = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01, max_grad_norm=0.0)
TDT = {1: torch.float16, 2: torch.bfloat16}


def f32(x):
    """Round a python float to the nearest fp32 value (what the C structs hold)."""
    return float(np.float32(x))


def hyper32(**kw):
    h = dict(HYPER)
    h.update(kw)
    return {k: f32(v) for k, v in h.items()}


def t2u16(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().cpu().view(torch.int16).numpy().view(np.uint16).copy()


def u16_to_t(a: np.ndarray, dt: int) -> torch.Tensor:
    return torch.from_numpy(a.view(np.int16).copy()).view(TDT[dt])


def ulp_dist(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Distance in fp32 ulps (monotone integer mapping of the bit patterns)."""
    def key(x):
        i = x.astype(np.float32).view(np.int32).astype(np.int64)
        return np.where(i < 0, -(i & 0x7FFFFFFF), i)
    return np.abs(key(a) - key(b))


def random_group(rng, max_tensors=5, max_numel=300):
    n = int(rng.integers(1, max_tensors + 1))
    return [int(x) for x in rng.integers(1, max_numel, n)]


def make_problem(numels, nd, dt, mode, seed, loss_scale=1.0, grad_std=1e-3, steps=3):
    """Seeded all-ranks problem: flat params, and per step nd full flat grads (padded with zeros)."""
    import oracle
    p = oracle.plan(numels, nd, mode)
    P = p["padded_total"]
    specs = [W.ParamSpec(f"t{i}", n) for i, n in enumerate(numels)]
    flat = torch.zeros(P, dtype=TDT[dt])
    W.init_params_(flat, specs, W.generator(seed, "cpu"))
    gens = [W.generator(seed + 1 + r, "cpu") for r in range(nd)]
    grads = []
    for _ in range(steps):
        step = []
        for r in range(nd):
            g = torch.zeros(P, dtype=TDT[dt])
            W.fill_grad_(g, specs, gens[r], lambda s: grad_std, loss_scale)
            step.append(t2u16(g))
        grads.append(step)
    return p, t2u16(flat), grads
