"""Seeded synthetic inputs for the ZeRO-DP partitioned optimizer step.

This module only describes parameter-group shapes and draws seeded random
tensors.  It holds none of the method's arithmetic (no averaging, no norm, no
Adam): the oracle and the CUDA path both receive the bytes it produces and
nothing else.  Tests and the benchmark import it; the library does not.

Workloads (all synthetic; the pages measure on no public data set):
  tiny-nd3           three tensors [257,129], [129], [1000,37] (Psi = 70,282),
                     N_d = 3, fp16, loss scale 1024, one +inf gradient at step 2
  gpt2-1.5b-nd8      GPT-2 1.5B-shaped group (48 layers, d = 1600, 4d MLP,
                     vocab 50257, context 1024, tied head), N_d = 8, all ranks
                     simulated, bf16
  llama3-8b-nd4-r1   Llama-3-8B-shaped group (32 layers, d = 4096, GQA 32q/8kv
                     heads of 128, SwiGLU 14336, vocab 128256, untied head),
                     N_d = 4, rank 1's shard only, bf16, global-norm clip 1.0
  gpt-7.5b-nd64-r63  GPT-like 7.5B shape (52 layers, d = 3456, 4d MLP, vocab
                     50257, context 1024), N_d = 64, rank 63's shard, fp16,
                     loss scale 65536, slice 0 holds exact zeros at every
                     100th element
  zero3-llama3-8b    the Llama-3-8B group as 34 ZeRO-3 units (embedding, 32
                     blocks, final norm + head), N_d = 4, rank 1

Random draws use torch generators seeded per rank / slice as listed with each
workload; a generator keeps drawing across steps, so every step gets fresh
gradients.  Values are drawn in fp32 (standard normal times the stated
standard deviation, times the loss scale where one is given) and rounded to the
16-bit dtype by torch.
"""
from __future__ import annotations

import json
import os
from dataclasses import dataclass, field

import torch

CHUNK = 1 << 26  # fp32 temporaries are bounded to 256 MB


@dataclass
class ParamSpec:
    name: str
    numel: int
    init: str = "normal"   # "normal" (std 0.02), "ones", "zeros"
    layer: int = 0         # depth index used by depth-scaled gradient std


# ------------------------------------------------------------------ shapes
def tiny_group():
    return [ParamSpec("w0", 257 * 129), ParamSpec("b0", 129), ParamSpec("w1", 1000 * 37)]


def gpt2_group(L=48, d=1600, V=50257, ctx=1024, wpe=True):
    """GPT-2 order: wte, wpe, h.0..h.{L-1}, ln_f; LayerNorm weight 1, bias 0; tied head."""
    out = [ParamSpec("wte", V * d, layer=0)]
    if wpe:
        out.append(ParamSpec("wpe", ctx * d, layer=0))
    for l in range(L):
        p = f"h.{l}."
        out += [ParamSpec(p + "ln_1.w", d, "ones", l), ParamSpec(p + "ln_1.b", d, "zeros", l),
                ParamSpec(p + "attn.c_attn.w", d * 3 * d, layer=l), ParamSpec(p + "attn.c_attn.b", 3 * d, layer=l),
                ParamSpec(p + "attn.c_proj.w", d * d, layer=l), ParamSpec(p + "attn.c_proj.b", d, layer=l),
                ParamSpec(p + "ln_2.w", d, "ones", l), ParamSpec(p + "ln_2.b", d, "zeros", l),
                ParamSpec(p + "mlp.c_fc.w", d * 4 * d, layer=l), ParamSpec(p + "mlp.c_fc.b", 4 * d, layer=l),
                ParamSpec(p + "mlp.c_proj.w", 4 * d * d, layer=l), ParamSpec(p + "mlp.c_proj.b", d, layer=l)]
    out += [ParamSpec("ln_f.w", d, "ones", L), ParamSpec("ln_f.b", d, "zeros", L)]
    return out


def llama_group(L=32, d=4096, hq=32, hkv=8, hd=128, ff=14336, V=128256):
    """Llama order: embed, layers (q, k, v, o, gate, up, down, in_norm, post_norm), norm, lm_head."""
    out = [ParamSpec("embed", V * d, layer=0)]
    for l in range(L):
        p = f"layers.{l}."
        out += [ParamSpec(p + "q", d * hq * hd, layer=l), ParamSpec(p + "k", d * hkv * hd, layer=l),
                ParamSpec(p + "v", d * hkv * hd, layer=l), ParamSpec(p + "o", hq * hd * d, layer=l),
                ParamSpec(p + "gate", d * ff, layer=l), ParamSpec(p + "up", d * ff, layer=l),
                ParamSpec(p + "down", ff * d, layer=l), ParamSpec(p + "in_norm", d, "ones", l),
                ParamSpec(p + "post_norm", d, "ones", l)]
    out += [ParamSpec("norm", d, "ones", L), ParamSpec("lm_head", V * d, layer=L)]
    return out


def llama_units(specs, L=32):
    """ZeRO-3 units: the embedding, each block, and (final norm + head)."""
    units = [[specs[0]]]
    per = (len(specs) - 3) // L
    for l in range(L):
        units.append(specs[1 + l * per: 1 + (l + 1) * per])
    units.append(specs[-2:])
    return [sum(s.numel for s in u) for u in units]


def numels(specs):
    return [s.numel for s in specs]


# ------------------------------------------------------------------ draws
def generator(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def fill_normal_(out: torch.Tensor, std: float, gen: torch.Generator, scale: float = 1.0):
    """out (1-D, 16-bit) <- round16(N(0,1) * std * scale), drawn in fp32 chunks."""
    n = out.numel()
    for s in range(0, n, CHUNK):
        e = min(n, s + CHUNK)
        x = torch.randn(e - s, generator=gen, device=out.device, dtype=torch.float32)
        x.mul_(std * scale)
        out[s:e].copy_(x)
    return out


def init_params_(flat: torch.Tensor, specs, gen: torch.Generator, std: float = 0.02):
    """Write the initial 16-bit parameters in flat order; padding stays 0."""
    flat.zero_()
    off = 0
    for s in specs:
        seg = flat[off:off + s.numel]
        if s.init == "normal":
            fill_normal_(seg, std, gen)
        elif s.init == "ones":
            seg.fill_(1.0)
        off += s.numel
    return flat


def fill_grad_(flat: torch.Tensor, specs, gen: torch.Generator, std_of, scale: float = 1.0):
    """One rank's full flat gradient: each tensor's segment ~ N(0, std_of(spec)) * scale."""
    flat.zero_()
    off = 0
    for s in specs:
        fill_normal_(flat[off:off + s.numel], std_of(s), gen, scale)
        off += s.numel
    return flat


def gpt2_grad_std(L=48):
    """std 1e-3 * (1 + layer/L): embeddings at depth 0, ln_f at depth L."""
    return lambda s: 1e-3 * (1.0 + s.layer / L)


DTYPES = {"f16": torch.float16, "bf16": torch.bfloat16}


@dataclass
class Workload:
    name: str
    specs: list
    nd: int
    dtype: str            # "f16" or "bf16" (grads and params)
    ranks: list           # simulated ranks whose shards the step updates
    loss_scale: float = 1.0
    max_grad_norm: float = 0.0
    hyper: dict = field(default_factory=lambda: dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8,
                                                     weight_decay=0.01))
    param_seed: int = 0
    grad_std: float = 1e-3
    notes: str = ""


def workload(name: str) -> Workload:
    if name == "tiny-nd3":
        return Workload(name, tiny_group(), 3, "f16", [0, 1, 2], loss_scale=1024.0,
                        notes="grads of rank r from seed 1+r; +inf at flat index 30000 of rank 0 at step 2")
    if name == "gpt2-1.5b-nd8":
        return Workload(name, gpt2_group(), 8, "bf16", list(range(8)),
                        notes="rank r grads from seed 1+r with std 1e-3*(1+layer/48)")
    if name == "llama3-8b-nd4-r1":
        return Workload(name, llama_group(), 4, "bf16", [1], max_grad_norm=1.0, grad_std=5e-4,
                        notes="slice j from seed 2+j, N(0,5e-4)")
    if name == "gpt-7.5b-nd64-r63":
        return Workload(name, gpt2_group(52, 3456, 50257, 1024), 64, "f16", [63], loss_scale=65536.0,
                        notes="slice j from seed 4+j, N(0,1e-3)*65536; slice 0 zero at j%100==0")
    if name == "zero3-llama3-8b":
        return Workload(name, llama_group(), 4, "bf16", [1], grad_std=5e-4, param_seed=3,
                        notes="per unit 4 buckets, bucket r from seed 5+r, N(0,5e-4)")
    raise KeyError(name)


OTHER_RANKS_SUMSQ = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tests", "golden",
                                 "other_ranks_sumsq.json")


def other_ranks_sumsq(wl: Workload) -> float:
    """The rank-local views need the other ranks' share of the global sum of
    squares (the operands of the norm's scalar all-reduce that this rank does
    not compute).  It is an input of the step, generated once from data:
    tests/golden/make_other_ranks_sumsq.py draws every other rank's staged
    slices with the workload's recipe from their own seeded generators and has
    the oracle reduce them and sum the squares exactly; the value is stored in
    tests/golden/other_ranks_sumsq.json with its recipe.  Workloads without a
    stored share (every rank simulated, or no clipping) take 0."""
    try:
        with open(OTHER_RANKS_SUMSQ) as f:
            return float(json.load(f)[wl.name]["value"])
    except (OSError, KeyError):
        return 0.0


# ------------------------------------------------------------------ device-side input sets
class GradStream:
    """Seeded gradient draws that continue across steps: one generator per
    rank (or staged slice), seeds as listed with each workload."""

    def __init__(self, seeds, device):
        self.gens = [generator(s, device) for s in seeds]

    def draw_flat(self, outs, specs, std_of, scale=1.0):
        """Full flat gradients (all-ranks view): rank r's buffer from generator r."""
        for g, o in zip(self.gens, outs):
            fill_grad_(o, specs, g, std_of, scale)
        return outs

    def draw_plain(self, outs, std, scale=1.0):
        """Staged slices (rank-local view): slice j ~ N(0, std) * scale from generator j."""
        for g, o in zip(self.gens, outs):
            fill_normal_(o, std, g, scale)
        return outs


def zero_every_100th_(t: torch.Tensor):
    """Exact zeros at every element whose index is a multiple of 100 (the 7.5B workload's slice 0)."""
    t[::100] = 0
    return t


def flat_params(specs, total: int, dtype, seed: int, device):
    """The group's 16-bit parameters laid out flat over `total` elements (the
    plan's padded length); padding is 0."""
    flat = torch.zeros(total, dtype=dtype, device=device)
    return init_params_(flat, specs, generator(seed, device))
