"""CPU oracle of the ZeRO-DP partitioned mixed-precision optimizer step.

TEST INFRASTRUCTURE ONLY.  The product path never imports this package: only
``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference legs of
``bench.py`` may.  It is a thin ctypes layer over ``zero_oracle.c`` (plain,
single-threaded C, scalar loops) and shares no code with the CUDA library.

Every function works on numpy arrays; 16-bit values travel as ``uint16`` bit
patterns.  dtype codes: 1 = fp16, 2 = bf16.

Which passage each function follows is stated in ``zero_oracle.c``.  Every
function here is pinned by a CPU test (``tests/test_oracle_*.py``) to something
other than itself: exhaustive comparison with numpy/torch conversions, Python's
correctly rounded ``math.fsum``, ``torch.optim.AdamW``, closed forms, the
memory figures printed on the pages, brute force on tiny inputs, and the
unpartitioned data-parallel step.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "zero_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboracle.so")

F16, BF16 = 1, 2
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile zero_oracle.c with gcc (IEEE fp32: no contraction, no fast-math)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
             "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _SO)
    return _SO


class Result(ctypes.Structure):
    _fields_ = [("overflow", ctypes.c_int32), ("applied", ctypes.c_int32),
                ("sumsq", ctypes.c_double), ("grad_norm", ctypes.c_double),
                ("clip_coef", ctypes.c_double), ("grad_mult", ctypes.c_float),
                ("pad", ctypes.c_float)]

    def as_dict(self):
        return {k: getattr(self, k) for k, _ in self._fields_ if k != "pad"}


class Scalars(ctypes.Structure):
    _fields_ = [(n, ctypes.c_float) for n in ("b1", "b2", "omb1", "omb2", "eps", "wdf", "ss", "rb2")]


_P = ctypes.c_void_p
_I64 = ctypes.c_int64


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_SO)
            sig = {
                "orc_f32_to_f16": (ctypes.c_uint16, [ctypes.c_float]),
                "orc_f32_to_bf16": (ctypes.c_uint16, [ctypes.c_float]),
                "orc_f16_to_f32": (ctypes.c_float, [ctypes.c_uint16]),
                "orc_bf16_to_f32": (ctypes.c_float, [ctypes.c_uint16]),
                "orc_round_array": (None, [_P, _P, _I64, ctypes.c_int]),
                "orc_widen_array": (None, [_P, _P, _I64, ctypes.c_int]),
                "orc_acc_size": (_I64, []),
                "orc_acc_clear": (None, [_P]),
                "orc_acc_add": (None, [_P, ctypes.c_double]),
                "orc_acc_merge": (None, [_P, _P]),
                "orc_acc_value": (ctypes.c_double, [_P]),
                "orc_exact_sum": (ctypes.c_double, [_P, _I64]),
                "orc_plan": (ctypes.c_int, [_P, ctypes.c_int, ctypes.c_int, ctypes.c_int, _P, _P, _P, _P, _P]),
                "orc_plan_intersections": (ctypes.c_int, [_P, _P, ctypes.c_int, _I64, _I64, _P]),
                "orc_mem_model": (ctypes.c_double, [ctypes.c_double, ctypes.c_double, ctypes.c_int, ctypes.c_int]),
                "orc_mem_model_plan": (ctypes.c_int, [ctypes.c_int64, ctypes.c_int64, ctypes.c_double, ctypes.c_int,
                                                      ctypes.c_int, ctypes.c_int64, ctypes.c_int64,
                                                      ctypes.POINTER(ctypes.c_double)]),
                "orc_make_scalars": (None, [ctypes.c_float] * 5 + [_I64, _P]),
                "orc_grad_multiplier": (ctypes.c_float, [ctypes.c_double] * 3 + [_P, _P]),
                "orc_reduce": (None, [_P, ctypes.c_int, ctypes.c_int, _I64, _I64, _P]),
                "orc_stats": (None, [_P, _I64, ctypes.c_int, _P, _P]),
                "orc_reduce_stats": (None, [_P, ctypes.c_int, ctypes.c_int, _I64, _I64, _P, _P]),
                "orc_apply": (None, [_P, ctypes.c_int, _P, _P, _P, _I64, _P, ctypes.c_int, ctypes.c_float, _P]),
                "orc_zero_step": (ctypes.c_int, [_P, ctypes.c_int, ctypes.c_int, ctypes.c_int, _P, _P, _P,
                                                 _P, _P, _P, _P, ctypes.c_int] + [ctypes.c_float] * 6 +
                                  [_I64, ctypes.c_double, ctypes.c_double, ctypes.c_int, _P, _P]),
                "orc_ddp_step": (ctypes.c_int, [_P, ctypes.c_int, ctypes.c_int, _I64, _P, _P, _P, _P, ctypes.c_int]
                                 + [ctypes.c_float] * 6 + [_I64, ctypes.c_double, _P]),
                "orc_zero3_gather": (None, [_P, ctypes.c_int, _I64, _P]),
                "orc_gather_segments": (None, [_P, _P, ctypes.c_int, _P]),
                "orc_comm_volume": (ctypes.c_double, [ctypes.c_double, ctypes.c_int, ctypes.c_int, ctypes.c_int]),
                "orc_round_robin": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, _P]),
                "orc_zero3_reduce": (None, [_P, ctypes.c_int, ctypes.c_int, _I64, ctypes.c_int, _P, _P, _P]),
            }
            for name, (res, args) in sig.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be contiguous"
    return a.ctypes.data


def _ptr_array(arrs, dtype=np.uint16):
    for a in arrs:
        assert a.dtype == dtype
    return (ctypes.c_void_p * max(1, len(arrs)))(*[_ptr(a) for a in arrs])


# ---------------------------------------------------------------- conversions
def round_to_16(x: np.ndarray, dt: int) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, np.uint16)
    lib().orc_round_array(_ptr(x), _ptr(out), x.size, dt)
    return out


def widen_16(h: np.ndarray, dt: int) -> np.ndarray:
    h = np.ascontiguousarray(h, dtype=np.uint16)
    out = np.empty(h.shape, np.float32)
    lib().orc_widen_array(_ptr(h), _ptr(out), h.size, dt)
    return out


# ---------------------------------------------------------------- exact sum
class ExactAccumulator:
    """Exact sum of non-negative doubles, rounded once on read."""

    def __init__(self):
        self.buf = ctypes.create_string_buffer(lib().orc_acc_size())
        lib().orc_acc_clear(self.buf)

    def add(self, x: float):
        lib().orc_acc_add(self.buf, float(x))

    def merge(self, other: "ExactAccumulator"):
        lib().orc_acc_merge(self.buf, other.buf)

    def value(self) -> float:
        return lib().orc_acc_value(self.buf)


def exact_sum(x: np.ndarray) -> float:
    x = np.ascontiguousarray(x, dtype=np.float64)
    return lib().orc_exact_sum(_ptr(x), x.size)


# ---------------------------------------------------------------- plan / memory
def plan(numels, world_size: int, mode: int = 0):
    numels = np.ascontiguousarray(numels, dtype=np.int64)
    n = numels.size
    t_off = np.zeros(max(n, 1), np.int64)
    r_off = np.zeros(world_size, np.int64)
    r_num = np.zeros(world_size, np.int64)
    padded = ctypes.c_int64()
    pad = ctypes.c_int64()
    rc = lib().orc_plan(_ptr(numels) if n else None, n, world_size, mode, _ptr(t_off), _ptr(r_off),
                        _ptr(r_num), ctypes.byref(padded), ctypes.byref(pad))
    if rc != 0:
        raise ValueError("invalid plan arguments")
    return {"tensor_offsets": t_off[:n], "rank_offsets": r_off, "rank_numels": r_num,
            "padded_total": padded.value, "padding": pad.value}


def plan_intersections(tensor_offsets, numels, rank_offset: int, rank_numel: int):
    t = np.ascontiguousarray(tensor_offsets, dtype=np.int64)
    n = np.ascontiguousarray(numels, dtype=np.int64)
    out = np.zeros((max(len(n), 1), 4), np.int64)
    k = lib().orc_plan_intersections(_ptr(t), _ptr(n), len(n), rank_offset, rank_numel, _ptr(out))
    return out[:k]


def mem_model(psi: float, K: float, nd: int, stage: int) -> float:
    return lib().orc_mem_model(psi, K, nd, stage)


def mem_model_plan(flat_numel: int, shard_numel: int, K: float, stage: int, sets: int = 1, fp32_temp: int = 0,
                   b16_temp: int = 0):
    """Plan-exact bytes of one rank: dict of params, grads, states, temp, total (None on a bad argument)."""
    out = (ctypes.c_double * 5)()
    if lib().orc_mem_model_plan(flat_numel, shard_numel, K, stage, sets, fp32_temp, b16_temp, out) != 0:
        return None
    return dict(zip(("params", "grads", "states", "temp", "total"), list(out)))


def comm_volume(psi: float, nd: int, stage: int, ring: bool = False) -> float:
    return lib().orc_comm_volume(psi, nd, stage, int(ring))


def round_robin(n: int, ws: int) -> np.ndarray:
    out = np.zeros(max(n, 1), np.int64)
    if lib().orc_round_robin(n, ws, _ptr(out)) != 0:
        raise ValueError("invalid round-robin arguments")
    return out[:n]


# ---------------------------------------------------------------- the step
def make_scalars(lr, beta1, beta2, eps, wd, t) -> Scalars:
    s = Scalars()
    lib().orc_make_scalars(lr, beta1, beta2, eps, wd, t, ctypes.byref(s))
    return s


def grad_multiplier(sumsq: float, loss_scale: float, max_norm: float):
    norm = ctypes.c_double()
    clip = ctypes.c_double()
    k = lib().orc_grad_multiplier(sumsq, loss_scale, max_norm, ctypes.byref(norm), ctypes.byref(clip))
    return k, norm.value, clip.value


def reduce(slices, gdt: int, off: int, numel: int) -> np.ndarray:
    out = np.empty(max(numel, 0), np.uint16)
    lib().orc_reduce(_ptr_array(slices), len(slices), gdt, off, numel, _ptr(out) if numel else None)
    return out


def stats(a: np.ndarray, gdt: int, acc: ExactAccumulator | None = None):
    acc = acc or ExactAccumulator()
    ovf = ctypes.c_int32(0)
    a = np.ascontiguousarray(a, dtype=np.uint16)
    lib().orc_stats(_ptr(a), a.size, gdt, acc.buf, ctypes.byref(ovf))
    return acc, ovf.value


def reduce_stats(slices, gdt: int, off: int, numel: int, acc: ExactAccumulator) -> int:
    """Accumulate the sum of squares of the reduced slices into acc; return the overflow flag."""
    ovf = ctypes.c_int32(0)
    lib().orc_reduce_stats(_ptr_array(slices), len(slices), gdt, off, numel, acc.buf, ctypes.byref(ovf))
    return ovf.value


def apply(a, gdt, master, m, v, param_out, pdt, k, scalars: Scalars):
    """AdamW on (master, m, v) in place; param_out (uint16) receives round_P(master)."""
    n = master.size
    assert a.size == n and m.size == n and v.size == n and param_out.size == n
    lib().orc_apply(_ptr(a), gdt, _ptr(master), _ptr(m), _ptr(v), n, _ptr(param_out), pdt, k,
                    ctypes.byref(scalars))


def zero_step(slices, gdt, shards, flat_param, pdt, hyper, t, loss_scale,
              extra_sumsq=0.0, extra_overflow=0, want_grad=False):
    """One partitioned step.  shards: list of dicts with numel, grad_off, param_off,
    master, m, v (fp32 arrays, updated in place when applied).  hyper: dict with
    lr, beta1, beta2, eps, weight_decay, max_grad_norm.  Returns (Result, [reduced])."""
    n = len(shards)
    numel = np.array([s["numel"] for s in shards] or [0], np.int64)
    goff = np.array([s["grad_off"] for s in shards] or [0], np.int64)
    poff = np.array([s["param_off"] for s in shards] or [0], np.int64)
    for s in shards:
        for k in ("master", "m", "v"):
            assert s[k].dtype == np.float32 and s[k].flags["C_CONTIGUOUS"]
    ms = _ptr_array([s["master"] for s in shards], np.float32)
    mm = _ptr_array([s["m"] for s in shards], np.float32)
    vv = _ptr_array([s["v"] for s in shards], np.float32)
    grads = [np.zeros(s["numel"], np.uint16) for s in shards] if want_grad else []
    gout = _ptr_array(grads) if want_grad else None
    res = Result()
    rc = lib().orc_zero_step(_ptr_array(slices), len(slices), gdt, n, _ptr(numel), _ptr(goff), _ptr(poff),
                             ms, mm, vv, _ptr(flat_param), pdt,
                             hyper["lr"], hyper["beta1"], hyper["beta2"], hyper["eps"],
                             hyper["weight_decay"], hyper.get("max_grad_norm", 0.0),
                             t, loss_scale, extra_sumsq, int(extra_overflow), gout, ctypes.byref(res))
    if rc != 0:
        raise MemoryError("oracle step failed")
    return res, grads


def ddp_step(grads, gdt, master, m, v, param, pdt, hyper, t, loss_scale):
    res = Result()
    lib().orc_ddp_step(_ptr_array(grads), len(grads), gdt, master.size, _ptr(master), _ptr(m), _ptr(v),
                       _ptr(param), pdt, hyper["lr"], hyper["beta1"], hyper["beta2"], hyper["eps"],
                       hyper["weight_decay"], hyper.get("max_grad_norm", 0.0), t, loss_scale,
                       ctypes.byref(res))
    return res


def zero3_gather(parts) -> np.ndarray:
    part = parts[0].size
    out = np.empty(part * len(parts), np.uint16)
    lib().orc_zero3_gather(_ptr_array(parts), len(parts), part, _ptr(out))
    return out


def gather_segments(segs) -> np.ndarray:
    lens = np.array([s.size for s in segs] or [0], np.int64)
    out = np.empty(int(lens.sum()), np.uint16)
    lib().orc_gather_segments(_ptr_array(segs), _ptr(lens), len(segs), _ptr(out) if out.size else None)
    return out


def zero3_reduce(buckets, owner: int, part_numel: int, gdt: int, acc: ExactAccumulator):
    out = np.empty(part_numel, np.uint16)
    ovf = ctypes.c_int32(0)
    lib().orc_zero3_reduce(_ptr_array(buckets), len(buckets), owner, part_numel, gdt, _ptr(out),
                           acc.buf, ctypes.byref(ovf))
    return out, ovf.value
