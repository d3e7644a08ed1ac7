"""GB300-native ZeRO-DP partitioned mixed-precision optimizer step.

A thin ctypes binding of ``libzero_gb300.so`` (C ABI in ``include/zero.h``):
the functions here have the C names and only marshal arguments -- every step
of the path runs in the library's CUDA kernels.  Pointers may be given as
torch tensors (their ``data_ptr()``) or as integers.  A nonzero status raises
``ZeroError`` with the library's message.

Importing this package loads the compiled library; if it has not been built
(``python zero_dp_partitioned_gb300/build.py``) the import fails -- there is
no fallback.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libzero_gb300.so")

ZERO_OK, ZERO_EINVAL, ZERO_EALIGN, ZERO_EWORKSPACE, ZERO_ECUDA, ZERO_ELIMIT = 0, -1, -2, -3, -4, -5
ZERO_F16, ZERO_BF16 = 1, 2
ZERO_PLAN_PADDED, ZERO_PLAN_UNPADDED = 0, 1
ZERO_MAX_SLICES = ZERO_MAX_SHARDS = 64


class ZeroError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"{msg} (status {code})")
        self.code = code


class zero_hyper(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_float), ("beta1", ctypes.c_float), ("beta2", ctypes.c_float),
                ("eps", ctypes.c_float), ("weight_decay", ctypes.c_float), ("max_grad_norm", ctypes.c_float),
                ("step", ctypes.c_int64)]


class zero_shard(ctypes.Structure):
    _fields_ = [("numel", ctypes.c_int64), ("grad_offset", ctypes.c_int64), ("param_offset", ctypes.c_int64),
                ("master_in", ctypes.c_void_p), ("m_in", ctypes.c_void_p), ("v_in", ctypes.c_void_p),
                ("master_out", ctypes.c_void_p), ("m_out", ctypes.c_void_p), ("v_out", ctypes.c_void_p),
                ("grad_shard", ctypes.c_void_p)]


class zero_stats(ctypes.Structure):
    _fields_ = [("sumsq", ctypes.c_double), ("overflow", ctypes.c_int32), ("reserved", ctypes.c_int32)]


class zero_chain(ctypes.Structure):
    _fields_ = [("cur", ctypes.c_int32), ("reserved", ctypes.c_int32), ("step", ctypes.c_int64),
                ("loss_scale", ctypes.c_double), ("applied", ctypes.c_int64), ("skipped", ctypes.c_int64),
                ("failed", ctypes.c_int64), ("min_loss_scale", ctypes.c_double)]

    def as_dict(self):
        return {k: getattr(self, k) for k, _ in self._fields_ if not k.startswith("reserved")}


class zero_result(ctypes.Structure):
    _fields_ = [("overflow", ctypes.c_int32), ("applied", ctypes.c_int32), ("path", ctypes.c_int32),
                ("status", ctypes.c_int32), ("sumsq", ctypes.c_double), ("grad_norm", ctypes.c_double),
                ("clip_coef", ctypes.c_double), ("grad_mult", ctypes.c_float), ("reserved", ctypes.c_float)]

    def as_dict(self):
        return {k: getattr(self, k) for k, _ in self._fields_ if not k.startswith("reserved")}


assert ctypes.sizeof(zero_hyper) == 32 and ctypes.sizeof(zero_shard) == 80
assert ctypes.sizeof(zero_stats) == 16 and ctypes.sizeof(zero_result) == 48 and ctypes.sizeof(zero_chain) == 56

_P, _I64, _I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
_SIGS = {
    "zero_plan": (_I, [_P, _I, _I, _I, _P, _P, _P, _P, _P]),
    "zero_plan_intersections": (_I, [_P, _P, _I, _I64, _I64, _P]),
    "zero_mem_model": (_I, [ctypes.c_double, ctypes.c_double, _I, _I, _P]),
    "zero_mem_model_plan": (_I, [_I64, _I64, ctypes.c_double, _I, _I, _I64, _I64, _P]),
    "zero_comm_volume": (_I, [ctypes.c_double, _I, _I, _I, _P]),
    "zero_plan_round_robin": (_I, [_I, _I, _P]),
    "zero_workspace_bytes": (ctypes.c_size_t, []),
    "zero_shard_step": (_I, [_P, _I, _I, _P, _I, _P, _I, _P, ctypes.c_float, ctypes.c_double, _I, _P,
                             ctypes.c_size_t, _P, _P]),
    "zero_shard_init": (_I, [_P, _I, _P, _I, _P]),
    "zero_shard_reduce": (_I, [_P, _I, _I, _P, _I, _I, _P, _P, ctypes.c_size_t, _P]),
    "zero_shard_apply": (_I, [_P, _I, _I, _P, _I, _P, ctypes.c_float, _P, ctypes.c_double, _I, _P, ctypes.c_size_t,
                              _P, _P]),
    "zero3_gather_layer": (_I, [_P, _I, _I64, _I, _P, _P]),
    "zero3_gather_segments": (_I, [_P, _P, _I, _I, _P, _P]),
    "zero3_gather_bulk": (_I, [_P, _P, _I, _I, _P, _I, _P, _P]),
    "zero3_reduce_bucket": (_I, [_P, _I, _I, _I64, _I, _P, _I, _P, _P, ctypes.c_size_t, _P]),
    "zero_shard_step_noalloc": (_I, [_P, _I, _I, _P, _I, _P, _I, _P, ctypes.c_float, ctypes.c_double, _I, _P, _P]),
    "zero_adam_scalar_table": (_I, [_P, _I64, _I64, _P]),
    "zero_shard_step_chained": (_I, [_P, _I, _I, _P, _I, _P, _I, _P, _P, _I64, _I64, _P, ctypes.c_double, _I, _P,
                                     ctypes.c_size_t, _P, _P]),
    "zero_shard_apply_chained": (_I, [_P, _I, _I, _P, _I, _P, _P, _I64, _I64, _P, _P, ctypes.c_double, _I, _P,
                                      ctypes.c_size_t, _P, _P]),
    "zero_shard_step_partial": (_I, [_P, _I, _I, _P, _I, _P, _I, _P, ctypes.c_float, _P, _I64, _I64, _P, _I, _P, _P,
                                     ctypes.c_size_t, _P]),
    "zero_shard_step_commit": (_I, [_P, _I, _P, _I, ctypes.c_float, _I64, _I64, _P, _P, ctypes.c_double, _I, _P, _P]),
    "zero_shard_step_host": (_I, [_P, _I, _I, _P, _I, _P, _I, _P, _P, ctypes.c_float, ctypes.c_double, _I, _P,
                                  ctypes.c_size_t, _P, ctypes.c_size_t, _P, _P]),
    "zero_last_error": (ctypes.c_char_p, []),
}
# every symbol include/zero.h declares
EXPORTS = tuple(_SIGS)


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with `python zero_dp_partitioned_gb300/build.py`")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


lib = _load()


def _ptr(x):
    if x is None:
        return None
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    return int(x)


def _stream(stream):
    if stream is not None:
        return _ptr(stream.cuda_stream if hasattr(stream, "cuda_stream") else stream)
    import torch
    return torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else None


def _check(rc):
    if rc < 0:
        raise ZeroError(rc, lib.zero_last_error().decode())
    return rc


def _ptrs(xs):
    return (ctypes.c_void_p * max(1, len(xs)))(*[_ptr(x) for x in xs])


# ------------------------------------------------------------------ host-only calls
def zero_plan(numels, world_size, mode=ZERO_PLAN_PADDED):
    n = len(numels)
    arr = (ctypes.c_int64 * max(1, n))(*numels)
    t_off = (ctypes.c_int64 * max(1, n))()
    r_off = (ctypes.c_int64 * world_size)()
    r_num = (ctypes.c_int64 * world_size)()
    padded, pad = ctypes.c_int64(), ctypes.c_int64()
    _check(lib.zero_plan(arr, n, world_size, mode, t_off, r_off, r_num, ctypes.byref(padded), ctypes.byref(pad)))
    return {"tensor_offsets": list(t_off)[:n], "rank_offsets": list(r_off), "rank_numels": list(r_num),
            "padded_total": padded.value, "padding": pad.value}


def zero_plan_intersections(tensor_offsets, numels, rank_offset, rank_numel):
    n = len(numels)
    t = (ctypes.c_int64 * max(1, n))(*tensor_offsets)
    m = (ctypes.c_int64 * max(1, n))(*numels)
    out = (ctypes.c_int64 * (4 * max(1, n)))()
    k = _check(lib.zero_plan_intersections(t, m, n, rank_offset, rank_numel, out))
    return [tuple(out[4 * i:4 * i + 4]) for i in range(k)]


def zero_mem_model(psi, K, n_d, stage):
    b = ctypes.c_double()
    _check(lib.zero_mem_model(psi, K, n_d, stage, ctypes.byref(b)))
    return b.value


def zero_mem_model_plan(flat_numel, shard_numel, K, stage, state_sets=1, fp32_temp_numel=0, b16_temp_numel=0):
    """Plan-exact bytes of one rank: dict of params, grads, states, temp, total."""
    out = (ctypes.c_double * 5)()
    _check(lib.zero_mem_model_plan(flat_numel, shard_numel, K, stage, state_sets, fp32_temp_numel, b16_temp_numel,
                                   out))
    return dict(zip(("params", "grads", "states", "temp", "total"), list(out)))


def zero_comm_volume(psi, n_d, stage, ring=False):
    v = ctypes.c_double()
    _check(lib.zero_comm_volume(psi, n_d, stage, int(ring), ctypes.byref(v)))
    return v.value


def zero_plan_round_robin(n_tensors, world_size):
    out = (ctypes.c_int64 * max(1, n_tensors))()
    _check(lib.zero_plan_round_robin(n_tensors, world_size, out))
    return list(out)[:n_tensors]


def zero_workspace_bytes():
    return lib.zero_workspace_bytes()


# ------------------------------------------------------------------ device calls
def shard(numel, grad_offset, param_offset, master_in, m_in, v_in, master_out=None, m_out=None, v_out=None,
          grad_shard=None) -> zero_shard:
    """A zero_shard; *_out default to *_in (in-place)."""
    return zero_shard(numel, grad_offset, param_offset, _ptr(master_in), _ptr(m_in), _ptr(v_in),
                      _ptr(master_out if master_out is not None else master_in),
                      _ptr(m_out if m_out is not None else m_in),
                      _ptr(v_out if v_out is not None else v_in), _ptr(grad_shard))


def hyper(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01, max_grad_norm=0.0, step=1) -> zero_hyper:
    return zero_hyper(lr, beta1, beta2, eps, weight_decay, max_grad_norm, step)


def zero_shard_step(grad_slices, grad_dtype, shards, flat_param, param_dtype, hyper, loss_scale,
                    extra_sumsq, extra_overflow, workspace, workspace_bytes, result, stream=None):
    sh = (zero_shard * max(1, len(shards)))(*shards)
    _check(lib.zero_shard_step(_ptrs(grad_slices), len(grad_slices), grad_dtype, sh, len(shards), _ptr(flat_param),
                               param_dtype, ctypes.byref(hyper), loss_scale, extra_sumsq, int(extra_overflow),
                               _ptr(workspace), workspace_bytes, _ptr(result), _stream(stream)))


def zero_shard_step_host(host_grad_slices, grad_dtype, shards, flat_param, param_dtype, host_param, hyper,
                         loss_scale, extra_sumsq, extra_overflow, staging, staging_bytes, workspace, workspace_bytes,
                         result, stream=None):
    """zero_shard_step with the gradients in page-locked host memory and the
    updated parameters copied back to page-locked host memory (host_param,
    laid out as flat_param; None = no copy down): the library copies the
    slices up chunk by chunk into the device ring `staging` while the chunks
    already up are reduced and updated."""
    sh = (zero_shard * max(1, len(shards)))(*shards)
    _check(lib.zero_shard_step_host(_ptrs(host_grad_slices), len(host_grad_slices), grad_dtype, sh, len(shards),
                                    _ptr(flat_param), param_dtype, _ptr(host_param), ctypes.byref(hyper), loss_scale,
                                    extra_sumsq, int(extra_overflow), _ptr(staging), staging_bytes, _ptr(workspace),
                                    workspace_bytes, _ptr(result), _stream(stream)))


def zero_shard_step_noalloc(grad_slices, grad_dtype, shards, flat_param, param_dtype, hyper, loss_scale,
                            extra_sumsq, extra_overflow, result, stream=None):
    """zero_shard_step without caller scratch (for callers that cannot allocate
    device memory): the library's built-in scratch array stands in for the
    workspace and the two-pass path's reduced-gradient buffers."""
    sh = (zero_shard * max(1, len(shards)))(*shards)
    _check(lib.zero_shard_step_noalloc(_ptrs(grad_slices), len(grad_slices), grad_dtype, sh, len(shards),
                                       _ptr(flat_param), param_dtype, ctypes.byref(hyper), loss_scale, extra_sumsq,
                                       int(extra_overflow), _ptr(result), _stream(stream)))


def zero_shard_init(shards, flat_param, param_dtype, stream=None):
    """Before the first step: every shard's master_in = fp32(its 16-bit
    parameters in flat_param), m_in = v_in = 0."""
    sh = (zero_shard * max(1, len(shards)))(*shards)
    _check(lib.zero_shard_init(sh, len(shards), _ptr(flat_param), param_dtype, _stream(stream)))


def zero_shard_reduce(grad_slices, grad_dtype, shards, accumulate, stats, workspace, workspace_bytes, stream=None):
    sh = (zero_shard * max(1, len(shards)))(*shards)
    _check(lib.zero_shard_reduce(_ptrs(grad_slices), len(grad_slices), grad_dtype, sh, len(shards), int(accumulate),
                                 _ptr(stats), _ptr(workspace), workspace_bytes, _stream(stream)))


def zero_shard_apply(shards, grad_dtype, flat_param, param_dtype, hyper, loss_scale, stats, extra_sumsq,
                     extra_overflow, workspace, workspace_bytes, result, stream=None):
    sh = (zero_shard * max(1, len(shards)))(*shards)
    _check(lib.zero_shard_apply(sh, len(shards), grad_dtype, _ptr(flat_param), param_dtype, ctypes.byref(hyper),
                                loss_scale, _ptr(stats), extra_sumsq, int(extra_overflow), _ptr(workspace),
                                workspace_bytes, _ptr(result), _stream(stream)))


def zero3_gather_layer(part_ptrs, unit_numel, dtype, layer_out, stream=None):
    _check(lib.zero3_gather_layer(_ptrs(part_ptrs), len(part_ptrs), unit_numel, dtype, _ptr(layer_out),
                                  _stream(stream)))


def zero3_gather_segments(segment_ptrs, segment_numels, dtype, layer_out, stream=None):
    n = len(segment_ptrs)
    lens = (ctypes.c_int64 * max(1, n))(*segment_numels)
    _check(lib.zero3_gather_segments(_ptrs(segment_ptrs), lens, n, dtype, _ptr(layer_out), _stream(stream)))


def zero3_gather_bulk(segment_ptrs, segment_numels, dtype, layer_out, n_ctas, status, stream=None):
    """The gather on at most n_ctas CTAs (0 = one per SM), moved by the TMA unit
    when every segment agrees with its slot modulo 16 bytes; status: device
    int32 (zero-filled by the caller), bit 0 set if a wait ran out."""
    n = len(segment_ptrs)
    lens = (ctypes.c_int64 * max(1, n))(*segment_numels)
    _check(lib.zero3_gather_bulk(_ptrs(segment_ptrs), lens, n, dtype, _ptr(layer_out), int(n_ctas), _ptr(status),
                                 _stream(stream)))


def zero3_reduce_bucket(bucket_ptrs, owner, unit_numel, grad_dtype, grad_part, accumulate, stats, workspace,
                        workspace_bytes, stream=None):
    _check(lib.zero3_reduce_bucket(_ptrs(bucket_ptrs), len(bucket_ptrs), owner, unit_numel, grad_dtype,
                                   _ptr(grad_part), int(accumulate), _ptr(stats), _ptr(workspace), workspace_bytes,
                                   _stream(stream)))


def zero_adam_scalar_table(hyper, t0, n):
    """The step-dependent AdamW scalars (lr / (1 - b1^t), 1 / sqrt(1 - b2^t)) for
    t = t0 .. t0 + n - 1, as a host float32 array of 2 n values."""
    import numpy as np
    out = np.zeros(2 * int(n), np.float32)
    _check(lib.zero_adam_scalar_table(ctypes.byref(hyper), int(t0), int(n), out.ctypes.data))
    return out


def chain(step=1, loss_scale=1.0, cur=0, min_loss_scale=0.0):
    """A zero_chain to copy to the device (56 bytes) as the start of a chain;
    min_loss_scale <= 0 leaves the library's floor of 2^-126."""
    return zero_chain(cur, 0, step, loss_scale, 0, 0, 0, min_loss_scale)


def read_chain(t) -> zero_chain:
    """A zero_chain from a 56-byte tensor (device or host)."""
    b = bytes(t.detach().cpu().view(-1).numpy().tobytes()) if hasattr(t, "detach") else bytes(t)
    return zero_chain.from_buffer_copy(b[:ctypes.sizeof(zero_chain)])


def zero_shard_step_chained(grad_slices, grad_dtype, shards, flat_param, param_dtype, hyper, scalar_table, table_t0,
                            n_table, chain_dev, extra_sumsq, extra_overflow, workspace, workspace_bytes, result,
                            stream=None):
    """One step with its bookkeeping (t, S, the state set in use) in the device
    zero_chain chain_dev; scalar_table: device float32, 2 n_table values."""
    sh = (zero_shard * max(1, len(shards)))(*shards)
    _check(lib.zero_shard_step_chained(_ptrs(grad_slices), len(grad_slices), grad_dtype, sh, len(shards),
                                       _ptr(flat_param), param_dtype, ctypes.byref(hyper), _ptr(scalar_table),
                                       int(table_t0), int(n_table), _ptr(chain_dev), extra_sumsq,
                                       int(extra_overflow), _ptr(workspace), workspace_bytes, _ptr(result),
                                       _stream(stream)))


def zero_shard_apply_chained(shards, grad_dtype, flat_param, param_dtype, hyper, scalar_table, table_t0, n_table,
                             chain_dev, stats, extra_sumsq, extra_overflow, workspace, workspace_bytes, result,
                             stream=None):
    """The apply pass with t, S and the state set in use read from the device
    zero_chain chain_dev, which it then updates; shards may update in place."""
    sh = (zero_shard * max(1, len(shards)))(*shards)
    _check(lib.zero_shard_apply_chained(sh, len(shards), grad_dtype, _ptr(flat_param), param_dtype,
                                        ctypes.byref(hyper), _ptr(scalar_table), int(table_t0), int(n_table),
                                        _ptr(chain_dev), _ptr(stats), extra_sumsq, int(extra_overflow),
                                        _ptr(workspace), workspace_bytes, _ptr(result), _stream(stream)))


def zero_shard_step_partial(grad_slices, grad_dtype, shards, flat_param, param_dtype, hyper, loss_scale, accumulate,
                            stats, workspace, workspace_bytes, scalar_table=None, table_t0=1, n_table=0,
                            chain_dev=None, stream=None):
    """A fused pass over some shards of a step, adding their statistics to
    stats; the step is decided later by zero_shard_step_commit.  With
    chain_dev, t, S and the state set in use come from the device chain."""
    sh = (zero_shard * max(1, len(shards)))(*shards)
    _check(lib.zero_shard_step_partial(_ptrs(grad_slices), len(grad_slices), grad_dtype, sh, len(shards),
                                       _ptr(flat_param), param_dtype, ctypes.byref(hyper), loss_scale,
                                       _ptr(scalar_table), int(table_t0), int(n_table), _ptr(chain_dev),
                                       int(accumulate), _ptr(stats), _ptr(workspace), workspace_bytes,
                                       _stream(stream)))


def zero_shard_step_commit(shards, flat_param, param_dtype, loss_scale, stats, extra_sumsq, extra_overflow, result,
                           table_t0=1, n_table=0, chain_dev=None, stream=None):
    """The decision of a step made of partial fused passes: the result from
    their statistics, the parameters restored on a skip, the chain updated."""
    sh = (zero_shard * max(1, len(shards)))(*shards)
    _check(lib.zero_shard_step_commit(sh, len(shards), _ptr(flat_param), param_dtype, loss_scale, int(table_t0),
                                      int(n_table), _ptr(chain_dev), _ptr(stats), extra_sumsq, int(extra_overflow),
                                      _ptr(result), _stream(stream)))


def read_result(t) -> zero_result:
    """A zero_result from a 48-byte tensor (device or host)."""
    b = bytes(t.detach().cpu().view(-1).numpy().tobytes()) if hasattr(t, "detach") else bytes(t)
    return zero_result.from_buffer_copy(b[:ctypes.sizeof(zero_result)])


def read_stats(t) -> zero_stats:
    b = bytes(t.detach().cpu().view(-1).numpy().tobytes())
    return zero_stats.from_buffer_copy(b[:ctypes.sizeof(zero_stats)])
