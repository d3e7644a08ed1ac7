"""Pins the oracle's IEEE 754 conversions (fp32 <-> fp16 / bf16, round to
nearest even) against numpy's float16 and torch's bfloat16 conversions, over
every one of the 2^32 binary32 bit patterns and every 16-bit pattern.
Mixed precision stores parameters and gradients in 16 bits (ZeRO paper,
Chinese translation, 3.1)."""
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

CHUNK = 1 << 24


def _check_chunk(orc, dt, c):
    u = np.arange(c * CHUNK, (c + 1) * CHUNK, dtype=np.uint64).astype(np.uint32)
    x = u.view(np.float32)
    mine = orc.round_to_16(x, dt)
    if dt == orc.F16:
        ref = torch.from_numpy(x.copy()).to(torch.float16).view(torch.int16).numpy().view(np.uint16)
        nan_mine = ((mine & 0x7C00) == 0x7C00) & ((mine & 0x03FF) != 0)
        nan_ref = ((ref & 0x7C00) == 0x7C00) & ((ref & 0x03FF) != 0)
        # second, independent reference on a strided subset: numpy's float16 cast
        sub = x[::251]
        with np.errstate(over="ignore", invalid="ignore"):
            ref_np = sub.astype(np.float16).view(np.uint16)
        m = ~np.isnan(sub)
        assert np.array_equal(mine[::251][m], ref_np[m]), f"numpy fp16 mismatch in chunk {c}"
    else:
        ref = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        nan_mine = ((mine & 0x7F80) == 0x7F80) & ((mine & 0x007F) != 0)
        nan_ref = ((ref & 0x7F80) == 0x7F80) & ((ref & 0x007F) != 0)
    assert np.array_equal(nan_mine, nan_ref), f"NaN mismatch in chunk {c}"
    ok = nan_mine | (mine == ref)
    if not ok.all():
        i = int(np.flatnonzero(~ok)[0])
        raise AssertionError(f"dt={dt} x=0x{u[i]:08x} mine=0x{mine[i]:04x} ref=0x{ref[i]:04x}")
    return True


def _exhaustive(orc, dt):
    with ThreadPoolExecutor(8) as ex:
        assert all(ex.map(lambda c: _check_chunk(orc, dt, c), range((1 << 32) // CHUNK)))


def test_f32_to_f16_all_bit_patterns(orc):
    _exhaustive(orc, orc.F16)


def test_f32_to_bf16_all_bit_patterns(orc):
    _exhaustive(orc, orc.BF16)


def test_widening_all_16bit_patterns(orc):
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    f16 = orc.widen_16(h, orc.F16)
    ref16 = h.view(np.float16).astype(np.float32)
    assert np.array_equal(np.isnan(f16), np.isnan(ref16))
    m = ~np.isnan(ref16)
    assert np.array_equal(f16[m].view(np.uint32), ref16[m].view(np.uint32))
    bf = orc.widen_16(h, orc.BF16)
    refbf = torch.from_numpy(h.view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    assert np.array_equal(np.isnan(bf), np.isnan(refbf))
    m = ~np.isnan(refbf)
    assert np.array_equal(bf[m].view(np.uint32), refbf[m].view(np.uint32))


def test_round_trip_is_identity(orc):
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    for dt in (orc.F16, orc.BF16):
        w = orc.widen_16(h, dt)
        back = orc.round_to_16(w, dt)
        m = ~np.isnan(w)
        assert np.array_equal(back[m], h[m])
