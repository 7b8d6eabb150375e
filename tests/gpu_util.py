"""Helpers shared by the GPU parity tests: sessions, host/device copies of
fp32 and bf16 buffers, guard bands around device buffers, and the acceptance
checks (bit-exact, the fp32 sum bound, one bf16 ulp)."""
import contextlib

import numpy as np
import torch

from gradient_sync_rcc_gb300 import rcc

DEV = "cuda:0"
GUARD_BYTES = 4096
GUARD_BYTE = 0x5A


@contextlib.contextmanager
def session(R, dtype=rcc.F32, deterministic=True, device=0):
    h = rcc.register(device, R, dtype, deterministic)
    try:
        yield h
    except BaseException:
        rcc.reset(h)
        raise
    else:
        rcc.finish(h)


def tdtype(dtype):
    return torch.float32 if dtype == rcc.F32 else torch.bfloat16


def to_dev(a: np.ndarray):
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16).copy()).to(DEV).view(torch.bfloat16)
    return torch.from_numpy(a.copy()).to(DEV)


def to_host(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16).copy()
    return t.cpu().numpy().copy()


class Guarded:
    """A device buffer with GUARD_BYTES of a fixed pattern on both sides.
    `offset_elems` shifts the view off 16-byte alignment when non-zero."""

    def __init__(self, n, dtype, offset_elems=0, fill=None):
        es = 4 if dtype == torch.float32 else 2
        self.g = GUARD_BYTES // es
        self.n = n
        self.off = offset_elems
        total = self.g + offset_elems + n + self.g
        raw = torch.empty(total * es, dtype=torch.uint8, device=DEV)
        raw.fill_(GUARD_BYTE)
        self.raw = raw
        self.full = raw.view(dtype)
        self.t = self.full[self.g + offset_elems: self.g + offset_elems + n]
        if fill is not None:
            self.t.copy_(fill)

    def guards_intact(self):
        es = self.full.element_size()
        lo = self.raw[: (self.g + self.off) * es]
        hi = self.raw[(self.g + self.off + self.n) * es:]
        return bool(torch.all(lo == GUARD_BYTE)) and bool(torch.all(hi == GUARD_BYTE))


# ---------------------------------------------------------------- checks

def bits_equal(a: np.ndarray, b: np.ndarray):
    return a.shape == b.shape and a.tobytes() == b.tobytes()


def within_fp32_bound(orc, gpu, xs, op):
    """|gpu - fp64| <= R 2^-23 sum_r |x_r| (sum) and that bound / R (mean)."""
    R = len(xs)
    d = orc.reduce_f64(xs, op)
    a = orc.abs_sum_f64(xs)
    bound = R * 2.0 ** -23 * a
    if op == "mean":
        bound = bound / R
    err = np.abs(gpu.astype(np.float64) - d)
    finite = np.isfinite(d)
    return bool(np.all(err[finite] <= bound[finite])), float(np.max(err[finite] - bound[finite],
                                                                    initial=-1.0))


def _ordered(b):
    b = b.astype(np.int64)
    return np.where(b & 0x8000, -(b & 0x7FFF), b)


def bf16_ulp(v):
    """bf16 spacing at |v| (2^(e-8) for |v| in [2^(e-1), 2^e); 2^-133 minimum)."""
    _, e = np.frexp(np.abs(v))
    return np.ldexp(1.0, np.maximum(e - 8, -133))


def within_one_bf16_ulp(orc, gpu_bits, xs_bits, op):
    """Within one bf16 ulp of the fp64 result rounded once to bf16.  Where the
    fp32 accumulation error bound itself exceeds half a bf16 ulp of the result
    (heavy cancellation), that element is held to the accumulation bound plus
    one ulp instead.  Returns (ok, number of such elements)."""
    R = len(xs_bits)
    d = orc.reduce_bf16_f64(xs_bits, op)
    ref = orc.f64_to_bf16(d)
    dist = np.abs(_ordered(gpu_bits) - _ordered(ref))
    wide = [orc.bf16_to_f32(x).astype(np.float64) for x in xs_bits]
    a = np.sum(np.abs(np.stack(wide)), axis=0)
    e32 = R * 2.0 ** -24 * a
    if op == "mean":
        e32 = e32 / R + 2.0 ** -24 * np.abs(d)
    loose = e32 > 0.5 * bf16_ulp(d)
    g = orc.bf16_to_f32(gpu_bits).astype(np.float64)
    ok_tight = dist <= 1
    ok_loose = np.abs(g - d) <= e32 + bf16_ulp(np.abs(d) + e32)
    ok = np.where(loose, ok_loose | ok_tight, ok_tight)
    return bool(np.all(ok)), int(np.sum(loose))
