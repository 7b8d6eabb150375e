"""Seeded random cases of every collective against the oracle.

Each case draws a collective (all_reduce, reduce, broadcast, reduce_scatter,
all_gather, all_to_all_single), a rank count from 1 to 64, an element type, a
reduction op, the summation mode, per-rank lengths (ragged, zero included) and
an offset of 0..9 elements for every buffer, so the vector, staged and scalar
paths and their seams are all reached in varied combinations.  Inputs are
uniform in [-1, 1); cases with the fixed rank order, or max/min, also carry
special values (NaN, +-Inf, +-0, subnormals).  Every output buffer sits between
guard bands that must come back untouched.

Acceptance as everywhere in the suite: bit-exact where the result is fixed
(rank order, max/min, copies, sums over at most three ranks, whose tree is the
fold); otherwise the fp32 bound R 2^-23 sum|x| (mean: / R) or one bf16 ulp of the
fp64 result.  A NaN produced by a sum matches any NaN (its payload is not
specified); max/min return the canonical quiet NaN bit for bit.
"""
import numpy as np
import pytest
import torch

from gradient_sync_rcc_gb300 import rcc, synth
from gpu_util import (DEV, Guarded, bits_equal, session, tdtype, to_dev, to_host,
                      within_fp32_bound, within_one_bf16_ulp)

pytestmark = pytest.mark.gpu

NCASES = 600
KINDS = ["all_reduce", "reduce", "broadcast", "reduce_scatter", "all_gather", "all_to_all"]
RANKS = [1, 2, 3, 4, 5, 6, 7, 8, 9, 12, 16, 33, 64]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gradient_sync_rcc_gb300 import build
    build.build()
    assert torch.cuda.is_available()


def _specials(dtype):
    f = np.array([np.nan, np.inf, -np.inf, 0.0, -0.0, 1e-40, -3e-39, 3.0e38], np.float32)
    if dtype == rcc.F32:
        return f
    return synth_bf16(f)


def synth_bf16(f):
    """bf16 bits of float32 values (round to nearest even through torch)."""
    return torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _draw(g, dtype, n, key, specials):
    if dtype == rcc.F32:
        x = synth.uniform_pm1(n, *key)
    else:
        x = synth.bf16_uniform_pm1(n, *key)
    if specials and n > 0:
        sp = _specials(dtype)
        k = int(g.integers(1, min(n, 6) + 1))
        x[g.integers(0, n, k)] = sp[g.integers(0, sp.size, k)]
    return x


def _is_nan(a, dtype):
    if dtype == rcc.F32:
        return np.isnan(a)
    b = a.astype(np.uint32)
    return ((b & 0x7F80) == 0x7F80) & ((b & 0x7F) != 0)


def _same(got, want, dtype, nan_any):
    if not nan_any:
        return bits_equal(got, want)
    ng, nw = _is_nan(got, dtype), _is_nan(want, dtype)
    return bool(np.array_equal(ng, nw)) and got[~nw].tobytes() == want[~nw].tobytes()


def _reduced_ok(orc, got, xs, op, dtype, exact, nan_any):
    """got (one output) against the oracle's reduction of the columns xs."""
    want = orc.reduce_f32(xs, op) if dtype == rcc.F32 else orc.reduce_bf16(xs, op)
    if exact:
        return _same(got, want, dtype, nan_any)
    if dtype == rcc.F32:
        return within_fp32_bound(orc, got, xs, op)[0]
    return within_one_bf16_ulp(orc, got, xs, op)[0]


def _case(i):
    g = synth.rng(0xCA5E, i)
    kind = KINDS[int(g.integers(len(KINDS)))]
    R = int(RANKS[int(g.integers(len(RANKS)))])
    dtype = rcc.F32 if g.random() < 0.6 else rcc.BF16
    op = ["sum", "mean", "max", "min"][int(g.integers(4))]
    det = bool(g.random() < 0.5)
    cap = max(8, 4096 // R)
    if kind in ("reduce_scatter", "all_to_all"):
        shard = int(g.integers(0, max(2, cap // R) + 1))
        n_in = R * shard
    elif kind == "broadcast":
        # the sender is the rank with a non-NULL buffer, and an empty tensor may
        # have none, so broadcasts carry at least one element
        n_in = int(g.integers(1, cap + 1))
    else:
        n_in = int(g.integers(0, cap + 1))
    specials = (det or op in ("max", "min")) and g.random() < 0.4
    return g, kind, R, dtype, op, det, n_in, specials


@pytest.mark.parametrize("i", range(NCASES))
def test_random_collective(orc, i):
    g, kind, R, dtype, op, det, n, specials = _case(i)
    td = tdtype(dtype)
    xs = [_draw(g, dtype, n, (0xCA5F, i, r), specials) for r in range(R)]
    offs = [int(v) for v in g.integers(0, 10, 2 * R)]
    ins = [Guarded(n, td, offset_elems=offs[r], fill=to_dev(xs[r]) if n else None)
           for r in range(R)]
    exact = det or op in ("max", "min") or R <= 3
    nan_any = op in ("sum", "mean")
    ok = True
    with session(R, dtype, det) as h:
        if kind == "all_reduce":
            outs = [Guarded(n, td, offset_elems=offs[R + r]) for r in range(R)]
            rcc.all_reduce(h, [x.t for x in ins], [o.t for o in outs], op)
        elif kind == "reduce":
            root = int(g.integers(R))
            outs = [Guarded(n, td, offset_elems=offs[R])]
            rcc.reduce(h, [x.t for x in ins], outs[0].t, root=root, op=op)
        elif kind == "broadcast":
            root = int(g.integers(R))
            outs = [Guarded(n, td, offset_elems=offs[R + r]) for r in range(R)]
            rcc.broadcast(h, ins[root].t, [o.t for o in outs], root=root)
        elif kind == "reduce_scatter":
            outs = [Guarded(n // R, td, offset_elems=offs[R + r]) for r in range(R)]
            rcc.reduce_scatter(h, [x.t for x in ins], [o.t for o in outs], op)
        elif kind == "all_gather":
            outs = [Guarded(n * R, td, offset_elems=offs[R + r]) for r in range(R)]
            rcc.all_gather(h, [x.t for x in ins], [o.t for o in outs])
        else:
            outs = [Guarded(n, td, offset_elems=offs[R + r]) for r in range(R)]
            rcc.all_to_all_single(h, [x.t for x in ins], [o.t for o in outs])
        torch.cuda.synchronize()
    got = [to_host(o.t) for o in outs]
    where = (kind, R, dtype, op, det, n, specials)
    for o in outs + ins:
        assert o.guards_intact(), where
    for x, gx in zip(xs, ins):                       # inputs are never written
        assert bits_equal(to_host(gx.t), x), where
    if kind == "all_reduce":
        for r in range(R):
            assert bits_equal(got[r], got[0]), where
        ok = _reduced_ok(orc, got[0], xs, op, dtype, exact, nan_any)
    elif kind == "reduce":
        ok = _reduced_ok(orc, got[0], xs, op, dtype, exact, nan_any)
    elif kind == "broadcast":
        ok = all(bits_equal(gr, xs[root]) for gr in got)
    elif kind == "reduce_scatter":
        m = n // R
        ok = all(_reduced_ok(orc, got[r], [x[r * m:(r + 1) * m] for x in xs], op, dtype, exact,
                             nan_any) for r in range(R))
    elif kind == "all_gather":
        ok = all(bits_equal(gr, np.concatenate(xs) if n else np.zeros(0, xs[0].dtype))
                 for gr in got)
    else:
        want = orc.all_to_all(xs) if n else [np.zeros(0, xs[0].dtype) for _ in xs]
        ok = all(bits_equal(a, b) for a, b in zip(got, want))
    assert ok, where
