"""ctypes binding of the CPU oracle (liboracle_rcc.so).

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's
CPU-baseline leg are the only callers.  The CUDA library never imports this
package.  Every function takes and returns numpy arrays; the arithmetic all
happens in rcc_oracle.cpp.
"""
import ctypes as C
import os

import numpy as np

from . import build as _build

F32, BF16 = 0, 1
SUM, MEAN, MAX, MIN = 0, 1, 2, 3
OPS = {"sum": SUM, "mean": MEAN, "max": MAX, "min": MIN}

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.LIB
        if not os.path.exists(path):
            _build.build()
        _lib = C.CDLL(path)
        _declare(_lib)
    return _lib


class Stats(C.Structure):
    _fields_ = [("sum", C.c_double), ("comp", C.c_double),
                ("nonfinite", C.c_uint64), ("count", C.c_uint64)]


class Decision(C.Structure):
    _fields_ = [("skip", C.c_int), ("norm", C.c_double), ("clip_coef", C.c_float)]


class AdamWScalars(C.Structure):
    _fields_ = [("step_size", C.c_float), ("inv_bc2_sqrt", C.c_float),
                ("decay", C.c_float), ("beta1", C.c_float),
                ("one_minus_beta1", C.c_float), ("beta2", C.c_float),
                ("one_minus_beta2", C.c_float), ("eps", C.c_float)]


class Scaler(C.Structure):
    _fields_ = [("scale", C.c_double), ("growth_factor", C.c_double),
                ("backoff_factor", C.c_double), ("growth_interval", C.c_int32),
                ("growth_tracker", C.c_int32)]


_P = C.c_void_p
_PP = C.POINTER(C.c_void_p)
_SZ = C.c_size_t


def _declare(L):
    sig = {
        "orc_bf16_to_f32": (C.c_float, [C.c_uint16]),
        "orc_f32_to_bf16_rne": (C.c_uint16, [C.c_float]),
        "orc_f64_to_bf16_rne": (C.c_uint16, [C.c_double]),
        "orc_f32_to_bf16_rne_n": (None, [_P, _SZ, _P]),
        "orc_f64_to_bf16_rne_n": (None, [_P, _SZ, _P]),
        "orc_reduce_f32": (None, [C.c_int, _PP, _SZ, C.c_int, _P]),
        "orc_reduce_f64": (None, [C.c_int, _PP, _SZ, C.c_int, _P]),
        "orc_reduce_bf16": (None, [C.c_int, _PP, _SZ, C.c_int, _P]),
        "orc_reduce_bf16_f64": (None, [C.c_int, _PP, _SZ, C.c_int, _P]),
        "orc_abs_sum_f64": (None, [C.c_int, _PP, _SZ, _P]),
        "orc_all_reduce": (C.c_int, [C.c_int, C.c_int, C.c_int, _PP, _PP, _SZ]),
        "orc_reduce": (C.c_int, [C.c_int, C.c_int, C.c_int, _PP, _P, _SZ]),
        "orc_broadcast": (C.c_int, [C.c_int, C.c_int, _P, _PP, _SZ]),
        "orc_reduce_scatter": (C.c_int, [C.c_int, C.c_int, C.c_int, _PP, _PP, _SZ]),
        "orc_all_gather": (C.c_int, [C.c_int, C.c_int, _PP, _PP, _SZ]),
        "orc_all_to_all": (C.c_int, [C.c_int, C.c_int, _PP, _PP, _SZ]),
        "orc_mean_unscale": (None, [C.c_int, _PP, _SZ, C.c_float, _P]),
        "orc_stats_accumulate": (None, [C.POINTER(Stats), _P, _SZ]),
        "orc_stats_value": (C.c_double, [C.POINTER(Stats)]),
        "orc_decide": (None, [C.POINTER(Stats), C.c_double, C.POINTER(Decision)]),
        "orc_adamw_scalars_for": (None, [C.c_double] * 5 + [C.c_int64, C.POINTER(AdamWScalars)]),
        "orc_adamw_update": (None, [_P, _SZ, C.c_float, C.POINTER(AdamWScalars), _P, _P, _P]),
        "orc_scaler_update": (None, [C.POINTER(Scaler), C.c_int]),
        "orc_grad_sync_adamw_step": (None, [C.c_int, C.c_int, _P, _PP, _PP, _PP, _PP]
                                     + [C.c_double] * 6
                                     + [C.POINTER(C.c_int64), C.POINTER(Scaler),
                                        C.POINTER(Stats), C.POINTER(Decision)]),
        "orc_report_pack": (None, [C.POINTER(Stats), C.POINTER(C.c_uint32)]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args


# ---------------------------------------------------------------- helpers

def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be contiguous"
    return C.c_void_p(a.ctypes.data)


def _ptrs(arrs):
    return (C.c_void_p * len(arrs))(*[a.ctypes.data for a in arrs])


def _dt(a):
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:
        return BF16
    raise TypeError("oracle dtypes: float32 or uint16 (bf16 bit patterns)")


def _check_ranks(xs):
    xs = [np.ascontiguousarray(x) for x in xs]
    n = xs[0].size
    assert all(x.size == n and x.dtype == xs[0].dtype for x in xs)
    return xs, n


# ---------------------------------------------------------------- conversions

def bf16_to_f32(b: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, np.uint16)
    lib().orc_f32_to_bf16_rne_n(_ptr(x), x.size, _ptr(out))
    return out


def f64_to_bf16(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(x.shape, np.uint16)
    lib().orc_f64_to_bf16_rne_n(_ptr(x), x.size, _ptr(out))
    return out


# ---------------------------------------------------------------- reductions

def reduce_f32(xs, op):
    xs, n = _check_ranks([np.asarray(x, np.float32) for x in xs])
    out = np.empty(n, np.float32)
    lib().orc_reduce_f32(len(xs), _ptrs(xs), n, OPS.get(op, op), _ptr(out))
    return out


def reduce_f64(xs, op):
    xs, n = _check_ranks([np.asarray(x, np.float32) for x in xs])
    out = np.empty(n, np.float64)
    lib().orc_reduce_f64(len(xs), _ptrs(xs), n, OPS.get(op, op), _ptr(out))
    return out


def reduce_bf16(xs, op):
    xs, n = _check_ranks([np.asarray(x, np.uint16) for x in xs])
    out = np.empty(n, np.uint16)
    lib().orc_reduce_bf16(len(xs), _ptrs(xs), n, OPS.get(op, op), _ptr(out))
    return out


def reduce_bf16_f64(xs, op):
    xs, n = _check_ranks([np.asarray(x, np.uint16) for x in xs])
    out = np.empty(n, np.float64)
    lib().orc_reduce_bf16_f64(len(xs), _ptrs(xs), n, OPS.get(op, op), _ptr(out))
    return out


def abs_sum_f64(xs):
    xs, n = _check_ranks([np.asarray(x, np.float32) for x in xs])
    out = np.empty(n, np.float64)
    lib().orc_abs_sum_f64(len(xs), _ptrs(xs), n, _ptr(out))
    return out


# ---------------------------------------------------------------- collectives

def all_reduce(xs, op, out=None):
    xs, n = _check_ranks(xs)
    out = out if out is not None else [np.empty_like(xs[0]) for _ in xs]
    rc = lib().orc_all_reduce(len(xs), _dt(xs[0]), OPS.get(op, op), _ptrs(xs), _ptrs(out), n)
    assert rc == 0
    return out


def reduce(xs, op, root_out):
    xs, n = _check_ranks(xs)
    rc = lib().orc_reduce(len(xs), _dt(xs[0]), OPS.get(op, op), _ptrs(xs), _ptr(root_out), n)
    assert rc == 0
    return root_out


def broadcast(root_send, outs):
    outs_p = (C.c_void_p * len(outs))(*[None if o is None else o.ctypes.data for o in outs])
    rc = lib().orc_broadcast(len(outs), _dt(root_send), _ptr(root_send), outs_p, root_send.size)
    assert rc == 0
    return outs


def reduce_scatter(xs, op):
    xs, n = _check_ranks(xs)
    R = len(xs)
    assert n % R == 0
    out = [np.empty(n // R, xs[0].dtype) for _ in xs]
    rc = lib().orc_reduce_scatter(R, _dt(xs[0]), OPS.get(op, op), _ptrs(xs), _ptrs(out), n)
    assert rc == 0
    return out


def all_gather(xs):
    xs, n = _check_ranks(xs)
    R = len(xs)
    out = [np.empty(n * R, xs[0].dtype) for _ in xs]
    rc = lib().orc_all_gather(R, _dt(xs[0]), _ptrs(xs), _ptrs(out), n)
    assert rc == 0
    return out


def all_to_all(xs):
    xs, n = _check_ranks(xs)
    R = len(xs)
    assert n % R == 0
    out = [np.empty(n, xs[0].dtype) for _ in xs]
    rc = lib().orc_all_to_all(R, _dt(xs[0]), _ptrs(xs), _ptrs(out), n)
    assert rc == 0
    return out


# ---------------------------------------------------------------- grad sync

def mean_unscale(grads, inv_scale):
    grads, n = _check_ranks([np.asarray(g, np.float32) for g in grads])
    out = np.empty(n, np.float32)
    lib().orc_mean_unscale(len(grads), _ptrs(grads), n, C.c_float(inv_scale), _ptr(out))
    return out


def stats_new():
    return Stats(0.0, 0.0, 0, 0)


def stats_accumulate(st, g):
    g = np.ascontiguousarray(g, np.float32)
    lib().orc_stats_accumulate(C.byref(st), _ptr(g), g.size)
    return st


def stats_value(st):
    return lib().orc_stats_value(C.byref(st))


def decide(st, max_grad_norm):
    d = Decision()
    lib().orc_decide(C.byref(st), max_grad_norm, C.byref(d))
    return d


def adamw_scalars(lr, beta1, beta2, eps, weight_decay, t):
    s = AdamWScalars()
    lib().orc_adamw_scalars_for(lr, beta1, beta2, eps, weight_decay, t, C.byref(s))
    return s


def adamw_update(g, clip_coef, scalars, p, m, v):
    """In-place update of the float32 arrays p, m, v."""
    for a in (g, p, m, v):
        assert a.dtype == np.float32 and a.flags["C_CONTIGUOUS"]
    lib().orc_adamw_update(_ptr(g), g.size, C.c_float(clip_coef), C.byref(scalars),
                           _ptr(p), _ptr(m), _ptr(v))


def scaler_new(scale=65536.0, growth_factor=2.0, backoff_factor=0.5, growth_interval=2000):
    return Scaler(scale, growth_factor, backoff_factor, growth_interval, 0)


def scaler_update(sc, found_inf):
    lib().orc_scaler_update(C.byref(sc), int(bool(found_inf)))


def grad_sync_adamw_step(grads, params, exp_avg, exp_avg_sq, *, lr, beta1, beta2, eps,
                         weight_decay, max_grad_norm, step, scaler):
    """grads[p][q]: rank q's scaled grad of tensor p.  Updates params/exp_avg/
    exp_avg_sq (lists of float32 arrays) in place; returns (step, stats, decision)."""
    P = len(params)
    R = len(grads[0])
    numel = (C.c_size_t * P)(*[params[p].size for p in range(P)])
    flat = [grads[p][q] for p in range(P) for q in range(R)]
    st, d = Stats(), Decision()
    t = C.c_int64(step)
    lib().orc_grad_sync_adamw_step(R, P, numel, _ptrs(flat), _ptrs(params), _ptrs(exp_avg),
                                   _ptrs(exp_avg_sq), lr, beta1, beta2, eps, weight_decay,
                                   max_grad_norm, C.byref(t), C.byref(scaler), C.byref(st),
                                   C.byref(d))
    return t.value, st, d


def report_pack(st):
    out = (C.c_uint32 * 3)()
    lib().orc_report_pack(C.byref(st), out)
    return list(out)
