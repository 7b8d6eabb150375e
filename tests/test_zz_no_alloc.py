"""rcc_grad_stats_noalloc: gradient statistics for callers that cannot allocate.

Some callers cannot allocate device memory at all: code enqueued while a
stream is being captured into a CUDA graph with allocation forbidden, or a
process whose device memory belongs to another runtime or a fixed pool.
rcc_grad_sync_adamw allocates session scratch on first use; this entry point
keeps its statistics rows in a static device array instead and writes only
into buffers the caller passes.

Through the C ABI, the report (sum of g^2, non-finite count) and the mean
gradient it produces must match rcc_grad_sync_adamw's for the same gradients,
within the tolerance the gradient-sync tests use (sum of squares 1e-12
relative; count and mean gradient exact), on two calls in a row -- one with
<= 1024 rows, one that needs the fan-in-1024 combine and carries a NaN.  Both
are also checked against the CPU oracle, and further cases cover 1, 3, 5, 8
and 12 ranks, views that allow only scalar accesses, and no stored mean.
"""
import ctypes as C

import numpy as np
import pytest
import torch

from gradient_sync_rcc_gb300 import rcc, synth
from gpu_util import DEV, session

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gradient_sync_rcc_gb300 import build
    build.build()
    assert torch.cuda.is_available()


def _reference(grads, scale):
    """Report and mean gradient from rcc_grad_sync_adamw (the existing entry point)."""
    n = grads[0].numel()
    mean = torch.empty(n, device=DEV)
    t = dict(grads=grads, params=[torch.zeros(n, device=DEV)], exp_avg=[torch.zeros(n, device=DEV)],
             exp_avg_sq=[torch.zeros(n, device=DEV)], mean_grad=mean)
    with session(len(grads)) as h:
        rep = rcc.grad_sync_adamw(h, rcc.ParamSets([t]), rcc.adamw_cfg(replicas=1),
                                  rcc.optim_state(scale=scale))
        torch.cuda.synchronize()
    return rep, mean


def _mean_matches(got, want):
    """Bit for bit, except that a NaN matches any NaN: the payload of a NaN
    produced by a sum is unspecified (only NaN-ness is compared)."""
    g = got.cpu().numpy()
    nan = np.isnan(want)
    return bool(np.array_equal(np.isnan(g), nan)) and \
        g[~nan].tobytes() == want[~nan].tobytes()


def _decode(report):
    w = report.cpu().numpy().view(np.uint32)
    return float(w[:2].copy().view(np.float64)[0]), int(w[2])


def test_noalloc_matches_grad_sync_on_two_calls(orc):
    R, scale = 4, 65536.0
    cases = [(3_000_001, None), (9_000_003, 12345)]      # 367 rows; 1099 rows + a NaN
    for call, (n, nan_at) in enumerate(cases):
        grads = [synth.gpu_draw("normal:1e-3", n, torch.float32, (40, call, r), DEV) * scale
                 for r in range(R)]
        if nan_at is not None:
            grads[1][nan_at] = float("nan")
        rep, mean_ref = _reference(grads, scale)
        report = torch.full((4,), -1, dtype=torch.int32, device=DEV)
        mean = torch.empty(n, device=DEV)
        rcc.grad_stats_noalloc(grads, scale, report, mean_grad=mean)
        torch.cuda.synchronize()
        sum_sq, nonfinite = _decode(report)
        assert abs(sum_sq - rep.sum_sq) <= 1e-12 * rep.sum_sq, (call, sum_sq, rep.sum_sq)
        assert nonfinite == rep.nonfinite == (0 if nan_at is None else 1)
        assert torch.equal(mean.view(torch.int32), mean_ref.view(torch.int32))
        # and both against the oracle
        want_mean = orc.mean_unscale([g.cpu().numpy() for g in grads], np.float32(1.0 / scale))
        st = orc.stats_accumulate(orc.stats_new(), want_mean)
        assert _mean_matches(mean, want_mean)
        assert abs(sum_sq - orc.stats_value(st)) <= 1e-12 * orc.stats_value(st)
        assert report.cpu().numpy().view(np.uint32)[2] == orc.report_pack(st)[2]


def _shifted(n, off, fill=None):
    """A float32 view `off` elements into a fresh allocation (off = 1: 4 bytes
    past a 256-byte boundary, so only the scalar path may touch it)."""
    base = torch.empty(n + off, device=DEV)
    v = base[off:off + n]
    if fill is not None:
        v.copy_(fill)
    return v


# (R, numel, view offset in elements, mean gradient stored, mean-gradient offset)
CASES = [
    (1, 1000, 0, True, 0),              # one rank: the mean is the unscaled gradient
    (3, 8192 * 1024 + 13, 1, False, 0),  # 1025 rows (one combine), misaligned: scalar path
    (4, 3_000_001, 0, True, 0),         # 16-byte vectors with a ragged tail
    (5, 20_000, 0, True, 1),            # aligned gradients, misaligned mean: scalar path
    (8, 65_541, 0, True, 0),            # compile-time eight ranks
    (12, 100_003, 0, True, 0),          # runtime rank count, vectors
    (12, 100_003, 1, True, 1),          # runtime rank count, scalar path
]


@pytest.mark.parametrize("R,n,off,store_mean,mean_off", CASES,
                         ids=["R%d-n%d-off%d-%s" % (c[0], c[1], c[2], "mean" if c[3] else "nomean")
                              for c in CASES])
def test_noalloc_against_oracle(orc, R, n, off, store_mean, mean_off):
    """Mean gradient bit for bit against the oracle's mean + unscale, the sum
    of squares within 1e-12 relative of the oracle's compensated fp64 sum, the
    non-finite count exactly, and the report's count word equal to the oracle's
    packing of its statistics; one NaN and one Inf are planted."""
    scale = 65536.0 if R != 3 else 1024.0
    grads = [_shifted(n, off, synth.gpu_draw("normal:1e-3", n, torch.float32, (41, R, r), DEV)
                      * scale) for r in range(R)]
    grads[R - 1][n // 2] = float("nan")
    grads[0][n - 1] = float("inf")
    mean = _shifted(n, mean_off) if store_mean else None
    report = torch.full((4,), -1, dtype=torch.int32, device=DEV)
    rcc.grad_stats_noalloc(grads, scale, report, mean_grad=mean)
    torch.cuda.synchronize()
    host = [g.cpu().numpy() for g in grads]
    want_mean = orc.mean_unscale(host, np.float32(1.0 / scale))
    st = orc.stats_accumulate(orc.stats_new(), want_mean)
    if store_mean:
        assert _mean_matches(mean, want_mean)
    sum_sq, nonfinite = _decode(report)
    want = orc.stats_value(st)
    assert nonfinite == st.nonfinite == 2
    assert abs(sum_sq - want) <= 1e-12 * want, (sum_sq, want)
    words = report.cpu().numpy().view(np.uint32)[:3].tolist()
    assert words[2] == orc.report_pack(st)[2]


def test_noalloc_rejects_sizes_beyond_the_static_array():
    # rejected on the host before any launch: the addresses are never used
    fake = rcc.ptr_array([0x7F0000000000 + r * (1 << 30) for r in range(4)])
    st = rcc.raw("rcc_grad_stats_noalloc", fake, 4, C.c_size_t(16384 * 8192 + 1), 1.0, None,
                 C.c_void_p(0x7E0000000000), None)
    assert st == rcc.ERR_INVALID_ARGUMENT
    assert "134217728" in rcc.last_error()
