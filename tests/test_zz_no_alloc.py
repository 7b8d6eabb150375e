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
<= 1024 rows, one that needs the fan-in-1024 combine and carries a NaN.
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


def _decode(report):
    w = report.cpu().numpy().view(np.uint32)
    return float(w[:2].copy().view(np.float64)[0]), int(w[2])


def test_noalloc_matches_grad_sync_on_two_calls():
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


def test_noalloc_rejects_sizes_beyond_the_static_array():
    # rejected on the host before any launch: the addresses are never used
    fake = rcc.ptr_array([0x7F0000000000 + r * (1 << 30) for r in range(4)])
    st = rcc.raw("rcc_grad_stats_noalloc", fake, 4, C.c_size_t(16384 * 8192 + 1), 1.0, None,
                 C.c_void_p(0x7E0000000000), None)
    assert st == rcc.ERR_INVALID_ARGUMENT
    assert "134217728" in rcc.last_error()
