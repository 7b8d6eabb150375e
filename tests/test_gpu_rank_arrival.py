"""Per-rank arrival on the GPU: one host thread and one CUDA stream per rank.

Each rank queues the copy of its input on its own stream just before it
arrives and reads its output on that stream right after the call returns, so
the result is correct only if the kernel waited for every rank's stream and
every rank's stream waited for the kernel.  Results must equal the oracle's
bit for bit (deterministic rank order).
"""
import threading

import numpy as np
import pytest
import torch

from gradient_sync_rcc_gb300 import rcc, synth
from gpu_util import DEV, bits_equal, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gradient_sync_rcc_gb300 import build
    build.build()
    assert torch.cuda.is_available()


def _threads(fn, R):
    errs = []

    def run(r):
        try:
            fn(r)
        except BaseException as e:  # surfaced below
            errs.append(e)

    ts = [threading.Thread(target=run, args=(r,)) for r in range(R)]
    for t in ts:
        t.start()
    for t in ts:
        t.join(120)
    assert not errs, errs


@pytest.mark.parametrize("R", [2, 4, 8])
def test_rank_threads_every_collective(orc, R):
    n = 4096 * 37 + 3                      # ragged
    N = n * R
    xs = synth.rank_buffers("uniform", R, N, 50, R)
    host_in = [torch.from_numpy(x).pin_memory() for x in xs]
    streams = [torch.cuda.Stream() for _ in range(R)]
    ins = [torch.zeros(N, device=DEV) for _ in range(R)]
    outs = {k: [None] * R for k in ("ar", "rs", "ag", "bc", "red")}
    h = rcc.register(0, R, rcc.F32, True)
    try:
        def rank(r):
            s = streams[r]
            with torch.cuda.stream(s):
                for rnd in range(3):
                    ins[r].copy_(host_in[r], non_blocking=True)     # queued before arrival
                    ar = torch.empty(N, device=DEV)
                    rcc.all_reduce_rank(h, r, ins[r], ar, "sum", stream=s)
                    rs = torch.empty(n, device=DEV)
                    rcc.reduce_scatter_rank(h, r, ins[r], rs, "mean", stream=s)
                    ag = torch.empty(N, device=DEV)
                    rcc.all_gather_rank(h, r, rs, ag, stream=s)
                    bc = torch.empty(N, device=DEV)
                    rcc.broadcast_rank(h, r, ins[r] if r == 1 else None, bc, N, stream=s)
                    red = torch.full((N,), 5.0, device=DEV)
                    rcc.reduce_rank(h, r, ins[r], red, root=R - 1, op="max", stream=s)
                    # read on this rank's stream right after the calls return
                    outs["ar"][r] = ar.clone()
                    outs["rs"][r] = rs.clone()
                    outs["ag"][r] = ag.clone()
                    outs["bc"][r] = bc.clone()
                    outs["red"][r] = red.clone()
                    ins[r].zero_()                               # next round refills it
        _threads(rank, R)
        torch.cuda.synchronize()
    finally:
        rcc.finish(h)
    ar_want = orc.reduce_f32(xs, "sum")
    rs_want = orc.reduce_scatter(xs, "mean")
    red_want = orc.reduce_f32(xs, "max")
    for r in range(R):
        assert bits_equal(to_host(outs["ar"][r]), ar_want)
        assert bits_equal(to_host(outs["rs"][r]), rs_want[r])
        assert bits_equal(to_host(outs["ag"][r]), np.concatenate(rs_want))
        assert bits_equal(to_host(outs["bc"][r]), xs[1])
        if r == R - 1:
            assert bits_equal(to_host(outs["red"][r]), red_want)
        else:
            assert bool(torch.all(outs["red"][r] == 5.0))   # non-roots untouched


def test_rank_threads_mismatch_launches_nothing():
    R, N = 4, 1000
    before = rcc.launch_count()
    bufs = [torch.zeros(N, device=DEV) for _ in range(R)]
    outs = [torch.zeros(N, device=DEV) for _ in range(R)]
    h = rcc.register(0, R, rcc.F32, True)
    status = [None] * R
    try:
        def rank(r):
            n = N if r != 2 else N - 1
            status[r] = rcc.lib().rcc_all_reduce_rank(h, r, bufs[r].data_ptr(), outs[r].data_ptr(),
                                                      n, 0, None)
        _threads(rank, R)
    finally:
        rcc.finish(h)
    assert status == [rcc.ERR_SHAPE_MISMATCH] * R
    assert rcc.launch_count() == before
