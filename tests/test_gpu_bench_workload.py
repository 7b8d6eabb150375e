"""Parity at the benchmark's full size and launch configuration.

The benchmark's step (8 logical ranks x 2^24 fp32, gradient-like values) is
built with bench.Workload itself and every row is checked against the oracle:
all_reduce sum/mean/max, reduce to root 7, broadcast from root 0,
reduce_scatter, all_gather, and the gradient-sync + AdamW step on the 8 rank
buffers as one tensor's gradients (one state copy, clip at 1.0).
"""
import numpy as np
import pytest
import torch

import bench
from gradient_sync_rcc_gb300 import rcc
from gpu_util import bits_equal, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def wl():
    from gradient_sync_rcc_gb300 import build
    build.build()
    return bench.Workload("cuda:0")


def test_every_row_of_the_bench_step(orc, wl):
    R = bench.R
    xs = [to_host(x) for x in wl.ins]
    p0 = to_host(wl.gs_tensors[0]["params"][0])
    h = rcc.register(0, R, rcc.F32, True)
    try:
        for op in ("sum", "mean", "max"):
            rcc.all_reduce(h, wl.ins, wl.ar, op)
            torch.cuda.synchronize()
            want = orc.reduce_f32(xs, op)
            for r in (0, R - 1):
                assert bits_equal(to_host(wl.ar[r]), want), op
        rcc.reduce(h, wl.ins, wl.red, root=R - 1, op="sum")
        rcc.broadcast(h, wl.ins[0], wl.bc, root=0)
        rcc.reduce_scatter(h, wl.ins, wl.rs, "sum")
        rcc.all_gather(h, wl.rs, wl.ag)
        torch.cuda.synchronize()
        s = orc.reduce_f32(xs, "sum")
        assert bits_equal(to_host(wl.red), s)
        for r in (0, 3, R - 1):
            assert bits_equal(to_host(wl.bc[r]), xs[0])
            assert bits_equal(to_host(wl.ag[r]), s)
        rs_want = orc.reduce_scatter(xs, "sum")
        for r in range(R):
            assert bits_equal(to_host(wl.rs[r]), rs_want[r])
        # the gradient-sync row, one step from the workload's initial state
        state = rcc.optim_state(scale=1.0)
        rep = rcc.grad_sync_adamw(h, wl.sets, wl.cfg, state)
        torch.cuda.synchronize()
    finally:
        rcc.finish(h)
    hp, hm, hv = [p0.copy()], [np.zeros_like(p0)], [np.zeros_like(p0)]
    sc = orc.scaler_new(1.0)
    step, st, d = orc.grad_sync_adamw_step([xs], hp, hm, hv, lr=wl.cfg.lr, beta1=wl.cfg.beta1,
                                           beta2=wl.cfg.beta2, eps=wl.cfg.eps,
                                           weight_decay=wl.cfg.weight_decay,
                                           max_grad_norm=wl.cfg.max_grad_norm, step=0, scaler=sc)
    assert rep.skipped == d.skip == 0 and state.step == step == 1
    assert abs(rep.sum_sq - orc.stats_value(st)) <= 1e-12 * orc.stats_value(st)
    assert rep.clip_coef < 1.0                     # the clip is active on this workload
    got = to_host(wl.gs_tensors[0]["params"][0]).astype(np.float64)
    assert np.all(np.abs(got - hp[0]) <= 1e-6 * np.maximum(np.abs(hp[0]), 1e-3))
    assert bits_equal(to_host(wl.gs_tensors[0]["mean_grad"]),
                      orc.mean_unscale(xs, np.float32(1.0)))
