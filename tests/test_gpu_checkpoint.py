"""Run versus resume, bit for bit ([ruCCL README §6, the collective_training
example]: two ranks on the same device; `run` saves each rank's model and
optimizer after the first update and performs the second; `resume` restores
that state and performs the second update).  The resumed second update must
reproduce the uninterrupted one exactly: parameters, moments, step count and
GradScaler state.  Both are also checked against the CPU oracle run over the
same two updates (parameters and moments within 1e-6 relative, step count and
scaler exact), so a fault common to both runs cannot pass."""
import numpy as np
import pytest
import torch

from gradient_sync_rcc_gb300 import checkpoint, rcc, synth
from gpu_util import DEV, session, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gradient_sync_rcc_gb300 import build
    build.build()
    assert torch.cuda.is_available()


R = 2
SIZES = [4096, 100003, 7]


def _model():
    return [dict(grads=[torch.empty(n, device=DEV) for _ in range(R)],
                 params=[synth.gpu_draw("normal:0.02", n, torch.float32, (60, i), DEV)
                         for _ in range(R)],
                 exp_avg=[torch.zeros(n, device=DEV) for _ in range(R)],
                 exp_avg_sq=[torch.zeros(n, device=DEV) for _ in range(R)],
                 mean_grad=torch.empty(n, device=DEV)) for i, n in enumerate(SIZES)]


def _grads(tensors, update, scale):
    for i, t in enumerate(tensors):
        for r in range(R):
            t["grads"][r].copy_(synth.gpu_draw("normal:1e-3", SIZES[i], torch.float32,
                                               (61, i, update, r), DEV) * scale)


def _oracle_two_updates(orc, cfg, scale0):
    """The oracle's state after updates 1 and 2 from the same initial
    parameters and gradients (drawn on the device exactly as the runs draw
    them, then copied to the host)."""
    hp = [to_host(synth.gpu_draw("normal:0.02", n, torch.float32, (60, i), DEV))
          for i, n in enumerate(SIZES)]
    hm = [np.zeros(n, np.float32) for n in SIZES]
    hv = [np.zeros(n, np.float32) for n in SIZES]
    sc = orc.scaler_new(scale0)
    step = 0
    for update in (1, 2):
        grads = [[to_host(synth.gpu_draw("normal:1e-3", n, torch.float32, (61, i, update, r), DEV)
                          * sc.scale) for r in range(R)] for i, n in enumerate(SIZES)]
        step, _, d = orc.grad_sync_adamw_step(
            grads, hp, hm, hv, lr=cfg.lr, beta1=cfg.beta1, beta2=cfg.beta2, eps=cfg.eps,
            weight_decay=cfg.weight_decay, max_grad_norm=cfg.max_grad_norm, step=step,
            scaler=sc)
        assert d.skip == 0
    return hp, hm, hv, step, sc


def _close(gpu, ref):
    return bool(np.all(np.abs(gpu.astype(np.float64) - ref) <= 1e-6 * np.maximum(np.abs(ref), 1e-3)))


@pytest.mark.parametrize("flags", [0, rcc.ADAMW_GRAPH])
def test_resume_reproduces_second_update(orc, tmp_path, flags):
    path = str(tmp_path / "collective-training-state.npz")
    # run: update 1, save, update 2
    run = _model()
    cfg = rcc.adamw_cfg(replicas=R, max_grad_norm=0.05, flags=flags)
    state = rcc.optim_state(scale=65536.0)
    with session(R) as h:
        sets = rcc.ParamSets(run)
        _grads(run, 1, state.scale)
        rcc.grad_sync_adamw(h, sets, cfg, state)
        torch.cuda.synchronize()
        checkpoint.save(path, checkpoint.state_dict(run, cfg, state))
        _grads(run, 2, state.scale)
        rep = rcc.grad_sync_adamw(h, sets, cfg, state)
        torch.cuda.synchronize()
    assert rep.skipped == 0 and state.step == 2
    # resume: fresh buffers, restore, update 2
    res = _model()
    for t in res:                                   # make sure nothing leaks from the draw
        for k in ("params", "exp_avg", "exp_avg_sq"):
            for x in t[k]:
                x.fill_(float("nan"))
    cfg2, state2 = checkpoint.load_state_dict(checkpoint.load(path), res, rcc)
    cfg2.flags = flags
    assert state2.step == 1
    with session(R) as h:
        _grads(res, 2, state2.scale)
        rcc.grad_sync_adamw(h, rcc.ParamSets(res), cfg2, state2)
        torch.cuda.synchronize()
    assert (state2.step, state2.scale, state2.growth_tracker) == \
        (state.step, state.scale, state.growth_tracker)
    for a, b in zip(run, res):
        for k in ("params", "exp_avg", "exp_avg_sq"):
            for x, y in zip(a[k], b[k]):
                assert torch.equal(x.view(torch.int32), y.view(torch.int32)), k
    # both against the oracle over the same two updates
    hp, hm, hv, ostep, sc = _oracle_two_updates(orc, cfg, 65536.0)
    assert (state2.step, state2.scale, state2.growth_tracker) == \
        (ostep, sc.scale, sc.growth_tracker)
    for i, t in enumerate(res):
        for k, ref in (("params", hp), ("exp_avg", hm), ("exp_avg_sq", hv)):
            for x in t[k]:
                assert _close(to_host(x), ref[i]), (i, k)
