"""Checkpoint state_dict handling on the CPU: round trip through a file,
step-options version 2, and the legacy rule (a state saved without options
restores with the fused step and hierarchical statistics off, hence no clip)
from the RUDA docs' native PyTorch section."""
import numpy as np
import pytest
import torch

from gradient_sync_rcc_gb300 import checkpoint, rcc


def _tensors():
    g = torch.Generator().manual_seed(5)
    return [dict(params=[torch.randn(n, generator=g) for _ in range(2)],
                 exp_avg=[torch.randn(n, generator=g) for _ in range(2)],
                 exp_avg_sq=[torch.rand(n, generator=g) for _ in range(2)]) for n in (7, 1000)]


def test_round_trip_through_file(tmp_path):
    ts = _tensors()
    cfg = rcc.adamw_cfg(lr=3e-4, max_grad_norm=0.5, replicas=2, elems_per_row=64)
    st = rcc.optim_state(scale=1024.0, step=17)
    st.growth_tracker = 5
    sd = checkpoint.state_dict(ts, cfg, st)
    path = str(tmp_path / "opt.npz")
    checkpoint.save(path, sd)
    back = checkpoint.load(path)
    assert back["step"] == 17 and back["scaler"]["growth_tracker"] == 5
    assert back["step_options"] == {"version": 2, "fused_step": True, "max_grad_norm": 0.5,
                                    "hierarchical_stats": True, "elems_per_row": 64}
    fresh = [{k: [torch.zeros_like(x) for x in v] for k, v in t.items()} for t in ts]
    cfg2, st2 = checkpoint.load_state_dict(back, fresh, rcc)
    for a, b in zip(ts, fresh):
        for k in a:
            for x, y in zip(a[k], b[k]):
                assert torch.equal(x, y)
    assert (cfg2.lr, cfg2.beta1, cfg2.beta2, cfg2.eps, cfg2.weight_decay) == \
        (cfg.lr, cfg.beta1, cfg.beta2, cfg.eps, cfg.weight_decay)
    assert cfg2.max_grad_norm == 0.5 and cfg2.replicas == 2 and cfg2.elems_per_row == 64
    assert (st2.step, st2.scale, st2.growth_tracker, st2.growth_interval) == (17, 1024.0, 5, 2000)


def test_legacy_state_restores_without_fused_options():
    ts = _tensors()
    sd = checkpoint.state_dict(ts, rcc.adamw_cfg(max_grad_norm=1.0, replicas=2), rcc.optim_state())
    del sd["step_options"]
    opts = checkpoint.step_options(sd)
    assert opts["fused_step"] is False and opts["hierarchical_stats"] is False
    cfg, _ = checkpoint.load_state_dict(sd, ts, rcc)
    assert cfg.max_grad_norm == 0.0 and cfg.hierarchical_stats == 0


def test_step_options_checks():
    sd = {"step_options": {"version": 1, "fused_step": True, "max_grad_norm": 1.0,
                           "hierarchical_stats": True, "elems_per_row": 0}}
    with pytest.raises(ValueError):
        checkpoint.step_options(sd)
    sd["step_options"].update(version=2, fused_step=False)
    with pytest.raises(ValueError):          # clipping requires the fused step
        checkpoint.step_options(sd)


def test_state_dict_does_not_alias_host_tensors():
    """A state taken from host tensors is a copy: changing the tensors after
    state_dict leaves the saved arrays as they were."""
    ts = _tensors()
    cfg = rcc.adamw_cfg(replicas=2)
    sd = checkpoint.state_dict(ts, cfg, rcc.optim_state())
    before = [{k: [a.copy() for a in v] for k, v in t.items()} for t in sd["tensors"]]
    for t in ts:
        for k in t:
            for x in t[k]:
                x.add_(1.0)
    for saved, ref in zip(sd["tensors"], before):
        for k in ref:
            for a, b in zip(saved[k], ref[k]):
                assert np.array_equal(a, b)
