"""Optimizer-state checkpoints for rcc_grad_sync_adamw.

[RUDA docs "Training and saving state", section "Native PyTorch training on
ruda:0"]: the model, optimizer and scaler state_dicts are saved together; the
optimizer stores fused_step and max_grad_norm, and hierarchical statistics use
step-options version 2; a state saved without these settings restores with
the fused step and hierarchical statistics disabled.  [ruCCL README §6]: the
collective_training example saves each rank's model and optimizer after the
first update and `resume` re-runs the second update from that state.

The state the gradient-sync step needs is the caller's: per tensor and replica
the fp32 params, exp_avg and exp_avg_sq, plus the step count and GradScaler
state (rcc_optim_state) and the step options (rcc_adamw_cfg).  A checkpoint is
a copy of those; this module moves them to and from host memory.  No method
arithmetic happens here.
"""
import numpy as np

STEP_OPTIONS_VERSION = 2


def _host_copy(x):
    """A host array that does not alias x: `.cpu()` of a device tensor is
    already a fresh host copy; of a host tensor it is the tensor itself."""
    a = x.detach().cpu().numpy()
    return a if x.is_cuda else a.copy()


def state_dict(tensors, cfg, state, fused_step=True):
    """Host copy of the optimizer state.  tensors: the dicts given to
    rcc.ParamSets (params / exp_avg / exp_avg_sq replica lists of device
    tensors); cfg: rcc.AdamWCfg; state: rcc.OptimState."""
    per = []
    for t in tensors:
        per.append({k: [_host_copy(x) for x in t[k]] for k in ("params", "exp_avg", "exp_avg_sq")})
    return {
        "tensors": per,
        "step": int(state.step),
        "scaler": {"scale": float(state.scale), "growth_factor": float(state.growth_factor),
                   "backoff_factor": float(state.backoff_factor),
                   "growth_interval": int(state.growth_interval),
                   "growth_tracker": int(state.growth_tracker)},
        "hyper": {"lr": cfg.lr, "betas": (cfg.beta1, cfg.beta2), "eps": cfg.eps,
                  "weight_decay": cfg.weight_decay, "replicas": int(cfg.replicas)},
        "step_options": {"version": STEP_OPTIONS_VERSION, "fused_step": bool(fused_step),
                         "max_grad_norm": float(cfg.max_grad_norm),
                         "hierarchical_stats": bool(cfg.hierarchical_stats),
                         "elems_per_row": int(cfg.elems_per_row)},
    }


def step_options(sd):
    """The step options a state restores with.  Without saved options (a
    legacy state) the fused step and hierarchical statistics are off, and with
    the fused step off there is no clipping."""
    opts = sd.get("step_options")
    if not opts:
        return {"version": 0, "fused_step": False, "max_grad_norm": 0.0,
                "hierarchical_stats": False, "elems_per_row": 0}
    if opts.get("version") != STEP_OPTIONS_VERSION:
        raise ValueError("unsupported step-options version %r" % (opts.get("version"),))
    if not opts["fused_step"] and opts["max_grad_norm"] > 0:
        raise ValueError("clipping requires fused_step=True")
    return dict(opts)


def load_state_dict(sd, tensors, rcc):
    """Copy a state_dict back into device tensors (same shapes) and return
    (cfg, state) for rcc_grad_sync_adamw."""
    import torch
    for t, saved in zip(tensors, sd["tensors"]):
        for k in ("params", "exp_avg", "exp_avg_sq"):
            for dst, src in zip(t[k], saved[k]):
                assert dst.numel() == src.size, "tensor shape changed since the checkpoint"
                dst.copy_(torch.from_numpy(np.ascontiguousarray(src)))
    opts = step_options(sd)
    h = sd["hyper"]
    cfg = rcc.adamw_cfg(lr=h["lr"], betas=tuple(h["betas"]), eps=h["eps"],
                        weight_decay=h["weight_decay"],
                        max_grad_norm=opts["max_grad_norm"] if opts["fused_step"] else 0.0,
                        replicas=h["replicas"], hierarchical_stats=opts["hierarchical_stats"],
                        elems_per_row=opts["elems_per_row"])
    sc = sd["scaler"]
    state = rcc.optim_state(scale=sc["scale"], growth_factor=sc["growth_factor"],
                            backoff_factor=sc["backoff_factor"],
                            growth_interval=sc["growth_interval"], step=sd["step"])
    state.growth_tracker = sc["growth_tracker"]
    return cfg, state


def save(path, sd):
    """Write a state_dict to an .npz file (arrays plus a JSON header)."""
    import json
    arrays = {}
    for i, t in enumerate(sd["tensors"]):
        for k, reps in t.items():
            for j, a in enumerate(reps):
                arrays["t%d_%s_%d" % (i, k, j)] = a
    meta = {k: v for k, v in sd.items() if k != "tensors"}
    meta["layout"] = [{k: len(reps) for k, reps in t.items()} for t in sd["tensors"]]
    np.savez(path, __meta__=np.frombuffer(json.dumps(meta).encode(), dtype=np.uint8), **arrays)


def load(path):
    import json
    with np.load(path) as z:
        meta = json.loads(bytes(z["__meta__"]).decode())
        tensors = []
        for i, lay in enumerate(meta.pop("layout")):
            tensors.append({k: [z["t%d_%s_%d" % (i, k, j)].copy() for j in range(n)]
                            for k, n in lay.items()})
    meta["tensors"] = tensors
    if "hyper" in meta:
        meta["hyper"]["betas"] = tuple(meta["hyper"]["betas"])
    return meta
