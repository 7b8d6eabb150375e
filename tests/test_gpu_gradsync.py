"""GPU parity of the gradient-sync + fused AdamW step against the CPU oracle.

[ruCCL README §6]: all_reduce Mean of the gradients, then the optimizer step.
[RUDA docs "Training and saving state", native PyTorch section]: unscale,
read-only analysis, global L2 clip at max_grad_norm, fan-in-1024 statistics
(no extra combine for <= 1024 rows, at most two, a reused region of at most
49,200 bytes), the 12-byte report read back, skip on non-finite, FP32 master
weights and moments, one update kernel per parameter.

Acceptance: parameters (and moments) within 1e-6 relative of the oracle,
|p_gpu - p_orc| <= 1e-6 * max(|p_orc|, 1e-3), after every step of a 10-step
run with one NaN injected at step 7 (that step skipped, the scale halved);
the sum of squares within 1e-12 relative; decisions and counters exact.
"""
import math
import struct

import numpy as np
import pytest
import torch

from gradient_sync_rcc_gb300 import rcc, synth
from gpu_util import DEV, bits_equal, session, to_dev, to_host

pytestmark = pytest.mark.gpu

LR, B1, B2, EPS, WD, MAXN = 1e-3, 0.9, 0.999, 1e-8, 0.01, 1.0
REL = 1e-6


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gradient_sync_rcc_gb300 import build
    build.build()
    assert torch.cuda.is_available()


def close(gpu, ref):
    return bool(np.all(np.abs(gpu.astype(np.float64) - ref) <= REL * np.maximum(np.abs(ref), 1e-3)))


def check_report_words(orc, rep, st):
    """The 12 bytes the call read back, word by word against the oracle's
    packing of its own statistics (RUDA docs, native PyTorch section: a 12-byte
    report read back before the update): the count word exactly, the two words
    of the fp64 sum of squares decoded within 1e-12 relative (the GPU sums in a
    different order)."""
    want = orc.report_pack(st)
    got = list(rep.report_words)
    assert got[2] == want[2], (got, want)
    s_gpu = struct.unpack("<d", struct.pack("<2I", got[0], got[1]))[0]
    s_orc = struct.unpack("<d", struct.pack("<2I", want[0], want[1]))[0]
    assert abs(s_gpu - s_orc) <= 1e-12 * s_orc, (s_gpu, s_orc)
    assert s_gpu == rep.sum_sq


class Problem:
    """Device state (replicas of p, m, v), persistent grad buffers, and the
    oracle's single host copy of the same state."""

    def __init__(self, R, sizes, seed, replicas, mean_grad=True):
        self.R, self.sizes, self.seed, self.rep = R, sizes, seed, replicas
        p0 = [synth.normal(n, 0.02, seed, 1, i) for i, n in enumerate(sizes)]
        self.hp = [x.copy() for x in p0]
        self.hm = [np.zeros(n, np.float32) for n in sizes]
        self.hv = [np.zeros(n, np.float32) for n in sizes]
        self.tensors = []
        for i, n in enumerate(sizes):
            self.tensors.append(dict(
                grads=[torch.empty(n, device=DEV) for _ in range(R)],
                params=[to_dev(p0[i]) for _ in range(replicas)],
                exp_avg=[torch.zeros(n, device=DEV) for _ in range(replicas)],
                exp_avg_sq=[torch.zeros(n, device=DEV) for _ in range(replicas)],
                mean_grad=torch.empty(n, device=DEV) if mean_grad else None))
        self.sets = rcc.ParamSets(self.tensors)

    def host_grads(self, step, scale, nan_at=None):
        out = []
        for i, n in enumerate(self.sizes):
            per = [(synth.normal(n, 1e-3, self.seed, 2, i, step, r) * np.float32(scale))
                   .astype(np.float32) for r in range(self.R)]
            out.append(per)
        if nan_at is not None and step == nan_at:
            out[0][0][0] = np.nan
        return out

    def load_grads(self, grads):
        for i, per in enumerate(grads):
            for r in range(self.R):
                self.tensors[i]["grads"][r].copy_(to_dev(per[r]))


def run_steps(orc, prob, steps, nan_at, cfg_kw, check_each=True, scale=65536.0, max_norm=MAXN):
    cfg = rcc.adamw_cfg(lr=LR, betas=(B1, B2), eps=EPS, weight_decay=WD, max_grad_norm=max_norm,
                        replicas=prob.rep, **cfg_kw)
    state = rcc.optim_state(scale=scale)
    sc = orc.scaler_new(scale)
    ostep = 0
    reports = []
    with session(prob.R, rcc.F32, True) as h:
        for k in range(1, steps + 1):
            grads = prob.host_grads(k, state.scale, nan_at)
            assert state.scale == sc.scale
            prob.load_grads(grads)
            rep = rcc.grad_sync_adamw(h, prob.sets, cfg, state)
            torch.cuda.synchronize()
            ostep, st, d = orc.grad_sync_adamw_step(
                grads, prob.hp, prob.hm, prob.hv, lr=LR, beta1=B1, beta2=B2, eps=EPS,
                weight_decay=WD, max_grad_norm=max_norm, step=ostep, scaler=sc)
            reports.append(rep)
            assert rep.skipped == d.skip
            assert rep.nonfinite == st.nonfinite
            check_report_words(orc, rep, st)
            assert state.step == ostep and state.scale == sc.scale
            if not d.skip:
                want = orc.stats_value(st)
                assert abs(rep.sum_sq - want) <= 1e-12 * want, (rep.sum_sq, want)
                assert abs(rep.clip_coef - d.clip_coef) <= 2e-7 * d.clip_coef
                per = 1 if cfg.flags & rcc.ADAMW_MULTI_TENSOR else len(prob.sizes)
                assert rep.update_launches == per
            else:   # the host flow launches nothing; the device flow's updates return at once
                per = 1 if cfg.flags & rcc.ADAMW_MULTI_TENSOR else len(prob.sizes)
                assert rep.update_launches == (per if rep.updates_before_readback else 0)
            on_device = cfg.flags & (rcc.ADAMW_DEVICE_DECISION | rcc.ADAMW_GRAPH)
            assert rep.updates_before_readback == (1 if on_device else 0)
            if check_each or k == steps:
                for i in range(len(prob.sizes)):
                    t = prob.tensors[i]
                    p0 = to_host(t["params"][0])
                    assert close(p0, prob.hp[i]), (k, i)
                    assert close(to_host(t["exp_avg"][0]), prob.hm[i]), (k, i)
                    assert close(to_host(t["exp_avg_sq"][0]), prob.hv[i]), (k, i)
                    for j in range(1, prob.rep):
                        for key in ("params", "exp_avg", "exp_avg_sq"):
                            assert torch.equal(t[key][j].view(torch.int32),
                                               t[key][0].view(torch.int32)), (k, i, j, key)
    return reports, state


MODES = {"host": 0, "device": rcc.ADAMW_DEVICE_DECISION, "graph": rcc.ADAMW_GRAPH,
         "multi": rcc.ADAMW_MULTI_TENSOR,
         "device_multi": rcc.ADAMW_DEVICE_DECISION | rcc.ADAMW_MULTI_TENSOR,
         "host_graph": rcc.ADAMW_HOST_GRAPH}


@pytest.mark.parametrize("mode", list(MODES))
@pytest.mark.parametrize("replicas", [1, 4])
@pytest.mark.parametrize("mean_grad", [True, False])
def test_ten_steps_nan_at_seven(orc, replicas, mean_grad, mode):
    sizes = synth.param_sizes(16, 1024, 65536, 10)
    prob = Problem(4, sizes, 11, replicas, mean_grad)
    # the unscaled mean gradient has norm ~0.2 here: max_grad_norm 0.1 keeps
    # the clip active on every applied step
    reports, state = run_steps(orc, prob, 10, 7, {"flags": MODES[mode]}, max_norm=0.1)
    assert [r.skipped for r in reports] == [0] * 6 + [1] + [0] * 3
    assert state.step == 9 and state.scale == 32768.0
    assert all(r.combine_launches == 0 for r in reports)      # <= 1024 rows
    assert all(r.clip_coef < 1.0 for r in reports if not r.skipped)


def test_decision_modes_bitwise_identical():
    """Host decision, device decision and the captured graph give the same bits."""
    sizes = synth.param_sizes(64, 1024, 200000, 30)
    finals = {}
    for mode, flags in MODES.items():
        prob = Problem(4, sizes, 31, 4, mode != "device")
        cfg = rcc.adamw_cfg(replicas=4, flags=flags)
        state = rcc.optim_state(scale=65536.0)
        with session(4) as h:
            for k in range(1, 7):
                prob.load_grads(prob.host_grads(k, state.scale, nan_at=4))
                rep = rcc.grad_sync_adamw(h, prob.sets, cfg, state)
                assert rep.skipped == (1 if k == 4 else 0)
            torch.cuda.synchronize()
        assert state.step == 5
        finals[mode] = [torch.cat([t["params"][1], t["exp_avg"][0], t["exp_avg_sq"][1]]).cpu()
                        for t in prob.tensors]
    for mode in (m for m in MODES if m != "host"):
        for a, b in zip(finals["host"], finals[mode]):
            assert torch.equal(a.view(torch.int32), b.view(torch.int32)), mode


@pytest.mark.parametrize("flags", [rcc.ADAMW_GRAPH, rcc.ADAMW_HOST_GRAPH])
def test_graph_recaptured_when_tensors_change(orc, flags):
    """New gradient buffers change the descriptor tables; the graph must follow."""
    sizes = [10000, 2000, 777]
    prob = Problem(2, sizes, 32, 1, True)
    run_steps(orc, prob, 2, None, {"flags": flags})
    for t in prob.tensors:
        t["grads"] = [torch.empty_like(g) for g in t["grads"]]
        t["mean_grad"] = torch.empty_like(t["mean_grad"])
    prob.sets = rcc.ParamSets(prob.tensors)
    run_steps(orc, prob, 2, None, {"flags": flags})


@pytest.mark.parametrize("R", [3, 4, 5, 8])
@pytest.mark.parametrize("scale", [65536.0, 1.0])
def test_mean_grad_output_bitwise(orc, R, scale):
    """The stored mean gradient, bit for bit: the division by R (a multiply by
    the exact reciprocal when R is a power of two) and the unscale.  At scale 1
    the subnormal sums below reach the output, so the rounding of s / R at the
    bottom of the range is checked too."""
    sizes = [1, 3, 4099, 70001]
    prob = Problem(R, sizes, 12, 1, True)
    grads = prob.host_grads(1, scale)
    tiny = np.array([1, 3, 7, 5, -9, 2, 11, 6], np.float32) * np.float32(2.0 ** -149)
    for r in range(R):
        grads[3][r][:8] = tiny * np.float32(r + 1)
    prob.load_grads(grads)
    cfg = rcc.adamw_cfg(replicas=1)
    with session(R) as h:
        rcc.grad_sync_adamw(h, prob.sets, cfg, rcc.optim_state(scale=scale))
        torch.cuda.synchronize()
    inv = np.float32(1.0 / scale)
    for i in range(len(sizes)):
        want = orc.mean_unscale(grads[i], inv)
        assert bits_equal(to_host(prob.tensors[i]["mean_grad"]), want)


def _levels(rows):
    return 0 if rows <= 1024 else (1 if rows <= 1024 * 1024 else 2)


@pytest.mark.parametrize("epr,sizes", [
    (8192, [5000, 70000]),                 # few rows: no combine
    (64, [300000, 123457]),                # > 1024 rows: one combine level
    (4, [3000000, 1500001]),               # > 1024^2 rows: two combine levels
])
def test_hierarchy_levels_and_region_bound(orc, epr, sizes):
    prob = Problem(2, sizes, 13, 1, True)
    reports, _ = run_steps(orc, prob, 2, None, {"elems_per_row": epr}, check_each=True)
    rows = sum(-(-n // epr) for n in sizes)
    for r in reports:
        assert r.stats_rows == rows
        assert r.combine_levels == _levels(rows)
        assert r.combine_launches == _levels(rows)
        assert r.combine_launches <= 2
        assert r.combine_region_bytes <= 49200


def test_flat_and_hierarchical_agree(orc):
    sizes = [3000000, 777777]
    out = {}
    for hier in (True, False):
        prob = Problem(4, sizes, 14, 1, True)
        reports, _ = run_steps(orc, prob, 1, None,
                               {"elems_per_row": 16, "hierarchical_stats": hier})
        out[hier] = reports[0]
    assert out[False].combine_levels == 0 and out[True].combine_levels == 1
    a, b = out[True].sum_sq, out[False].sum_sq
    assert abs(a - b) <= 1e-13 * a


def test_no_clip_below_threshold(orc):
    """Tiny gradients: the norm stays below max_grad_norm, no clipping."""
    sizes = [4096, 1000]
    prob = Problem(2, sizes, 15, 2, True)
    cfg = rcc.adamw_cfg(replicas=2, max_grad_norm=MAXN)
    grads = prob.host_grads(1, 1.0)      # scale 1: unscaled std 1e-3/sqrt(2), norm ~ 0.05
    prob.load_grads(grads)
    with session(2) as h:
        rep = rcc.grad_sync_adamw(h, prob.sets, cfg, rcc.optim_state(scale=1.0))
        torch.cuda.synchronize()
    assert rep.grad_norm < MAXN and rep.clip_coef == 1.0 and rep.skipped == 0
    sc = orc.scaler_new(1.0)
    orc.grad_sync_adamw_step(grads, prob.hp, prob.hm, prob.hv, lr=LR, beta1=B1, beta2=B2,
                             eps=EPS, weight_decay=WD, max_grad_norm=MAXN, step=0, scaler=sc)
    for i in range(len(sizes)):
        assert close(to_host(prob.tensors[i]["params"][1]), prob.hp[i])


def test_descriptor_cache_follows_pointer_changes(orc):
    """Re-running with different gradient buffers (new pointers) must use them."""
    sizes = [10000, 2000]
    prob = Problem(2, sizes, 16, 1, True)
    run_steps(orc, prob, 2, None, {})
    # swap in fresh gradient tensors: the descriptor must be re-uploaded
    for t in prob.tensors:
        t["grads"] = [torch.empty_like(g) for g in t["grads"]]
    prob.sets = rcc.ParamSets(prob.tensors)
    run_steps(orc, prob, 1, None, {})


def test_full_1024_tensors_ten_steps(orc):
    """1024 fp32 tensors, sizes log-uniform in [1024, 4194304], R = 4, grads
    N(0, 1e-3) x 65536, 10 steps, NaN at step 7.  The oracle runs streamed per
    tensor on host copies of the same device-generated gradients."""
    R, P = 4, 1024
    sizes = synth.param_sizes(P, 1024, 4194304, 20)
    rep_count = 4
    p_dev, m_dev, v_dev, g_dev, mg_dev = [], [], [], [], []
    hp, hm, hv = [], [], []
    for i, n in enumerate(sizes):
        p0 = synth.gpu_draw("normal:0.02", n, torch.float32, (21, i), DEV)
        p_dev.append([p0.clone() for _ in range(rep_count)])
        m_dev.append([torch.zeros(n, device=DEV) for _ in range(rep_count)])
        v_dev.append([torch.zeros(n, device=DEV) for _ in range(rep_count)])
        g_dev.append([torch.empty(n, device=DEV) for _ in range(R)])
        mg_dev.append(torch.empty(n, device=DEV))
        hp.append(to_host(p0))
        hm.append(np.zeros(n, np.float32))
        hv.append(np.zeros(n, np.float32))
    sets = rcc.ParamSets([dict(grads=g_dev[i], params=p_dev[i], exp_avg=m_dev[i],
                               exp_avg_sq=v_dev[i], mean_grad=mg_dev[i]) for i in range(P)])
    cfg = rcc.adamw_cfg(lr=LR, betas=(B1, B2), eps=EPS, weight_decay=WD, max_grad_norm=MAXN,
                        replicas=rep_count)
    state = rcc.optim_state(scale=65536.0)
    sc = orc.scaler_new(65536.0)
    t = 0
    with session(R) as h:
        for k in range(1, 11):
            for i, n in enumerate(sizes):
                for r in range(R):
                    g_dev[i][r].copy_(synth.gpu_draw("normal:1e-3", n, torch.float32,
                                                     (22, i, k, r), DEV) * state.scale)
            if k == 7:
                g_dev[0][0][0] = float("nan")
            rep = rcc.grad_sync_adamw(h, sets, cfg, state)
            torch.cuda.synchronize()
            # oracle, streamed per tensor
            inv = np.float32(1.0 / sc.scale)
            st = orc.stats_new()
            means = []
            for i in range(P):
                mean = orc.mean_unscale([to_host(g) for g in g_dev[i]], inv)
                orc.stats_accumulate(st, mean)
                means.append(mean)
            d = orc.decide(st, MAXN)
            assert rep.skipped == d.skip and rep.nonfinite == st.nonfinite
            check_report_words(orc, rep, st)
            if d.skip:
                orc.scaler_update(sc, True)
            else:
                want = orc.stats_value(st)
                assert abs(rep.sum_sq - want) <= 1e-12 * want
                t += 1
                s = orc.adamw_scalars(LR, B1, B2, EPS, WD, t)
                for i in range(P):
                    orc.adamw_update(means[i], d.clip_coef, s, hp[i], hm[i], hv[i])
                orc.scaler_update(sc, False)
            assert state.step == t and state.scale == sc.scale
            assert rep.combine_levels == _levels(rep.stats_rows)
    assert t == 9 and state.scale == 32768.0
    bad = []
    for i in range(P):
        for name, dev_list, ref in (("p", p_dev, hp), ("m", m_dev, hm), ("v", v_dev, hv)):
            if not close(to_host(dev_list[i][0]), ref[i]):
                bad.append((name, i))
            for j in range(1, rep_count):
                assert torch.equal(dev_list[i][j].view(torch.int32),
                                   dev_list[i][0].view(torch.int32)), (name, i, j)
    assert not bad, bad[:10]
    assert math.isfinite(rep.grad_norm)


def test_overlapping_outputs_rejected_shared_grads_allowed():
    """Updates of different tensors may run concurrently, so written buffers
    (params, moments, mean gradient) must be disjoint from every other buffer;
    gradients are only read and may be shared."""
    R, n = 2, 1000
    g = torch.randn(n, device=DEV)
    base = torch.zeros(5 * n, device=DEV)
    t1 = dict(grads=[g, g], params=[base[:n]], exp_avg=[base[n:2 * n]],
              exp_avg_sq=[base[2 * n:3 * n]], mean_grad=None)
    clash = dict(grads=[g, g], params=[base[2 * n + 8:3 * n + 8]],
                 exp_avg=[torch.zeros(n, device=DEV)], exp_avg_sq=[torch.zeros(n, device=DEV)],
                 mean_grad=None)
    fine = dict(grads=[g, g], params=[base[3 * n:4 * n]], exp_avg=[torch.zeros(n, device=DEV)],
                exp_avg_sq=[torch.zeros(n, device=DEV)], mean_grad=None)
    mean_on_grad = dict(fine, mean_grad=g)
    cfg = rcc.adamw_cfg(replicas=1)
    with session(R) as h:
        for bad in (clash, mean_on_grad):
            with pytest.raises(rcc.RccError) as ei:
                rcc.grad_sync_adamw(h, rcc.ParamSets([t1, bad]), cfg, rcc.optim_state(scale=1.0))
            assert ei.value.status == rcc.ERR_INVALID_ARGUMENT
        rep = rcc.grad_sync_adamw(h, rcc.ParamSets([t1, fine]), cfg, rcc.optim_state(scale=1.0))
        torch.cuda.synchronize()
    assert rep.update_launches == 2


@pytest.mark.parametrize("R", [3, 6])
@pytest.mark.parametrize("mean_grad", [True, False])
@pytest.mark.parametrize("per_rank_state", [False, True])
def test_rank_counts_that_are_not_powers_of_two(orc, R, mean_grad, per_rank_state):
    """R = 3 and 6 divide (no exact reciprocal); with no stored mean gradient
    the update recomputes the mean with the same arithmetic.  With R state
    copies the update kernels take their runtime replica-count path."""
    sizes = [5000, 1023, 64]
    prob = Problem(R, sizes, 17, R if per_rank_state else 1, mean_grad)
    run_steps(orc, prob, 3, None, {})
    if per_rank_state:
        prob2 = Problem(R, sizes, 17, R, mean_grad)
        run_steps(orc, prob2, 2, None, {"flags": MODES["device_multi"]})


_CHAIN_CHECK = """
import sys
sys.path.insert(0, {tests!r})
import oracle
oracle.build.build()
import test_gpu_gradsync as t
from gradient_sync_rcc_gb300 import rcc, synth
for flags in (0, rcc.ADAMW_GRAPH, rcc.ADAMW_HOST_GRAPH):
    prob = t.Problem(4, synth.param_sizes(9, 1024, 40000, 17), 18, 1, True)
    t.run_steps(oracle, prob, 3, None, {{"flags": flags}})
print("chains ok")
"""


@pytest.mark.parametrize("chains", ["1", "3"])
def test_chain_counts_update_every_tensor(chains):
    """The chain count is read once per process (RCC_CHAINS), so other counts
    run in a child process: every tensor must still be updated, in every
    per-tensor flow."""
    import os
    import subprocess
    import sys
    tests = os.path.dirname(os.path.abspath(__file__))
    env = dict(os.environ, RCC_CHAINS=chains)
    out = subprocess.run([sys.executable, "-c", _CHAIN_CHECK.format(tests=tests)], env=env,
                         cwd=os.path.dirname(tests), capture_output=True, text=True, timeout=600)
    assert out.returncode == 0 and "chains ok" in out.stdout, out.stdout + out.stderr


@pytest.mark.parametrize("off", [1, 4, 8])
@pytest.mark.parametrize("mode", ["host", "device_multi"])
def test_misaligned_tensors(orc, off, mode):
    """Every buffer a view `off` floats into a larger allocation: 4 bytes
    (scalar paths), 16 bytes (16-byte vectors) or 32 bytes (32-byte statistics
    vectors) past a 256-byte boundary."""
    sizes = [5000, 1027, 64, 8195]
    prob = Problem(4, sizes, 19, 1, True)

    def shift(t):
        base = torch.empty(t.numel() + off, device=DEV)
        v = base[off:off + t.numel()]
        v.copy_(t)
        return v

    for t in prob.tensors:
        t["grads"] = [shift(g) for g in t["grads"]]
        for key in ("params", "exp_avg", "exp_avg_sq"):
            t[key] = [shift(x) for x in t[key]]
        t["mean_grad"] = shift(t["mean_grad"])
    prob.sets = rcc.ParamSets(prob.tensors)
    run_steps(orc, prob, 3, None, {"flags": MODES[mode]})


def test_readback_timeout_applies_nothing_and_the_next_call_steps(orc, monkeypatch):
    """A report that does not come back within RCC_WAIT_LIMIT_MS: the call
    returns RCC_ERR_TIMEOUT with nothing applied (the default flow launches no
    update before its decision) and the optimizer state unchanged.  The next
    call waits for the queued work of the abandoned one before reusing its
    staging memory, then steps exactly as the oracle does."""
    sizes = [200000, 5000]
    prob = Problem(4, sizes, 23, 1, True)
    cfg = rcc.adamw_cfg(lr=LR, betas=(B1, B2), eps=EPS, weight_decay=WD, max_grad_norm=MAXN,
                        replicas=1)
    state = rcc.optim_state(scale=65536.0)
    grads = prob.host_grads(1, state.scale)
    prob.load_grads(grads)
    p_before = [to_host(t["params"][0]) for t in prob.tensors]
    busy = torch.empty(1 << 28, device=DEV)
    busy.fill_(1.0)
    with session(4) as h:
        torch.cuda.synchronize()
        for _ in range(40):                  # tens of ms of work ahead on the stream
            busy.mul_(1.0)
        monkeypatch.setenv("RCC_WAIT_LIMIT_MS", "1")
        with pytest.raises(rcc.RccError) as err:
            rcc.grad_sync_adamw(h, prob.sets, cfg, state)
        assert err.value.status == rcc.ERR_TIMEOUT
        assert state.step == 0 and state.scale == 65536.0
        monkeypatch.delenv("RCC_WAIT_LIMIT_MS")
        torch.cuda.synchronize()
        for i, t in enumerate(prob.tensors):
            assert bits_equal(to_host(t["params"][0]), p_before[i])
        rep = rcc.grad_sync_adamw(h, prob.sets, cfg, state)
        torch.cuda.synchronize()
    assert rep.skipped == 0 and state.step == 1
    sc = orc.scaler_new(65536.0)
    orc.grad_sync_adamw_step(grads, prob.hp, prob.hm, prob.hv, lr=LR, beta1=B1, beta2=B2,
                             eps=EPS, weight_decay=WD, max_grad_norm=MAXN, step=0, scaler=sc)
    for i in range(len(sizes)):
        assert close(to_host(prob.tensors[i]["params"][0]), prob.hp[i])


def test_step_times_split_the_call(orc):
    """RCC_STEP_TIMING: the four phase times of a grad-sync call are positive and
    add up to about the time between CUDA events around the call (the
    statistics kernel the longest phase at this size)."""
    sizes = [2_000_003]
    prob = Problem(4, sizes, 34, 1, True)
    prob.load_grads(prob.host_grads(1, 65536.0))
    cfg = rcc.adamw_cfg(replicas=1)
    state = rcc.optim_state(scale=65536.0)
    h = rcc.register(0, 4, rcc.F32, True, step_timing=True)
    try:
        for _ in range(3):
            rcc.grad_sync_adamw(h, prob.sets, cfg, state)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        rcc.grad_sync_adamw(h, prob.sets, cfg, state)
        b.record()
        t = rcc.last_step_times(h)
        torch.cuda.synchronize()
        total = a.elapsed_time(b)
        rcc.set_flags(h, True, step_timing=False)
        rcc.grad_sync_adamw(h, prob.sets, cfg, state)
        with pytest.raises(rcc.RccError):       # the last call was not timed
            rcc.last_step_times(h)
    finally:
        rcc.finish(h)
    assert all(x >= 0.0 for x in t) and t[0] > 0.0 and t[3] > 0.0, t
    assert sum(t) <= total * 1.01 + 0.005, (t, total)
    assert sum(t) >= 0.5 * total, (t, total)


@pytest.mark.parametrize("mean_mode", ["aligned", "offset", "none"])
def test_skipped_host_step_stores_the_mean_and_applies_nothing(orc, mean_mode):
    """A skipped step in the host flow launches the statistics and report
    kernels only (no update kernel), whether the mean gradient goes through
    the 32-byte statistics path, the 16-byte one, or is not stored.  The
    stored mean gradient still equals the oracle's bit for bit (its NaN by
    position, not payload), and the state is untouched."""
    R, n = 4, 300_000
    hg = [synth.normal(n, 1e-3, 35, r) * np.float32(1024.0) for r in range(R)]
    hg[2][777] = np.nan
    grads = [to_dev(x) for x in hg]
    p = to_dev(synth.normal(n, 0.02, 35, 9))
    p_before = p.clone()
    base = torch.empty(n + 8, device=DEV)
    mean = {"aligned": base[:n], "offset": base[1:n + 1], "none": None}[mean_mode]
    sets = rcc.ParamSets([dict(grads=grads, params=[p], exp_avg=[torch.zeros_like(p)],
                               exp_avg_sq=[torch.zeros_like(p)], mean_grad=mean)])
    cfg = rcc.adamw_cfg(replicas=1)
    state = rcc.optim_state(scale=1024.0)
    with session(R) as h:
        rcc.grad_sync_adamw(h, sets, cfg, state)     # uploads the tables; skipped too
        torch.cuda.synchronize()
        scale = state.scale                          # backed off by that skip
        before = rcc.launch_count()
        rep = rcc.grad_sync_adamw(h, sets, cfg, state)
        torch.cuda.synchronize()
        launched = rcc.launch_count() - before
    assert rep.skipped == 1 and rep.update_launches == 0
    assert launched == 2 + rep.combine_launches
    assert torch.equal(p.view(torch.int32), p_before.view(torch.int32))
    if mean is not None:
        # a NaN's payload is not fixed (the GPU adds to the canonical NaN)
        want = orc.mean_unscale(hg, np.float32(1.0 / scale))
        got = to_host(mean)
        nan = np.isnan(want)
        assert np.array_equal(np.isnan(got), nan) and nan[777]
        assert bits_equal(got[~nan], want[~nan])
