"""Seeded random cases of the gradient-sync + AdamW step against the oracle.

Each case draws 1-12 parameter tensors of 1..70,000 elements (tiny ragged ones
included), 1-8 ranks, one or R state copies, a stored or recomputed mean
gradient, buffer offsets of 0..9 elements (so 32-byte, 16-byte and scalar paths
mix within one call), a statistics row size (a multiple of 4 from 4 to 8192), a
flow (host decision, device decision, captured graph, multi-tensor, host graph)
and sometimes a NaN or an Inf in one gradient.  Two steps run; after each the
parameters and moments of every tensor (every state copy bit-identical to the
first) must be within 1e-6 relative of the oracle, the decision and counters
exact, the sum of squares within 1e-12 relative and the 12 report bytes equal to
the oracle's packing of its statistics (count exactly, sum within 1e-12).
"""
import struct

import numpy as np
import pytest
import torch

from gradient_sync_rcc_gb300 import rcc, synth
from gpu_util import DEV, session, to_dev, to_host

pytestmark = pytest.mark.gpu

NCASES = 60
LR, B1, B2, EPS, WD = 1e-3, 0.9, 0.999, 1e-8, 0.01
FLOWS = [0, rcc.ADAMW_DEVICE_DECISION, rcc.ADAMW_GRAPH, rcc.ADAMW_MULTI_TENSOR,
         rcc.ADAMW_DEVICE_DECISION | rcc.ADAMW_MULTI_TENSOR, rcc.ADAMW_HOST_GRAPH]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gradient_sync_rcc_gb300 import build
    build.build()
    assert torch.cuda.is_available()


def _close(gpu, ref):
    return bool(np.all(np.abs(gpu.astype(np.float64) - ref) <= 1e-6 * np.maximum(np.abs(ref), 1e-3)))


def _view(n, off, fill=None):
    base = torch.empty(n + off, device=DEV)
    v = base[off:off + n]
    if fill is not None:
        v.copy_(fill)
    return v


@pytest.mark.parametrize("i", range(NCASES))
def test_random_grad_sync(orc, i):
    g = synth.rng(0x6A5, i)
    P = int(g.integers(1, 13))
    R = int(g.integers(1, 9))
    rep = R if g.random() < 0.4 else 1
    mean = bool(g.random() < 0.7)
    flags = FLOWS[int(g.integers(len(FLOWS)))]
    epr = int(g.choice([4, 8, 12, 64, 1000, 4096, 8192]))
    sizes = [int(v) for v in np.where(g.random(P) < 0.3, g.integers(1, 8, P),
                                      g.integers(1, 70001, P))]
    max_norm = float(g.choice([0.0, 0.05, 1.0, 100.0]))
    where = (P, R, rep, mean, flags, epr, sizes, max_norm)
    hp = [synth.normal(n, 0.02, 0x6A6, i, k) for k, n in enumerate(sizes)]
    hm = [np.zeros(n, np.float32) for n in sizes]
    hv = [np.zeros(n, np.float32) for n in sizes]
    tensors = []
    for k, n in enumerate(sizes):
        o = [int(v) for v in g.integers(0, 10, R + 3 * rep + 1)]
        tensors.append(dict(
            grads=[_view(n, o[r]) for r in range(R)],
            params=[_view(n, o[R + j], to_dev(hp[k])) for j in range(rep)],
            exp_avg=[_view(n, o[R + rep + j], torch.zeros(n, device=DEV)) for j in range(rep)],
            exp_avg_sq=[_view(n, o[R + 2 * rep + j], torch.zeros(n, device=DEV))
                        for j in range(rep)],
            mean_grad=_view(n, o[-1]) if mean else None))
    sets = rcc.ParamSets(tensors)
    cfg = rcc.adamw_cfg(lr=LR, betas=(B1, B2), eps=EPS, weight_decay=WD, max_grad_norm=max_norm,
                        replicas=rep, elems_per_row=epr, flags=flags)
    state = rcc.optim_state(scale=1024.0)
    sc = orc.scaler_new(1024.0)
    ostep = 0
    with session(R) as h:
        for step in (1, 2):
            grads = [[(synth.normal(n, 1e-3, 0x6A7, i, k, step, r) * np.float32(sc.scale))
                      .astype(np.float32) for r in range(R)] for k, n in enumerate(sizes)]
            if g.random() < 0.25:
                k = int(g.integers(P))
                grads[k][int(g.integers(R))][int(g.integers(sizes[k]))] = \
                    [np.nan, np.inf, -np.inf][int(g.integers(3))]
            for k in range(P):
                for r in range(R):
                    tensors[k]["grads"][r].copy_(to_dev(grads[k][r]))
            rep_ = rcc.grad_sync_adamw(h, sets, cfg, state)
            torch.cuda.synchronize()
            ostep, st, d = orc.grad_sync_adamw_step(
                grads, hp, hm, hv, lr=LR, beta1=B1, beta2=B2, eps=EPS, weight_decay=WD,
                max_grad_norm=max_norm, step=ostep, scaler=sc)
            assert rep_.skipped == d.skip and rep_.nonfinite == st.nonfinite, where
            assert state.step == ostep and state.scale == sc.scale, where
            want = orc.stats_value(st)
            assert abs(rep_.sum_sq - want) <= 1e-12 * want, where
            words = list(rep_.report_words)
            assert words[2] == orc.report_pack(st)[2], where
            assert struct.unpack("<d", struct.pack("<2I", words[0], words[1]))[0] == rep_.sum_sq
            if not d.skip:
                assert abs(rep_.clip_coef - d.clip_coef) <= 2e-7 * d.clip_coef, where
            for k in range(P):
                t = tensors[k]
                assert _close(to_host(t["params"][0]), hp[k]), (where, step, k)
                assert _close(to_host(t["exp_avg"][0]), hm[k]), (where, step, k)
                assert _close(to_host(t["exp_avg_sq"][0]), hv[k]), (where, step, k)
                for j in range(1, rep):
                    for key in ("params", "exp_avg", "exp_avg_sq"):
                        assert torch.equal(t[key][j].view(torch.int32),
                                           t[key][0].view(torch.int32)), (where, step, k, key)
