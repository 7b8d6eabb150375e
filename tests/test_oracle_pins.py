"""Pins for the CPU oracle: each check ties it to something other than itself.

Collectives (ruCCL README §2, §5; Monarch "Struct Communicator"):
  * the pages' worked example (4 ranks, 257 FP32, sum and mean, inputs kept),
    exact on integer-valued inputs, within the fp32 bound on uniform inputs;
  * exact rational sums (fractions) and correctly rounded quotients;
  * hand-derived rounding cases that fix the rank order of the fold;
  * numpy's max/min on finite data, hand cases for NaN and signed zeros;
  * torch's CPU bf16 conversion for the fp32 -> bf16 rounding;
  * exact nearest-even rounding (fractions) for fp64 -> bf16;
  * collective identities (reduce_scatter concatenated == all_reduce, ...);
  * brute force on tiny R and N.
"""
import json
import math
import os
import struct
from fractions import Fraction

import numpy as np
import pytest
import torch

from gradient_sync_rcc_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
U24 = 2.0 ** -24


def f32(x):
    return np.float32(x)


def bits32(x):
    return struct.unpack("<I", struct.pack("<f", float(x)))[0]


# ----------------------------------------------------------- page example

def test_page_example_integer_variant_exact(orc):
    spec = json.load(open(os.path.join(GOLDEN, "page_example.json")))
    R, N = spec["ranks"], spec["elements"]
    xs = synth.rank_buffers("int", R, N, 1, 0)
    before = [x.copy() for x in xs]
    s = orc.all_reduce(xs, "sum")
    m = orc.all_reduce(xs, "mean")
    exact = [sum(int(x[i]) for x in xs) for i in range(N)]
    for r in range(R):
        assert [int(v) for v in s[r]] == exact
        assert [Fraction(float(v)) for v in m[r]] == [Fraction(e, R) for e in exact]
    if spec["inputs_unchanged"]:
        for a, b in zip(xs, before):
            assert a.tobytes() == b.tobytes()


def test_page_example_uniform_within_bound(orc):
    spec = json.load(open(os.path.join(GOLDEN, "page_example.json")))
    R, N = spec["ranks"], spec["elements"]
    xs = synth.rank_buffers("uniform", R, N, 1, 1)
    before = [x.copy() for x in xs]
    s = orc.all_reduce(xs, "sum")[0]
    m = orc.all_reduce(xs, "mean")[0]
    for i in range(N):
        exact = sum(Fraction(float(x[i])) for x in xs)
        scale = sum(abs(Fraction(float(x[i]))) for x in xs)
        bound = R * Fraction(2) ** -23 * scale
        assert abs(Fraction(float(s[i])) - exact) <= bound
        assert abs(Fraction(float(m[i])) - exact / R) <= bound / R
    # values on the 2^-23 grid with |sum| < 4 need at most 25 bits: the fp64 path is exact
    d = orc.reduce_f64(xs, "sum")
    for i in range(N):
        assert Fraction(float(d[i])) == sum(Fraction(float(x[i])) for x in xs)
    for a, b in zip(xs, before):
        assert a.tobytes() == b.tobytes()


# ----------------------------------------------------------- rank order

def test_rank_order_fixes_rounding(orc):
    one, tiny = f32(1.0), f32(U24)
    # left fold: (1 + 2^-24) ties to 1, again to 1
    fwd = orc.reduce_f32([np.array([one]), np.array([tiny]), np.array([tiny])], "sum")
    assert fwd[0] == f32(1.0)
    # reversed ranks: 2^-24 + 2^-24 = 2^-23 exactly, then 1 + 2^-23 is representable
    rev = orc.reduce_f32([np.array([tiny]), np.array([tiny]), np.array([one])], "sum")
    assert rev[0] == f32(1.0 + 2.0 ** -23)
    # four ranks: a pairwise tree would give 1 + 2^-23; the left fold gives 1
    four = orc.reduce_f32([np.array([one])] + [np.array([tiny])] * 3, "sum")
    assert four[0] == f32(1.0)


def test_mean_is_one_ieee_division(orc):
    R = 3
    xs = synth.rank_buffers("uniform", R, 4096, 2, 0)
    s = orc.reduce_f32(xs, "sum")
    m = orc.reduce_f32(xs, "mean")
    # fp64 quotient rounded to fp32 is the correctly rounded fp32 quotient
    # (53 >= 2*24 + 2), an independent route to fl32(sum / 3)
    want = (s.astype(np.float64) / 3.0).astype(np.float32)
    assert m.tobytes() == want.tobytes()
    # and it is not the reciprocal multiply on every element
    recip = s * np.float32(1.0 / 3.0)
    assert np.any(recip != m)


# ----------------------------------------------------------- max / min

def test_max_min_vs_numpy(orc):
    for R in (1, 2, 3, 5, 8):
        xs = synth.rank_buffers("grad", R, 3000, 3, R)
        stack = np.stack(xs)
        assert orc.reduce_f32(xs, "max").tobytes() == stack.max(0).tobytes()
        assert orc.reduce_f32(xs, "min").tobytes() == stack.min(0).tobytes()


def test_max_min_special_values(orc):
    nan, inf = np.float32(np.nan), np.float32(np.inf)

    def red(vals, op):
        return orc.reduce_f32([np.array([v], np.float32) for v in vals], op)[0]

    for op in ("max", "min"):
        assert bits32(red([1.0, nan, 2.0], op)) == 0x7FC00000
        assert bits32(red([nan, 1.0], op)) == 0x7FC00000
    # signed zeros compare equal: the lowest rank's value is kept
    assert bits32(red([-0.0, 0.0], "max")) == 0x80000000
    assert bits32(red([0.0, -0.0], "max")) == 0x00000000
    assert bits32(red([-0.0, 0.0], "min")) == 0x80000000
    assert red([-inf, 1.0], "max") == 1.0
    assert red([inf, 1.0], "min") == 1.0
    assert red([-inf, -inf], "max") == -inf


# ----------------------------------------------------------- special values, fp64 path

def test_sum_special_values(orc):
    inf = np.float32(np.inf)
    fmax = np.finfo(np.float32).max

    def s32(vals):
        return orc.reduce_f32([np.array([v], np.float32) for v in vals], "sum")[0]

    def s64(vals):
        return orc.reduce_f64([np.array([v], np.float32) for v in vals], "sum")[0]

    assert s32([inf, 1.0]) == inf
    assert np.isnan(s32([inf, -inf]))
    assert s32([fmax, fmax]) == inf                       # fp32 overflow
    assert s64([fmax, fmax]) == 2.0 * float(fmax)         # fp64 does not
    sub = np.array([1], np.uint32).view(np.float32)[0]   # smallest subnormal 2^-149
    assert bits32(s32([sub, sub])) == 2                   # 2^-148 exactly
    assert s32([sub, -sub]) == 0.0


def test_f64_path_exact_on_grid(orc):
    for R in (2, 5, 8):
        xs = synth.rank_buffers("uniform", R, 500, 4, R)
        d = orc.reduce_f64(xs, "sum")
        for i in range(0, 500, 7):
            assert Fraction(float(d[i])) == sum(Fraction(float(x[i])) for x in xs)
        dm = orc.reduce_f64(xs, "mean")
        for i in range(0, 500, 11):
            exact = sum(Fraction(float(x[i])) for x in xs) / R
            assert abs(Fraction(float(dm[i])) - exact) <= abs(exact) * Fraction(2) ** -53


def test_fp32_error_bound_gradient_like(orc):
    for R in (2, 4, 8):
        xs = synth.rank_buffers("grad", R, 20000, 5, R)
        s = orc.reduce_f32(xs, "sum").astype(np.float64)
        d = orc.reduce_f64(xs, "sum")
        a = orc.abs_sum_f64(xs)
        assert np.all(np.abs(s - d) <= R * 2.0 ** -23 * a)
        ab = np.sum(np.abs(np.stack(xs).astype(np.float64)), axis=0)
        assert np.allclose(a, ab, rtol=1e-15, atol=0)


# ----------------------------------------------------------- bf16 rounding

def test_f32_to_bf16_matches_torch(orc):
    g = synth.rng(6)
    patterns = g.integers(0, 1 << 32, size=1 << 20, dtype=np.uint64).astype(np.uint32)
    # every exponent with the tie pattern (low half exactly 0x8000), odd and even kept bits
    ties = []
    for e in range(256):
        for hi in (0, 1, 2, 3, 0x7F):
            for lo in (0x8000, 0x7FFF, 0x8001, 0):
                for s in (0, 1):
                    ties.append((s << 31) | (e << 23) | (hi << 16) | lo)
    patterns = np.concatenate([patterns, np.array(ties, np.uint32)])
    x = patterns.view(np.float32)
    ours = orc.f32_to_bf16(x)
    ref = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    isnan = np.isnan(x)
    assert np.array_equal(ours[~isnan], ref[~isnan])
    # NaN stays NaN (quiet)
    back = orc.bf16_to_f32(ours[isnan])
    assert np.all(np.isnan(back))


def _exact_bf16_round(d: float) -> float:
    """Nearest bf16 value to d with ties to even, by exhaustive comparison."""
    if d == 0:
        return d
    fr = Fraction(d)
    a = abs(fr)
    e = math.frexp(abs(d))[1]           # a in [2^(e-1), 2^e)
    q = max(e - 8, -133)
    ulp = Fraction(2) ** q
    lo = (a / ulp).__floor__() * ulp
    hi = lo + ulp
    if a - lo < hi - a:
        r = lo
    elif a - lo > hi - a:
        r = hi
    else:
        r = lo if (lo / ulp) % 2 == 0 else hi
    if r >= Fraction(2) ** 128:
        return math.copysign(math.inf, d)
    return math.copysign(float(r), d)


def test_f64_to_bf16_single_rounding(orc):
    g = synth.rng(7)
    vals = list(g.standard_normal(2000) * np.exp(g.uniform(-60, 60, 2000)))
    # cases where rounding through fp32 first would land on a tie and go the other way
    vals += [1.0 + 2.0 ** -8 + 2.0 ** -40, -(1.0 + 2.0 ** -8 + 2.0 ** -40),
             1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, 2.0 ** -130 + 2.0 ** -134,
             3.3895313892515355e38, 3.39e38, 1e-45, 5e-41]
    x = np.array(vals, np.float64)
    ours = orc.f64_to_bf16(x)
    for v, b in zip(vals, ours):
        got = float(orc.bf16_to_f32(np.array([b], np.uint16))[0])
        assert got == _exact_bf16_round(v), (v, got)


def test_bf16_reduce_vs_torch_and_f64(orc):
    for R in (2, 3, 8):
        xs = synth.rank_buffers("bf16_normal", R, 5000, 8, R)
        ours = orc.reduce_bf16(xs, "sum")
        # torch CPU: widen, add rank by rank in fp32, one conversion to bf16
        ts = [torch.from_numpy(x.view(np.int16).copy()).view(torch.bfloat16).float() for x in xs]
        acc = ts[0].clone()
        for t in ts[1:]:
            acc = acc + t
        ref = acc.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(ours, ref)
        # within one bf16 ulp of the fp64 result rounded once
        d = orc.reduce_bf16_f64(xs, "sum")
        r64 = orc.f64_to_bf16(d)

        def ordered(b):
            b = b.astype(np.int32)
            return np.where(b & 0x8000, -(b & 0x7FFF), b)
        assert np.max(np.abs(ordered(ours) - ordered(r64))) <= 1
        # max/min are a choice among the inputs
        stack = np.stack([orc.bf16_to_f32(x) for x in xs])
        assert np.array_equal(orc.bf16_to_f32(orc.reduce_bf16(xs, "max")), stack.max(0))
        assert np.array_equal(orc.bf16_to_f32(orc.reduce_bf16(xs, "min")), stack.min(0))


# ----------------------------------------------------------- collective identities

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("R", [1, 2, 3, 4, 8])
def test_collective_identities(orc, dtype, R):
    n = R * 37
    xs = (synth.rank_buffers("uniform", R, n, 9, R) if dtype == "f32"
          else synth.rank_buffers("bf16_uniform", R, n, 9, R))
    before = [x.copy() for x in xs]
    for op in ("sum", "mean", "max", "min"):
        ar = orc.all_reduce(xs, op)
        for r in range(1, R):
            assert ar[r].tobytes() == ar[0].tobytes()
        rs = orc.reduce_scatter(xs, op)
        assert np.concatenate(rs).tobytes() == ar[0].tobytes()
        ag = orc.all_gather(rs)
        for r in range(R):
            assert ag[r].tobytes() == ar[r].tobytes()
        root = R - 1
        out = [np.full_like(x, 7) for x in xs]
        orc.reduce(xs, op, out[root])
        assert out[root].tobytes() == ar[0].tobytes()
        for r in range(R):
            if r != root:
                assert np.all(out[r] == 7)
    for root in range(R):
        outs = [np.zeros_like(xs[0]) for _ in range(R)]
        orc.broadcast(xs[root], outs)
        for o in outs:
            assert o.tobytes() == xs[root].tobytes()
    if R & (R - 1) == 0:
        s = orc.all_reduce(xs, "sum")[0]
        m = orc.all_reduce(xs, "mean")[0]
        if dtype == "f32":
            assert m.tobytes() == (s / np.float32(R)).astype(np.float32).tobytes()
    for a, b in zip(xs, before):
        assert a.tobytes() == b.tobytes()


@pytest.mark.parametrize("R", [1, 2, 3, 5, 8])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_all_to_all_is_a_block_transpose(orc, R, dtype):
    """Monarch all_to_all_single with equal splits: viewing rank q's buffer as
    R chunks, out[r] chunk q = in[q] chunk r, i.e. numpy's transpose of the
    (rank, chunk) axes; applying it twice gives the input back."""
    n = 41
    kind = "uniform" if dtype == "f32" else "bf16_uniform"
    xs = synth.rank_buffers(kind, R, R * n, 26, R)
    out = orc.all_to_all(xs)
    X = np.stack(xs).reshape(R, R, n)
    want = np.transpose(X, (1, 0, 2)).reshape(R, R * n)
    for r in range(R):
        assert out[r].tobytes() == want[r].tobytes()
    back = orc.all_to_all(out)
    for a, b in zip(back, xs):
        assert a.tobytes() == b.tobytes()


def test_all_reduce_in_place(orc):
    xs = synth.rank_buffers("uniform", 4, 100, 10, 0)
    copy = [x.copy() for x in xs]
    want = orc.all_reduce(copy, "sum")
    orc.all_reduce(xs, "sum", out=xs)
    for a, b in zip(xs, want):
        assert a.tobytes() == b.tobytes()


@pytest.mark.parametrize("R", [1, 2, 3, 5, 8])
@pytest.mark.parametrize("N", [0, 1, 3, 4, 5, 7, 8, 9, 31, 33])
def test_brute_force_tiny(orc, R, N):
    xs = synth.rank_buffers("grad", R, N, 11, R, N)
    if N == 0:
        out = orc.all_reduce(xs, "sum")
        assert all(o.size == 0 for o in out)
        return
    if R == 1:
        for op in ("sum", "mean", "max", "min"):
            assert orc.all_reduce(xs, op)[0].tobytes() == xs[0].tobytes()
    s = orc.all_reduce(xs, "sum")[0]
    m = orc.all_reduce(xs, "mean")[0]
    mx = orc.all_reduce(xs, "max")[0]
    mn = orc.all_reduce(xs, "min")[0]
    for i in range(N):
        col = [Fraction(float(x[i])) for x in xs]
        exact = sum(col)
        bound = R * Fraction(2) ** -23 * sum(abs(c) for c in col)
        assert abs(Fraction(float(s[i])) - exact) <= bound
        assert abs(Fraction(float(m[i])) - exact / R) <= bound / R
        assert Fraction(float(mx[i])) == max(col)
        assert Fraction(float(mn[i])) == min(col)


# ----------------------------------------------------------- gradient sync + AdamW

LR, B1, B2, EPS, WD = 1e-3, 0.9, 0.999, 1e-8, 0.01


def test_mean_unscale_exact_on_integers(orc):
    R, S = 4, 65536.0
    ints = [synth.int_pm1000(999, 12, r) for r in range(R)]
    grads = [(x * np.float32(S)).astype(np.float32) for x in ints]
    g = orc.mean_unscale(grads, np.float32(1.0 / S))
    for i in range(999):
        exact = sum(Fraction(int(x[i])) for x in ints) / R
        assert Fraction(float(g[i])) == exact


def test_stats_vs_fsum(orc):
    g = synth.normal(50000, 5e-4, 13)
    g[17] = np.nan
    g[99] = np.inf
    st = orc.stats_accumulate(orc.stats_new(), g)
    finite = g[np.isfinite(g)]
    want = math.fsum(float(v) * float(v) for v in finite)
    assert abs(orc.stats_value(st) - want) <= 4e-16 * want
    assert st.nonfinite == 2 and st.count == g.size


def test_clip_decision(orc):
    g = np.array([0.75, 1.0], np.float32)         # norm exactly 1.25
    st = orc.stats_accumulate(orc.stats_new(), g)
    d = orc.decide(st, 1.25)
    assert d.norm == 1.25 and d.skip == 0 and d.clip_coef == 1.0   # not clipped at equality
    d = orc.decide(st, 2.0)
    assert d.clip_coef == 1.0
    d = orc.decide(st, 1.0)
    assert d.clip_coef == np.float32(0.8)
    d = orc.decide(st, 0.0)                        # no clipping configured
    assert d.clip_coef == 1.0
    # after clipping the global norm equals max_grad_norm
    big = synth.normal(10000, 1.0, 14)
    st = orc.stats_accumulate(orc.stats_new(), big)
    d = orc.decide(st, 1.0)
    clipped = big.astype(np.float64) * float(d.clip_coef)
    assert abs(math.sqrt(math.fsum(clipped * clipped)) - 1.0) < 1e-6
    bad = np.array([1.0, np.nan], np.float32)
    d = orc.decide(orc.stats_accumulate(orc.stats_new(), bad), 1.0)
    assert d.skip == 1


def test_adamw_constant_gradient_closed_form(orc):
    """With a constant gradient the bias-corrected moments are g and g^2 at
    every step, so p_t = a p_{t-1} - c with a = 1 - lr*wd, c = lr*g/(|g|+eps):
    p_t = a^t p_0 - c (1 - a^t) / (1 - a)."""
    n = 64
    g = synth.normal(n, 1e-3, 15)
    p0 = synth.normal(n, 0.02, 16)
    p, m, v = p0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    for t in range(1, 11):
        s = orc.adamw_scalars(LR, B1, B2, EPS, WD, t)
        orc.adamw_update(g, 1.0, s, p, m, v)
        a = 1.0 - LR * WD
        gd = g.astype(np.float64)
        c = LR * gd / (np.abs(gd) + EPS)
        want = a ** t * p0.astype(np.float64) - c * (1 - a ** t) / (1 - a)
        # fp32 against exact: each step rounds p about 4 times (decay, quotient,
        # product, difference), so allow t * 4 half-ulps of |p| plus a little
        # for the moments' own rounding
        tol = t * 4 * 2.0 ** -24 * np.maximum(np.abs(want), 1e-3) + 1e-10
        assert np.all(np.abs(p - want) <= tol), t


def test_adamw_two_distinct_gradients_closed_form(orc):
    """m^_2 = (b1 g1 + g2)/(1 + b1), v^_2 = (b2 g1^2 + g2^2)/(1 + b2)."""
    n = 64
    g1 = synth.normal(n, 1e-3, 17)
    g2 = synth.normal(n, 1e-3, 18)
    p0 = synth.normal(n, 0.02, 19)
    p, m, v = p0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    orc.adamw_update(g1, 1.0, orc.adamw_scalars(LR, B1, B2, EPS, WD, 1), p, m, v)
    orc.adamw_update(g2, 1.0, orc.adamw_scalars(LR, B1, B2, EPS, WD, 2), p, m, v)
    a = 1.0 - LR * WD
    G1, G2, P0 = (x.astype(np.float64) for x in (g1, g2, p0))
    p1 = a * P0 - LR * G1 / (np.abs(G1) + EPS)
    mh = (B1 * G1 + G2) / (1 + B1)
    vh = (B2 * G1 * G1 + G2 * G2) / (1 + B2)
    p2 = a * p1 - LR * mh / (np.sqrt(vh) + EPS)
    assert np.all(np.abs(p - p2) <= 1e-6 * np.maximum(np.abs(p2), 1e-3))
    assert np.allclose(m, (1 - B1) * (B1 * G1 + G2), rtol=1e-6, atol=0)
    assert np.allclose(v, (1 - B2) * (B2 * G1 * G1 + G2 * G2), rtol=1e-6, atol=0)


def test_adamw_first_step_with_clip(orc):
    n = 256
    g = synth.normal(n, 1e-3, 20)
    p0 = synth.normal(n, 0.02, 21)
    p, m, v = p0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    coef = np.float32(0.25)
    orc.adamw_update(g, coef, orc.adamw_scalars(LR, B1, B2, EPS, WD, 1), p, m, v)
    gp = g.astype(np.float64) * float(coef)
    want = (1 - LR * WD) * p0.astype(np.float64) - LR * gp / (np.abs(gp) + EPS)
    assert np.all(np.abs(p - want) <= 1e-6 * np.maximum(np.abs(want), 1e-3))


def _small_problem(R=4, P=6, seed=22):
    sizes = synth.param_sizes(P, 16, 2048, seed)
    params = [synth.normal(n, 0.02, seed, 1, i) for i, n in enumerate(sizes)]
    return R, sizes, params


def _grads(R, sizes, step, scale, seed, nan_at=None):
    grads = []
    for i, n in enumerate(sizes):
        per = [(synth.normal(n, 1e-3, seed, 2, i, step, r) * np.float32(scale)).astype(np.float32)
               for r in range(R)]
        grads.append(per)
    if nan_at is not None and step == nan_at:
        grads[0][0][0] = np.nan
    return grads


def test_skip_on_nonfinite_and_scaler(orc):
    R, sizes, params = _small_problem()
    m = [np.zeros_like(p) for p in params]
    v = [np.zeros_like(p) for p in params]
    sc = orc.scaler_new(65536.0)
    step = 0
    for k in range(1, 11):
        grads = _grads(R, sizes, k, sc.scale, 23, nan_at=7)
        snap = [a.copy() for a in params + m + v]
        scale_before = sc.scale
        step_before = step
        step, st, d = orc.grad_sync_adamw_step(grads, params, m, v, lr=LR, beta1=B1, beta2=B2,
                                               eps=EPS, weight_decay=WD, max_grad_norm=1.0,
                                               step=step, scaler=sc)
        if k == 7:
            assert d.skip == 1 and st.nonfinite == 1
            assert step == step_before
            for a, b in zip(params + m + v, snap):
                assert a.tobytes() == b.tobytes()
            assert sc.scale == scale_before * 0.5 and sc.growth_tracker == 0
        else:
            assert d.skip == 0 and step == step_before + 1
    assert step == 9 and sc.scale == 32768.0


def test_scaler_growth_interval(orc):
    sc = orc.scaler_new(1024.0, growth_interval=3)
    for _ in range(2):
        orc.scaler_update(sc, False)
    assert sc.scale == 1024.0 and sc.growth_tracker == 2
    orc.scaler_update(sc, False)
    assert sc.scale == 2048.0 and sc.growth_tracker == 0
    orc.scaler_update(sc, True)
    assert sc.scale == 1024.0 and sc.growth_tracker == 0


def test_clip_applies_after_unscale(orc):
    """Scaled gradients have a huge norm; unscaled ones have norm < max_norm,
    so no clipping may happen."""
    R, S = 2, 65536.0
    g = np.full(4, 0.125, np.float32)            # unscaled mean norm = 0.25
    grads = [[(g * np.float32(S)).astype(np.float32) for _ in range(R)]]
    p = [np.ones(4, np.float32)]
    m = [np.zeros(4, np.float32)]
    v = [np.zeros(4, np.float32)]
    sc = orc.scaler_new(S)
    step, st, d = orc.grad_sync_adamw_step(grads, p, m, v, lr=LR, beta1=B1, beta2=B2, eps=EPS,
                                           weight_decay=WD, max_grad_norm=1.0, step=0, scaler=sc)
    assert d.skip == 0 and d.clip_coef == 1.0 and d.norm == 0.25
    assert orc.stats_value(st) == 0.0625


def test_full_step_matches_piecewise_closed_form(orc):
    """First step of the full driver: every element obeys the first-step closed
    form with the clip coefficient computed from the global norm."""
    R, sizes, params = _small_problem(P=5, seed=24)
    p0 = [p.copy() for p in params]
    m = [np.zeros_like(p) for p in params]
    v = [np.zeros_like(p) for p in params]
    sc = orc.scaler_new(65536.0)
    grads = _grads(R, sizes, 1, sc.scale, 25)
    # unscaled mean gradients in fp64 (exact here: powers of two, fp32 sums of 4)
    means = [np.sum(np.stack(gs).astype(np.float64), axis=0) / R / 65536.0 for gs in grads]
    norm = math.sqrt(math.fsum(float(x) ** 2 for g in means for x in g))
    step, st, d = orc.grad_sync_adamw_step(grads, params, m, v, lr=LR, beta1=B1, beta2=B2,
                                           eps=EPS, weight_decay=WD, max_grad_norm=1e-3,
                                           step=0, scaler=sc)
    assert abs(d.norm - norm) <= 1e-6 * norm
    assert d.clip_coef == np.float32(1e-3 / d.norm)
    for pp, q0, g in zip(params, p0, means):
        gp = g * float(d.clip_coef)
        want = (1 - LR * WD) * q0.astype(np.float64) - LR * gp / (np.abs(gp) + EPS)
        assert np.all(np.abs(pp - want) <= 1e-6 * np.maximum(np.abs(want), 1e-3))


# ----------------------------------------------------------- the 12-byte report

def test_report_pack_layout(orc):
    """The report read back before the update (RUDA docs "Training and saving
    state", native PyTorch section) is fixed by the page only in size: 12 bytes.
    This build reads it as the fp64 sum of squares followed by the u32 count of
    non-finite gradients, little-endian, with the count saturated at 2^32 - 1
    (any non-zero count skips the step either way).  Pinned against the byte
    layout that struct.pack writes for "<dI" and against hand-decoded words."""
    cases = [(1.25, 0.0, 3), (math.pi, 0.0, 0), (1.0, 0.5, 7), (5e-324, 0.0, 1),
             (float("inf"), 0.0, 2 ** 32 - 1), (12345.678, -0.078, 65536)]
    for total, comp, nonfinite in cases:
        st = orc.Stats(total, comp, nonfinite, 0)
        want = list(struct.unpack("<3I", struct.pack("<dI", total + comp, nonfinite)))
        assert orc.report_pack(st) == want, (total, comp, nonfinite)
    # hand-decoded: 1.25 = 0x3FF4000000000000; pi = 0x400921FB54442D18
    assert orc.report_pack(orc.Stats(1.25, 0.0, 3, 0)) == [0x00000000, 0x3FF40000, 3]
    assert orc.report_pack(orc.Stats(math.pi, 0.0, 9, 0)) == [0x54442D18, 0x400921FB, 9]
    # the value packed is the compensated sum (sum + compensation)
    assert orc.report_pack(orc.Stats(1.0, 0.5, 0, 0))[:2] == [0x00000000, 0x3FF80000]
    # counts beyond 32 bits saturate instead of wrapping to a small (or zero) count
    assert orc.report_pack(orc.Stats(1.0, 0.0, 2 ** 33, 0))[2] == 0xFFFFFFFF
    assert orc.report_pack(orc.Stats(1.0, 0.0, 2 ** 32 + 5, 0))[2] == 0xFFFFFFFF
