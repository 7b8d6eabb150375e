"""GPU parity of the five collectives against the CPU oracle, through the C ABI.

Workloads follow the pages' example and the sizes the benchmark uses:
  * 4 logical ranks, 257 FP32 elements, sum and mean, inputs unchanged, the
    session closed afterwards (ruCCL README §5 "CUDA example");
  * 8 ranks x 2^24 FP32 gradient-like values, sum/mean/max in deterministic
    and fast modes (the benchmark's workload, checked in full);
  * reduce_scatter then all_gather of 8 x 2^26 bf16 values with fp32
    accumulation (Monarch reduce_scatter_tensor / all_gather_into_tensor);
  * a size sweep R in {2,4,8}, N = 257*4^k up to 2^28: all_reduce mean (fp32,
    bf16), broadcast from root 0, reduce to root R-1;
  * edge cases: empty, ragged and misaligned buffers, R = 1 and R beyond the
    specialised counts, in-place forms, NaN/Inf/signed zeros.
Acceptance: deterministic mode and max/min bit-exact; integer-valued fp32
bit-exact in every mode; fp32 sum/mean within R 2^-23 sum|x| of fp64 (the mean
bound divided by R); bf16 within one bf16 ulp of the fp64 result rounded once.
"""
import math

import numpy as np
import pytest
import torch

from gradient_sync_rcc_gb300 import rcc, synth
from gpu_util import (DEV, Guarded, bits_equal, session, tdtype, to_dev, to_host,
                      within_fp32_bound, within_one_bf16_ulp)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gradient_sync_rcc_gb300 import build
    build.build()
    assert torch.cuda.is_available()


def host_ranks(kind, R, n, *key):
    return synth.rank_buffers(kind, R, n, *key)


# ---------------------------------------------------------------- page example

@pytest.mark.parametrize("kind", ["uniform", "int"])
@pytest.mark.parametrize("det", [True, False])
def test_page_example_4_ranks_257_fp32(orc, kind, det):
    R, N = 4, 257
    xs = host_ranks(kind, R, N, 100, 0 if kind == "uniform" else 1)
    ins = [Guarded(N, torch.float32, fill=to_dev(x)) for x in xs]
    before = [to_host(g.t) for g in ins]
    for op in ("sum", "mean"):
        outs = [Guarded(N, torch.float32) for _ in range(R)]
        with session(R, rcc.F32, det) as h:
            rcc.all_reduce(h, [g.t for g in ins], [o.t for o in outs], op)
            torch.cuda.synchronize()
        got = [to_host(o.t) for o in outs]
        want = orc.all_reduce(xs, op)
        for r in range(R):
            assert bits_equal(got[r], got[0])
            assert outs[r].guards_intact()
        if det or kind == "int":
            assert bits_equal(got[0], want[0])
        else:
            ok, worst = within_fp32_bound(orc, got[0], xs, op)
            assert ok, worst
    for g, b in zip(ins, before):
        assert bits_equal(to_host(g.t), b)       # inputs unchanged
        assert g.guards_intact()


def test_session_closed_after_example():
    with session(4) as h:
        pass
    with pytest.raises(rcc.RccError) as ei:
        rcc.reset(h)
    assert ei.value.status == rcc.ERR_MISSING_REGISTRATION


# ---------------------------------------------------------------- 8 x 2^24 fp32

@pytest.fixture(scope="module")
def cfg_8x2p24():
    R, N = 8, 1 << 24
    xs = host_ranks("grad", R, N, 200)
    dev = [to_dev(x) for x in xs]
    return xs, dev


@pytest.mark.parametrize("op", ["sum", "mean", "max"])
@pytest.mark.parametrize("det", [True, False])
def test_all_reduce_8_ranks_2p24(orc, cfg_8x2p24, op, det):
    xs, dev = cfg_8x2p24
    R, N = len(xs), xs[0].size
    outs = [torch.empty(N, dtype=torch.float32, device=DEV) for _ in range(R)]
    with session(R, rcc.F32, det) as h:
        rcc.all_reduce(h, dev, outs, op)
        torch.cuda.synchronize()
    for r in range(1, R):
        assert torch.equal(outs[r].view(torch.int32), outs[0].view(torch.int32))
    got = to_host(outs[0])
    if det or op == "max":
        assert bits_equal(got, orc.reduce_f32(xs, op))
    else:
        ok, worst = within_fp32_bound(orc, got, xs, op)
        assert ok, worst


# ---------------------------------------------------------------- RS -> AG, 8 x 2^26 bf16

@pytest.mark.parametrize("det", [True, False])
def test_reduce_scatter_all_gather_8_ranks_2p26_bf16(orc, det):
    R, N = 8, 1 << 26
    n = N // R
    dev = synth.gpu_rank_buffers("normal1", R, N, torch.bfloat16, (300,), DEV)
    rs = [torch.empty(n, dtype=torch.bfloat16, device=DEV) for _ in range(R)]
    ag = [torch.empty(N, dtype=torch.bfloat16, device=DEV) for _ in range(R)]
    ar = [torch.empty(N, dtype=torch.bfloat16, device=DEV) for _ in range(R)]
    with session(R, rcc.BF16, det) as h:
        rcc.reduce_scatter(h, dev, rs, "sum")
        rcc.all_gather(h, rs, ag)
        rcc.all_reduce(h, dev, ar, "sum")
        torch.cuda.synchronize()
    # all_gather of reduce_scatter == all_reduce, bitwise, on every rank
    for r in range(R):
        assert torch.equal(ag[r].view(torch.int16), ar[r].view(torch.int16))
        assert torch.equal(torch.cat(rs).view(torch.int16), ar[r].view(torch.int16))
    xs = [to_host(x) for x in dev]
    got = np.concatenate([to_host(x) for x in rs])
    if det:
        want = np.concatenate(orc.reduce_scatter(xs, "sum"))
        assert bits_equal(got, want)
    ok, loose = within_one_bf16_ulp(orc, got, xs, "sum")
    assert ok
    # Elements held to the accumulation bound instead of one ulp.  An element
    # is held so only if R 2^-24 sum|x| > ulp(y)/2, and ulp(y) > |y| 2^-8, so
    # only if |y| < 2^-12 sum|x|.  For R independent N(0,1) inputs y ~ N(0, R)
    # (density at most 1/sqrt(2 pi R)) and E sum|x| = R sqrt(2/pi), so the
    # expected fraction is at most p = 2 R sqrt(2/pi) 2^-12 / sqrt(2 pi R),
    # 4.4e-4 at R = 8 (a CPU draw of 2^22 elements gave 1.2e-4).  Allow six
    # binomial standard deviations above p N.
    p = 2 * R * math.sqrt(2 / math.pi) * 2.0 ** -12 / math.sqrt(2 * math.pi * R)
    assert loose <= p * N + 6 * math.sqrt(p * N), (loose, p * N)


# ---------------------------------------------------------------- size sweep

SWEEP_N = [257 * 4 ** k for k in range(10)] + [1 << 28]
FULL_CHECK_MAX = 257 * 4 ** 6        # the oracle checks every element up to here


def _sample_idx(N, key):
    if N <= FULL_CHECK_MAX:
        return None
    g = synth.rng(*key)
    idx = np.unique(np.concatenate([np.arange(4096), np.arange(N - 4096, N),
                                    g.integers(0, N, 65536)]))
    return torch.from_numpy(idx).to(DEV)


def _cols(ts, idx):
    return [to_host(t if idx is None else t[idx]) for t in ts]


@pytest.mark.parametrize("R", [2, 4, 8])
@pytest.mark.parametrize("N", SWEEP_N)
@pytest.mark.parametrize("dtype", [rcc.F32, rcc.BF16])
def test_sweep_all_reduce_mean(orc, R, N, dtype):
    td = tdtype(dtype)
    dev = synth.gpu_rank_buffers("uniform", R, N, td, (400, R, N), DEV)
    outs = [torch.empty(N, dtype=td, device=DEV) for _ in range(R)]
    with session(R, dtype, True) as h:
        rcc.all_reduce(h, dev, outs, "mean")
        torch.cuda.synchronize()
    for r in range(1, R):
        assert torch.equal(outs[r].view(torch.int16 if dtype else torch.int32),
                           outs[0].view(torch.int16 if dtype else torch.int32))
    idx = _sample_idx(N, (401, R, N))
    xs = _cols(dev, idx)
    got = _cols([outs[0]], idx)[0]
    if dtype == rcc.F32:
        assert bits_equal(got, orc.reduce_f32(xs, "mean"))
        ok, worst = within_fp32_bound(orc, got, xs, "mean")
        assert ok, worst
    else:
        assert bits_equal(got, orc.reduce_bf16(xs, "mean"))
        ok, _ = within_one_bf16_ulp(orc, got, xs, "mean")
        assert ok
    del dev, outs
    torch.cuda.empty_cache()


@pytest.mark.parametrize("R", [2, 4, 8])
@pytest.mark.parametrize("N", SWEEP_N)
def test_sweep_broadcast_root0_reduce_rootlast(orc, R, N):
    dev = synth.gpu_rank_buffers("uniform", R, N, torch.float32, (500, R, N), DEV)
    outs = [torch.full((N,), 7.0, dtype=torch.float32, device=DEV) for _ in range(R)]
    red = [torch.full((N,), -3.0, dtype=torch.float32, device=DEV) for _ in range(R)]
    with session(R, rcc.F32, True) as h:
        rcc.broadcast(h, dev[0], outs, root=0)
        rcc.reduce(h, dev, red[R - 1], root=R - 1, op="sum")
        torch.cuda.synchronize()
    for r in range(R):
        assert torch.equal(outs[r].view(torch.int32), dev[0].view(torch.int32))
    for r in range(R - 1):
        assert bool(torch.all(red[r] == -3.0))      # non-roots untouched
    idx = _sample_idx(N, (501, R, N))
    xs = _cols(dev, idx)
    assert bits_equal(_cols([red[R - 1]], idx)[0], orc.reduce_f32(xs, "sum"))
    del dev, outs, red
    torch.cuda.empty_cache()


# ---------------------------------------------------------------- edge cases

RAGGED = [1, 2, 3, 5, 7, 255, 257, 1023, 4097, 65537]


@pytest.mark.parametrize("R", [1, 2, 3, 5, 7, 8, 12, 64])
@pytest.mark.parametrize("dtype", [rcc.F32, rcc.BF16])
def test_ragged_and_rank_counts(orc, R, dtype):
    td = tdtype(dtype)
    for N in RAGGED:
        kind = "uniform" if dtype == rcc.F32 else "bf16_uniform"
        xs = host_ranks(kind, R, N, 600, R, N)
        ins = [to_dev(x) for x in xs]
        for op in ("sum", "mean", "max", "min"):
            for det in (True, False):
                outs = [Guarded(N, td) for _ in range(R)]
                with session(R, dtype, det) as h:
                    rcc.all_reduce(h, ins, [o.t for o in outs], op)
                    torch.cuda.synchronize()
                got = [to_host(o.t) for o in outs]
                for r in range(R):
                    assert outs[r].guards_intact()
                    assert bits_equal(got[r], got[0])
                if dtype == rcc.F32:
                    if det or op in ("max", "min") or R <= 3:
                        assert bits_equal(got[0], orc.reduce_f32(xs, op)), (N, op, det)
                    else:
                        assert within_fp32_bound(orc, got[0], xs, op)[0]
                else:
                    if det or op in ("max", "min") or R <= 3:
                        assert bits_equal(got[0], orc.reduce_bf16(xs, op)), (N, op, det)
                    assert within_one_bf16_ulp(orc, got[0], xs, op)[0]


@pytest.mark.parametrize("dtype", [rcc.F32, rcc.BF16])
def test_misaligned_views(orc, dtype):
    """Buffers shifted off 16-byte alignment take the scalar path."""
    td = tdtype(dtype)
    R, N = 4, 5000
    kind = "uniform" if dtype == rcc.F32 else "bf16_uniform"
    xs = host_ranks(kind, R, N, 700)
    for offs in ([1, 1, 1, 1], [0, 1, 2, 3], [0, 0, 0, 1]):
        ins = [Guarded(N, td, offset_elems=o, fill=to_dev(x)) for o, x in zip(offs, xs)]
        outs = [Guarded(N, td, offset_elems=(o + 1) % 4) for o in offs]
        with session(R, dtype, True) as h:
            rcc.all_reduce(h, [g.t for g in ins], [o.t for o in outs], "sum")
            torch.cuda.synchronize()
        want = orc.reduce_f32(xs, "sum") if dtype == rcc.F32 else orc.reduce_bf16(xs, "sum")
        for o in outs:
            assert o.guards_intact()
            assert bits_equal(to_host(o.t), want)


def test_zero_count_is_noop():
    R = 4
    before = rcc.launch_count()
    e = [torch.empty(0, device=DEV) for _ in range(R)]
    with session(R) as h:
        rcc.all_reduce(h, e, e, "sum")
        rcc.reduce_scatter(h, e, e, "sum")
        rcc.all_gather(h, e, e)
    assert rcc.launch_count() == before


def test_integer_inputs_bit_exact_in_every_mode(orc):
    for R in (3, 5, 8):
        xs = host_ranks("int", R, 100003, 800, R)
        ins = [to_dev(x) for x in xs]
        for det in (True, False):
            for op in ("sum", "mean"):
                outs = [torch.empty_like(ins[0]) for _ in range(R)]
                with session(R, rcc.F32, det) as h:
                    rcc.all_reduce(h, ins, outs, op)
                    torch.cuda.synchronize()
                # integer sums are exact in any order, so every mode gives the
                # oracle's bits (the mean is then one correctly rounded division)
                assert bits_equal(to_host(outs[0]), orc.reduce_f32(xs, op))


def test_in_place_all_reduce(orc):
    R, N = 4, 10007
    xs = host_ranks("uniform", R, N, 900)
    want = orc.reduce_f32(xs, "sum")
    bufs = [to_dev(x) for x in xs]
    with session(R, rcc.F32, True) as h:
        rcc.all_reduce(h, bufs, bufs, "sum")
        torch.cuda.synchronize()
    for b in bufs:
        assert bits_equal(to_host(b), want)
    # partly in place
    bufs = [to_dev(x) for x in xs]
    outs = [bufs[0], torch.empty_like(bufs[1]), bufs[2], torch.empty_like(bufs[3])]
    with session(R, rcc.F32, True) as h:
        rcc.all_reduce(h, bufs, outs, "sum")
        torch.cuda.synchronize()
    for o in outs:
        assert bits_equal(to_host(o), want)


def test_special_values_max_min_sum(orc):
    R = 5
    vals = np.array([0.0, -0.0, np.inf, -np.inf, np.nan, 1.0, -1.0, 3e38, -3e38, 1e-45],
                    np.float32)
    g = synth.rng(1000)
    N = 4099
    xs = [vals[g.integers(0, len(vals), N)] for _ in range(R)]
    ins = [to_dev(x) for x in xs]
    for op in ("max", "min", "sum"):
        outs = [torch.empty_like(ins[0]) for _ in range(R)]
        with session(R, rcc.F32, True) as h:
            rcc.all_reduce(h, ins, outs, op)
            torch.cuda.synchronize()
        got = to_host(outs[0])
        want = orc.reduce_f32(xs, op)
        if op == "sum":       # NaN payloads are not specified: compare NaN-ness and the rest
            assert np.array_equal(np.isnan(got), np.isnan(want))
            m = ~np.isnan(want)
            assert bits_equal(got[m], want[m])
        else:
            assert bits_equal(got, want)
    # bf16
    xb = [orc.f32_to_bf16(x) for x in xs]
    insb = [to_dev(x) for x in xb]
    for op in ("max", "min"):
        outs = [torch.empty_like(insb[0]) for _ in range(R)]
        with session(R, rcc.BF16, True) as h:
            rcc.all_reduce(h, insb, outs, op)
            torch.cuda.synchronize()
        assert bits_equal(to_host(outs[0]), orc.reduce_bf16(xb, op))


# shards whose offsets s*n break 16-byte alignment go through the staged
# kernels; the large ones there cover many full tiles plus head and tail
@pytest.mark.parametrize("R,n", [(3, 257), (4, 1), (8, 4096), (5, 33), (64, 40),
                                 (8, 262145), (3, 100003), (12, 65537), (4, 131074)])
@pytest.mark.parametrize("dtype", [rcc.F32, rcc.BF16])
def test_reduce_scatter_all_gather_shapes(orc, R, n, dtype):
    td = tdtype(dtype)
    N = R * n
    kind = "uniform" if dtype == rcc.F32 else "bf16_uniform"
    xs = host_ranks(kind, R, N, 1100, R, n)
    ins = [to_dev(x) for x in xs]
    rs = [Guarded(n, td) for _ in range(R)]
    ag = [Guarded(N, td) for _ in range(R)]
    with session(R, dtype, True) as h:
        rcc.reduce_scatter(h, ins, [g.t for g in rs], "mean")
        rcc.all_gather(h, [g.t for g in rs], [g.t for g in ag])
        torch.cuda.synchronize()
    want = orc.reduce_scatter(xs, "mean")
    for r in range(R):
        assert rs[r].guards_intact() and ag[r].guards_intact()
        assert bits_equal(to_host(rs[r].t), want[r])
        assert bits_equal(to_host(ag[r].t), np.concatenate(want))


@pytest.mark.parametrize("op", ["sum", "max", "min"])
@pytest.mark.parametrize("det", [True, False])
def test_reduce_scatter_odd_shards_every_op(orc, op, det):
    """The staged reduction at an odd shard, each op, both summation modes."""
    R, n = 8, 65537
    N = R * n
    xs = host_ranks("uniform", R, N, 1101, R, n)
    ins = [to_dev(x) for x in xs]
    rs = [Guarded(n, torch.float32) for _ in range(R)]
    with session(R, rcc.F32, det) as h:
        rcc.reduce_scatter(h, ins, [g.t for g in rs], op)
        torch.cuda.synchronize()
    want = orc.reduce_scatter(xs, op)
    exact = np.sum([x.astype(np.float64) for x in xs], axis=0)
    mag = np.sum([np.abs(x.astype(np.float64)) for x in xs], axis=0)
    for r in range(R):
        assert rs[r].guards_intact()
        got = to_host(rs[r].t)
        if det or op != "sum":
            assert bits_equal(got, want[r])
        else:                                  # pairwise tree: within the fp32 bound
            lo, hi = r * n, (r + 1) * n
            assert np.all(np.abs(got.astype(np.float64) - exact[lo:hi])
                          <= R * 2.0 ** -23 * mag[lo:hi])


def test_all_gather_in_place(orc):
    R, n = 4, 1000
    xs = host_ranks("uniform", R, n, 1200)
    outs = [torch.zeros(R * n, device=DEV) for _ in range(R)]
    for q in range(R):
        outs[q][q * n:(q + 1) * n].copy_(to_dev(xs[q]))
    send = [outs[q][q * n:(q + 1) * n] for q in range(R)]
    with session(R, rcc.F32, True) as h:
        rcc.all_gather(h, send, outs)
        torch.cuda.synchronize()
    for r in range(R):
        assert bits_equal(to_host(outs[r]), np.concatenate(xs))


def test_broadcast_root_alias_and_none(orc):
    R, N = 4, 3001
    x = host_ranks("uniform", 1, N, 1300)[0]
    src = to_dev(x)
    outs = [torch.zeros(N, device=DEV) for _ in range(R)]
    outs[2] = src                                  # the root's recv aliases its send
    with session(R, rcc.F32, True) as h:
        rcc.broadcast(h, src, outs, root=2)
        torch.cuda.synchronize()
    for o in outs:
        assert bits_equal(to_host(o), x)


def test_finish_then_reregister_and_reset_with_pending_work():
    R, N = 8, 1 << 22
    ins = [torch.ones(N, device=DEV) for _ in range(R)]
    outs = [torch.empty(N, device=DEV) for _ in range(R)]
    h = rcc.register(0, R, rcc.F32, True)
    with pytest.raises(rcc.RccError) as ei:
        rcc.register(0, R, rcc.F32, True)
    assert ei.value.status == rcc.ERR_DUPLICATE_REGISTRATION
    for _ in range(10):
        rcc.all_reduce(h, ins, outs, "sum")
    rcc.reset(h)                                  # discards the session at once
    h2 = rcc.register(0, R, rcc.F32, True)
    rcc.all_reduce(h2, ins, outs, "sum")
    rcc.finish(h2)
    assert bool(torch.all(outs[0] == 8.0))


# ---------------------------------------------------------------- all_to_all_single, list all_gather

@pytest.mark.parametrize("R,n", [(1, 100), (2, 4099), (3, 257), (4, 1 << 16), (8, 33), (8, 1 << 18),
                                 (8, 262145), (4, 65539)])
@pytest.mark.parametrize("dtype", [rcc.F32, rcc.BF16])
def test_all_to_all_single(orc, R, n, dtype):
    td = tdtype(dtype)
    N = R * n
    kind = "uniform" if dtype == rcc.F32 else "bf16_uniform"
    xs = host_ranks(kind, R, N, 1400, R, n)
    ins = [to_dev(x) for x in xs]
    outs = [Guarded(N, td) for _ in range(R)]
    with session(R, dtype, True) as h:
        rcc.all_to_all_single(h, ins, [o.t for o in outs])
        torch.cuda.synchronize()
    want = orc.all_to_all(xs)
    for r in range(R):
        assert outs[r].guards_intact()
        assert bits_equal(to_host(outs[r].t), want[r])


def test_all_to_all_single_misaligned(orc):
    R, n = 4, 1001
    xs = host_ranks("uniform", R, R * n, 1401)
    ins = [Guarded(R * n, torch.float32, offset_elems=1, fill=to_dev(x)) for x in xs]
    outs = [Guarded(R * n, torch.float32, offset_elems=3) for _ in range(R)]
    with session(R) as h:
        rcc.all_to_all_single(h, [g.t for g in ins], [o.t for o in outs])
        torch.cuda.synchronize()
    want = orc.all_to_all(xs)
    for r in range(R):
        assert outs[r].guards_intact() and bits_equal(to_host(outs[r].t), want[r])


@pytest.mark.parametrize("R,n", [(2, 1000), (4, 4097), (8, 1 << 16)])
def test_all_gather_list(orc, R, n):
    xs = host_ranks("uniform", R, n, 1402, R)
    ins = [to_dev(x) for x in xs]
    lists = [[Guarded(n, torch.float32) for _ in range(R)] for _ in range(R)]
    # rank 1 gathers its own tensor in place
    lists[1][1] = None
    recv = [[g.t if g is not None else None for g in row] for row in lists]
    recv[1][1] = ins[1]
    with session(R) as h:
        rcc.all_gather_list(h, ins, recv)
        torch.cuda.synchronize()
    for r in range(R):
        for q in range(R):
            got = to_host(recv[r][q])
            assert bits_equal(got, xs[q]), (r, q)
            if lists[r][q] is not None:
                assert lists[r][q].guards_intact()


@pytest.mark.parametrize("kind", ["reduce_scatter", "all_gather", "all_to_all"])
@pytest.mark.parametrize("dtype", [rcc.F32, rcc.BF16])
@pytest.mark.parametrize("out_off16", [True, False])
def test_staged_kernels_on_16_byte_bases(orc, kind, dtype, out_off16):
    """Odd shards whose buffers start 16 bytes past a 32-byte boundary: the
    staged kernels' 16-byte-vector form, over many tiles plus head and tail,
    bit for bit against the oracle, with the guard bands intact."""
    R, n = 8, 65537
    td = tdtype(dtype)
    es = 4 if dtype == rcc.F32 else 2
    off16 = 16 // es                               # elements in 16 bytes
    kind_draw = "uniform" if dtype == rcc.F32 else "bf16_uniform"
    out_off = off16 if out_off16 else 0
    if kind == "all_gather":
        xs = host_ranks(kind_draw, R, n, 1500, R, n)
        ins = [Guarded(n, td, offset_elems=off16, fill=to_dev(x)) for x in xs]
        outs = [Guarded(R * n, td, offset_elems=out_off) for _ in range(R)]
        want = [np.concatenate(xs)] * R
    else:
        xs = host_ranks(kind_draw, R, R * n, 1501, R, n)
        ins = [Guarded(R * n, td, offset_elems=off16, fill=to_dev(x)) for x in xs]
        if kind == "reduce_scatter":
            outs = [Guarded(n, td, offset_elems=out_off) for _ in range(R)]
            want = orc.reduce_scatter(xs, "sum")
        else:
            outs = [Guarded(R * n, td, offset_elems=out_off) for _ in range(R)]
            want = orc.all_to_all(xs)
    with session(R, dtype, True) as h:
        if kind == "reduce_scatter":
            rcc.reduce_scatter(h, [g.t for g in ins], [o.t for o in outs], "sum")
        elif kind == "all_gather":
            rcc.all_gather(h, [g.t for g in ins], [o.t for o in outs])
        else:
            rcc.all_to_all_single(h, [g.t for g in ins], [o.t for o in outs])
        torch.cuda.synchronize()
    for r in range(R):
        assert outs[r].guards_intact() and ins[r].guards_intact()
        assert bits_equal(to_host(outs[r].t), want[r]), (kind, r)
