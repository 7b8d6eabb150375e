"""Per-rank arrival on the host (no GPU): each logical rank is its own thread.

[ruCCL README introduction and §1: the in_process implementation runs logical
ranks inside one process; §3: every rank calls matching collectives in the
same order with matching shape, op and root; §4: reset discards in-flight
operation state.]
The last rank to arrive checks the set and launches; every rank returns the
same status.  Sessions are registered on device ordinal 63 (never current),
so an agreeing set stops at the device check and launches nothing; the fake
addresses are never dereferenced.
"""
import ctypes as C
import os
import threading
import time

import pytest

DEV = 63
BASE = 0x7F0000000000


@pytest.fixture
def L(rcc_lib):
    return rcc_lib


@pytest.fixture
def comm(L):
    made = []

    def make(R=4):
        h = C.c_void_p()
        assert L.raw("rcc_register", DEV, R, 0, 1, C.byref(h)) == L.OK
        made.append(h.value)
        return h.value

    yield make
    for h in made:
        L.raw("rcc_reset", h)


@pytest.fixture
def short_wait():
    old = os.environ.get("RCC_WAIT_LIMIT_MS")
    os.environ["RCC_WAIT_LIMIT_MS"] = "400"
    yield
    if old is None:
        del os.environ["RCC_WAIT_LIMIT_MS"]
    else:
        os.environ["RCC_WAIT_LIMIT_MS"] = old


def run_ranks(calls):
    """Run each zero-argument callable in its own thread; return their results."""
    out = [None] * len(calls)

    def go(i):
        out[i] = calls[i]()

    ts = [threading.Thread(target=go, args=(i,)) for i in range(len(calls))]
    for t in ts:
        t.start()
    for t in ts:
        t.join(30)
        assert not t.is_alive()
    return out


def ar(L, h, r, count=1024, op=0, send=None, recv=None):
    s = BASE + r * (1 << 24) if send is None else send
    d = BASE * 2 + r * (1 << 24) if recv is None else recv
    return lambda: L.raw("rcc_all_reduce_rank", h, r, s, d, count, op, None)


def stopped_at_device(L, st):
    return st in (L.ERR_CUDA, L.ERR_INVALID_ARGUMENT)


def test_agreeing_ranks_share_one_outcome(L, comm):
    h = comm(4)
    res = run_ranks([ar(L, h, r) for r in range(4)])
    assert len(set(res)) == 1 and stopped_at_device(L, res[0])
    # a zero-count collective completes (no launch) with RCC_OK for everyone
    assert run_ranks([ar(L, h, r, count=0) for r in range(4)]) == [L.OK] * 4


def test_mismatches_reported_to_every_rank(L, comm):
    h = comm(4)
    res = run_ranks([ar(L, h, r, count=1024 if r != 2 else 1000) for r in range(4)])
    assert res == [L.ERR_SHAPE_MISMATCH] * 4
    res = run_ranks([ar(L, h, r, op=0 if r != 1 else 2) for r in range(4)])
    assert res == [L.ERR_INCONSISTENT_OP] * 4
    # rank 3 calls a different collective
    calls = [ar(L, h, r) for r in range(3)]
    calls.append(lambda: L.raw("rcc_all_gather_rank", h, 3, BASE, BASE * 3, 256, None))
    assert run_ranks(calls) == [L.ERR_INCONSISTENT_OP] * 4
    # reduce with different roots
    red = [lambda r=r: L.raw("rcc_reduce_rank", h, r, BASE + r * (1 << 24), BASE * 2, 64, 0,
                             3 if r else 2, None) for r in range(4)]
    assert run_ranks(red) == [L.ERR_INCONSISTENT_ROOT] * 4
    # broadcast with two senders, then with none
    two = [lambda r=r: L.raw("rcc_broadcast_rank", h, r, BASE + r * 4096 if r < 2 else None,
                             BASE * 2 + r * (1 << 24), 64, None) for r in range(4)]
    assert run_ranks(two) == [L.ERR_BROADCAST_SENDERS] * 4
    none = [lambda r=r: L.raw("rcc_broadcast_rank", h, r, None, BASE * 2 + r * (1 << 24), 64,
                              None) for r in range(4)]
    assert run_ranks(none) == [L.ERR_BROADCAST_SENDERS] * 4
    # after all that, an agreeing round still works
    res = run_ranks([ar(L, h, r) for r in range(4)])
    assert len(set(res)) == 1 and stopped_at_device(L, res[0])


def test_bad_rank_index(L, comm):
    h = comm(2)
    assert L.raw("rcc_all_reduce_rank", h, 2, BASE, BASE * 2, 8, 0, None) == L.ERR_INVALID_ARGUMENT
    assert L.raw("rcc_all_reduce_rank", h, -1, BASE, BASE * 2, 8, 0, None) == L.ERR_INVALID_ARGUMENT


def test_duplicate_arrival_rejected(L, comm, short_wait):
    h = comm(3)
    first = []
    t = threading.Thread(target=lambda: first.append(ar(L, h, 0)()))
    t.start()
    time.sleep(0.05)
    assert ar(L, h, 0)() == L.ERR_INVALID_ARGUMENT          # same rank again
    assert "twice" in L.last_error()
    rest = run_ranks([ar(L, h, 1), ar(L, h, 2)])             # the others complete the set
    t.join(10)
    assert len(set(rest + first)) == 1 and stopped_at_device(L, rest[0])


def test_missing_rank_times_out_for_everyone(L, comm, short_wait):
    h = comm(4)
    t0 = time.time()
    res = run_ranks([ar(L, h, r) for r in range(3)])         # rank 3 never comes
    assert res == [L.ERR_TIMEOUT] * 3
    assert time.time() - t0 < 5
    # the discarded collective leaves the session usable
    res = run_ranks([ar(L, h, r) for r in range(4)])
    assert len(set(res)) == 1 and stopped_at_device(L, res[0])


def test_reset_wakes_waiting_ranks(L, comm):
    h = comm(4)
    out = []
    ts = [threading.Thread(target=lambda r=r: out.append(ar(L, h, r)())) for r in range(2)]
    for t in ts:
        t.start()
    time.sleep(0.1)
    assert L.raw("rcc_reset", h) == L.OK
    for t in ts:
        t.join(10)
        assert not t.is_alive()
    assert out == [L.ERR_MISSING_REGISTRATION] * 2


def test_many_rounds_in_order(L, comm):
    h = comm(4)

    def rank_loop(r):
        return [L.raw("rcc_all_reduce_rank", h, r, BASE + r * (1 << 24), BASE * 2 + r * (1 << 24),
                      0 if k % 2 else 512, 0, None) for k in range(20)]
    res = run_ranks([lambda r=r: rank_loop(r) for r in range(4)])
    for k in range(20):
        col = {res[r][k] for r in range(4)}
        assert len(col) == 1
        assert (col.pop() == L.OK) if k % 2 else True
