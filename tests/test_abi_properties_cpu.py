"""Property test of the host-side validation order (CPU only).

Random per-rank counts, ops, roots and missing buffers; the status returned
must be the one the documented order gives: shape, op, root, broadcast
senders, zero-count no-op, missing buffers, then the device check.  Sessions
live on device ordinal 63 so nothing is ever launched; the addresses are fake
and never dereferenced.
"""
import ctypes as C

import pytest

hyp = pytest.importorskip("hypothesis")
st = pytest.importorskip("hypothesis.strategies")
from hypothesis import given, settings  # noqa: E402

DEV = 63
BASE = 0x7F0000000000


@pytest.fixture(scope="module")
def L():
    from gradient_sync_rcc_gb300 import build, rcc
    build.build()
    return rcc


def _session(L, R):
    h = C.c_void_p()
    assert L.raw("rcc_register", DEV, R, 0, 1, C.byref(h)) == L.OK
    return h.value


def _device(L, status):
    return status in (L.ERR_CUDA, L.ERR_INVALID_ARGUMENT)


rank_case = st.integers(1, 8).flatmap(lambda R: st.fixed_dictionaries({
    "R": st.just(R),
    "counts": st.lists(st.sampled_from([0, 64, 64, 64, 65]), min_size=R, max_size=R),
    "ops": st.lists(st.sampled_from([0, 0, 0, 1, 2, 7]), min_size=R, max_size=R),
    "roots": st.lists(st.sampled_from([0, 0, R - 1, R]), min_size=R, max_size=R),
    "send_null": st.lists(st.sampled_from([False, False, False, True]), min_size=R, max_size=R),
    "recv_null": st.lists(st.sampled_from([False, False, False, True]), min_size=R, max_size=R),
}))


def _model_all_reduce(c):
    R = c["R"]
    if any(n != c["counts"][0] for n in c["counts"]):
        return "shape"
    if any(o not in (0, 1, 2, 3) or o != c["ops"][0] for o in c["ops"]):
        return "op"
    if c["counts"][0] == 0:
        return "ok"
    if any(c["send_null"][r] or c["recv_null"][r] for r in range(R)):
        return "missing"
    return "device"


def _model_reduce(c):
    R = c["R"]
    if any(n != c["counts"][0] for n in c["counts"]):
        return "shape"
    if any(o not in (0, 1, 2, 3) or o != c["ops"][0] for o in c["ops"]):
        return "op"
    if any(not (0 <= x < R) or x != c["roots"][0] for x in c["roots"]):
        return "root"
    if c["counts"][0] == 0:
        return "ok"
    if any(c["send_null"]) or c["recv_null"][c["roots"][0]]:
        return "missing"
    return "device"


def _check(L, want, got):
    table = {"shape": L.ERR_SHAPE_MISMATCH, "op": L.ERR_INCONSISTENT_OP,
             "root": L.ERR_INCONSISTENT_ROOT, "missing": L.ERR_MISSING_REGISTRATION,
             "ok": L.OK, "senders": L.ERR_BROADCAST_SENDERS}
    if want == "device":
        assert _device(L, got), got
    else:
        assert got == table[want], (want, got)


@settings(max_examples=300, deadline=None)
@given(rank_case)
def test_all_reduce_and_reduce_follow_the_documented_order(L, c):
    R = c["R"]
    h = _session(L, R)
    try:
        send = [None if c["send_null"][r] else BASE + r * (1 << 24) for r in range(R)]
        recv = [None if c["recv_null"][r] else BASE * 2 + r * (1 << 24) for r in range(R)]
        got = L.raw("rcc_all_reduce", h, L.ptr_array(send), L.ptr_array(recv),
                    L.size_array(c["counts"]), L.int_array(c["ops"]), None)
        _check(L, _model_all_reduce(c), got)
        got = L.raw("rcc_reduce", h, L.ptr_array(send), L.ptr_array(recv),
                    L.size_array(c["counts"]), L.int_array(c["ops"]), L.int_array(c["roots"]),
                    None)
        _check(L, _model_reduce(c), got)
    finally:
        L.raw("rcc_reset", h)


@settings(max_examples=200, deadline=None)
@given(st.integers(1, 8).flatmap(lambda R: st.tuples(
    st.just(R), st.lists(st.booleans(), min_size=R, max_size=R),
    st.lists(st.sampled_from([128, 128, 129]), min_size=R, max_size=R),
    st.lists(st.sampled_from([False, False, True]), min_size=R, max_size=R))))
def test_broadcast_sender_rule(L, case):
    R, senders, counts, recv_null = case
    h = _session(L, R)
    try:
        send = [BASE + r * 4096 if senders[r] else None for r in range(R)]
        recv = [None if recv_null[r] else BASE * 2 + r * (1 << 24) for r in range(R)]
        got = L.raw("rcc_broadcast", h, L.ptr_array(send), L.ptr_array(recv),
                    L.size_array(counts), None)
        if any(n != counts[0] for n in counts):
            want = "shape"
        elif sum(senders) != 1:
            want = "senders"
        else:
            root = senders.index(True)
            if any(recv_null[r] for r in range(R) if r != root):
                want = "missing"
            elif all(recv_null[r] or r == root for r in range(R)) and recv_null[root]:
                want = "ok"                   # nobody to write to
            else:
                want = "device"
        _check(L, want, got)
    finally:
        L.raw("rcc_reset", h)
