"""C-ABI host-side tests (no GPU needed).

The library loads, exports every function include/rcc.h declares, and rejects
each malformed call with the status the ruCCL README's CollectiveError cases
name (duplicate or missing registration, shape mismatch, inconsistent op or
root, broadcast sender count != 1), in the documented order, before any CUDA
call.  Sessions here are registered on device ordinal 63, which is never the
current device: a call that passes validation stops at the device check
(RCC_ERR_CUDA without a GPU, RCC_ERR_INVALID_ARGUMENT with one) and launches
nothing, so the fake addresses below are never dereferenced.
"""
import ctypes as C
import os
import re

import pytest

DEV = 63
BASE = 0x7F0000000000  # fake, 256-byte aligned "device" addresses (never dereferenced)


@pytest.fixture
def L(rcc_lib):
    return rcc_lib


@pytest.fixture
def comm(L):
    sessions = []

    def make(R=4, dtype=0, device=DEV, flags=1):
        h = C.c_void_p()
        st = L.raw("rcc_register", device, R, dtype, flags, C.byref(h))
        assert st == L.OK, L.last_error()
        sessions.append(h.value)
        return h.value

    yield make
    for h in sessions:
        L.raw("rcc_reset", h)   # may already be gone


def addrs(R, stride=1 << 24, base=BASE):
    return [base + r * stride for r in range(R)]


def reached_device_check(L, st):
    # validation passed; the call stopped at the device check without launching
    return st in (L.ERR_CUDA, L.ERR_INVALID_ARGUMENT) and (
        "device" in L.last_error() or "cuda" in L.last_error().lower())


# ---------------------------------------------------------------- exports

def test_exports_every_declared_symbol(L):
    hdr = open(os.path.join(os.path.dirname(__file__), "..", "include", "rcc.h")).read()
    declared = set(re.findall(r"^[A-Za-z0-9_ *]*?\b(rcc_[a-z_]+)\s*\(", hdr, re.M))
    assert declared, "no declarations parsed"
    assert declared == set(L.SYMBOLS)
    lib = L.lib()
    for name in declared:
        assert hasattr(lib, name), name


def test_status_strings(L):
    for code in range(10):
        assert L.lib().rcc_status_string(code).decode().startswith("RCC_")


# ---------------------------------------------------------------- lifecycle

def test_register_validation(L):
    h = C.c_void_p()
    assert L.raw("rcc_register", -1, 4, 0, 1, C.byref(h)) == L.ERR_INVALID_ARGUMENT
    assert L.raw("rcc_register", DEV, 0, 0, 1, C.byref(h)) == L.ERR_INVALID_ARGUMENT
    assert L.raw("rcc_register", DEV, 65, 0, 1, C.byref(h)) == L.ERR_INVALID_ARGUMENT
    assert L.raw("rcc_register", DEV, 4, 7, 1, C.byref(h)) == L.ERR_INVALID_ARGUMENT
    assert L.raw("rcc_register", DEV, 4, 0, 0x10, C.byref(h)) == L.ERR_INVALID_ARGUMENT
    assert L.raw("rcc_register", DEV, 4, 0, 1, None) == L.ERR_INVALID_ARGUMENT


def test_duplicate_registration(L, comm):
    a = comm(device=DEV)
    h = C.c_void_p()
    assert L.raw("rcc_register", DEV, 2, 0, 1, C.byref(h)) == L.ERR_DUPLICATE_REGISTRATION
    assert "already" in L.last_error()
    b = comm(device=DEV - 1)            # another device is independent
    assert a != b


def test_reset_then_missing_then_reregister(L, comm):
    a = comm()
    assert L.raw("rcc_reset", a) == L.OK
    assert L.raw("rcc_reset", a) == L.ERR_MISSING_REGISTRATION
    assert L.raw("rcc_set_flags", a, 0) == L.ERR_MISSING_REGISTRATION
    R = 4
    st = L.raw("rcc_all_reduce", a, L.ptr_array(addrs(R)), L.ptr_array(addrs(R, base=BASE * 2)),
               L.size_array([8] * R), L.int_array([0] * R), None)
    assert st == L.ERR_MISSING_REGISTRATION
    b = comm()
    assert b != a                       # a fresh handle; the stale one stays dead
    assert L.raw("rcc_set_flags", a, 0) == L.ERR_MISSING_REGISTRATION
    assert L.raw("rcc_set_flags", b, 0) == L.OK


def test_null_and_forged_handles(L):
    assert L.raw("rcc_reset", None) == L.ERR_MISSING_REGISTRATION
    assert L.raw("rcc_reset", 0x12345) == L.ERR_MISSING_REGISTRATION
    assert L.raw("rcc_finish", None, None) == L.ERR_MISSING_REGISTRATION


def test_set_flags_validation(L, comm):
    a = comm()
    assert L.raw("rcc_set_flags", a, 0x4) == L.ERR_INVALID_ARGUMENT
    assert L.raw("rcc_set_flags", a, 0) == L.OK
    assert L.raw("rcc_set_flags", a, 1) == L.OK
    assert L.raw("rcc_set_flags", a, L.DETERMINISTIC | L.STEP_TIMING) == L.OK


def test_step_times_need_a_timed_call(L, comm):
    a = comm()
    out = (C.c_float * 4)()
    assert L.raw("rcc_last_step_times", a, out) == L.ERR_INVALID_ARGUMENT
    assert "RCC_STEP_TIMING" in L.last_error()
    assert L.raw("rcc_last_step_times", a, None) == L.ERR_INVALID_ARGUMENT
    assert L.raw("rcc_last_step_times", None, out) == L.ERR_MISSING_REGISTRATION


# ---------------------------------------------------------------- all_reduce

def _ar(L, h, send, recv, counts, ops):
    return L.raw("rcc_all_reduce", h, send, recv, counts, ops, None)


def test_all_reduce_errors(L, comm):
    R = 4
    h = comm(R)
    s, r = addrs(R), addrs(R, base=BASE * 2)
    S, Rv = L.ptr_array(s), L.ptr_array(r)
    n = L.size_array([1000] * R)
    ops = L.int_array([L.SUM] * R)
    assert _ar(L, h, None, Rv, n, ops) == L.ERR_INVALID_ARGUMENT
    assert _ar(L, h, S, Rv, None, ops) == L.ERR_INVALID_ARGUMENT
    assert _ar(L, h, S, Rv, L.size_array([1000, 1000, 999, 1000]), ops) == L.ERR_SHAPE_MISMATCH
    assert _ar(L, h, S, Rv, n, L.int_array([0, 0, 1, 0])) == L.ERR_INCONSISTENT_OP
    assert _ar(L, h, S, Rv, n, L.int_array([9] * R)) == L.ERR_INCONSISTENT_OP
    missing = list(s)
    missing[2] = None
    assert _ar(L, h, L.ptr_array(missing), Rv, n, ops) == L.ERR_MISSING_REGISTRATION
    missing = list(r)
    missing[3] = None
    assert _ar(L, h, S, L.ptr_array(missing), n, ops) == L.ERR_MISSING_REGISTRATION
    # recv buffers overlapping each other / another rank's input
    ov = list(r)
    ov[1] = r[0] + 64
    assert _ar(L, h, S, L.ptr_array(ov), n, ops) == L.ERR_INVALID_ARGUMENT
    ov = list(r)
    ov[1] = s[0]
    assert _ar(L, h, S, L.ptr_array(ov), n, ops) == L.ERR_INVALID_ARGUMENT
    # valid calls (out of place, in place) pass validation
    assert reached_device_check(L, _ar(L, h, S, Rv, n, ops))
    assert reached_device_check(L, _ar(L, h, S, S, n, ops))
    # count 0 is a no-op even without buffers
    assert _ar(L, h, L.ptr_array([None] * R), L.ptr_array([None] * R),
               L.size_array([0] * R), ops) == L.OK


def test_check_order(L, comm):
    R = 4
    h = comm(R)
    S, Rv = L.ptr_array(addrs(R)), L.ptr_array(addrs(R, base=BASE * 2))
    bad_n = L.size_array([8, 9, 8, 8])
    bad_ops = L.int_array([0, 1, 0, 0])
    # shape before op
    assert _ar(L, h, S, Rv, bad_n, bad_ops) == L.ERR_SHAPE_MISMATCH
    # handle before shape
    assert _ar(L, 0x999, S, Rv, bad_n, bad_ops) == L.ERR_MISSING_REGISTRATION
    # op before missing buffers
    assert _ar(L, h, L.ptr_array([None] * R), Rv, L.size_array([8] * R), bad_ops) == \
        L.ERR_INCONSISTENT_OP


# ---------------------------------------------------------------- reduce

def test_reduce_errors(L, comm):
    R = 4
    h = comm(R)
    s = addrs(R)
    S = L.ptr_array(s)
    n = L.size_array([64] * R)
    ops = L.int_array([L.MAX] * R)
    out = [None] * R
    out[3] = BASE * 2

    def red(recv, roots, ops=ops, send=S):
        return L.raw("rcc_reduce", h, send, L.ptr_array(recv), n, ops, L.int_array(roots), None)

    assert red(out, [3, 3, 2, 3]) == L.ERR_INCONSISTENT_ROOT
    assert red(out, [4] * R) == L.ERR_INCONSISTENT_ROOT
    assert red(out, [-1] * R) == L.ERR_INCONSISTENT_ROOT
    assert red([None] * R, [3] * R) == L.ERR_MISSING_REGISTRATION
    assert red(out, [3] * R, ops=L.int_array([2, 2, 3, 2])) == L.ERR_INCONSISTENT_OP
    ov = list(out)
    ov[3] = s[1] + 16
    assert red(ov, [3] * R) == L.ERR_INVALID_ARGUMENT
    assert reached_device_check(L, red(out, [3] * R))
    inplace = [None] * R
    inplace[3] = s[3]
    assert reached_device_check(L, red(inplace, [3] * R))


# ---------------------------------------------------------------- broadcast

def test_broadcast_errors(L, comm):
    R = 4
    h = comm(R)
    r = addrs(R, base=BASE * 2)
    n = L.size_array([100] * R)

    def bc(send, recv=r, counts=n):
        return L.raw("rcc_broadcast", h, L.ptr_array(send), L.ptr_array(recv), counts, None)

    assert bc([None] * R) == L.ERR_BROADCAST_SENDERS
    assert bc([BASE, BASE + 4096, None, None]) == L.ERR_BROADCAST_SENDERS
    one = [None, BASE, None, None]
    assert bc(one, counts=L.size_array([100, 100, 100, 7])) == L.ERR_SHAPE_MISMATCH
    recv = list(r)
    recv[2] = None
    assert bc(one, recv) == L.ERR_MISSING_REGISTRATION
    recv = list(r)
    recv[1] = None                       # the root keeps its own tensor
    assert reached_device_check(L, bc(one, recv))
    recv = list(r)
    recv[1] = BASE                       # the root's recv aliases its send: skipped
    assert reached_device_check(L, bc(one, recv))
    recv = list(r)
    recv[2] = BASE + 8                   # overlaps the root's input
    assert bc(one, recv) == L.ERR_INVALID_ARGUMENT


# ---------------------------------------------------------------- reduce_scatter / all_gather

def test_reduce_scatter_errors(L, comm):
    R = 4
    h = comm(R)
    S, Rv = L.ptr_array(addrs(R)), L.ptr_array(addrs(R, base=BASE * 2))
    ops = L.int_array([L.SUM] * R)

    def rs(counts, recv=Rv):
        return L.raw("rcc_reduce_scatter", h, S, recv, L.size_array(counts), ops, None)

    assert rs([1002] * R) == L.ERR_SHAPE_MISMATCH           # 1002 % 4 != 0
    assert rs([1000, 1000, 1000, 996]) == L.ERR_SHAPE_MISMATCH
    assert reached_device_check(L, rs([1000] * R))
    ov = addrs(R, base=BASE * 2)
    ov[2] = ov[1] + 400                                      # shards of 250 fp32 overlap
    assert rs([1000] * R, L.ptr_array(ov)) == L.ERR_INVALID_ARGUMENT


def test_all_gather_errors_and_in_place(L, comm):
    R = 4
    h = comm(R)
    n = 256
    recv = addrs(R, base=BASE * 2)

    def ag(send, recv=recv):
        return L.raw("rcc_all_gather", h, L.ptr_array(send), L.ptr_array(recv),
                     L.size_array([n] * R), None)

    assert reached_device_check(L, ag(addrs(R)))
    # in place: rank q's input is slot q of its own output
    own = [recv[q] + q * n * 4 for q in range(R)]
    assert reached_device_check(L, ag(own))
    bad = list(own)
    bad[1] = recv[1] + 2 * n * 4                             # not its own slot
    assert ag(bad) == L.ERR_INVALID_ARGUMENT
    assert ag([None] + addrs(R)[1:]) == L.ERR_MISSING_REGISTRATION


# ---------------------------------------------------------------- grad sync

def _param_sets(L, R, rep, numel=1000, P=2, grads_null=None, rank_numel=None):
    keep = []
    arr = (L.ParamSet * P)()
    for p in range(P):
        g = [BASE + (p * 64 + r) * (1 << 24) for r in range(R)]
        if grads_null is not None and p == 1:
            g[grads_null] = None
        st = [BASE * 2 + (p * 64 + k) * (1 << 24) for k in range(3 * rep)]
        ga, pa = L.ptr_array(g), L.ptr_array(st[:rep])
        ma, va = L.ptr_array(st[rep:2 * rep]), L.ptr_array(st[2 * rep:])
        rn = L.size_array(rank_numel) if (rank_numel is not None and p == 1) else None
        keep += [ga, pa, ma, va, rn]
        arr[p] = L.ParamSet(numel, rn, ga, pa, ma, va, None)
    return arr, keep


def test_grad_sync_validation(L, comm):
    R = 4
    h = comm(R)
    cfg = L.adamw_cfg(replicas=R)
    state = L.optim_state()
    rep = L.StepReport()

    def gs(arr, P=2, cfg=cfg, state=state, h=h):
        return L.raw("rcc_grad_sync_adamw", h, arr, P, C.byref(cfg), C.byref(state),
                     C.byref(rep), None)

    arr, keep = _param_sets(L, R, R)
    assert reached_device_check(L, gs(arr))
    empty, keepe = _param_sets(L, R, R, numel=0)
    assert gs(empty) == L.ERR_INVALID_ARGUMENT and "0 elements" in L.last_error()
    assert gs(arr, P=0) == L.ERR_INVALID_ARGUMENT
    assert gs(arr, h=0x4242) == L.ERR_MISSING_REGISTRATION
    arr2, keep2 = _param_sets(L, R, R, rank_numel=[1000, 1000, 999, 1000])
    assert gs(arr2) == L.ERR_SHAPE_MISMATCH
    arr3, keep3 = _param_sets(L, R, R, grads_null=2)
    assert gs(arr3) == L.ERR_MISSING_REGISTRATION
    assert gs(arr, cfg=L.adamw_cfg(replicas=3)) == L.ERR_INVALID_ARGUMENT
    assert gs(arr, cfg=L.adamw_cfg(replicas=R, elems_per_row=6)) == L.ERR_INVALID_ARGUMENT
    assert gs(arr, cfg=L.adamw_cfg(replicas=R, eps=0.0)) == L.ERR_INVALID_ARGUMENT
    assert gs(arr, cfg=L.adamw_cfg(replicas=R, betas=(1.0, 0.999))) == L.ERR_INVALID_ARGUMENT
    assert gs(arr, cfg=L.adamw_cfg(replicas=R, flags=0x10)) == L.ERR_INVALID_ARGUMENT
    for bad in (2, -1):
        assert gs(arr, cfg=L.adamw_cfg(replicas=R, hierarchical_stats=bad)) == \
            L.ERR_INVALID_ARGUMENT
    for ok in (0, 1):
        assert reached_device_check(L, gs(arr, cfg=L.adamw_cfg(replicas=R, hierarchical_stats=ok)))
    for other in (L.ADAMW_DEVICE_DECISION, L.ADAMW_GRAPH, L.ADAMW_MULTI_TENSOR):
        assert gs(arr, cfg=L.adamw_cfg(replicas=R, flags=L.ADAMW_HOST_GRAPH | other)) == \
            L.ERR_INVALID_ARGUMENT
    assert reached_device_check(L, gs(arr, cfg=L.adamw_cfg(replicas=R, flags=L.ADAMW_HOST_GRAPH)))
    assert gs(arr, cfg=L.adamw_cfg(replicas=R, flags=L.ADAMW_GRAPH | L.ADAMW_MULTI_TENSOR)) == \
        L.ERR_INVALID_ARGUMENT
    assert reached_device_check(L, gs(arr, cfg=L.adamw_cfg(replicas=R, flags=L.ADAMW_MULTI_TENSOR)))
    assert reached_device_check(L, gs(arr, cfg=L.adamw_cfg(replicas=R, flags=L.ADAMW_GRAPH)))
    assert gs(arr, state=L.optim_state(scale=0.0)) == L.ERR_INVALID_ARGUMENT
    assert gs(arr, state=L.optim_state(scale=float("inf"))) == L.ERR_INVALID_ARGUMENT
    # more statistics rows than two fan-in-1024 levels can take
    big, keepb = _param_sets(L, R, R, numel=(4096 * 1024 + 1) * 4, P=1)
    assert gs(big, P=1, cfg=L.adamw_cfg(replicas=R, elems_per_row=4)) == L.ERR_INVALID_ARGUMENT
    assert "elems_per_row" in L.last_error()
    # exactly at the limit is accepted
    ok, keepo = _param_sets(L, R, R, numel=4096 * 1024 * 4, P=1)
    assert reached_device_check(L, gs(ok, P=1, cfg=L.adamw_cfg(replicas=R, elems_per_row=4)))


def test_grad_sync_needs_f32_session(L, comm):
    R = 2
    h = comm(R, dtype=L.BF16)
    arr, keep = _param_sets(L, R, 1)
    cfg, state, rep = L.adamw_cfg(replicas=1), L.optim_state(), L.StepReport()
    st = L.raw("rcc_grad_sync_adamw", h, arr, 2, C.byref(cfg), C.byref(state), C.byref(rep), None)
    assert st == L.ERR_INVALID_ARGUMENT and "F32" in L.last_error()


def test_no_kernel_launched_by_validation(L, comm):
    before = L.launch_count()
    R = 8
    h = comm(R)
    S, Rv = L.ptr_array(addrs(R)), L.ptr_array(addrs(R, base=BASE * 2))
    n = L.size_array([4096] * R)
    for op in range(4):
        _ar(L, h, S, Rv, n, L.int_array([op] * R))
        L.raw("rcc_reduce_scatter", h, S, Rv, n, L.int_array([op] * R), None)
    L.raw("rcc_all_gather", h, S, Rv, n, None)
    assert L.launch_count() == before


# ---------------------------------------------------------------- all_to_all / list all_gather

def test_all_to_all_single_errors(L, comm):
    R = 4
    h = comm(R)
    S, Rv = L.ptr_array(addrs(R)), L.ptr_array(addrs(R, base=BASE * 2))

    def a2a(counts, recv=Rv, send=S):
        return L.raw("rcc_all_to_all_single", h, send, recv, L.size_array(counts), None)

    assert a2a([1002] * R) == L.ERR_SHAPE_MISMATCH
    assert a2a([1000, 1000, 1000, 996]) == L.ERR_SHAPE_MISMATCH
    assert a2a([0] * R, recv=L.ptr_array([None] * R)) == L.OK
    assert a2a([1000] * R, recv=L.ptr_array([None] + addrs(R, base=BASE * 2)[1:])) == \
        L.ERR_MISSING_REGISTRATION
    ov = addrs(R, base=BASE * 2)
    ov[3] = ov[2] + 64
    assert a2a([1000] * R, recv=L.ptr_array(ov)) == L.ERR_INVALID_ARGUMENT
    assert a2a([1000] * R, recv=S) == L.ERR_INVALID_ARGUMENT        # no in-place form
    assert reached_device_check(L, a2a([1000] * R))


def test_all_gather_list_errors(L, comm):
    R = 3
    h = comm(R)
    n = 100
    send = addrs(R)
    recv = [BASE * 2 + i * 4096 for i in range(R * R)]

    def agl(recv=recv, send=send):
        return L.raw("rcc_all_gather_list", h, L.ptr_array(send), L.ptr_array(recv),
                     L.size_array([n] * R), None)

    assert reached_device_check(L, agl())
    inplace = list(recv)
    for r in range(R):
        inplace[r * R + r] = send[r]                    # own entry is the input
    assert reached_device_check(L, agl(inplace))
    bad = list(recv)
    bad[5] = recv[4] + 8                                # two list entries overlap
    assert agl(bad) == L.ERR_INVALID_ARGUMENT
    bad = list(recv)
    bad[1] = send[1]                                    # rank 0's entry aliases rank 1's input
    assert agl(bad) == L.ERR_INVALID_ARGUMENT
    bad = list(recv)
    bad[7] = None
    assert agl(bad) == L.ERR_MISSING_REGISTRATION


def test_noalloc_wrapper_rejects_what_the_abi_cannot_see(L):
    """rcc_grad_stats_noalloc takes bare pointers and one element count, so the
    binding checks what the C call cannot: dtype, contiguity, equal sizes and
    the report's size (all rejected before any call into the library)."""
    import torch
    a = torch.zeros(8)
    rep = torch.zeros(3, dtype=torch.int32)
    bad = [([a, torch.zeros(7)], rep, None),                       # sizes differ
           ([a, torch.zeros(8, dtype=torch.bfloat16)], rep, None),  # not float32
           ([a, torch.zeros(16)[::2]], rep, None),                  # not contiguous
           ([a, a], torch.zeros(2, dtype=torch.int32), None),       # report < 12 bytes
           ([a, a], rep, torch.zeros(9)),                           # mean of another size
           ([], rep, None)]
    for grads, report, mean in bad:
        with pytest.raises(ValueError):
            L.grad_stats_noalloc(grads, 1.0, report, mean_grad=mean)


def test_nvtx_ranges_do_not_change_behaviour():
    """With RCC_NVTX=1 every call opens and closes an NVTX range (read once per
    process, so in a child process); statuses and messages stay the same."""
    import os
    import subprocess
    import sys
    code = (
        "import ctypes as C\n"
        "from gradient_sync_rcc_gb300 import rcc as L\n"
        "h = C.c_void_p()\n"
        "assert L.raw('rcc_register', 63, 4, 0, 1, C.byref(h)) == L.OK\n"
        "assert L.raw('rcc_register', 63, 4, 0, 1, C.byref(C.c_void_p())) == "
        "L.ERR_DUPLICATE_REGISTRATION\n"
        "assert L.raw('rcc_set_flags', h, 0x4) == L.ERR_INVALID_ARGUMENT\n"
        "assert L.raw('rcc_reset', h) == L.OK\n"
        "print('nvtx ok')\n")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    out = subprocess.run([sys.executable, "-c", code], cwd=root, capture_output=True, text=True,
                         env=dict(os.environ, RCC_NVTX="1"), timeout=120)
    assert out.returncode == 0 and "nvtx ok" in out.stdout, out.stdout + out.stderr


def test_marshalling_arrays():
    """The binding's argument arrays: pointer arrays map None and 0 to NULL;
    count and op arrays, which the library only reads, are shared between
    calls with the same contents and never between different contents."""
    from gradient_sync_rcc_gb300 import rcc
    p = rcc.ptr_array([0, None, 4096])
    assert list(p) == [None, None, 4096]
    a = rcc.size_array([8, 8, 7])
    assert list(a) == [8, 8, 7]
    assert rcc.size_array([8, 8, 7]) is a
    assert list(rcc.size_array([8, 8, 8])) == [8, 8, 8]
    assert rcc.int_array([8, 8, 7]) is not a and list(rcc.int_array([8, 8, 7])) == [8, 8, 7]
    for k in range(300):                      # the table is cleared, contents stay right
        assert list(rcc.size_array([k, k + 1])) == [k, k + 1]
