"""Python binding of librcc's C ABI (include/rcc.h): argument marshalling only.

Every collective and the gradient-sync step run inside librcc.so's CUDA
kernels; this module turns torch tensors into device pointers, element
counts and the current CUDA stream, calls the C entry point of the same name
and raises RccError on a non-zero status.  There is no fallback: if
librcc.so is missing, loading raises.

Low-level `raw_*` helpers pass arbitrary per-rank arrays straight through and
return the status code, for exercising the validation paths.
"""
import ctypes as C
import os

HERE = os.path.dirname(os.path.abspath(__file__))
# RCC_LIBRARY may name another build of the same library (e.g. one compiled
# with different tuning macros); there is no fallback either way.
LIB_PATH = os.environ.get("RCC_LIBRARY") or os.path.join(HERE, "librcc.so")

# status codes, dtypes, ops, flags (mirrors include/rcc.h)
OK = 0
ERR_DUPLICATE_REGISTRATION = 1
ERR_MISSING_REGISTRATION = 2
ERR_SHAPE_MISMATCH = 3
ERR_INCONSISTENT_OP = 4
ERR_INCONSISTENT_ROOT = 5
ERR_BROADCAST_SENDERS = 6
ERR_INVALID_ARGUMENT = 7
ERR_TIMEOUT = 8
ERR_CUDA = 9
F32, BF16 = 0, 1
SUM, MEAN, MAX, MIN = 0, 1, 2, 3
OPS = {"sum": SUM, "mean": MEAN, "max": MAX, "min": MIN}
DETERMINISTIC = 0x1
STEP_TIMING = 0x2
ADAMW_DEVICE_DECISION = 0x1
ADAMW_GRAPH = 0x2
ADAMW_MULTI_TENSOR = 0x4
ADAMW_HOST_GRAPH = 0x8
MAX_RANKS = 64

# every symbol include/rcc.h declares
SYMBOLS = ["rcc_register", "rcc_set_flags", "rcc_finish", "rcc_reset", "rcc_all_reduce",
           "rcc_reduce", "rcc_broadcast", "rcc_reduce_scatter", "rcc_all_gather",
           "rcc_grad_sync_adamw", "rcc_grad_stats_noalloc", "rcc_last_error_message",
           "rcc_status_string", "rcc_kernel_launch_count", "rcc_all_reduce_rank",
           "rcc_reduce_rank", "rcc_broadcast_rank", "rcc_reduce_scatter_rank",
           "rcc_all_gather_rank", "rcc_all_to_all_single", "rcc_all_gather_list",
           "rcc_last_step_times"]


class ParamSet(C.Structure):
    _fields_ = [("numel", C.c_size_t), ("rank_numel", C.POINTER(C.c_size_t)),
                ("grads", C.POINTER(C.c_void_p)), ("params", C.POINTER(C.c_void_p)),
                ("exp_avg", C.POINTER(C.c_void_p)), ("exp_avg_sq", C.POINTER(C.c_void_p)),
                ("mean_grad", C.c_void_p)]


class AdamWCfg(C.Structure):
    _fields_ = [("lr", C.c_double), ("beta1", C.c_double), ("beta2", C.c_double),
                ("eps", C.c_double), ("weight_decay", C.c_double),
                ("max_grad_norm", C.c_double), ("replicas", C.c_int32),
                ("hierarchical_stats", C.c_int32), ("elems_per_row", C.c_uint32),
                ("flags", C.c_uint32)]


class OptimState(C.Structure):
    _fields_ = [("step", C.c_int64), ("scale", C.c_double), ("growth_factor", C.c_double),
                ("backoff_factor", C.c_double), ("growth_interval", C.c_int32),
                ("growth_tracker", C.c_int32)]


class StepReport(C.Structure):
    _fields_ = [("sum_sq", C.c_double), ("grad_norm", C.c_double), ("scale_used", C.c_double),
                ("nonfinite", C.c_uint32), ("skipped", C.c_int32), ("clip_coef", C.c_float),
                ("combine_launches", C.c_int32), ("stats_rows", C.c_uint64),
                ("combine_region_bytes", C.c_uint64), ("update_launches", C.c_uint64),
                ("report_words", C.c_uint32 * 3), ("combine_levels", C.c_int32),
                ("updates_before_readback", C.c_int32)]


_lib = None
_PP = C.POINTER(C.c_void_p)


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                "librcc.so is not built (%s); build it with gradient_sync_rcc_gb300.build.build()"
                % LIB_PATH)
        L = C.CDLL(LIB_PATH)
        st = C.c_int
        L.rcc_register.argtypes = [C.c_int, C.c_int, C.c_int, C.c_uint, _PP]
        L.rcc_set_flags.argtypes = [C.c_void_p, C.c_uint]
        L.rcc_finish.argtypes = [C.c_void_p, C.c_void_p]
        L.rcc_reset.argtypes = [C.c_void_p]
        L.rcc_all_reduce.argtypes = [C.c_void_p, _PP, _PP, C.POINTER(C.c_size_t),
                                     C.POINTER(C.c_int), C.c_void_p]
        L.rcc_reduce.argtypes = [C.c_void_p, _PP, _PP, C.POINTER(C.c_size_t),
                                 C.POINTER(C.c_int), C.POINTER(C.c_int), C.c_void_p]
        L.rcc_broadcast.argtypes = [C.c_void_p, _PP, _PP, C.POINTER(C.c_size_t), C.c_void_p]
        L.rcc_reduce_scatter.argtypes = [C.c_void_p, _PP, _PP, C.POINTER(C.c_size_t),
                                         C.POINTER(C.c_int), C.c_void_p]
        L.rcc_all_gather.argtypes = [C.c_void_p, _PP, _PP, C.POINTER(C.c_size_t), C.c_void_p]
        L.rcc_grad_sync_adamw.argtypes = [C.c_void_p, C.POINTER(ParamSet), C.c_int,
                                          C.POINTER(AdamWCfg), C.POINTER(OptimState),
                                          C.POINTER(StepReport), C.c_void_p]
        L.rcc_grad_stats_noalloc.argtypes = [_PP, C.c_int, C.c_size_t, C.c_double, C.c_void_p,
                                             C.c_void_p, C.c_void_p]
        vp, sz = C.c_void_p, C.c_size_t
        L.rcc_all_reduce_rank.argtypes = [vp, C.c_int, vp, vp, sz, C.c_int, vp]
        L.rcc_reduce_rank.argtypes = [vp, C.c_int, vp, vp, sz, C.c_int, C.c_int, vp]
        L.rcc_broadcast_rank.argtypes = [vp, C.c_int, vp, vp, sz, vp]
        L.rcc_reduce_scatter_rank.argtypes = [vp, C.c_int, vp, vp, sz, C.c_int, vp]
        L.rcc_all_gather_rank.argtypes = [vp, C.c_int, vp, vp, sz, vp]
        L.rcc_all_to_all_single.argtypes = [vp, _PP, _PP, C.POINTER(C.c_size_t), vp]
        L.rcc_all_gather_list.argtypes = [vp, _PP, _PP, C.POINTER(C.c_size_t), vp]
        L.rcc_last_step_times.argtypes = [vp, C.POINTER(C.c_float)]
        for name in ("rcc_register", "rcc_set_flags", "rcc_finish", "rcc_reset", "rcc_all_reduce",
                     "rcc_reduce", "rcc_broadcast", "rcc_reduce_scatter", "rcc_all_gather",
                     "rcc_grad_sync_adamw", "rcc_grad_stats_noalloc", "rcc_all_reduce_rank",
                     "rcc_reduce_rank", "rcc_broadcast_rank", "rcc_reduce_scatter_rank",
                     "rcc_all_gather_rank", "rcc_all_to_all_single", "rcc_all_gather_list",
                     "rcc_last_step_times"):
            getattr(L, name).restype = st
        L.rcc_last_error_message.restype = C.c_char_p
        L.rcc_last_error_message.argtypes = []
        L.rcc_status_string.restype = C.c_char_p
        L.rcc_status_string.argtypes = [C.c_int]
        L.rcc_kernel_launch_count.restype = C.c_uint64
        L.rcc_kernel_launch_count.argtypes = []
        _lib = L
    return _lib


class RccError(RuntimeError):
    def __init__(self, status, message):
        self.status = status
        name = lib().rcc_status_string(status).decode()
        super().__init__("%s: %s" % (name, message))


def last_error():
    return lib().rcc_last_error_message().decode()


def _check(status):
    if status != OK:
        raise RccError(status, last_error())
    return status


def launch_count():
    return int(lib().rcc_kernel_launch_count())


# ------------------------------------------------------------- marshalling

_PTR_TYPES = {}
_CONST_ARRAYS = {}


def ptr_array(ptrs):
    """A void* array (None and 0 are NULL)."""
    ty = _PTR_TYPES.get(len(ptrs))
    if ty is None:
        ty = _PTR_TYPES[len(ptrs)] = C.c_void_p * len(ptrs)
    return ty(*ptrs)


def _const_array(ctype, vals):
    # count and op arrays repeat from call to call and the library only reads
    # them: one array per distinct content (the table is cleared past 256)
    key = (ctype, tuple(vals))
    arr = _CONST_ARRAYS.get(key)
    if arr is None:
        if len(_CONST_ARRAYS) > 256:
            _CONST_ARRAYS.clear()
        arr = _CONST_ARRAYS[key] = (ctype * len(vals))(*vals)
    return arr


def size_array(vals):
    """A read-only size_t array for the library's count arguments."""
    return _const_array(C.c_size_t, vals)


def int_array(vals):
    """A read-only int array for the library's op and root arguments."""
    return _const_array(C.c_int, vals)


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return C.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return C.c_void_p(stream)
    return C.c_void_p(stream.cuda_stream)


def _op(op):
    return OPS[op] if isinstance(op, str) else int(op)


# ------------------------------------------------------------- sessions

def _flags(deterministic, step_timing):
    return (DETERMINISTIC if deterministic else 0) | (STEP_TIMING if step_timing else 0)


def register(device=0, num_ranks=4, dtype=F32, deterministic=True, step_timing=False):
    """rcc_register; returns the session handle (an int)."""
    h = C.c_void_p()
    _check(lib().rcc_register(device, num_ranks, dtype, _flags(deterministic, step_timing),
                              C.byref(h)))
    return h.value


def set_flags(comm, deterministic=True, step_timing=False):
    _check(lib().rcc_set_flags(comm, _flags(deterministic, step_timing)))


def last_step_times(comm):
    """rcc_last_step_times: ms of the last timed grad-sync call's phases
    (statistics kernel, combines + report, report to first update launch,
    updates)."""
    out = (C.c_float * 4)()
    _check(lib().rcc_last_step_times(comm, out))
    return list(out)


def finish(comm, stream=None):
    _check(lib().rcc_finish(comm, _stream(stream)))


def reset(comm):
    _check(lib().rcc_reset(comm))


# ------------------------------------------------------------- collectives (torch tensors)

def all_reduce(comm, send, recv, op="sum", stream=None):
    R = len(send)
    _check(lib().rcc_all_reduce(comm, ptr_array([_ptr(t) for t in send]),
                                ptr_array([_ptr(t) for t in recv]),
                                size_array([t.numel() for t in send]),
                                int_array([_op(op)] * R), _stream(stream)))


def reduce(comm, send, recv_root, root, op="sum", stream=None):
    R = len(send)
    recv = [None] * R
    recv[root] = recv_root
    _check(lib().rcc_reduce(comm, ptr_array([_ptr(t) for t in send]),
                            ptr_array([_ptr(t) for t in recv]),
                            size_array([t.numel() for t in send]), int_array([_op(op)] * R),
                            int_array([root] * R), _stream(stream)))


def broadcast(comm, root_send, recv, root, stream=None):
    R = len(recv)
    send = [None] * R
    send[root] = root_send
    _check(lib().rcc_broadcast(comm, ptr_array([_ptr(t) for t in send]),
                               ptr_array([_ptr(t) for t in recv]),
                               size_array([root_send.numel()] * R), _stream(stream)))


def reduce_scatter(comm, send, recv, op="sum", stream=None):
    R = len(send)
    _check(lib().rcc_reduce_scatter(comm, ptr_array([_ptr(t) for t in send]),
                                    ptr_array([_ptr(t) for t in recv]),
                                    size_array([t.numel() for t in send]),
                                    int_array([_op(op)] * R), _stream(stream)))


def all_gather(comm, send, recv, stream=None):
    _check(lib().rcc_all_gather(comm, ptr_array([_ptr(t) for t in send]),
                                ptr_array([_ptr(t) for t in recv]),
                                size_array([t.numel() for t in send]), _stream(stream)))


def all_to_all_single(comm, send, recv, stream=None):
    _check(lib().rcc_all_to_all_single(comm, ptr_array([_ptr(t) for t in send]),
                                       ptr_array([_ptr(t) for t in recv]),
                                       size_array([t.numel() for t in send]), _stream(stream)))


def all_gather_list(comm, send, recv_lists, stream=None):
    """recv_lists[r][q] receives send[q]."""
    R = len(send)
    flat = [_ptr(recv_lists[r][q]) for r in range(R) for q in range(R)]
    _check(lib().rcc_all_gather_list(comm, ptr_array([_ptr(t) for t in send]), ptr_array(flat),
                                     size_array([t.numel() for t in send]), _stream(stream)))


# ------------------------------------------------------------- per-rank arrival (one thread per rank)

def all_reduce_rank(comm, rank, send, recv, op="sum", stream=None):
    _check(lib().rcc_all_reduce_rank(comm, rank, _ptr(send), _ptr(recv), send.numel(), _op(op),
                                     _stream(stream)))


def reduce_rank(comm, rank, send, recv, root, op="sum", stream=None):
    _check(lib().rcc_reduce_rank(comm, rank, _ptr(send), _ptr(recv), send.numel(), _op(op), root,
                                 _stream(stream)))


def broadcast_rank(comm, rank, send, recv, count, stream=None):
    _check(lib().rcc_broadcast_rank(comm, rank, _ptr(send), _ptr(recv), count, _stream(stream)))


def reduce_scatter_rank(comm, rank, send, recv, op="sum", stream=None):
    _check(lib().rcc_reduce_scatter_rank(comm, rank, _ptr(send), _ptr(recv), send.numel(),
                                         _op(op), _stream(stream)))


def all_gather_rank(comm, rank, send, recv, stream=None):
    _check(lib().rcc_all_gather_rank(comm, rank, _ptr(send), _ptr(recv), send.numel(),
                                     _stream(stream)))


# ------------------------------------------------------------- gradient sync

def adamw_cfg(lr=1e-3, betas=(0.9, 0.999), eps=1e-8, weight_decay=0.01, max_grad_norm=1.0,
              replicas=1, hierarchical_stats=True, elems_per_row=0, flags=0):
    return AdamWCfg(lr, betas[0], betas[1], eps, weight_decay, max_grad_norm, replicas,
                    int(hierarchical_stats), elems_per_row, flags)


def optim_state(scale=65536.0, growth_factor=2.0, backoff_factor=0.5, growth_interval=2000,
                step=0):
    return OptimState(step, scale, growth_factor, backoff_factor, growth_interval, 0)


class ParamSets:
    """Keeps the ctypes arrays of a list of parameter tensors alive.

    tensors: list of dicts with keys grads (R tensors), params, exp_avg,
    exp_avg_sq (replica lists) and optional mean_grad."""

    def __init__(self, tensors):
        self._keep = []
        self.arr = (ParamSet * len(tensors))()
        for i, t in enumerate(tensors):
            g = ptr_array([x.data_ptr() for x in t["grads"]])
            p = ptr_array([x.data_ptr() for x in t["params"]])
            m = ptr_array([x.data_ptr() for x in t["exp_avg"]])
            v = ptr_array([x.data_ptr() for x in t["exp_avg_sq"]])
            self._keep += [g, p, m, v]
            mg = t.get("mean_grad")
            self.arr[i] = ParamSet(t["params"][0].numel(), None, g, p, m, v,
                                   None if mg is None else mg.data_ptr())

    def __len__(self):
        return len(self.arr)


def grad_sync_adamw(comm, param_sets, cfg, state, stream=None):
    """rcc_grad_sync_adamw over a ParamSets; updates `state` in place and
    returns the StepReport."""
    rep = StepReport()
    _check(lib().rcc_grad_sync_adamw(comm, param_sets.arr, len(param_sets), C.byref(cfg),
                                     C.byref(state), C.byref(rep), _stream(stream)))
    return rep


def grad_stats_noalloc(grads, loss_scale, report, mean_grad=None, stream=None):
    """rcc_grad_stats_noalloc for one tensor: grads are R device tensors,
    report a device tensor of at least 12 bytes (e.g. torch.int32 x 3).

    The C call receives bare pointers and one element count, so it cannot
    see a short, strided or bf16 rank tensor; those are rejected here."""
    import torch
    if not grads:
        raise ValueError("grads is empty")
    n, dev = grads[0].numel(), grads[0].device
    for t in list(grads) + ([mean_grad] if mean_grad is not None else []):
        if t.dtype != torch.float32 or not t.is_contiguous():
            raise ValueError("gradients and mean_grad must be contiguous float32 tensors")
        if t.numel() != n or t.device != dev:
            raise ValueError("every gradient and mean_grad must have %d elements on %s" % (n, dev))
    if report.device != dev or not report.is_contiguous() or \
            report.numel() * report.element_size() < 12:
        raise ValueError("report must be a contiguous device tensor of at least 12 bytes on %s"
                         % dev)
    _check(lib().rcc_grad_stats_noalloc(ptr_array([g.data_ptr() for g in grads]), len(grads),
                                        n, float(loss_scale), _ptr(mean_grad),
                                        report.data_ptr(), _stream(stream)))


# ------------------------------------------------------------- raw calls (status only)

def raw(name, *args):
    return getattr(lib(), name)(*args)
