"""ctypes binding of the OpenMP CPU baseline (rcc_oracle_omp.cpp), built into
oracle/liboracle_rcc_omp.so on first use.

Benchmark infrastructure: only the benchmark's CPU-baseline leg calls it.  No
test takes it as a reference; the reference is the single-threaded oracle.
"""
import ctypes as C
import os
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "rcc_oracle_omp.cpp")
LIB = os.path.join(HERE, "liboracle_rcc_omp.so")
CXXFLAGS = ["-std=c++17", "-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
            "-fno-fast-math"]
OPS = {"sum": 0, "mean": 1, "max": 2, "min": 3}

_lib = None


def build(force=False):
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    tmp = LIB + ".tmp%d" % os.getpid()
    subprocess.run(["g++", *CXXFLAGS, SRC, "-o", tmp], check=True, capture_output=True)
    os.replace(tmp, LIB)
    return LIB


def lib():
    global _lib
    if _lib is None:
        L = C.CDLL(build())
        L.orc_omp_all_reduce_f32.argtypes = [C.c_int, C.POINTER(C.c_void_p),
                                             C.POINTER(C.c_void_p), C.c_size_t, C.c_int, C.c_int]
        L.orc_omp_all_reduce_f32.restype = C.c_int
        _lib = L
    return _lib


def all_reduce(xs, outs, op, threads):
    """outs[r][:] = op over xs (float32 arrays of equal size), on `threads` threads."""
    for a in list(xs) + list(outs):
        assert a.dtype == np.float32 and a.flags["C_CONTIGUOUS"] and a.size == xs[0].size
    send = (C.c_void_p * len(xs))(*[a.ctypes.data for a in xs])
    recv = (C.c_void_p * len(outs))(*[a.ctypes.data for a in outs])
    st = lib().orc_omp_all_reduce_f32(len(xs), send, recv, xs[0].size, OPS[op], threads)
    if st != 0:
        raise ValueError("bad arguments")
