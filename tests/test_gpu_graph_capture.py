"""Collectives captured into a CUDA graph by the caller, then replayed.

Every kernel of the library is launched with programmatic dependent launch, so
a captured stream records programmatic edges between consecutive kernels.  The
graph here chains a reduce_scatter into an all_gather that reads its output,
then an all_reduce and a broadcast, and is replayed on fresh inputs written
into the same buffers: each replay must match the oracle bit for bit
(deterministic rank order), as the same calls do outside a graph.
"""
import numpy as np
import pytest
import torch

import oracle as orc
from gradient_sync_rcc_gb300 import rcc, synth
from gpu_util import DEV, session, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gradient_sync_rcc_gb300 import build
    build.build()
    orc.build.build()
    assert torch.cuda.is_available()


def test_collectives_replayed_from_a_cuda_graph():
    R, N = 4, 4 * 65539                       # ragged: N / R is odd
    ins = [torch.empty(N, device=DEV) for _ in range(R)]
    rs = [torch.empty(N // R, device=DEV) for _ in range(R)]
    ag = [torch.empty(N, device=DEV) for _ in range(R)]
    ar = [torch.empty(N, device=DEV) for _ in range(R)]
    bc = [torch.empty(N, device=DEV) for _ in range(R)]

    def calls(h):
        rcc.reduce_scatter(h, ins, rs, "sum")
        rcc.all_gather(h, rs, ag)             # reads what reduce_scatter wrote
        rcc.all_reduce(h, ins, ar, "mean")
        rcc.broadcast(h, ins[1], bc, root=1)

    with session(R) as h:
        stream = torch.cuda.Stream()
        with torch.cuda.stream(stream):       # warm-up outside the capture
            calls(h)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            calls(h)
        torch.cuda.synchronize()
        for trial in range(3):
            xs = synth.rank_buffers("uniform", R, N, 41, trial)
            for t, x in zip(ins, xs):
                t.copy_(torch.from_numpy(x))
            torch.cuda.synchronize()
            graph.replay()
            torch.cuda.synchronize()
            want_rs = orc.reduce_scatter(xs, "sum")
            for a, b in zip(rs, want_rs):
                assert to_host(a).tobytes() == b.tobytes(), trial
            want_ag = np.concatenate(want_rs)
            for a in ag:
                assert to_host(a).tobytes() == want_ag.tobytes(), trial
            want_ar = orc.reduce_f32(xs, "mean")
            for a in ar:
                assert to_host(a).tobytes() == want_ar.tobytes(), trial
            for a in bc:
                assert to_host(a).tobytes() == xs[1].tobytes(), trial
        del graph
