"""GPU parity of the tensor-core M = 1 path under concurrency, through the C
ABI, against the CPU oracle.

When a 128-row output tile is split between CTAs, the kernels publish partial
sums in a static scratch array of the library, in a slot chosen on the device
from the launch's grid identifier, each word tagged with its launch.  These
tests run many such launches at the same time -- more calls in flight on
separate streams than there are slots near each other, and two captured CUDA
graphs replayed concurrently -- and check every output against the oracle and
that no wait ran out (fault word 0).
"""
import numpy as np
import pytest

import synth
from tolerance import check_matvec, to_f64

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

# 8192 x 5376 Q4_0 (24.8 MB) takes the tensor-core kernel; 5376 = 21 K-groups
# per tile and 1344 units over 152 CTAs, so most tiles are split between CTAs.
N, K = 8192, 5376
NMAT = 3


def dev_u8(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def dev_act(a):
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16).cuda()
    return torch.from_numpy(a.copy()).cuda()


@pytest.fixture(scope="module")
def mats():
    return [synth.q4_0_weights(N, K, seed=900 + i) for i in range(NMAT)]


def gate(stream_list, cycles=20_000_000):
    """Hold every stream behind one event recorded after a long sleep, so the
    calls queued behind it are released together."""
    side = torch.cuda.Stream()
    ev = torch.cuda.Event()
    with torch.cuda.stream(side):
        torch.cuda._sleep(cycles)
        ev.record(side)
    for s in stream_list:
        s.wait_event(ev)


def oracle_refs(oracle, w_np, xs):
    return [oracle.qmv("q4_0", w_np, x, N, K) for x in xs]


def test_many_streams_in_flight(qbw, oracle, mats):
    calls = 40      # more than the scratch's 32 slots
    assert qbw.fault_read(clear=True) == 0
    w_dev = [dev_u8(w) for w in mats]
    xs = [synth.activations(K, seed=1000 + i, dtype="bf16" if i % 4 else "f32") for i in range(calls)]
    x_dev = [dev_act(x) for x in xs]
    ys = [torch.full((N,), float("nan"), dtype=torch.float32, device="cuda") for _ in range(calls)]
    streams = [torch.cuda.Stream() for _ in range(calls)]
    torch.cuda.synchronize()
    gate(streams)
    for i in range(calls):
        qbw.qmv_q4_0(w_dev[i % NMAT], x_dev[i], ys[i], 1, N, K, stream=streams[i])
    torch.cuda.synchronize()
    assert qbw.fault_read(clear=True) == 0
    for i in range(calls):
        y_ref, S = oracle.qmv("q4_0", mats[i % NMAT], xs[i], N, K)
        check_matvec(to_f64(ys[i]), y_ref, S, what=f"stream call {i}")


def test_two_graphs_replayed_concurrently(qbw, oracle, mats):
    per_graph = 12
    assert qbw.fault_read(clear=True) == 0
    w_dev = [dev_u8(w) for w in mats]
    xs = [[synth.activations(K, seed=2000 + 100 * g + i, dtype="bf16") for i in range(per_graph)] for g in range(2)]
    x_dev = [[dev_act(x) for x in row] for row in xs]
    ys = [[torch.full((N,), float("nan"), dtype=torch.float32, device="cuda") for _ in range(per_graph)]
          for _ in range(2)]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    graphs = []
    for g in range(2):
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=streams[g]):
            for i in range(per_graph):
                qbw.qmv_q4_0(w_dev[(g + i) % NMAT], x_dev[g][i], ys[g][i], 1, N, K, stream=streams[g])
        graphs.append(graph)
    torch.cuda.synchronize()
    for y_row in ys:
        for y in y_row:
            y.fill_(float("nan"))
    for _ in range(4):
        gate(streams)
        for g in range(2):
            with torch.cuda.stream(streams[g]):
                graphs[g].replay()
    torch.cuda.synchronize()
    assert qbw.fault_read(clear=True) == 0
    for g in range(2):
        for i in range(per_graph):
            y_ref, S = oracle.qmv("q4_0", mats[(g + i) % NMAT], xs[g][i], N, K)
            check_matvec(to_f64(ys[g][i]), y_ref, S, what=f"graph {g} call {i}")
