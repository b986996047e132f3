"""Failure detection on the GPU, without a GPU fault.

Every wait in the kernels is bounded: when a wait runs out, the kernel records
a code in the library's fault word and returns, so the context stays usable and
the host learns of it through qbw_fault_read.  qbw_selftest_wait runs each kind
of wait on something nothing will complete, with a short limit (a flag that
nothing sets), so the timeout path itself is exercised.
"""
import time

import numpy as np
import pytest

import synth
from tolerance import check_matvec, to_f64

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.mark.parametrize("which,bit", [(0, 1 << 1), (1, 1 << 4)])
def test_bounded_wait_reports_and_returns(qbw, oracle, which, bit):
    qbw.fault_read(clear=True)
    limit_us = 20000
    t0 = time.perf_counter()
    qbw.selftest_wait(which, limit_us)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert qbw.fault_read(clear=True) == bit
    assert dt >= limit_us * 1e-6          # the wait did wait, then gave up
    assert qbw.fault_read(clear=True) == 0
    # the context still runs the library's kernels correctly
    N, K = 300, 2304
    w = synth.q4_0_weights(N, K, seed=9)
    x = synth.activations(K, seed=9)
    y = torch.empty(N, device="cuda")
    qbw.qmv_q4_0(torch.from_numpy(w).cuda(), torch.from_numpy(x).cuda(), y, 1, N, K)
    torch.cuda.synchronize()
    y_ref, S = oracle.qmv("q4_0", w, x, N, K)
    check_matvec(to_f64(y), y_ref, S, what="after a timed-out wait")
    assert qbw.fault_read(clear=True) == 0
