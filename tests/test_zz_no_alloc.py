"""GPU tests of qmm_q4_0_smallM_noalloc, the small-M product whose split-K
scratch is a static array inside the library.  The file name sorts last so that
the call's one-time set-up also runs after every other test has used the
library; it passes alone in a fresh process too.

Each case makes two noalloc calls in a row (the second one depends on the first
leaving the arrival counters at zero) and compares both with
qmm_q4_0_smallM on a caller workspace.  The header promises bit-identical
results, which is stricter than the parity tolerance.
"""
import numpy as np
import pytest

import synth
from tolerance import check_matvec, to_f64

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def dev_u8(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def dev_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16).copy()).view(torch.bfloat16).cuda()


def bits(Y):
    return Y.view(torch.int16) if Y.dtype == torch.bfloat16 else Y.view(torch.int32)


def compare_with_workspace_path(qbw, M, N, K, odt, seed):
    w = dev_u8(synth.q4_0_weights(N, K, seed=seed))
    X = dev_bf16(synth.activations((M, K), seed=seed, dtype="bf16"))
    need = qbw.qmm_q4_0_smallM_workspace_bytes(M, N, K)
    ws = torch.zeros(max(need, 256), dtype=torch.uint8, device="cuda")
    Y_ws = torch.empty(M, N, dtype=odt, device="cuda")
    qbw.qmm_q4_0_smallM(w, X, Y_ws, M, N, K, workspace=ws)
    outs = []
    for _ in range(2):
        Y = torch.full((M, N), float("nan"), dtype=odt, device="cuda")
        qbw.qmm_q4_0_smallM_noalloc(w, X, Y, M, N, K)
        outs.append(Y)
    torch.cuda.synchronize()
    assert qbw.fault_read(clear=True) == 0
    for Y in outs:
        assert torch.equal(bits(Y), bits(Y_ws))
    return w, X, outs[0], need


@pytest.mark.parametrize("M,N,K", [(8, 5376, 5376), (16, 5376, 5376), (32, 5376, 5376),
                                   (17, 256, 2048), (32, 128, 21504), (8, 4000, 21504)])
@pytest.mark.parametrize("odt", [torch.bfloat16, torch.float32])
def test_noalloc_matches_workspace_entry(qbw, M, N, K, odt):
    # on a 152-SM part the 5376-row shapes split K inside one cluster (no
    # scratch), the next two take the workspace path and the last one is a
    # stream-K plan (its shares in the scratch)
    _, _, _, need = compare_with_workspace_path(qbw, M, N, K, odt, seed=M + N + K)
    assert need <= qbw.NOALLOC_SCRATCH_BYTES
    if (M, N, K) == (8, 4000, 21504):
        # only the stream-K layout has this size: the 4096-byte counter region,
        # then one tagged 8-byte word per CTA (one per SM), token column and row
        sms = torch.cuda.get_device_properties(0).multi_processor_count
        assert need == 4096 + (sms * 8 * 128 * 8 + 255) // 256 * 256, "the case no longer takes the stream-K plan"


def test_noalloc_after_reported_fault(qbw):
    # A reported fault makes the next call zero-fill the static scratch again
    # before it runs; the calls after it must still match the workspace path.
    # The fault is the library's own bounded-wait self-test (a 20 ms wait on a
    # word nothing writes), not a GPU fault.
    qbw.selftest_wait(1, 20000)
    torch.cuda.synchronize()
    assert qbw.fault_read(clear=True) == 1 << 4
    for M, N, K in ((8, 4000, 21504), (17, 256, 2048)):
        compare_with_workspace_path(qbw, M, N, K, torch.bfloat16, seed=3 * M + K)


def test_noalloc_against_oracle(qbw, oracle):
    M, N, K = 16, 640, 4096
    w, X, Y, need = compare_with_workspace_path(qbw, M, N, K, torch.float32, seed=5)
    assert need > 0
    Y_ref, S = oracle.qmm_q4_0(w.cpu().numpy(), synth.activations((M, K), seed=5, dtype="bf16"), M, N, K)
    check_matvec(to_f64(Y), Y_ref, S, rel=1e-2, what="noalloc")


@pytest.mark.parametrize("M,N,K", [(8, 21504, 5376), (4, 100, 96)])
def test_noalloc_paths_without_scratch(qbw, M, N, K):
    # one split per tile, or the CUDA-core path: the call forwards unchanged
    assert qbw.qmm_q4_0_smallM_workspace_bytes(M, N, K) == 0
    compare_with_workspace_path(qbw, M, N, K, torch.bfloat16, seed=7)


def test_noalloc_largest_plans_fit(qbw):
    # The split plan keeps splits * tiles <= SM count, so the partial sums are at
    # most SMs * 32 * 128 * 4 bytes; on this part that is under the static limit.
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    worst = max(qbw.qmm_q4_0_smallM_workspace_bytes(32, N, 65536) for N in (128, 256, 384, 1024, 2048, 5376))
    assert worst <= sms * 32 * 128 * 4 + 4096
    if sms * 32 * 128 * 4 + 4096 <= qbw.NOALLOC_SCRATCH_BYTES:
        assert worst <= qbw.NOALLOC_SCRATCH_BYTES


def test_noalloc_rejects_bad_arguments(qbw):
    w = torch.zeros(256 * 8 * 18, dtype=torch.uint8, device="cuda")
    X = torch.zeros(8, 256, dtype=torch.bfloat16, device="cuda")
    Y = torch.empty(8, 256, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(qbw.QbwError) as e:
        qbw.qmm_q4_0_smallM_noalloc(w, X, Y, 33, 256, 256)
    assert e.value.status == 2
    with pytest.raises(qbw.QbwError) as e:
        qbw.qmm_q4_0_smallM_noalloc(w, X.float(), Y, 8, 256, 256)
    assert e.value.status == 3
