"""GPU parity of the Q4_K entry points (qmv_q4_k, qdequant_q4_k) against the CPU
oracle on the same seeded bytes.

Q4_K products are summed per 32-weight sub-block by the pages' algebraic split,
d sc_j * sum(q x) - dmin m_j * sum(x) (jouleclaw-loader-gguf BENCHMARKS, the
NEON Q4_K kernel).  The two sums are formed separately, so the rounding of a
row scales with S2 = sum (|d sc_j q| + |dmin m_j|) |x| rather than with
sum |w x|, which is 0 where a weight cancels exactly.  The bound is 2e-3 * S2
(plus the bf16 output term); S2 = 0 still demands exactly 0.

Aligned weights take the tensor-core kernel (exact codes, scales and mins
applied per sub-block in fp32); a weight pointer off 16 bytes takes the
exact CUDA-core kernel.
"""
import numpy as np
import pytest

import synth
from tolerance import check_matvec, to_f64

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def dev_u8(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def dev_act(a):
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16).cuda()
    return torch.from_numpy(a.copy()).cuda()


ODT = {"f32": torch.float32, "bf16": torch.bfloat16}


def run(qbw, w, x, N, K, odt, offset=0):
    if offset:
        buf = torch.zeros(w.size + 64, dtype=torch.uint8, device="cuda")
        buf[offset:offset + w.size] = dev_u8(w)
        wd = buf[offset:offset + w.size]
    else:
        wd = dev_u8(w)
    y = torch.full((N,), float("nan"), dtype=ODT[odt], device="cuda")
    qbw.qmv_q4_k(wd, dev_act(x), y, 1, N, K)
    torch.cuda.synchronize()
    assert qbw.fault_read(clear=True) == 0
    return to_f64(y)


@pytest.mark.parametrize("N,K", [(1, 256), (37, 512), (300, 2304), (1000, 5376), (129, 8192), (5413, 5376),
                                 (600, 65536)])
@pytest.mark.parametrize("xdt,odt", [("f32", "f32"), ("bf16", "bf16"), ("bf16", "f32")])
def test_qmv_q4_k(qbw, oracle, N, K, xdt, odt):
    w = synth.q4_k_weights(N, K, seed=N + K)
    x = synth.activations(K, seed=K + 5, dtype=xdt)
    y_ref, _ = oracle.qmv("q4_k", w, x, N, K)
    S2 = oracle.q4k_split_scale(w, x, N, K)
    for _ in range(2):    # the second call must find the split-tile scratch consumed
        y = run(qbw, w, x, N, K, odt)
        check_matvec(y, y_ref, S2, out_bf16=(odt == "bf16"), what=f"q4_k N={N} K={K}")


@pytest.mark.parametrize("offset", [2, 8])
def test_qmv_q4_k_misaligned_weights(qbw, oracle, offset):
    N, K = 200, 2048
    w = synth.q4_k_weights(N, K, seed=77)
    x = synth.activations(K, seed=78)
    y = run(qbw, w, x, N, K, "f32", offset=offset)
    y_ref, _ = oracle.qmv("q4_k", w, x, N, K)
    check_matvec(y, y_ref, oracle.q4k_split_scale(w, x, N, K), what="q4_k misaligned")


def test_qmv_q4_k_full_21504x5376(qbw, oracle):
    N, K = 21504, 5376
    w = synth.q4_k_weights(N, K, seed=1)
    x = synth.activations(K, seed=1)
    y = run(qbw, w, x, N, K, "f32")
    y_ref, _ = oracle.qmv("q4_k", w, x, N, K)
    worst = check_matvec(y, y_ref, oracle.q4k_split_scale(w, x, N, K), what="q4_k 21504x5376")
    assert worst < 1e-4


def test_qmv_q4_k_table_too_small_takes_bf16_code_form(qbw, oracle):
    # each CTA's units touch up to 55 super-block columns, more than the 8-bit form's
    # activation table holds (48): the bf16-code instantiation runs
    N, K = 4000, 65536
    w = synth.q4_k_weights(N, K, seed=65)
    x = synth.activations(K, seed=65)
    y = run(qbw, w, x, N, K, "f32")
    y_ref, _ = oracle.qmv("q4_k", w, x, N, K)
    check_matvec(y, y_ref, oracle.q4k_split_scale(w, x, N, K), what="q4_k K=65536 bf16-code form")


def test_qmv_q4_k_cancelling_weights(qbw, oracle):
    # d sc q = dmin m in every sub-block: every weight is exactly 0, while the
    # two split sums are not; the result must stay within 2e-3 of S2
    N, K = 64, 1024
    nb = N * K // 256
    half = np.array([0.25], dtype=np.float16).view(np.uint16)[0]
    eighth = np.array([0.125], dtype=np.float16).view(np.uint16)[0]
    # sc = 1, m = 4, q = 2: 0.25 * 1 * 2 - 0.125 * 4 = 0
    scales = np.array([1, 1, 1, 1, 4, 4, 4, 4, 0x11, 0x11, 0x11, 0x11], dtype=np.uint8)  # sc 4..7 = 1, m 4..7 = 1
    scales[8:] = 0x41                                                                   # m 4..7 = 4
    w = synth.q4_k_records([half] * nb, [eighth] * nb, np.tile(scales, nb), np.full(nb * 128, 0x22, np.uint8))
    assert np.all(oracle.dequant("q4_k", w, N, K) == 0.0)
    x = synth.activations(K, seed=3)
    y = run(qbw, w, x, N, K, "f32")
    S2 = oracle.q4k_split_scale(w, x, N, K)
    assert np.all(S2 > 0)
    check_matvec(y, np.zeros(N), S2, what="q4_k cancelling")


def test_qmv_q4_k_deterministic(qbw):
    N, K = 3000, 5376
    w = dev_u8(synth.q4_k_weights(N, K, seed=5))
    x = dev_act(synth.activations(K, seed=5))
    y1 = torch.empty(N, device="cuda")
    y2 = torch.empty(N, device="cuda")
    qbw.qmv_q4_k(w, x, y1, 1, N, K)
    qbw.qmv_q4_k(w, x, y2, 1, N, K)
    torch.cuda.synchronize()
    assert torch.equal(y1.view(torch.int32), y2.view(torch.int32))


@pytest.mark.parametrize("N,K", [(3, 256), (129, 2048), (50, 5376)])
def test_qdequant_q4_k_bit_exact(qbw, oracle, N, K):
    w = synth.q4_k_weights(N, K, seed=N * K)
    out = torch.empty(N, K, device="cuda")
    qbw.qdequant_q4_k(dev_u8(w), out, N, K)
    torch.cuda.synchronize()
    ref = oracle.dequant("q4_k", w, N, K)
    assert np.array_equal(out.cpu().numpy().view(np.uint32), ref.view(np.uint32))
