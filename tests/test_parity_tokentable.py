"""GPU parity of the Q8_0 token table: the row gather qembed_q8_0 (bit-exact
against the oracle's dequantized rows; bf16 rounded to nearest even from
them) and the tied LM head, qmv_q8_0 over the whole table (2e-3 of
sum |w x| per output, checked on sampled row ranges at full size).

The full-size table is the token table of the 31B profile: 262144 rows of
5376 inputs (1.5 GB of Q8_0 blocks), generated once for the module.
"""
import numpy as np
import pytest

import synth
from tolerance import check_matvec, to_f64

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

VOCAB, HIDDEN = 262144, 5376


@pytest.fixture(scope="module")
def table():
    w = synth.q8_0_weights(VOCAB, HIDDEN, seed=12)
    return w, torch.from_numpy(w).cuda()


def ids_dev(ids):
    return torch.from_numpy(np.asarray(ids, dtype=np.int32)).cuda()


def expected_rows(oracle, w, N, K, ids):
    rb = synth.row_bytes("q8_0", K)
    rows = np.stack([np.frombuffer(w, dtype=np.uint8)[i * rb:(i + 1) * rb] for i in ids])
    return oracle.dequant("q8_0", rows.reshape(-1), len(ids), K).reshape(len(ids), K)


@pytest.mark.parametrize("N,K", [(1000, 2048), (37, 96), (5, 32)])
def test_embed_bit_exact_small(qbw, oracle, N, K):
    w = synth.q8_0_weights(N, K, seed=N + K)
    rng = np.random.default_rng(N)
    ids = np.concatenate([[0, N - 1, N - 1], rng.integers(0, N, 20)]).astype(np.int32)
    wd = torch.from_numpy(w).cuda()
    ref = expected_rows(oracle, w, N, K, ids)
    out32 = torch.full((len(ids), K), float("nan"), device="cuda")
    qbw.qembed_q8_0(wd, ids_dev(ids), out32, N, K)
    out16 = torch.empty(len(ids), K, dtype=torch.bfloat16, device="cuda")
    qbw.qembed_q8_0(wd, ids_dev(ids), out16, N, K)
    torch.cuda.synchronize()
    assert qbw.fault_read(clear=True) == 0
    got32 = out32.cpu().numpy()
    assert np.array_equal(got32.view(np.uint32), ref.astype(np.float32).view(np.uint32))
    got16 = out16.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(got16, oracle.round_bf16(ref.reshape(-1)).reshape(ref.shape))


def test_embed_full_size_table(qbw, oracle, table):
    w, wd = table
    ids = np.array([0, 1, 2, 131071, 200000, VOCAB - 2, VOCAB - 1, 7], dtype=np.int32)
    out = torch.empty(len(ids), HIDDEN, device="cuda")
    qbw.qembed_q8_0(wd, ids_dev(ids), out, VOCAB, HIDDEN)
    torch.cuda.synchronize()
    assert qbw.fault_read(clear=True) == 0
    ref = expected_rows(oracle, w, VOCAB, HIDDEN, ids)
    assert np.array_equal(out.cpu().numpy().view(np.uint32), ref.astype(np.float32).view(np.uint32))


def test_lm_head_full_size_sampled(qbw, oracle, table):
    # the tied LM head: logits = W_table h, one token, bf16 activations
    w, wd = table
    x = synth.activations(HIDDEN, seed=12, dtype="bf16")
    xd = torch.from_numpy(x.view(np.int16).copy()).view(torch.bfloat16).cuda()
    y = torch.empty(VOCAB, device="cuda")
    qbw.qmv_q8_0(wd, xd, y, 1, VOCAB, HIDDEN)
    torch.cuda.synchronize()
    assert qbw.fault_read(clear=True) == 0
    got = to_f64(y)
    for n0, n1 in ((0, 256), (131000, 131256), (VOCAB - 256, VOCAB)):
        y_ref, S = oracle.qmv_rows("q8_0", w, x, n0, n1, HIDDEN)
        check_matvec(got[n0:n1], y_ref, S, what=f"lm head rows {n0}..{n1}")


def test_embed_index_out_of_range(qbw):
    N, K = 64, 256
    wd = torch.from_numpy(synth.q8_0_weights(N, K, seed=3)).cuda()
    ids = ids_dev([5, -1, N, 6])
    out = torch.full((4, K), float("nan"), device="cuda")
    qbw.fault_read(clear=True)
    qbw.qembed_q8_0(wd, ids, out, N, K)
    torch.cuda.synchronize()
    assert qbw.fault_read(clear=True) == (1 << 3)
    got = out.cpu().numpy()
    assert np.all(got[1] == 0) and np.all(got[2] == 0)
    assert np.all(np.isfinite(got[0])) and np.all(np.isfinite(got[3]))


def test_embed_empty_and_rejects(qbw):
    N, K = 8, 64
    wd = torch.from_numpy(synth.q8_0_weights(N, K, seed=4)).cuda()
    out = torch.empty(0, K, device="cuda")
    qbw.qembed_q8_0(wd, ids_dev([]), out, N, K)
    bad = torch.empty(2, K, dtype=torch.float16, device="cuda")
    with pytest.raises(qbw.QbwError) as e:
        qbw.qembed_q8_0(wd, ids_dev([0, 1]), bad, N, K)
    assert e.value.status == 3
    with pytest.raises(qbw.QbwError) as e:
        qbw.qembed_q8_0(wd, ids_dev([0, 1]), torch.empty(2, 48, device="cuda"), N, 48)
    assert e.value.status == 2
