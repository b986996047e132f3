"""Pins of the oracle's Q4_K decode and product (CPU only).

The jouleclaw-loader-gguf BENCHMARKS page ("Q4_K matmul -- scalar fused vs
AMX-tiled", and the NEON follow-up) fixes what a Q4_K product computes: per
32-weight sub-block, w = d_sub * q - m_sub, summed as
d_sub * sum(a * q) - m_sub * sum(a).  The page gives no byte layout; the oracle
reads the GGUF block_q4_K record.  These tests pin the oracle to things other
than itself:

* a packer written here, statement by statement from the record's
  description, whose fields the oracle's unpacker must return;
* hand-built super-blocks whose every weight is computed here from the
  chosen fields;
* the closed form of constant blocks;
* the algebraic split, evaluated here from the fields;
* a dense fp64 product of the oracle's own dequantized matrix (accumulation
  and indexing).
"""
import numpy as np
import pytest

import synth

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def pack_scales(sc, m):
    """12 scale bytes from six-bit sub-block scales sc[0..7] and mins m[0..7]:
    bytes 0..3 hold sc[0..3] in their low six bits and the top two bits of
    sc[4..7] above them; bytes 4..7 the same for m; bytes 8..11 hold the low
    four bits of sc[4..7] (low nibble) and of m[4..7] (high nibble)."""
    s = [0] * 12
    for j in range(4):
        s[j] = (sc[j] & 63) | ((sc[j + 4] >> 4) << 6)
        s[j + 4] = (m[j] & 63) | ((m[j + 4] >> 4) << 6)
        s[j + 8] = (sc[j + 4] & 15) | ((m[j + 4] & 15) << 4)
    return np.array(s, dtype=np.uint8)


def pack_codes(q):
    """128 nibble bytes from 256 codes: chunk i (64 codes) keeps codes
    64i .. 64i + 31 in the low nibbles of bytes 32i .. 32i + 31 and codes
    64i + 32 .. 64i + 63 in their high nibbles."""
    out = np.zeros(128, dtype=np.uint8)
    for i in range(4):
        for l in range(32):
            out[32 * i + l] = (q[64 * i + l] & 15) | ((q[64 * i + 32 + l] & 15) << 4)
    return out


def unpack_code(qs, e):
    """Code of weight e, read here independently of the oracle."""
    byte = int(qs[32 * (e // 64) + (e % 32)])
    return byte & 15 if (e % 64) < 32 else byte >> 4


def f16_bits(v):
    return np.array([v], dtype=np.float16).view(np.uint16)[0]


def test_scale_fields_round_trip(oracle):
    rng = np.random.default_rng(5)
    cases = [(list(range(0, 64, 8)), list(range(63, 0, -8))), ([63] * 8, [0] * 8), ([0] * 8, [63] * 8),
             ([32, 31, 16, 15, 48, 47, 1, 62], [62, 1, 47, 48, 15, 16, 31, 32])]
    cases += [(list(rng.integers(0, 64, 8)), list(rng.integers(0, 64, 8))) for _ in range(50)]
    for sc, m in cases:
        s = pack_scales(sc, m)
        for j in range(8):
            assert oracle.q4k_scale_min(s, j) == (sc[j], m[j]), (sc, m, j)


def test_handbuilt_superblocks_dequant(oracle):
    # two super-blocks in one row (K = 512), every weight computed here
    blocks, expect = [], []
    for b, (d, dmin) in enumerate([(0.5, 0.25), (2.0 ** -10, 3.0 * 2.0 ** -12)]):
        sc = [(7 * j + 3 * b + 1) % 64 for j in range(8)]
        m = [(11 * j + 5 * b + 2) % 64 for j in range(8)]
        q = [(e * 7 + b) % 16 for e in range(256)]
        blocks.append(synth.q4_k_records([f16_bits(d)], [f16_bits(dmin)], pack_scales(sc, m), pack_codes(q)))
        expect += [d * sc[e // 32] * q[e] - dmin * m[e // 32] for e in range(256)]
    w = np.concatenate(blocks)
    got = oracle.dequant("q4_k", w, 1, 512)[0]
    ref = np.array(expect, dtype=np.float64).astype(np.float32)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("c,sc,m", [(0, 5, 0), (15, 63, 63), (8, 1, 8), (3, 40, 7)])
def test_constant_blocks_closed_form(oracle, c, sc, m):
    N, K = 3, 768
    d, dmin = 0.125, 0.0625
    nb = N * K // 256
    w = synth.q4_k_records([f16_bits(d)] * nb, [f16_bits(dmin)] * nb,
                           np.tile(pack_scales([sc] * 8, [m] * 8), nb), np.tile(pack_codes([c] * 256), nb))
    x = synth.activations(K, seed=c + sc)
    y, S = oracle.qmv("q4_k", w, x, N, K)
    wv = d * sc * c - dmin * m
    xs = x.astype(np.float64)
    np.testing.assert_allclose(y, wv * xs.sum(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(S, abs(wv) * np.abs(xs).sum(), rtol=1e-12, atol=1e-15)
    # d_sub q = m_sub exactly: every weight is 0, the sum is exactly 0
    if d * sc * c == dmin * m:
        assert np.all(y == 0.0) and np.all(S == 0.0)


def test_algebraic_split(oracle):
    # y = sum_j d sc_j sum(q x) - dmin m_j sum(x), evaluated here from the fields
    N, K = 5, 1024
    w = synth.q4_k_weights(N, K, seed=21)
    x = synth.activations(K, seed=22)
    y, _ = oracle.qmv("q4_k", w, x, N, K)
    xs = x.astype(np.float64)
    rec = w.reshape(N, K // 256, 144)
    for n in range(N):
        acc = 0.0
        for b in range(K // 256):
            blk = rec[n, b]
            d = float(np.frombuffer(blk[0:2].tobytes(), dtype="<f2")[0])
            dmin = float(np.frombuffer(blk[2:4].tobytes(), dtype="<f2")[0])
            for j in range(8):
                sc, m = oracle.q4k_scale_min(blk[4:16], j)
                seg = xs[b * 256 + 32 * j: b * 256 + 32 * j + 32]
                qx = sum(unpack_code(blk[16:], 32 * j + t) * seg[t] for t in range(32))
                acc += d * sc * qx - dmin * m * seg.sum()
        assert abs(acc - y[n]) <= 1e-12 * max(1.0, abs(y[n])), (n, acc, y[n])


@pytest.mark.parametrize("N,K", [(1, 256), (7, 512), (33, 1280)])
def test_product_matches_dense(oracle, N, K):
    w = synth.q4_k_weights(N, K, seed=N + K)
    for xdt in ("f32", "bf16"):
        x = synth.activations(K, seed=K, dtype=xdt)
        xs = oracle.bf16_to_f64(x) if xdt == "bf16" else x.astype(np.float64)
        y, S = oracle.qmv("q4_k", w, x, N, K)
        W = oracle.dequant("q4_k", w, N, K).astype(np.float64)
        np.testing.assert_allclose(y, W @ xs, rtol=1e-6, atol=1e-9)
        np.testing.assert_allclose(S, np.abs(W) @ np.abs(xs), rtol=1e-6, atol=1e-9)
        y2, _ = oracle.qmv_rows("q4_k", w, x, 1 if N > 1 else 0, N, K)
        np.testing.assert_array_equal(y2, y[1 if N > 1 else 0:])


def test_split_scale_definition(oracle):
    N, K = 4, 512
    w = synth.q4_k_weights(N, K, seed=30)
    x = synth.activations(K, seed=31)
    _, S = oracle.qmv("q4_k", w, x, N, K)
    S2 = oracle.q4k_split_scale(w, x, N, K)
    assert np.all(S2 >= S * (1 - 1e-12))
    # dmin = 0: |d_sub q| + 0 = |w|, so S2 = S
    rec = w.copy().reshape(-1, 144)
    rec[:, 2:4] = 0
    w0 = rec.reshape(-1)
    _, S0 = oracle.qmv("q4_k", w0, x, N, K)
    np.testing.assert_allclose(oracle.q4k_split_scale(w0, x, N, K), S0, rtol=1e-12)


def test_rejects_k_not_multiple_of_256(oracle):
    w = synth.q4_k_weights(1, 256, seed=1)
    with pytest.raises(ValueError):
        oracle.qmv("q4_k", w, synth.activations(288, seed=1), 1, 288)


def test_split_scale_handworked(oracle):
    """S2 of a hand-built super-block, worked out here by hand.

    The split forms d sc_j * sum(q x) and dmin m_j * sum(x) separately
    (jouleclaw-loader-gguf BENCHMARKS, "Q4_K matmul -- scalar fused vs
    AMX-tiled"), so its error scale takes |d sc_j q_k| and |dmin m_j| apart:
    S2 = sum_j sum_k (|d sc_j q_k| + |dmin m_j|) |x_k|.

    Fields: d = 1/2, dmin = 1/4, sc_j = j + 1, m_j = 2 j, every code of
    sub-block j equal to j, and x_k = +-1 (sign alternating), so |x_k| = 1.
    Sub-block j then adds 32 * (j (j + 1) / 2 + j / 2) = 16 j^2 + 32 j, and
    over j = 0..7: 16 * 140 + 32 * 28 = 2240 + 896 = 3136.  The plain scale
    sum |w x| differs: weight d sc_j q - dmin m_j = j (j + 1) / 2 - j / 2
    = j^2 / 2, so S = 32 * sum_j j^2 / 2 = 16 * 140 = 2240.

    A second row sets every code to 8 and sc_j = 1, m_j = 8 with d = dmin =
    1/4: each weight is 1/4 * 8 - 1/4 * 8 = 0, so S = 0, but S2 = 256 *
    (2 + 2) = 1024 (both terms of the split are nonzero and cancel).
    """
    rows = []
    sc = [j + 1 for j in range(8)]
    m = [2 * j for j in range(8)]
    q = [e // 32 for e in range(256)]
    rows.append(synth.q4_k_records([f16_bits(0.5)], [f16_bits(0.25)], pack_scales(sc, m), pack_codes(q)))
    rows.append(synth.q4_k_records([f16_bits(0.25)], [f16_bits(0.25)], pack_scales([1] * 8, [8] * 8),
                                   pack_codes([8] * 256)))
    w = np.concatenate(rows)
    x = np.array([1.0 if k % 2 == 0 else -1.0 for k in range(256)], dtype=np.float32)
    S2 = oracle.q4k_split_scale(w, x, 2, 256)
    assert S2[0] == 3136.0 and S2[1] == 1024.0, S2
    y, S = oracle.qmv("q4_k", w, x, 2, 256)
    assert S[0] == 2240.0 and S[1] == 0.0 and y[1] == 0.0, (S, y)
