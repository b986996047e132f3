"""Pins of the oracle's mixed-bit formats (CPU only).

The Core AI model zoo page on the Gemma-4-E2B raw-Metal port ("What shipped",
"Architecture") names three weight formats for its hand-written matrix-vector
kernels: int2-symmetric, int4-affine and int8, stored as quantized words qp,
scales sc and biases bi.  It gives no byte layout; the library documents one
(fields packed lowest bits first into 32-bit words, row after row; one fp16
scale, and for int4 one fp16 bias, per group of G weights of a row).  These
tests pin the oracle to things other than itself:

* rows worked out here by hand, field by field, from chosen words;
* the closed form of constant fields;
* an unpacker written here with numpy (its own shifts and sign handling) and
  a dense fp64 product;
* the definition of the affine split's scale S2 on a hand-built row.
"""
import numpy as np
import pytest

import synth


def f16(v):
    return np.array([v], dtype=np.float16).view(np.uint16)[0]


def test_handworked_int4_affine(oracle):
    # words 0x76543210, 0xFEDCBA98, 0x01234567, 0x89ABCDEF: fields lowest bits
    # first give codes 0..7, 8..15, 7..0, 15..8; scale 1, bias -8: w = c - 8
    qp = np.array([0x76543210, 0xFEDCBA98, 0x01234567, 0x89ABCDEF], dtype=np.uint32)
    sc = np.array([f16(1.0)], dtype=np.uint16)
    bi = np.array([f16(-8.0)], dtype=np.uint16)
    w = oracle.mixbit_dequant(4, qp, sc, bi, 32, 1, 32)[0]
    expect = list(range(-8, 0)) + list(range(0, 8)) + list(range(-1, -9, -1)) + list(range(7, -1, -1))
    assert w.tolist() == [float(v) for v in expect]
    x = np.ones(32, dtype=np.float32)
    y, S, S2 = oracle.qmv_mixbit(4, qp, sc, bi, 32, x, 1, 32)
    # sum of w: (-36) + 28 + (-36) + 28 = -16; sum |w| = 36 + 28 + 36 + 28 = 128;
    # S2 = sum (|c| + |bi|) = (0 + .. + 15) * 2 + 32 * 8 = 240 + 256 = 496
    assert y[0] == -16.0 and S[0] == 128.0 and S2[0] == 496.0


def test_handworked_int2_symmetric(oracle):
    # byte 0xE4 = 11 10 01 00: fields 0, 1, 2, 3 -> q = 0, 1, -2, -1;
    # byte 0x1B = 00 01 10 11: fields 3, 2, 1, 0 -> q = -1, -2, 1, 0.
    # Two groups of 16: scale 1/2 on the first word, 2 on the second.
    qp = np.array([0xE4E4E4E4, 0x1B1B1B1B], dtype=np.uint32)
    sc = np.array([f16(0.5), f16(2.0)], dtype=np.uint16)
    w = oracle.mixbit_dequant(2, qp, sc, None, 16, 1, 32)[0]
    expect = [0.0, 0.5, -1.0, -0.5] * 4 + [-2.0, -4.0, 2.0, 0.0] * 4
    assert w.tolist() == expect
    x = np.arange(32, dtype=np.float32)
    y, S, S2 = oracle.qmv_mixbit(2, qp, sc, None, 16, x, 1, 32)
    assert y[0] == float(np.dot(np.array(expect, dtype=np.float64), np.arange(32.0)))
    assert S[0] == S2[0]                      # no bias: the split's scale is S


def test_handworked_int8(oracle):
    # bytes 01 7F FF 80 02 FE 00 00 -> q = 1, 127, -1, -128, 2, -2, 0, 0; scale 1/4
    qp = np.array([0x80FF7F01, 0x0000FE02], dtype=np.uint32)
    sc = np.array([f16(0.25)], dtype=np.uint16)
    w = oracle.mixbit_dequant(8, qp, sc, None, 8, 1, 8)[0]
    assert w.tolist() == [0.25, 31.75, -0.25, -32.0, 0.5, -0.5, 0.0, 0.0]


def test_fp16_subnormal_scale_and_exact_rounding(oracle):
    # scale 2^-24 (fp16 0x0001) times code 127 is exact; an affine weight
    # sc * c + bi is rounded to fp32 once
    qp = np.array([0x7F7F7F7F], dtype=np.uint32)
    w = oracle.mixbit_dequant(8, qp, np.array([1], np.uint16), None, 4, 1, 4)[0]
    assert w.tolist() == [127 * 2.0 ** -24] * 4
    qp4 = np.array([0x00000001], dtype=np.uint32)          # codes 1, 0, 0, ...
    sc = np.array([f16(1.0 + 2.0 ** -10)], np.uint16)
    bi = np.array([f16(2.0 ** 11)], np.uint16)
    w4 = oracle.mixbit_dequant(4, qp4, sc, bi, 8, 1, 8)[0]
    exact = (1.0 + 2.0 ** -10) + 2.0 ** 11                 # 2049.0009765625
    assert w4[0] == np.float32(exact) and w4[1] == np.float32(2.0 ** 11)


@pytest.mark.parametrize("bits,field,value", [(2, 0, 0), (2, 1, 1), (2, 2, -2), (2, 3, -1),
                                              (4, 0, 0), (4, 9, 9), (4, 15, 15),
                                              (8, 5, 5), (8, 128, -128), (8, 255, -1)])
def test_constant_fields_closed_form(oracle, bits, field, value):
    N, K, G = 3, 128, 32
    fields = np.full((N, K), field, dtype=np.uint32)
    qp = synth.pack_fields(fields, bits)
    rng = np.random.default_rng(bits * 1000 + field)
    sc_v = (rng.uniform(0.5, 2.0, N * K // G)).astype(np.float16)
    bi_v = (rng.uniform(-8.0, 8.0, N * K // G)).astype(np.float16)
    x = synth.activations(K, seed=field)
    y, S, _ = oracle.qmv_mixbit(bits, qp, sc_v.view(np.uint16), bi_v.view(np.uint16) if bits == 4 else None,
                                G, x, N, K)
    xs = x.astype(np.float64).reshape(K // G, G).sum(axis=1)
    for n in range(N):
        s = sc_v[n * K // G:(n + 1) * K // G].astype(np.float64)
        wv = s * value + (bi_v[n * K // G:(n + 1) * K // G].astype(np.float64) if bits == 4 else 0.0)
        assert abs(y[n] - float((wv * xs).sum())) <= 1e-12 * max(1.0, abs(y[n]))


def numpy_weights(bits, qp, sc, bi, G, N, K):
    """Independent unpacker: every field by shifting its own word."""
    words = qp.reshape(N, K * bits // 32).astype(np.uint64)
    k = np.arange(K)
    word = words[:, (k * bits) // 32]
    field = (word >> ((k * bits) % 32).astype(np.uint64)) & ((1 << bits) - 1)
    field = field.astype(np.int64)
    if bits in (2, 8):
        field = np.where(field >= (1 << (bits - 1)), field - (1 << bits), field)
    scale = sc.view(np.float16).astype(np.float64).reshape(N, K // G).repeat(G, axis=1)
    w = scale * field
    if bits == 4:
        w = w + bi.view(np.float16).astype(np.float64).reshape(N, K // G).repeat(G, axis=1)
    return w, scale, field


@pytest.mark.parametrize("bits", [2, 4, 8])
@pytest.mark.parametrize("N,K,G", [(1, 64, 32), (5, 128, 64), (7, 256, 256), (3, 192, 16)])
def test_product_matches_numpy(oracle, bits, N, K, G):
    qp, sc, bi = synth.mixbit_weights(bits, N, K, G, seed=N + K + bits)
    W, scale, field = numpy_weights(bits, qp, sc, bi, G, N, K)
    np.testing.assert_array_equal(oracle.mixbit_dequant(bits, qp, sc, bi, G, N, K), W.astype(np.float32))
    for xdt in ("f32", "bf16"):
        x = synth.activations(K, seed=K + 1, dtype=xdt)
        xs = oracle.bf16_to_f64(x) if xdt == "bf16" else x.astype(np.float64)
        y, S, S2 = oracle.qmv_mixbit(bits, qp, sc, bi, G, x, N, K)
        np.testing.assert_allclose(y, W @ xs, rtol=1e-12, atol=1e-15)
        np.testing.assert_allclose(S, np.abs(W) @ np.abs(xs), rtol=1e-12, atol=1e-15)
        split = np.abs(scale * field)
        if bits == 4:
            split = split + np.abs(bi.view(np.float16).astype(np.float64).reshape(N, K // G).repeat(G, axis=1))
        np.testing.assert_allclose(S2, split @ np.abs(xs), rtol=1e-12, atol=1e-15)


def test_rejects_bad_shapes(oracle):
    qp, sc, bi = synth.mixbit_weights(4, 1, 64, 32, seed=1)
    with pytest.raises(ValueError):
        oracle.qmv_mixbit(4, qp, sc, bi, 48, synth.activations(64, seed=1), 1, 64)    # 64 % 48
    with pytest.raises(ValueError):
        oracle.qmv_mixbit(3, qp, sc, bi, 32, synth.activations(64, seed=1), 1, 64)
