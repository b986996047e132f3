"""Pins for the oracle's products (dequant, matvec, gate+up, small-M).

The oracle is checked against what the pages and the mathematics fix:
hand-worked single blocks (tests/golden), the closed form for constant
blocks, a brute-force dense fp64 GEMV built from an independent numpy decode
of the same bytes, and invariants (exact dequant, linearity, row
permutation).  None of these reuse the oracle's own code.
"""
import json
import math
import os

import numpy as np
import pytest

import synth
from conftest import GOLDEN


# ------------------------------------------------------------ independent decode
def numpy_dense(fmt, w, N, K):
    """Dense fp64 W [N, K] from raw blocks, decoded with numpy only."""
    nb = K // 32
    bpb = synth.block_bytes(fmt)
    blk = np.asarray(w, dtype=np.uint8).reshape(N, nb, bpb)
    d = np.ascontiguousarray(blk[:, :, 0:2]).view("<f2")[..., 0].astype(np.float64)
    if fmt == "q8_0":
        q = np.ascontiguousarray(blk[:, :, 2:]).view(np.int8).astype(np.float64)
    else:
        qs = blk[:, :, 2:]
        q = np.concatenate([qs & 0x0F, qs >> 4], axis=2).astype(np.float64) - 8.0
    return (d[:, :, None] * q).reshape(N, K)


def widen(x):
    x = np.asarray(x)
    if x.dtype == np.uint16:
        return (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return x.astype(np.float64)


# ------------------------------------------------------------ golden blocks
def test_handworked_blocks(oracle):
    doc = json.load(open(os.path.join(GOLDEN, "handworked_blocks.json")))
    assert len(doc["cases"]) >= 15
    for c in doc["cases"]:
        w = np.frombuffer(bytes.fromhex(c["block_hex"]), dtype=np.uint8).copy()
        assert w.size == synth.block_bytes(c["fmt"])
        x = np.array(c["x"], dtype=np.float32)
        y, S = oracle.qmv(c["fmt"], w, x, 1, 32)
        assert y[0] == c["y"], (c["name"], y[0], c["y"])


def test_handworked_one_hots_agree_with_dequant(oracle):
    doc = json.load(open(os.path.join(GOLDEN, "handworked_blocks.json")))
    for c in doc["cases"]:
        x = np.array(c["x"])
        if np.count_nonzero(x) != 1 or x.max() != 1.0:
            continue
        w = np.frombuffer(bytes.fromhex(c["block_hex"]), dtype=np.uint8).copy()
        deq = oracle.dequant(c["fmt"], w, 1, 32)
        assert deq[0, int(np.argmax(x))] == c["y"], c["name"]


# ------------------------------------------------------------ closed form
@pytest.mark.parametrize("fmt,d_bits,code", [
    ("q8_0", 0x3C00, 5), ("q8_0", 0x0003, -128), ("q8_0", 0xB555, 127),
    ("q4_0", 0x2E66, 13), ("q4_0", 0x0001, 0), ("q4_0", 0x3800, 8), ("q4_0", 0xC000, 3)])
def test_constant_blocks_closed_form(oracle, fmt, d_bits, code):
    N, K = 5, 288
    w = synth.constant_blocks(fmt, N, K, d_bits, code)
    x = synth.activations(K, seed=11)
    y, S = oracle.qmv(fmt, w, x, N, K)
    d = float(np.array([d_bits], dtype=np.uint16).view(np.float16)[0])
    c = code if fmt == "q8_0" else code - 8
    exact = d * c * math.fsum(float(v) for v in x)
    sabs = abs(d * c) * math.fsum(abs(float(v)) for v in x)
    for n in range(N):
        assert abs(y[n] - exact) <= 1e-13 * max(sabs, 1e-300)
        assert abs(S[n] - sabs) <= 1e-13 * max(sabs, 1e-300)


def test_constant_blocks_gateup_closed_form(oracle):
    N, K = 3, 96
    wg = synth.constant_blocks("q4_0", N, K, 0x3C00, 12)   # w = +4
    wu = synth.constant_blocks("q4_0", N, K, 0x3800, 2)    # w = 0.5 * -6 = -3
    x = synth.activations(K, seed=3, dtype="bf16")
    sx = math.fsum(widen(x))
    r = oracle.gateup_q4_0(wg, wu, x, N, K)
    g, u = 4.0 * sx, -3.0 * sx
    gelu = 0.5 * g * (1.0 + math.tanh(math.sqrt(2.0 / math.pi) * (g + 0.044715 * g ** 3)))
    assert np.allclose(r["g"], g, rtol=1e-13) and np.allclose(r["u"], u, rtol=1e-13)
    assert np.allclose(r["out"], gelu * u, rtol=1e-12)


# ------------------------------------------------------------ brute force
SHAPES = [(1, 32), (3, 64), (8, 96), (8, 288), (5, 512)]


def _random_weights(fmt, N, K, seed):
    if seed % 2:
        return synth.weights(fmt, N, K, seed=seed)
    # edge scales: subnormals, zero, negative zero, largest finite, negatives
    pool = np.array([0x0001, 0x03FF, 0x0400, 0x0000, 0x8000, 0x7BFF, 0xFBFF, 0x3C00, 0x1234, 0x9234],
                    dtype=np.uint16)
    return synth.random_with_scale_bits(fmt, N, K, seed, pool)


@pytest.mark.parametrize("fmt", ["q8_0", "q4_0"])
@pytest.mark.parametrize("N,K", SHAPES)
@pytest.mark.parametrize("xdt", ["f32", "bf16"])
def test_brute_force_dense_gemv(oracle, fmt, N, K, xdt):
    for seed in (1, 2):
        w = _random_weights(fmt, N, K, seed)
        x = synth.activations(K, seed=seed + 100, dtype=xdt)
        W = numpy_dense(fmt, w, N, K)
        xd = widen(x)
        y_ref = W @ xd
        S_ref = np.abs(W * xd[None, :]).sum(axis=1)
        y, S = oracle.qmv(fmt, w, x, N, K)
        tol = 1e-12 * S_ref + 1e-300
        assert np.all(np.abs(y - y_ref) <= tol)
        assert np.allclose(S, S_ref, rtol=1e-12, atol=0)


@pytest.mark.parametrize("fmt", ["q8_0", "q4_0"])
def test_dequant_exact_in_fp32(oracle, fmt):
    # Every decoded weight is exactly representable in fp32 (11-bit scale times
    # a code of at most 8 bits), including subnormal and extreme scales.
    for seed in (1, 2, 4):
        N, K = 7, 256
        w = _random_weights(fmt, N, K, seed)
        deq = oracle.dequant(fmt, w, N, K)
        W = numpy_dense(fmt, w, N, K)
        assert np.array_equal(deq.astype(np.float64), W)


# ------------------------------------------------------------ invariants
@pytest.mark.parametrize("fmt", ["q8_0", "q4_0"])
def test_linearity(oracle, fmt):
    N, K = 6, 320
    w = synth.weights(fmt, N, K, seed=9)
    x1 = synth.activations(K, seed=1)
    x2 = synth.activations(K, seed=2)
    a, b = np.float32(0.75), np.float32(-2.0)   # exact scalings keep a*x1 + b*x2 close to exact
    xs = (a * x1.astype(np.float64) + b * x2.astype(np.float64))
    y1, S1 = oracle.qmv(fmt, w, x1, N, K)
    y2, S2 = oracle.qmv(fmt, w, x2, N, K)
    y3, _ = oracle.qmv(fmt, w, xs.astype(np.float32), N, K)
    # x3 itself is rounded to fp32 once: allow that rounding plus fp64 noise
    bound = 2 ** -23 * (abs(a) * S1 + abs(b) * S2) + 1e-12 * (S1 + S2)
    assert np.all(np.abs(y3 - (a * y1 + b * y2)) <= bound)


@pytest.mark.parametrize("fmt", ["q8_0", "q4_0"])
def test_row_permutation(oracle, fmt):
    N, K = 9, 160
    w = synth.weights(fmt, N, K, seed=4)
    rb = synth.row_bytes(fmt, K)
    perm = np.random.default_rng(0).permutation(N)
    wp = w.reshape(N, rb)[perm].reshape(-1)
    x = synth.activations(K, seed=5, dtype="bf16")
    y, S = oracle.qmv(fmt, w, x, N, K)
    yp, Sp = oracle.qmv(fmt, wp, x, N, K)
    assert np.array_equal(yp, y[perm]) and np.array_equal(Sp, S[perm])


def test_qmv_rows_matches_full(oracle):
    N, K = 10, 256
    w = synth.weights("q4_0", N, K, seed=12)
    x = synth.activations(K, seed=13)
    y, S = oracle.qmv("q4_0", w, x, N, K)
    ys, Ss = oracle.qmv_rows("q4_0", w, x, 3, 8, K)
    assert np.array_equal(ys, y[3:8]) and np.array_equal(Ss, S[3:8])


# ------------------------------------------------------------ small-M and gate+up
@pytest.mark.parametrize("M", [1, 3, 8])
def test_qmm_brute_force(oracle, M):
    N, K = 6, 192
    w = synth.weights("q4_0", N, K, seed=21)
    X = synth.activations((M, K), seed=22, dtype="bf16")
    Y, S = oracle.qmm_q4_0(w, X, M, N, K)
    W = numpy_dense("q4_0", w, N, K)
    Xd = widen(X)
    Y_ref = Xd @ W.T
    S_ref = np.abs(Xd)[:, None, :] * np.abs(W)[None, :, :]
    S_ref = S_ref.sum(axis=2)
    assert np.all(np.abs(Y - Y_ref) <= 1e-12 * S_ref + 1e-300)
    assert np.allclose(S, S_ref, rtol=1e-12)
    for m in range(M):
        y, s = oracle.qmv("q4_0", w, X[m], N, K)
        assert np.array_equal(Y[m], y) and np.array_equal(S[m], s)


def test_gateup_brute_force(oracle):
    torch = pytest.importorskip("torch")
    N, K = 7, 256
    wg = synth.weights("q4_0", N, K, seed=2, stream=0)
    wu = synth.weights("q4_0", N, K, seed=2, stream=1)
    x = synth.activations(K, seed=2, dtype="bf16")
    r = oracle.gateup_q4_0(wg, wu, x, N, K)
    xd = widen(x)
    g = numpy_dense("q4_0", wg, N, K) @ xd
    u = numpy_dense("q4_0", wu, N, K) @ xd
    out = torch.nn.functional.gelu(torch.from_numpy(g), approximate="tanh").numpy() * u
    scale = np.abs(numpy_dense("q4_0", wg, N, K) * xd).sum(1) + np.abs(numpy_dense("q4_0", wu, N, K) * xd).sum(1)
    assert np.all(np.abs(r["g"] - g) <= 1e-12 * scale)
    assert np.all(np.abs(r["u"] - u) <= 1e-12 * scale)
    assert np.all(np.abs(r["out"] - out) <= 1e-10 * (np.abs(out) + scale))
