"""GPU parity of the mixed-bit matrices (int2-symmetric, int4-affine, int8)
through the C ABI, against the CPU oracle on the same seeded words, scales and
biases.

* Dequantization is bit-exact: sc q is exact in fp32, and sc c + bi is rounded
  once on both sides.
* y = W x is compared element by element with the matvec rule on the split's
  scale: |y - y_ref| <= 2e-3 S2 (+ the bf16 output rounding), S2 = sum (|sc q|
  + |bi|) |x| (S2 = S for the symmetric formats; the int4 kernel forms
  sc * sum(c x) and bi * sum(x) apart).
Shapes cover one and two rows per warp item, ragged row counts, rows shorter
than one pass of the warp, groups smaller and larger than a 16-byte word
group, per-channel scales (group = K), and the 31B profile's 5376 x 21504 and
21504 x 5376 shapes in full.

int4-affine, int2-symmetric and int8 matrices with groups of 32 (or a larger
power of two) take the tensor-core 8-bit form, with bf16 or fp32 x, from 5 MB
(int4), 4 MB (int2) or 16 MB (int8) of codes (10, 5 and 64 MB for K <= 4096):
the test_tc* cases cover ragged tiles, short and long rows,
constant fields, zero scales, repeatability and the fallback to the CUDA-core
kernel for scale arrays that are not 16-byte aligned.
"""
import numpy as np
import pytest

import synth
from tolerance import check_matvec, to_f64

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def dev(a):
    if a is None:
        return None
    return torch.from_numpy(np.ascontiguousarray(a).view(np.uint8).copy()).cuda()


def dev_act(a):
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16).cuda()
    return torch.from_numpy(a.copy()).cuda()


def run(qbw, bits, qp, sc, bi, G, x, N, K, odt=torch.float32):
    y = torch.full((N,), float("nan"), dtype=odt, device="cuda")
    qbw.qmv_mixbit(bits, dev(qp), dev(sc), dev(bi), G, dev_act(x), y, 1, N, K)
    torch.cuda.synchronize()
    assert qbw.fault_read(clear=True) == 0
    return y


SHAPES = [(1, 64, 32), (7, 128, 16), (2, 256, 256), (300, 2304, 32), (33, 1024, 64), (1000, 5376, 32),
          (129, 4096, 128), (64, 512, 512)]


@pytest.mark.parametrize("bits", [2, 4, 8])
@pytest.mark.parametrize("N,K,G", SHAPES)
def test_dequant_bit_exact(qbw, oracle, bits, N, K, G):
    qp, sc, bi = synth.mixbit_weights(bits, N, K, G, seed=N + K + G + bits)
    out = torch.empty(N, K, dtype=torch.float32, device="cuda")
    qbw.qdequant_mixbit(bits, dev(qp), dev(sc), dev(bi), G, out, N, K)
    torch.cuda.synchronize()
    ref = oracle.mixbit_dequant(bits, qp, sc, bi, G, N, K)
    assert np.array_equal(out.cpu().numpy().view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("bits", [2, 4, 8])
@pytest.mark.parametrize("N,K,G", SHAPES)
@pytest.mark.parametrize("xdt,odt", [("f32", torch.float32), ("bf16", torch.bfloat16), ("bf16", torch.float32)])
def test_qmv_small(qbw, oracle, bits, N, K, G, xdt, odt):
    qp, sc, bi = synth.mixbit_weights(bits, N, K, G, seed=3 * N + K + bits)
    x = synth.activations(K, seed=K + bits, dtype=xdt)
    y = run(qbw, bits, qp, sc, bi, G, x, N, K, odt)
    y_ref, _, S2 = oracle.qmv_mixbit(bits, qp, sc, bi, G, x, N, K)
    check_matvec(to_f64(y), y_ref, S2, out_bf16=(odt == torch.bfloat16), what=f"mixbit{bits} N={N} K={K} G={G}")


@pytest.mark.parametrize("bits", [2, 4, 8])
@pytest.mark.parametrize("N,K", [(21504, 5376), (5376, 21504)])
def test_qmv_full_size(qbw, oracle, bits, N, K):
    # the 31B profile's FFN shapes, groups of 32, every row compared
    qp, sc, bi = synth.mixbit_weights(bits, N, K, 32, seed=7 + bits)
    x = synth.activations(K, seed=8, dtype="bf16")
    y = run(qbw, bits, qp, sc, bi, 32, x, N, K)
    y_ref, _, S2 = oracle.qmv_mixbit(bits, qp, sc, bi, 32, x, N, K)
    check_matvec(to_f64(y), y_ref, S2, what=f"mixbit{bits} full {N}x{K}")


@pytest.mark.parametrize("bits,field,value", [(2, 2, -2), (2, 1, 1), (4, 15, 15), (4, 0, 0), (8, 128, -128)])
def test_constant_fields(qbw, oracle, bits, field, value):
    # every field equal: y[n] = sum over groups of (sc value + bi) * sum(x over the group)
    N, K, G = 130, 1024, 64
    qp = synth.pack_fields(np.full((N, K), field, dtype=np.uint32), bits)
    _, sc, bi = synth.mixbit_weights(bits, N, K, G, seed=field + 1)
    x = synth.activations(K, seed=field + 2)
    y = to_f64(run(qbw, bits, qp, sc, bi, G, x, N, K))
    xs = x.astype(np.float64).reshape(K // G, G).sum(axis=1)
    s = sc.view(np.float16).astype(np.float64).reshape(N, K // G)
    wv = s * value + (bi.view(np.float16).astype(np.float64).reshape(N, K // G) if bits == 4 else 0.0)
    ref = (wv * xs).sum(axis=1)
    _, _, S2 = oracle.qmv_mixbit(bits, qp, sc, bi, G, x, N, K)
    check_matvec(y, ref, S2, what=f"constant mixbit{bits}")


def test_zero_scales_give_exact_zero(qbw):
    N, K, G = 66, 512, 32
    for bits in (2, 4, 8):
        qp, sc, bi = synth.mixbit_weights(bits, N, K, G, seed=bits)
        sc = np.zeros_like(sc)
        bi = np.zeros_like(bi) if bi is not None else None
        y = run(qbw, bits, qp, sc, bi, G, synth.activations(K, seed=1), N, K)
        assert torch.all(y == 0)


def test_deterministic(qbw):
    N, K, G = 3000, 4096, 32
    for bits in (2, 4, 8):
        qp, sc, bi = synth.mixbit_weights(bits, N, K, G, seed=11)
        x = synth.activations(K, seed=12, dtype="bf16")
        a = run(qbw, bits, qp, sc, bi, G, x, N, K)
        b = run(qbw, bits, qp, sc, bi, G, x, N, K)
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))


@pytest.mark.parametrize("bits,K", [(2, 41728), (4, 36864), (8, 47872)])
def test_largest_k(qbw, oracle, bits, K):
    # the longest rows each format takes with groups of 16 (the activations and
    # the copy rings fill one CTA's 227 KB of shared memory), and one step more
    # is rejected
    N, G = 300, 16
    qp, sc, bi = synth.mixbit_weights(bits, N, K, G, seed=bits + 40)
    x = synth.activations(K, seed=bits + 41, dtype="bf16")
    y = run(qbw, bits, qp, sc, bi, G, x, N, K)
    y_ref, _, S2 = oracle.qmv_mixbit(bits, qp, sc, bi, G, x, N, K)
    check_matvec(to_f64(y), y_ref, S2, what=f"mixbit{bits} K={K}")
    K2 = K + 256
    qp2, sc2, bi2 = synth.mixbit_weights(bits, 2, K2, G, seed=1)
    y2 = torch.empty(2, dtype=torch.float32, device="cuda")
    with pytest.raises(qbw.QbwError) as err:
        qbw.qmv_mixbit(bits, dev(qp2), dev(sc2), dev(bi2), G, dev_act(synth.activations(K2, seed=2, dtype="bf16")),
                       y2, 1, 2, K2)
    assert err.value.status == 2           # QBW_ESHAPE


# int4-affine, int2-symmetric and int8, groups of 32, bf16 x, at least 5 MB
# (int4), 4 MB (int2) or 16 MB (int8) of codes (10, 5 and 64 MB for K <= 4096):
# the tensor-core form.
# (rows, K): a ragged last tile, the shortest rows (one K-group; int8: two, as
# one K-group would need more rows than the split plan's tile limit allows
# at its size threshold), the 31B profile's K, and long rows (84 K-groups)
TC_SHAPES = {4: [(3077, 5376), (80001, 256), (14000, 1536), (4000, 21504)],
             2: [(3077, 5376), (78200, 256), (24000, 1536), (4000, 21504)],
             8: [(3077, 5376), (125001, 512), (42000, 1536), (2000, 21504)]}
TC_CASES = [(b, N, K) for b in (4, 2, 8) for N, K in TC_SHAPES[b]]


def two_complement(field, bits):
    return field - (1 << bits) if bits != 4 and field >= (1 << (bits - 1)) else field


def route(qbw, bits, qp, sc, bi, G, x, N, K):
    """Whether the call takes the tensor-core form (asked of the library)."""
    return qbw.qmv_mixbit_route(bits, dev(qp), dev(sc), dev(bi), G, dev_act(x), N, K)


@pytest.mark.parametrize("bits,N,K", TC_CASES)
@pytest.mark.parametrize("xdt,odt", [("bf16", torch.float32), ("bf16", torch.bfloat16), ("f32", torch.float32)])
def test_tc(qbw, oracle, bits, N, K, xdt, odt):
    # bf16 x: two pieces per activation; fp32 x: three, the third in a second B
    # (int2 and int4 then read their scales from global memory)
    qp, sc, bi = synth.mixbit_weights(bits, N, K, 32, seed=N + K + bits)
    x = synth.activations(K, seed=K + 5, dtype=xdt)
    assert route(qbw, bits, qp, sc, bi, 32, x, N, K), "the case no longer takes the tensor-core form"
    y = run(qbw, bits, qp, sc, bi, 32, x, N, K, odt)
    y_ref, _, S2 = oracle.qmv_mixbit(bits, qp, sc, bi, 32, x, N, K)
    check_matvec(to_f64(y), y_ref, S2, out_bf16=(odt == torch.bfloat16), what=f"tc int{bits} {N}x{K}")


@pytest.mark.parametrize("bits,field", [(4, 0), (4, 15), (4, 8), (2, 0), (2, 1), (2, 2), (2, 3), (8, 0), (8, 127),
                                        (8, 128), (8, 255), (8, 17)])
def test_tc_constant_fields(qbw, oracle, bits, field):
    # every code equal: y[n] = sum over groups of (sc q + bi) * sum(x over the group)
    N, K, G = 3077, 5376, 32
    qp = synth.pack_fields(np.full((N, K), field, dtype=np.uint32), bits)
    _, sc, bi = synth.mixbit_weights(bits, N, K, G, seed=field + 3)
    x = synth.activations(K, seed=field + 4, dtype="bf16")
    assert route(qbw, bits, qp, sc, bi, G, x, N, K)
    y = to_f64(run(qbw, bits, qp, sc, bi, G, x, N, K))
    xs = (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64).reshape(K // G, G).sum(axis=1)
    s = sc.view(np.float16).astype(np.float64).reshape(N, K // G)
    b = bi.view(np.float16).astype(np.float64).reshape(N, K // G) if bits == 4 else 0.0
    ref = ((s * two_complement(field, bits) + b) * xs).sum(axis=1)
    _, _, S2 = oracle.qmv_mixbit(bits, qp, sc, bi, G, x, N, K)
    if bits != 4 and field == 0:
        assert np.all(y == 0)          # every weight is 0
    check_matvec(y, ref, S2, what=f"tc constant int{bits} {field}")


@pytest.mark.parametrize("bits", [4, 2, 8])
def test_tc_zero_scales(qbw, bits):
    N, K = 3077, 5376
    qp, sc, bi = synth.mixbit_weights(bits, N, K, 32, seed=2)
    y = run(qbw, bits, qp, np.zeros_like(sc), None if bi is None else np.zeros_like(bi), 32,
            synth.activations(K, seed=3, dtype="bf16"), N, K)
    assert torch.all(y == 0)


@pytest.mark.parametrize("bits", [4, 2, 8])
def test_tc_deterministic(qbw, bits):
    N, K = 21504, 5376
    qp, sc, bi = synth.mixbit_weights(bits, N, K, 32, seed=21)
    x = synth.activations(K, seed=22, dtype="bf16")
    a = run(qbw, bits, qp, sc, bi, 32, x, N, K)
    b = run(qbw, bits, qp, sc, bi, 32, x, N, K)
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))


@pytest.mark.parametrize("bits", [4, 2, 8])
def test_tc_unaligned_scales_fall_back(qbw, oracle, bits):
    # scales (and biases) 4 bytes past a 16-byte boundary: the CUDA-core kernel
    N, K = 3077, 5376
    qp, sc, bi = synth.mixbit_weights(bits, N, K, 32, seed=31)
    x = synth.activations(K, seed=32, dtype="bf16")

    def shifted(a):
        buf = torch.zeros(a.nbytes + 16, dtype=torch.uint8, device="cuda")
        buf[4:4 + a.nbytes] = dev(a)
        return buf[4:4 + a.nbytes]

    sc_s, bi_s = shifted(sc), None if bi is None else shifted(bi)
    assert route(qbw, bits, qp, sc, bi, 32, x, N, K)                   # aligned: tensor cores
    assert not qbw.qmv_mixbit_route(bits, dev(qp), sc_s, bi_s, 32, dev_act(x), N, K)
    y = torch.full((N,), float("nan"), dtype=torch.float32, device="cuda")
    qbw.qmv_mixbit(bits, dev(qp), sc_s, bi_s, 32, dev_act(x), y, 1, N, K)
    torch.cuda.synchronize()
    assert qbw.fault_read(clear=True) == 0
    y_ref, _, S2 = oracle.qmv_mixbit(bits, qp, sc, bi, 32, x, N, K)
    check_matvec(to_f64(y), y_ref, S2, what=f"int{bits} unaligned scales")


@pytest.mark.parametrize("bits", [4, 2, 8])
def test_tc_long_rows(qbw, oracle, bits):
    # K = 86016 (336 K-groups): beyond what the CUDA-core kernel can stage,
    # taken by the tensor-core form (every 128-row tile split across about 67
    # CTAs), with bf16 and fp32 x; the same rows with groups of 16 (CUDA cores
    # only) are rejected
    N, K = 200, 86016
    qp, sc, bi = synth.mixbit_weights(bits, N, K, 32, seed=71 + bits)
    for xdt in ("bf16", "f32"):
        x = synth.activations(K, seed=72, dtype=xdt)
        assert route(qbw, bits, qp, sc, bi, 32, x, N, K)
        y = run(qbw, bits, qp, sc, bi, 32, x, N, K)
        y_ref, _, S2 = oracle.qmv_mixbit(bits, qp, sc, bi, 32, x, N, K)
        check_matvec(to_f64(y), y_ref, S2, what=f"tc int{bits} K={K} {xdt}")
    qp16, sc16, bi16 = synth.mixbit_weights(bits, N, K, 16, seed=73)
    y32 = torch.empty(N, dtype=torch.float32, device="cuda")
    with pytest.raises(qbw.QbwError) as err:
        qbw.qmv_mixbit(bits, dev(qp16), dev(sc16), dev(bi16), 16, dev_act(synth.activations(K, seed=72, dtype="bf16")),
                       y32, 1, N, K)
    assert err.value.status == 2           # QBW_ESHAPE


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_route_cuda_core_cases(qbw, bits):
    # what stays on the CUDA-core kernel: groups below 32 or not a power of two,
    # rows not a multiple of 256, and matrices below the size thresholds
    N, K = 21504, 5376
    qp, sc, bi = synth.mixbit_weights(bits, N, K, 32, seed=91)
    xb = synth.activations(K, seed=92, dtype="bf16")
    assert route(qbw, bits, qp, sc, bi, 32, xb, N, K)
    assert route(qbw, bits, qp, sc, bi, 32, synth.activations(K, seed=92), N, K)      # fp32 x too
    for G in (16, 48):                                         # not a power of two of at least 32
        qpg, scg, big = synth.mixbit_weights(bits, N, K, G, seed=93)
        assert not route(qbw, bits, qpg, scg, big, G, xb, N, K)
    K2 = 5376 - 64                                             # 5312: K % 256 != 0
    qp2, sc2, bi2 = synth.mixbit_weights(bits, N, K2, 32, seed=94)
    assert not route(qbw, bits, qp2, sc2, bi2, 32, synth.activations(K2, seed=95, dtype="bf16"), N, K2)
    qs, ss, bs = synth.mixbit_weights(bits, 300, K, 32, seed=96)
    assert not route(qbw, bits, qs, ss, bs, 32, xb, 300, K)


# larger groups (a power of two): the threads read the scales and biases from
# global memory; K = 6144 for groups of 512 (5376 is not a multiple of 512)
GROUP_CASES = [(b, G, 3077, 5376) for b in (2, 4, 8) for G in (64, 128, 256)] + \
              [(b, 512, 3000, 6144) for b in (2, 4, 8)]


@pytest.mark.parametrize("bits,G,N,K", GROUP_CASES)
@pytest.mark.parametrize("xdt", ["bf16", "f32"])
def test_tc_larger_groups(qbw, oracle, bits, G, N, K, xdt):
    qp, sc, bi = synth.mixbit_weights(bits, N, K, G, seed=G + bits)
    x = synth.activations(K, seed=G + 1, dtype=xdt)
    assert route(qbw, bits, qp, sc, bi, G, x, N, K), "the case no longer takes the tensor-core form"
    y = run(qbw, bits, qp, sc, bi, G, x, N, K)
    y_ref, _, S2 = oracle.qmv_mixbit(bits, qp, sc, bi, G, x, N, K)
    check_matvec(to_f64(y), y_ref, S2, what=f"tc int{bits} G={G} {N}x{K}")


@pytest.mark.parametrize("bits", [4, 2, 8])
def test_tc_larger_groups_constant_fields(qbw, oracle, bits):
    N, K, G = 3077, 5376, 128
    field = {4: 11, 2: 3, 8: 200}[bits]
    qp = synth.pack_fields(np.full((N, K), field, dtype=np.uint32), bits)
    _, sc, bi = synth.mixbit_weights(bits, N, K, G, seed=5)
    x = synth.activations(K, seed=6, dtype="bf16")
    assert route(qbw, bits, qp, sc, bi, G, x, N, K)
    y = to_f64(run(qbw, bits, qp, sc, bi, G, x, N, K))
    xs = (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64).reshape(K // G, G).sum(axis=1)
    s = sc.view(np.float16).astype(np.float64).reshape(N, K // G)
    b = bi.view(np.float16).astype(np.float64).reshape(N, K // G) if bits == 4 else 0.0
    ref = ((s * two_complement(field, bits) + b) * xs).sum(axis=1)
    _, _, S2 = oracle.qmv_mixbit(bits, qp, sc, bi, G, x, N, K)
    check_matvec(y, ref, S2, what=f"tc constant int{bits} G={G}")
