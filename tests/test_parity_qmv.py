"""GPU parity of the M = 1 entry points (qmv_q8_0, qmv_q4_0, qmv_gateup_q4_0)
and of the dequantizers, through the C ABI, against the CPU oracle on the same
seeded bytes.  Small shapes compare every element and cover several tasks,
full 64-block chunks, ragged final chunks and the fallback path; the full-size
workloads (2048 x 2048 Q8_0, 21504 x 5376 Q4_0, gate+up of two 21504 x 5376
Q4_0 matrices) are compared element by element too, since the oracle finishes
them in well under a second each.
"""
import numpy as np
import pytest

import synth
from tolerance import check_gateup, check_matvec, to_f64

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

GUARD = 64


def dev_u8(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def dev_act(a):
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16).cuda()
    return torch.from_numpy(a.copy()).cuda()


class Guarded:
    """An output tensor with sentinel-filled guard regions on both sides."""

    def __init__(self, shape, dtype):
        n = int(np.prod(shape))
        self.buf = torch.full((n + 2 * GUARD,), -12345.0, dtype=dtype, device="cuda")
        self.t = self.buf[GUARD:GUARD + n].view(*shape)
        self.t.fill_(float("nan"))

    def check(self):
        head = self.buf[:GUARD]
        tail = self.buf[-GUARD:]
        assert torch.all(head == -12345.0) and torch.all(tail == -12345.0), "output guard region overwritten"


ODT = {"f32": torch.float32, "bf16": torch.bfloat16}

# (N, K): fast path shapes with and without a ragged final chunk, many tasks,
# single task, and shapes the fallback kernel takes (K % 256 != 0).
SHAPES = [(1, 256), (7, 256), (37, 512), (300, 2304), (513, 2048), (1000, 5376), (129, 8192), (64, 4352),
          (5, 32), (33, 96), (70, 800)]


def run_qmv(qbw, fmt, w_np, x_np, N, K, odt):
    out = Guarded((N,), ODT[odt])
    f = qbw.qmv_q8_0 if fmt == "q8_0" else qbw.qmv_q4_0
    f(dev_u8(w_np), dev_act(x_np), out.t, 1, N, K)
    torch.cuda.synchronize()
    out.check()
    return to_f64(out.t)


@pytest.mark.parametrize("fmt", ["q8_0", "q4_0"])
@pytest.mark.parametrize("N,K", SHAPES)
@pytest.mark.parametrize("xdt,odt", [("f32", "f32"), ("bf16", "bf16"), ("bf16", "f32"), ("f32", "bf16")])
def test_qmv_small(qbw, oracle, fmt, N, K, xdt, odt):
    w = synth.weights(fmt, N, K, seed=N * 7 + K)
    x = synth.activations(K, seed=K + 3, dtype=xdt)
    y = run_qmv(qbw, fmt, w, x, N, K, odt)
    y_ref, S = oracle.qmv(fmt, w, x, N, K)
    check_matvec(y, y_ref, S, out_bf16=(odt == "bf16"), what=f"{fmt} N={N} K={K}")


def test_qmv_q8_0_full_2048(qbw, oracle):
    N = K = 2048
    w = synth.q8_0_weights(N, K, seed=0)
    x = synth.activations(K, seed=0)
    y = run_qmv(qbw, "q8_0", w, x, N, K, "f32")
    y_ref, S = oracle.qmv("q8_0", w, x, N, K)
    worst = check_matvec(y, y_ref, S, what="q8_0 2048x2048")
    assert worst < 1e-4


def test_qmv_q4_0_full_21504x5376(qbw, oracle):
    N, K = 21504, 5376
    w = synth.q4_0_weights(N, K, seed=1)
    x = synth.activations(K, seed=1)
    y = run_qmv(qbw, "q4_0", w, x, N, K, "f32")
    y_ref, S = oracle.qmv("q4_0", w, x, N, K)
    worst = check_matvec(y, y_ref, S, what="q4_0 21504x5376")
    assert worst < 1e-4


# Shapes that take the tensor-core path (K % 256 == 0, at least 15 MB of Q4_0
# weights, 32 MB for gate+up): a ragged last 128-row tile, K-groups split over
# many CTAs (N = 600, K = 65536: every tile is shared by about 30 CTAs), and
# both activation and output dtypes.
TC_SHAPES = [(5413, 5376), (3000, 10240), (600, 65536)]


@pytest.mark.parametrize("N,K", TC_SHAPES)
@pytest.mark.parametrize("xdt,odt", [("f32", "f32"), ("bf16", "bf16")])
def test_qmv_q4_0_tensor_core_shapes(qbw, oracle, N, K, xdt, odt):
    w = synth.q4_0_weights(N, K, seed=N + K)
    x = synth.activations(K, seed=K + 11, dtype=xdt)
    y_ref, S = oracle.qmv("q4_0", w, x, N, K)
    for _ in range(2):   # the second call must find the split-tile scratch consumed
        y = run_qmv(qbw, "q4_0", w, x, N, K, odt)
        check_matvec(y, y_ref, S, out_bf16=(odt == "bf16"), what=f"q4_0 tc N={N} K={K}")
    assert qbw.fault_read(clear=True) == 0


# The tensor-core path's one-token Q4_0 products take the 8-bit operand form:
# codes c & 7 and the bit-3 indicator as e4m3 bytes (both 0 where c = 8), each
# activation as e4m3 pieces under a power-of-two scale per 32-element block
# (two pieces for bf16 activations, three for fp32).  15.1 MB of weights (the
# tensor-core path), a last tile of 8 rows.
F8_N, F8_K = 5000, 5376


@pytest.mark.parametrize("xdt", ["bf16", "f32"])
@pytest.mark.parametrize("code", [0, 7, 8, 9, 15])
def test_tc_8bit_constant_blocks(qbw, oracle, code, xdt):
    # code 8 is weight 0 everywhere: S = 0 and the output must be exactly 0
    w = synth.constant_blocks("q4_0", F8_N, F8_K, 0x3555, code)
    x = synth.activations(F8_K, seed=6, dtype=xdt)
    y = run_qmv(qbw, "q4_0", w, x, F8_N, F8_K, "f32")
    y_ref, S = oracle.qmv("q4_0", w, x, F8_N, F8_K)
    check_matvec(y, y_ref, S, what=f"tc 8-bit {xdt} constant code {code}")
    if code == 8:
        assert np.all(y == 0.0)


@pytest.mark.parametrize("xdt,odt", [("bf16", "f32"), ("bf16", "bf16"), ("f32", "f32")])
def test_tc_8bit_activation_ranges(qbw, oracle, xdt, odt):
    # Each 32-element block of x gets its own factor 10^-30 .. 10^30, a tenth
    # of the blocks are all zero, and a quarter carry one element 1000 times
    # the rest (an outlier channel): the per-block scale must place every
    # block in e4m3's range and keep the small elements of outlier blocks.
    N, K = F8_N, F8_K
    g = np.random.default_rng(61)
    x = g.standard_normal(K).astype(np.float32)
    nb = K // 32
    x *= np.repeat(10.0 ** g.integers(-30, 31, size=nb), 32).astype(np.float32)
    x.reshape(nb, 32)[g.random(nb) < 0.1] = 0.0
    out_blocks = np.flatnonzero(g.random(nb) < 0.25)
    x.reshape(nb, 32)[out_blocks, g.integers(0, 32, size=out_blocks.size)] *= 1000.0
    xin = synth.f32_to_bf16_bits(x) if xdt == "bf16" else x
    w = synth.q4_0_weights(N, K, seed=61)
    y_ref, S = oracle.qmv("q4_0", w, xin, N, K)
    y = run_qmv(qbw, "q4_0", w, xin, N, K, odt)
    worst = check_matvec(y, y_ref, S, out_bf16=(odt == "bf16"), what=f"tc 8-bit {xdt} activation ranges")
    if xdt == "f32" and odt == "f32":
        assert worst < 5e-4      # three pieces carry fp32 x to about 2^-12


@pytest.mark.parametrize("xdt", ["bf16", "f32"])
def test_tc_8bit_edge_scales(qbw, oracle, xdt):
    pool = np.array([0x0000, 0x8000, 0x0001, 0x03FF, 0x0400, 0x7BFF, 0xFBFF, 0x3C00, 0x2E66, 0xA123],
                    dtype=np.uint16)
    w = synth.random_with_scale_bits("q4_0", F8_N, F8_K, 18, pool)
    x = synth.activations(F8_K, seed=18, dtype=xdt)
    y = run_qmv(qbw, "q4_0", w, x, F8_N, F8_K, "f32")
    y_ref, S = oracle.qmv("q4_0", w, x, F8_N, F8_K)
    check_matvec(y, y_ref, S, what=f"tc 8-bit {xdt} edge scales")


@pytest.mark.parametrize("xdt", ["bf16", "f32"])
def test_tc_8bit_one_group_per_tile(qbw, oracle, xdt):
    # K = 256 with 15.8 MB of weights: every 128-row tile is a single unit,
    # so no tile is split and the activation table holds one group
    N, K = 110000, 256
    w = synth.q4_0_weights(N, K, seed=63)
    x = synth.activations(K, seed=63, dtype=xdt)
    y = run_qmv(qbw, "q4_0", w, x, N, K, "f32")
    y_ref, S = oracle.qmv("q4_0", w, x, N, K)
    check_matvec(y, y_ref, S, what=f"tc 8-bit K=256 {xdt}")


@pytest.mark.parametrize("xdt", ["bf16", "f32"])
def test_tc_table_too_small_takes_bf16_code_form(qbw, oracle, xdt):
    # K = 65536 over 32 tiles: each CTA's units touch up to 55 K-groups, more than
    # the 8-bit form's activation table holds (48), so the bf16-code form runs
    N, K = 4000, 65536
    w = synth.q4_0_weights(N, K, seed=64)
    x = synth.activations(K, seed=64, dtype=xdt)
    y = run_qmv(qbw, "q4_0", w, x, N, K, "f32")
    y_ref, S = oracle.qmv("q4_0", w, x, N, K)
    check_matvec(y, y_ref, S, what=f"tc bf16-code form K=65536 {xdt}")


def test_tc_fp32_gateup(qbw, oracle):
    # gate+up with fp32 activations: the 8-bit form with three pieces
    N, K = 5413, 5376
    wg = synth.q4_0_weights(N, K, seed=52, stream=0)
    wu = synth.q4_0_weights(N, K, seed=52, stream=1)
    x = synth.activations(K, seed=52, dtype="f32")
    o = run_gateup(qbw, wg, wu, x, N, K, "f32")
    ref = oracle.gateup_q4_0(wg, wu, x, N, K)
    check_gateup(o, ref, oracle, what="gateup fp32 x")


def run_gateup(qbw, wg, wu, x, N, K, odt):
    out = Guarded((N,), ODT[odt])
    qbw.qmv_gateup_q4_0(dev_u8(wg), dev_u8(wu), dev_act(x), out.t, 1, N, K)
    torch.cuda.synchronize()
    out.check()
    return to_f64(out.t)


@pytest.mark.parametrize("N,K", [(1, 256), (9, 512), (300, 2304), (1000, 5376), (40, 96)])
@pytest.mark.parametrize("odt", ["f32", "bf16"])
def test_gateup_small(qbw, oracle, N, K, odt):
    wg = synth.q4_0_weights(N, K, seed=2, stream=0)
    wu = synth.q4_0_weights(N, K, seed=2, stream=1)
    x = synth.activations(K, seed=2, dtype="bf16")
    o = run_gateup(qbw, wg, wu, x, N, K, odt)
    ref = oracle.gateup_q4_0(wg, wu, x, N, K)
    check_gateup(o, ref, oracle, out_bf16=(odt == "bf16"), what=f"gateup N={N} K={K}")


def test_gateup_full_21504x5376(qbw, oracle):
    N, K = 21504, 5376
    wg = synth.q4_0_weights(N, K, seed=2, stream=0)
    wu = synth.q4_0_weights(N, K, seed=2, stream=1)
    x = synth.activations(K, seed=2, dtype="bf16")
    o = run_gateup(qbw, wg, wu, x, N, K, "f32")
    ref = oracle.gateup_q4_0(wg, wu, x, N, K)
    check_gateup(o, ref, oracle, what="gateup full")


@pytest.mark.parametrize("odt", ["f32", "bf16"])
def test_gateup_tensor_core_ragged(qbw, oracle, odt):
    # 5413 rows: the last 128-row tile holds 37; 2 x 16.4 MB of weights
    N, K = 5413, 5376
    wg = synth.q4_0_weights(N, K, seed=51, stream=0)
    wu = synth.q4_0_weights(N, K, seed=51, stream=1)
    x = synth.activations(K, seed=51, dtype="bf16")
    o = run_gateup(qbw, wg, wu, x, N, K, odt)
    ref = oracle.gateup_q4_0(wg, wu, x, N, K)
    check_gateup(o, ref, oracle, out_bf16=(odt == "bf16"), what="gateup tc ragged")


def test_gateup_fused_buffer_and_large_gate(qbw, oracle):
    # One [gate ; up] buffer passed as two views.  Gate = up = 30 must give 900
    # (the large-gate regression), and gates in the thousands must stay finite.
    N, K = 64, 256
    rb = synth.row_bytes("q4_0", K)
    ones = synth.constant_blocks("q4_0", N, K, 0x3C00, 9)          # every weight +1
    x = np.zeros(K, dtype=np.float32)
    x[0] = 30.0
    fw = dev_u8(np.concatenate([ones, ones]))
    out = Guarded((N,), torch.float32)
    qbw.qmv_gateup_q4_0(fw[:N * rb], fw[N * rb:], dev_act(x), out.t, 1, N, K)
    torch.cuda.synchronize()
    out.check()
    assert np.all(to_f64(out.t) == 900.0)

    wg = synth.q4_0_weights(N, K, seed=12, stream=0)
    wu = synth.q4_0_weights(N, K, seed=12, stream=1)
    xl = (synth.activations(K, seed=12) * 3000.0).astype(np.float32)
    fw = dev_u8(np.concatenate([wg, wu]))
    out = Guarded((N,), torch.float32)
    qbw.qmv_gateup_q4_0(fw[:N * rb], fw[N * rb:], dev_act(xl), out.t, 1, N, K)
    torch.cuda.synchronize()
    out.check()
    o = to_f64(out.t)
    ref = oracle.gateup_q4_0(wg, wu, xl, N, K)
    assert np.abs(ref["g"]).max() > 100.0
    assert np.all(np.isfinite(o))
    check_gateup(o, ref, oracle, what="gateup large gates")


@pytest.mark.parametrize("fmt", ["q8_0", "q4_0"])
def test_deterministic(qbw, fmt):
    N, K = 3000, 5376
    w = dev_u8(synth.weights(fmt, N, K, seed=5))
    x = dev_act(synth.activations(K, seed=5))
    y1 = torch.empty(N, device="cuda")
    y2 = torch.empty(N, device="cuda")
    f = qbw.qmv_q8_0 if fmt == "q8_0" else qbw.qmv_q4_0
    f(w, x, y1, 1, N, K)
    f(w, x, y2, 1, N, K)
    torch.cuda.synchronize()
    assert torch.equal(y1.view(torch.int32), y2.view(torch.int32))


@pytest.mark.parametrize("fmt", ["q8_0", "q4_0"])
@pytest.mark.parametrize("offset", [2, 6])
def test_misaligned_weights_take_the_exact_fallback(qbw, oracle, fmt, offset):
    N, K = 100, 2048
    w = synth.weights(fmt, N, K, seed=8)
    buf = torch.zeros(w.size + 64, dtype=torch.uint8, device="cuda")
    buf[offset:offset + w.size] = dev_u8(w)
    x = synth.activations(K, seed=8)
    y = torch.empty(N, device="cuda")
    f = qbw.qmv_q8_0 if fmt == "q8_0" else qbw.qmv_q4_0
    f(buf[offset:offset + w.size], dev_act(x), y, 1, N, K)
    torch.cuda.synchronize()
    y_ref, S = oracle.qmv(fmt, w, x, N, K)
    check_matvec(to_f64(y), y_ref, S, what="misaligned")


@pytest.mark.parametrize("fmt", ["q8_0", "q4_0"])
def test_edge_scales(qbw, oracle, fmt):
    # zero, negative zero, subnormal, largest and negative fp16 scales
    pool = np.array([0x0000, 0x8000, 0x0001, 0x03FF, 0x0400, 0x7BFF, 0xFBFF, 0x3C00, 0x2E66, 0xA123],
                    dtype=np.uint16)
    N, K = 257, 2304
    w = synth.random_with_scale_bits(fmt, N, K, 17, pool)
    x = synth.activations(K, seed=17)
    y = run_qmv(qbw, fmt, w, x, N, K, "f32")
    y_ref, S = oracle.qmv(fmt, w, x, N, K)
    check_matvec(y, y_ref, S, what="edge scales")


@pytest.mark.parametrize("fmt,code", [("q8_0", 0), ("q4_0", 8), ("q8_0", -128), ("q4_0", 0), ("q4_0", 15)])
def test_constant_blocks(qbw, oracle, fmt, code):
    N, K = 96, 2048
    w = synth.constant_blocks(fmt, N, K, 0x3555, code)
    x = synth.activations(K, seed=4)
    y = run_qmv(qbw, fmt, w, x, N, K, "f32")
    y_ref, S = oracle.qmv(fmt, w, x, N, K)
    check_matvec(y, y_ref, S, what="constant blocks")
    if S.max() == 0:
        assert np.all(y == 0)


def test_large_k_beyond_shared_memory(qbw, oracle):
    # K = 65536: the staged fp32 activations alone exceed shared memory, so
    # the planner declines the streaming kernel and the fallback runs.
    N, K = 48, 65536
    w = synth.q4_0_weights(N, K, seed=30)
    x = synth.activations(K, seed=30, dtype="bf16")
    y = run_qmv(qbw, "q4_0", w, x, N, K, "f32")
    y_ref, S = oracle.qmv("q4_0", w, x, N, K)
    check_matvec(y, y_ref, S, what="K=65536")


@pytest.mark.parametrize("fmt", ["q8_0", "q4_0"])
@pytest.mark.parametrize("N,K", [(3, 32), (129, 2048), (50, 5376)])
def test_dequant_bit_exact(qbw, oracle, fmt, N, K):
    pool = np.array([0x0001, 0x03FF, 0x0000, 0x8000, 0x7BFF, 0xFBFF, 0x3C00, 0x1234], dtype=np.uint16)
    for w in (synth.weights(fmt, N, K, seed=3), synth.random_with_scale_bits(fmt, N, K, 9, pool)):
        out = Guarded((N, K), torch.float32)
        f = qbw.qdequant_q8_0 if fmt == "q8_0" else qbw.qdequant_q4_0
        f(dev_u8(w), out.t, N, K)
        torch.cuda.synchronize()
        out.check()
        ref = oracle.dequant(fmt, w, N, K)
        got = out.t.cpu().numpy()
        assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


def test_no_fault_recorded(qbw):
    assert qbw.fault_read(clear=True) == 0


@pytest.mark.parametrize("xdt,offset", [("f32", 1), ("f32", 2), ("bf16", 1), ("bf16", 3)])
def test_activations_not_vector_aligned(qbw, oracle, xdt, offset):
    # x aligned to its dtype only: the staging falls back to scalar loads
    N, K = 300, 2304
    w = synth.q4_0_weights(N, K, seed=40)
    x = synth.activations(K, seed=40, dtype=xdt)
    full = dev_act(np.concatenate([x[:offset], x]))   # x starts `offset` elements in
    y = torch.empty(N, device="cuda")
    qbw.qmv_q4_0(dev_u8(w), full[offset:], y, 1, N, K)
    torch.cuda.synchronize()
    y_ref, S = oracle.qmv("q4_0", w, x, N, K)
    check_matvec(to_f64(y), y_ref, S, what=f"x offset {offset}")
