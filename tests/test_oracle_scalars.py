"""Pins for the oracle's scalar building blocks: fp16/bf16 decoding, bf16
rounding and GELU-tanh.  Each is checked against something other than the
oracle itself: numpy's IEEE half type, the bf16 bit layout as fp32's top
half, exact rational arithmetic, PyTorch's tanh-GELU and erf-GELU.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

from conftest import GOLDEN


def test_fp16_decoder_all_patterns(oracle):
    # Every one of the 65536 binary16 patterns (incl. 2046 subnormals, +-0,
    # +-inf, NaNs) against numpy's own float16 -> float64 widening.
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.fp16_to_f64(bits)
    ref = bits.view(np.float16).astype(np.float64)
    finite = np.isfinite(ref)
    assert finite.sum() == 63488
    assert np.array_equal(got[finite], ref[finite])
    assert np.array_equal(np.signbit(got[finite]), np.signbit(ref[finite]))
    assert np.array_equal(np.isinf(got), np.isinf(ref))
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    # smallest subnormal and largest finite, from the format's definition
    assert oracle.fp16_to_f64(np.array([0x0001]))[0] == 2.0 ** -24
    assert oracle.fp16_to_f64(np.array([0x7BFF]))[0] == 65504.0


def test_bf16_decoder_all_patterns(oracle):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.bf16_to_f64(bits)
    with np.errstate(invalid="ignore"):
        ref = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    finite = np.isfinite(ref)
    assert np.array_equal(got[finite], ref[finite])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(np.isinf(got), np.isinf(ref))


def _bf16_float(b) -> float:
    return float((np.array([b], dtype=np.uint32) << 16).view(np.float32)[0])


def _bf16_value(b):
    return Fraction(_bf16_float(b))


def _round_bf16_exact(v: float) -> int:
    """Nearest-even bf16 by exhaustive comparison with exact rationals."""
    fv = Fraction(v)
    # candidates: bf16 values bracketing v, found through float32 truncation
    f32 = np.array([v], dtype=np.float32)  # nearby float32 (only used to find neighbours)
    top = int(f32.view(np.uint32)[0] >> 16)
    cands = {(top + d) & 0xFFFF for d in (-2, -1, 0, 1, 2)}
    best = None
    for c in sorted(cands):
        if not math.isfinite(_bf16_float(c)):
            continue
        cv = _bf16_value(c)
        err = abs(cv - fv)
        key = (err, (c & 1))  # ties: even mantissa (lowest bit 0) wins
        if best is None or key < best[0]:
            best = (key, c)
    return best[1]


def test_round_bf16_against_exact_rationals(oracle):
    g = np.random.default_rng(123)
    vals = list(g.standard_normal(3000) * np.exp(g.uniform(-40, 40, 3000)))
    # exact ties between two bf16 neighbours (both parities), and subnormals
    for b in (0x3F80, 0x3F81, 0x4000, 0x0001, 0x0002, 0x007F, 0x0080, 0x7F7E):
        lo = _bf16_value(b)
        hi = _bf16_value(b + 1)
        vals.append(float((lo + hi) / 2))
        vals.append(float(lo + (hi - lo) / 3))
        vals.append(-float((lo + hi) / 2))
    vals += [1e-45, -3e-41, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -9]
    got = oracle.round_bf16(np.array(vals))
    for v, b in zip(vals, got):
        exp = _round_bf16_exact(abs(v))
        if v < 0:
            exp |= 0x8000
        assert int(b) == exp, (v, hex(int(b)), hex(exp))


def test_round_bf16_matches_torch_for_fp32_inputs(oracle):
    torch = pytest.importorskip("torch")
    g = np.random.default_rng(5)
    v = (g.standard_normal(20000) * np.exp(g.uniform(-30, 30, 20000))).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.round_bf16(v.astype(np.float64))
    assert np.array_equal(got, ref)
    assert oracle.round_bf16(np.array([3.5e38]))[0] == 0x7F80  # beyond bf16 max -> inf


def test_gelu_golden_pins(oracle):
    doc = json.load(open(os.path.join(GOLDEN, "gelu_pins.json")))
    for c in doc["cases"]:
        out = oracle.gelu_tanh(np.array([c["gate"]]))[0] * c["up"]
        assert out == c["out"], c["name"]


def test_gelu_matches_torch_tanh_form(oracle):
    torch = pytest.importorskip("torch")
    v = np.concatenate([np.linspace(-12, 12, 4001), [-1e4, -88.0, -30.0, 30.0, 88.0, 1e4]])
    ref = torch.nn.functional.gelu(torch.from_numpy(v), approximate="tanh").numpy()
    got = oracle.gelu_tanh(v)
    # same formula, different evaluation order: agree to a few ulp of max(1, |v|)
    assert np.all(np.abs(got - ref) <= 4e-15 * np.maximum(1.0, np.abs(v)))


def test_gelu_is_tanh_form_not_erf_form(oracle):
    v = np.linspace(-6, 6, 2401)
    got = oracle.gelu_tanh(v)
    erf_form = np.array([0.5 * t * (1.0 + math.erf(t / math.sqrt(2.0))) for t in v])
    diff = np.abs(got - erf_form)
    # the two forms differ by a few 1e-4 at most, but do differ
    assert diff.max() < 1e-3
    assert diff.max() > 1e-5


def test_gelu_properties(oracle):
    v = np.linspace(-20, 20, 801)
    g = oracle.gelu_tanh(v)
    gm = oracle.gelu_tanh(-v)
    # gelu(v) - gelu(-v) = v for the tanh form (tanh is odd)
    assert np.allclose(g - gm, v, rtol=0, atol=1e-12)
    assert oracle.gelu_tanh(np.array([0.0]))[0] == 0.0
    big = oracle.gelu_tanh(np.array([1e4, -1e4, 1e30, -1e30]))
    assert np.all(np.isfinite(big))
    assert big[0] == 1e4 and big[1] == 0.0


def test_gelu_derivative_by_differences(oracle):
    v = np.linspace(-8, 8, 321)
    h = 1e-6
    fd = (oracle.gelu_tanh(v + h) - oracle.gelu_tanh(v - h)) / (2 * h)
    assert np.allclose(oracle.gelu_tanh_deriv(v), fd, rtol=0, atol=1e-7)
