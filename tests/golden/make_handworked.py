"""Writes handworked_blocks.json and gelu_pins.json.

Every expected value here is worked out by hand in its ``derivation`` string
from the block definitions (w = d*q for Q8_0, w = d*(q-8) for Q4_0) and the
GELU formula; the script calls neither the oracle nor the CUDA library.
Run it from the repository root: ``python tests/golden/make_handworked.py``.
"""
import json
import os

HERE = os.path.dirname(os.path.abspath(__file__))


def hexb(bs):
    return bytes(bs).hex()


def onehot(k):
    return [1.0 if i == k else 0.0 for i in range(32)]


def blocks():
    cases = []
    # Q4_0, d = 1.0, qs[j] = j | (15-j) << 4: element j<16 has code j, element 16+j has code 15-j.
    blk = [0x00, 0x3C] + [(j & 0xF) | (((15 - j) & 0xF) << 4) for j in range(16)]
    for k, exp, why in [(0, -8.0, "element 0 = low nibble of qs[0] = 0; w = 1*(0-8)"),
                        (5, -3.0, "element 5 = low nibble of qs[5] = 5; w = 5-8"),
                        (15, 7.0, "element 15 = low nibble of qs[15] = 15; w = 15-8"),
                        (16, 7.0, "element 16 = high nibble of qs[0] = 15; w = 15-8"),
                        (20, 3.0, "element 20 = high nibble of qs[4] = 11; w = 11-8"),
                        (31, -8.0, "element 31 = high nibble of qs[15] = 0; w = 0-8")]:
        cases.append(dict(name=f"q4_0_nibble_position_e{k}", fmt="q4_0", block_hex=hexb(blk),
                          x=onehot(k), y=exp, derivation=why))
    cases.append(dict(
        name="q4_0_x_is_k", fmt="q4_0", block_hex=hexb(blk), x=[float(i) for i in range(32)], y=-248.0,
        derivation="sum_{j<16} (j-8)*j = 1240-960 = 280; sum_{j<16} (7-j)*(16+j) = 1792-1080-1240 = -528; "
                   "total -248 (a sum check only: the swapped nibble order gives the same total, the "
                   "one-hot cases pin the order)"))
    blk2 = [0x00, 0x3C] + [0xE1] * 16
    cases.append(dict(name="q4_0_low_half", fmt="q4_0", block_hex=hexb(blk2), x=[1.0] * 16 + [0.0] * 16,
                      y=-112.0, derivation="elements 0..15 take the low nibbles (code 1): 16*(1-8) = -112"))
    cases.append(dict(name="q4_0_high_half", fmt="q4_0", block_hex=hexb(blk2), x=[0.0] * 16 + [1.0] * 16,
                      y=96.0, derivation="elements 16..31 take the high nibbles (code 14): 16*(14-8) = 96"))
    blk3 = [0x00, 0x40] + [0x00] * 16
    cases.append(dict(name="q4_0_code0_is_minus8d", fmt="q4_0", block_hex=hexb(blk3), x=[1.0] * 32, y=-512.0,
                      derivation="d = 0x4000 = 2.0 (bytes 00 40, little-endian, first two bytes); code 0 -> "
                                 "w = 2*(0-8) = -16; 32*(-16) = -512"))
    blk4 = [0x00, 0x3C] + [0x88] * 16
    cases.append(dict(name="q4_0_code8_is_zero", fmt="q4_0", block_hex=hexb(blk4),
                      x=[float(i + 1) for i in range(32)], y=0.0, derivation="every code is 8 -> every weight is 0"))
    blk5 = [0x00, 0xBC] + [0xFF] * 16
    cases.append(dict(name="q4_0_negative_scale", fmt="q4_0", block_hex=hexb(blk5), x=[1.0] * 32, y=-224.0,
                      derivation="d = 0xBC00 = -1.0; code 15 -> w = -1*(15-8) = -7; 32*(-7) = -224"))
    blk6 = [0x01, 0x00] + [0xF0] * 16
    cases.append(dict(name="q4_0_subnormal_scale", fmt="q4_0", block_hex=hexb(blk6), x=[1.0] * 32,
                      y=(16 * (-8) + 16 * 7) * 2.0 ** -24,
                      derivation="d = 0x0001 = 2^-24 (smallest fp16 subnormal); low nibbles 0 -> -8, high "
                                 "nibbles 15 -> 7; 16*(-8)+16*7 = -16; y = -16 * 2^-24"))
    blk8 = [0x00, 0x3C] + [(k - 16) & 0xFF for k in range(32)]
    cases.append(dict(name="q8_0_ramp_sum", fmt="q8_0", block_hex=hexb(blk8), x=[1.0] * 32, y=-16.0,
                      derivation="d = 1.0, q[k] = k-16: sum_{k=0}^{31} (k-16) = 496 - 512 = -16"))
    cases.append(dict(name="q8_0_ramp_e0", fmt="q8_0", block_hex=hexb(blk8), x=onehot(0), y=-16.0,
                      derivation="q[0] = -16 (byte 0xF0, signed)"))
    cases.append(dict(name="q8_0_ramp_e31", fmt="q8_0", block_hex=hexb(blk8), x=onehot(31), y=15.0,
                      derivation="q[31] = 15"))
    blk9 = [0x00, 0x38] + [127] * 32
    cases.append(dict(name="q8_0_half_scale_max_code", fmt="q8_0", block_hex=hexb(blk9), x=[1.0] * 32,
                      y=2032.0, derivation="d = 0x3800 = 0.5; 0.5*127*32 = 2032"))
    blk10 = [0x01, 0x00] + [127] + [0] * 31
    cases.append(dict(name="q8_0_subnormal_scale", fmt="q8_0", block_hex=hexb(blk10), x=onehot(0),
                      y=127 * 2.0 ** -24, derivation="d = 0x0001 = 2^-24; q[0] = 127 -> 127 * 2^-24 exactly"))
    blk11 = [0x00, 0x3C] + [0x80] + [0xFF] * 31
    cases.append(dict(name="q8_0_minus128_and_minus1", fmt="q8_0", block_hex=hexb(blk11), x=[1.0] * 32,
                      y=-159.0, derivation="byte 0x80 is -128, bytes 0xFF are -1: -128 + 31*(-1) = -159"))
    return {
        "about": "Hand-worked single-block examples (N=1, K=32): y = sum_k w_k x_k.",
        "sources": [
            "gem docs/research/architecture.md, 'M4 Max operating assumptions': Q4_0 is a 32-element/18-byte "
            "block, Q8_0 the token-table/baseline format",
            "block layout read as the GGUF records block_q8_0 {fp16 d; int8 qs[32]} and block_q4_0 {fp16 d; "
            "uint8 qs[16]}, code j in the low nibble of qs[j], code j+16 in the high nibble (the pages name "
            "GGUF but do not print the record)",
            "w = d*q (Q8_0) and w = d*(q-8) (Q4_0) as the method defines them",
            "jouleclaw-loader-gguf BENCHMARKS, 'Half-width GPU residents + the BF16 negative result': fp16 "
            "subnormal scales must decode exactly (known-answer bit patterns)"],
        "cases": cases}


def gelu():
    return {
        "about": "GELU-tanh pins.",
        "sources": [
            "SafeC Gemma 4 design notes, 'Gated FFN': gelu_tanh(x) = 0.5 x (1 + tanh(sqrt(2/pi)(x + "
            "0.044715 x^3))), the tanh form, not the erf form",
            "SafeC Gemma 4 design notes, 'Further optimization: QKV projection fusion, fully GPU-chained "
            "FFN': large-gate regression, gate = up = 30 gives 900 (previously NaN)"],
        "cases": [
            {"name": "large_gate_regression", "gate": 30.0, "up": 30.0, "out": 900.0,
             "derivation": "tanh(sqrt(2/pi)*(30 + 0.044715*27000)) = 1 to double precision, so gelu(30) = 30 "
                           "and 30*30 = 900"},
            {"name": "zero_gate", "gate": 0.0, "up": 5.0, "out": 0.0, "derivation": "gelu(0) = 0"}]}


if __name__ == "__main__":
    with open(os.path.join(HERE, "handworked_blocks.json"), "w") as f:
        json.dump(blocks(), f, indent=1)
    with open(os.path.join(HERE, "gelu_pins.json"), "w") as f:
        json.dump(gelu(), f, indent=1)
