"""The oracle's pins must catch plausible mistakes.

Each case copies the oracle source, plants one mistake (a swapped nibble
order, a dropped term, a wrong sign, index, bias or constant), compiles the
copy with gcc and runs the oracle pin tests against it in a subprocess.  The
pins pass on the real oracle and must fail on every mutant.  Everything
happens on the CPU.
"""
import os
import subprocess
import sys

import pytest

from conftest import ROOT

SRC = os.path.join(ROOT, "oracle", "qbw_oracle.c")

MUTANTS = {
    "nibble_order_swapped": ("int code = (k < 16) ? (byte & 0x0f) : (byte >> 4);",
                             "int code = (k < 16) ? (byte >> 4) : (byte & 0x0f);"),
    "q4_offset_dropped": ("w[k] = d * (double)(code - 8);", "w[k] = d * (double)(code);"),
    "q4_offset_sign": ("w[k] = d * (double)(code - 8);", "w[k] = d * (double)(code + 8);"),
    "q8_unsigned_codes": ("w[k] = d * (double)(int)(int8_t)blk[2 + k];", "w[k] = d * (double)(int)blk[2 + k];"),
    "q4_byte_index_off": ("uint8_t byte = blk[2 + (k % 16)];", "uint8_t byte = blk[1 + (k % 16)];"),
    "scale_read_at_end": ("double d = oracle_fp16_to_f64(read_u16le(blk));\n    for (int k = 0; k < ORACLE_QK; k++) {",
                          "double d = oracle_fp16_to_f64(read_u16le(blk + 16));\n    for (int k = 0; k < ORACLE_QK; k++) {"),
    "fp16_subnormal_scale": ("v = ldexp((double)m, -24);", "v = ldexp((double)m, -14);"),
    "fp16_bias_off_by_one": ("v = ldexp((double)(1024 + m), e - 25);", "v = ldexp((double)(1024 + m), e - 24);"),
    "fp16_implicit_bit_dropped": ("v = ldexp((double)(1024 + m), e - 25);", "v = ldexp((double)(m), e - 25);"),
    "bf16_bias_off_by_one": ("v = ldexp((double)(128 + m), e - 134);", "v = ldexp((double)(128 + m), e - 133);"),
    "round_ties_away": ("(frac == 0.5 && fmod(fl, 2.0) != 0.0)", "(frac == 0.5)"),
    "abs_dropped_from_scale": ("                sabs += fabs(p);", "                sabs += p;"),
    "mixbit_abs_dropped_from_scale": ("            sabs += fabs(p);\n            int64_t g", "            sabs += p;\n            int64_t g"),
    "first_block_skipped": ("for (int64_t b = 0; b < nb; b++) {\n            decode_block(fmt, w + (n * nb + b) * "
                            "block_size(fmt), wb);\n            for (int k = 0; k < be; k++) {\n                double p",
                            "for (int64_t b = 1; b < nb; b++) {\n            decode_block(fmt, w + (n * nb + b) * "
                            "block_size(fmt), wb);\n            for (int k = 0; k < be; k++) {\n                double p"),
    "dequant_block_index": ("out[n * K + b * be + k] = (float)wb[k];", "out[n * K + b + k] = (float)wb[k];"),
    "gelu_cubic_constant": ("return 0.5 * v * (1.0 + tanh(c * (v + 0.044715 * v * v * v)));",
                            "return 0.5 * v * (1.0 + tanh(c * (v + 0.04715 * v * v * v)));"),
    "gelu_linear_term_dropped": ("return 0.5 * v * (1.0 + tanh(c * (v + 0.044715 * v * v * v)));",
                                 "return 0.5 * v * (1.0 + tanh(c * (0.044715 * v * v * v)));"),
    "gelu_erf_form": ("return 0.5 * v * (1.0 + tanh(c * (v + 0.044715 * v * v * v)));",
                      "return 0.5 * v * (1.0 + erf(v / sqrt(2.0)));"),
    "qmm_operand_transposed": ("matvec_rows(1, w, xd + m * K, 0, N, K, Y + m * N, S + m * N);",
                               "matvec_rows(1, w, xd + m, 0, N, K, Y + m * N, S + m * N);"),
    "gateup_gate_on_up": ("out[n] = oracle_gelu_tanh(g[n]) * u[n];", "out[n] = oracle_gelu_tanh(u[n]) * g[n];"),
    "q4k_scale_min_swapped": ("*sc = s[j] & 63;\n        *m = s[j + 4] & 63;", "*sc = s[j + 4] & 63;\n        *m = s[j] & 63;"),
    "q4k_high_bits_from_wrong_byte": ("*sc = (s[j + 4] & 0x0f) | ((s[j - 4] >> 6) << 4);",
                                      "*sc = (s[j + 4] & 0x0f) | ((s[j] >> 6) << 4);"),
    "q4k_min_nibble_low": ("*m = (s[j + 4] >> 4) | ((s[j] >> 6) << 4);", "*m = (s[j + 4] & 0x0f) | ((s[j] >> 6) << 4);"),
    "q4k_nibble_halves_swapped": ("return (l < 32) ? (byte & 0x0f) : (byte >> 4);",
                                  "return (l < 32) ? (byte >> 4) : (byte & 0x0f);"),
    "q4k_chunk_stride": ("uint8_t byte = qs[32 * chunk + (l % 32)];", "uint8_t byte = qs[16 * chunk + (l % 32)];"),
    "q4k_min_added": ("w[e] = d * (double)sc * (double)q4k_code(blk + 16, e) - dmin * (double)m;",
                      "w[e] = d * (double)sc * (double)q4k_code(blk + 16, e) + dmin * (double)m;"),
    "q4k_min_unscaled": ("w[e] = d * (double)sc * (double)q4k_code(blk + 16, e) - dmin * (double)m;",
                         "w[e] = d * (double)sc * (double)q4k_code(blk + 16, e) - (double)m;"),
    "q4k_dmin_read_as_d": ("double dmin = oracle_fp16_to_f64(read_u16le(blk + 2));\n        for (int e = 0; e < ORACLE_QK_K; e++) {\n            int sc, m;\n            oracle_q4k_scale_min(blk + 4, e / 32, &sc, &m);\n            w[e]",
                           "double dmin = oracle_fp16_to_f64(read_u16le(blk));\n        for (int e = 0; e < ORACLE_QK_K; e++) {\n            int sc, m;\n            oracle_q4k_scale_min(blk + 4, e / 32, &sc, &m);\n            w[e]"),
    "q4k_subblock_of_64": ("oracle_q4k_scale_min(blk + 4, e / 32, &sc, &m);\n            w[e]",
                           "oracle_q4k_scale_min(blk + 4, e / 64, &sc, &m);\n            w[e]"),
    "q4k_split_min_doubled": ("fabs(dmin * (double)m);\n                s2 +=", "fabs(2.0 * dmin * (double)m);\n                s2 +="),
    "q4k_split_min_dropped": ("double t = fabs(d * (double)sc * (double)q4k_code(blk + 16, e)) + fabs(dmin * (double)m);",
                              "double t = fabs(d * (double)sc * (double)q4k_code(blk + 16, e));"),
    "mixbit_fields_msb_first": ("int v = (int)((word >> (bit % 32)) & ((1u << bits) - 1u));",
                                "int v = (int)((word >> (32 - bits - bit % 32)) & ((1u << bits) - 1u));"),
    "mixbit_int2_unsigned": ("if (bits != 4 && v >= (1 << (bits - 1)))", "if (bits == 8 && v >= (1 << (bits - 1)))"),
    "mixbit_int8_unsigned": ("if (bits != 4 && v >= (1 << (bits - 1)))", "if (bits == 2 && v >= (1 << (bits - 1)))"),
    "mixbit_int4_signed": ("if (bits != 4 && v >= (1 << (bits - 1)))", "if (v >= (1 << (bits - 1)))"),
    "mixbit_bias_dropped": ("    if (bits == 4)\n        v += oracle_fp16_to_f64(bi[g]);",
                            "    if (bits == 4)\n        v += 0.0;"),
    "mixbit_bias_sign": ("    if (bits == 4)\n        v += oracle_fp16_to_f64(bi[g]);",
                         "    if (bits == 4)\n        v -= oracle_fp16_to_f64(bi[g]);"),
    "mixbit_group_without_row": ("const uint32_t *row = qp + n * (K * bits / 32);\n    int64_t g = n * (K / group) + k / group;",
                                 "const uint32_t *row = qp + n * (K * bits / 32);\n    int64_t g = k / group;"),
    "mixbit_row_stride": ("const uint32_t *row = qp + n * (K * bits / 32);\n    int64_t g",
                          "const uint32_t *row = qp + n * (K / 32);\n    int64_t g"),
    "mixbit_split_bias_dropped": ("t += fabs(oracle_fp16_to_f64(bi[g]));", "t += 0.0;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    before, after = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(before) == 1, f"pattern for {name} not found exactly once"
    mutated = src.replace(before, after)
    c = tmp_path / "mutant.c"
    so = tmp_path / "libmutant.so"
    c.write_text(mutated)
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-w",
                           "-o", str(so), str(c), "-lm"])
    env = dict(os.environ, QBW_ORACLE_LIB=str(so))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_scalars.py"),
                        os.path.join(ROOT, "tests", "test_oracle_products.py"),
                        os.path.join(ROOT, "tests", "test_oracle_q4k.py"),
                        os.path.join(ROOT, "tests", "test_oracle_mixbit.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"mutant {name} survived the pins:\n{r.stdout[-2000:]}"
