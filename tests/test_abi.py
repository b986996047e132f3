"""The C ABI on the CPU: the library loads, exports every entry point that
include/qbw.h declares, and rejects invalid arguments on the host before
touching a GPU (validation returns before any CUDA call)."""
import ctypes
import os
import re
import subprocess

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "qbw.h")


@pytest.fixture(scope="module")
def lib():
    import block_quantized_weight_gb300 as qbw
    if not os.path.exists(qbw.lib_path()):
        from block_quantized_weight_gb300 import build as b
        b.build()
    return qbw.load()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w\s\*]+?\b(\w+)\s*\(", src, flags=re.M)) - {"if"})


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("qmv_q8_0", "qmv_q4_0", "qmv_gateup_q4_0", "qmm_q4_0_smallM", "qmm_q4_0_smallM_workspace_bytes",
              "qdequant_q8_0", "qdequant_q4_0", "qmv_q4_k", "qdequant_q4_k", "qbw_status_str", "qbw_version",
              "qbw_fault_read", "qmv_mixbit", "qdequant_mixbit"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    import block_quantized_weight_gb300 as qbw
    out = subprocess.run(["nm", "-D", "--defined-only", qbw.lib_path()], capture_output=True, text=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for n in declared_functions():
        assert n in exported, n
        assert getattr(lib, n) is not None


def test_library_has_no_oracle_code(lib):
    import block_quantized_weight_gb300 as qbw
    out = subprocess.run(["nm", "-D", qbw.lib_path()], capture_output=True, text=True).stdout
    assert "oracle" not in out
    csrc = os.path.join(ROOT, "block_quantized_weight_gb300", "csrc")
    for f in os.listdir(csrc):
        assert "oracle" not in open(os.path.join(csrc, f)).read().lower(), f


def test_status_strings(lib):
    import block_quantized_weight_gb300 as qbw
    for s in range(8):
        assert qbw.status_str(s).startswith("QBW_")
    assert qbw.version() >= 0x10000


F32, BF16 = 0, 1
P = ctypes.c_void_p
ADDR = 0x7F0000000000  # never dereferenced: every case below fails validation first


def qmv(lib, name, w=ADDR, x=ADDR + (1 << 30), xt=F32, y=ADDR + (2 << 30), yt=F32, M=1, N=16, K=256):
    return getattr(lib, name)(P(w) if w else None, P(x) if x else None, xt, P(y) if y else None, yt, M, N, K, None)


@pytest.mark.parametrize("name", ["qmv_q8_0", "qmv_q4_0", "qmv_q4_k"])
def test_qmv_validation(lib, name):
    assert qmv(lib, name, w=0) == 1
    assert qmv(lib, name, x=0) == 1
    assert qmv(lib, name, y=0) == 1
    assert qmv(lib, name, xt=7) == 3
    assert qmv(lib, name, yt=-1) == 3
    assert qmv(lib, name, M=2) == 2
    assert qmv(lib, name, M=0) == 2
    assert qmv(lib, name, N=0) == 2
    assert qmv(lib, name, K=0) == 2
    assert qmv(lib, name, K=48) == 2
    assert qmv(lib, name, K=1 << 25) == 2
    assert qmv(lib, name, N=1 << 31) == 2
    assert qmv(lib, name, x=ADDR + (1 << 30) + 2, xt=F32) == 4
    assert qmv(lib, name, y=ADDR + (2 << 30) + 1, yt=BF16) == 4
    # output overlapping the activations or the weights
    assert qmv(lib, name, y=ADDR + (1 << 30) + 64) == 1
    assert qmv(lib, name, y=ADDR + 16) == 1


def test_q4k_needs_whole_super_blocks(lib):
    # Q4_K super-blocks hold 256 weights: K = 288 is a whole number of 32-weight
    # blocks but not of super-blocks
    assert qmv(lib, "qmv_q4_k", K=288) == 2
    assert qmv(lib, "qmv_q4_k", K=512, y=ADDR + 16 * 144 - 8) == 1      # y overlaps the 16 x 512 weights
    f = lib.qdequant_q4_k
    assert f(None, P(ADDR + (1 << 30)), 4, 256, None) == 1
    assert f(P(ADDR), P(ADDR + (1 << 30)), 4, 288, None) == 2
    assert f(P(ADDR), P(ADDR + (1 << 30) + 2), 4, 256, None) == 4
    assert f(P(ADDR), P(ADDR + 8), 4, 256, None) == 1


def test_selftest_wait_validation(lib):
    # rejected before any device work
    assert lib.qbw_selftest_wait(2, 1000, None) == 1
    assert lib.qbw_selftest_wait(-1, 1000, None) == 1
    assert lib.qbw_selftest_wait(0, 0, None) == 1
    assert lib.qbw_selftest_wait(0, 2000001, None) == 1


def test_gateup_validation(lib):
    f = lib.qmv_gateup_q4_0
    a, b, x, y = ADDR, ADDR + (1 << 28), ADDR + (1 << 30), ADDR + (2 << 30)
    assert f(P(a), None, P(x), F32, P(y), F32, 1, 16, 256, None) == 1
    assert f(P(a), P(b), P(x), F32, P(y), F32, 3, 16, 256, None) == 2
    assert f(P(a), P(b), P(x), F32, P(b + 8), F32, 1, 16, 256, None) == 1


def test_qmm_validation(lib):
    f = lib.qmm_q4_0_smallM
    w, X, Y = ADDR, ADDR + (1 << 30), ADDR + (2 << 30)
    assert f(None, P(X), BF16, P(Y), BF16, 8, 64, 256, None, 0, None) == 1
    assert f(P(w), P(X), F32, P(Y), BF16, 8, 64, 256, None, 0, None) == 3
    assert f(P(w), P(X), BF16, P(Y), BF16, 0, 64, 256, None, 0, None) == 2
    assert f(P(w), P(X), BF16, P(Y), BF16, 33, 64, 256, None, 0, None) == 2
    assert f(P(w), P(X), BF16, P(Y), BF16, 8, 64, 100, None, 0, None) == 2
    assert f(P(w), P(X + 1), BF16, P(Y), BF16, 8, 64, 256, None, 0, None) == 4


def test_dequant_validation(lib):
    for name in ("qdequant_q8_0", "qdequant_q4_0"):
        f = getattr(lib, name)
        assert f(None, P(ADDR + (1 << 30)), 4, 64, None) == 1
        assert f(P(ADDR), P(ADDR + (1 << 30)), 4, 40, None) == 2
        assert f(P(ADDR), P(ADDR + (1 << 30) + 2), 4, 64, None) == 4
        assert f(P(ADDR), P(ADDR + 8), 4, 64, None) == 1


def test_chain_calls_reject_null_arguments_before_touching_a_device(lib):
    import ctypes
    import block_quantized_weight_gb300 as qbw
    L = qbw.load()
    h = ctypes.c_void_p()
    assert L.qbw_chain_create(None, 1, ctypes.byref(h)) == 1          # QBW_EINVAL
    assert L.qbw_chain_create(None, 0, ctypes.byref(h)) == 1
    assert not h.value
    assert L.qbw_chain_create(None, 1, None) == 1
    assert L.qbw_chain_run(None, None) == 1
    assert L.qbw_chain_destroy(None) == 1


def test_mixbit_validation(lib):
    f = lib.qmv_mixbit
    w, sc, bi, x, y = P(ADDR), P(ADDR + (1 << 28)), P(ADDR + (1 << 29)), P(ADDR + (1 << 30)), P(ADDR + (3 << 30))
    assert f(3, w, sc, bi, 32, x, F32, y, F32, 1, 16, 256, None) == 1          # unknown kind
    assert f(4, w, sc, None, 32, x, F32, y, F32, 1, 16, 256, None) == 1        # int4 needs biases
    assert f(2, w, sc, None, 32, x, F32, y, F32, 1, 16, 96, None) == 2         # 96 * 2 bits: not whole word groups
    assert f(8, w, sc, None, 24, x, F32, y, F32, 1, 16, 96, None) == 2         # group not a multiple of 16
    assert f(8, w, sc, None, 64, x, F32, y, F32, 1, 16, 96, None) == 2         # 96 % 64
    assert f(8, w, sc, None, 32, x, F32, y, F32, 2, 16, 256, None) == 2        # M != 1
    assert f(8, w, sc, None, 64, x, F32, y, F32, 1, 16, 65536, None) == 2      # x does not fit shared memory
    assert f(8, P(ADDR + 8), sc, None, 32, x, F32, y, F32, 1, 16, 256, None) == 4
    assert f(8, w, sc, None, 32, P(ADDR + (1 << 30) + 4), F32, y, F32, 1, 16, 256, None) == 4
    assert f(8, w, sc, None, 32, x, 7, y, F32, 1, 16, 256, None) == 3
    assert f(8, w, sc, None, 32, x, F32, P(ADDR + 64), F32, 1, 16, 256, None) == 1    # y overlaps the words
    r = lib.qmv_mixbit_route                                                     # no device needed for these
    tc = ctypes.c_int(-1)
    assert r(3, w, sc, bi, 32, F32, 16, 256, ctypes.byref(tc)) == 1             # unknown kind
    assert r(8, w, sc, None, 32, F32, 16, 256, None) == 1                        # no result pointer
    assert r(8, w, sc, None, 32, 7, 16, 256, ctypes.byref(tc)) == 3              # unknown activation type
    assert r(8, w, sc, None, 64, BF16, 16, 65536, ctypes.byref(tc)) == 2         # neither kernel takes it
    assert r(8, P(ADDR + 8), sc, None, 32, BF16, 16, 256, ctypes.byref(tc)) == 4
    assert tc.value == -1                                                          # untouched on error
    g = lib.qdequant_mixbit
    assert g(4, w, sc, None, 32, y, 16, 256, None) == 1
    assert g(2, w, sc, None, 32, P(ADDR + (3 << 30) + 2), 16, 256, None) == 4
    assert g(8, w, P(ADDR + (1 << 28) + 2), None, 32, y, 16, 256, None) == 4       # scales 4-byte aligned
