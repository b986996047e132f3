"""CPU oracle for block-quantized matvec -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never does: it
has no CPU fallback, and it shares no code with this oracle.

The arithmetic lives in ``qbw_oracle.c`` (scalar C, fp64 accumulation in
ascending k).  This module only compiles it with gcc and marshals numpy
arrays through ctypes.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qbw_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

F32, BF16 = 0, 1
_FMT = {"q8_0": 0, "q4_0": 1, "q4_k": 2}


_LIB_MT_PATH = os.path.join(_OUT_DIR, "liboracle_mt.so")
_lib_mt = None


def build(force: bool = False, mt: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/liboracle.so`` (plain gcc, no SIMD
    flags), or with ``mt`` the same source with OpenMP into ``liboracle_mt.so``
    (rows of a product split over threads; used only for the all-core CPU
    baseline)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    path = _LIB_MT_PATH if mt else _LIB_PATH
    if force or not os.path.exists(path) or os.path.getmtime(path) < os.path.getmtime(_SRC):
        tmp = path + f".{os.getpid()}.tmp"
        subprocess.check_call([
            "gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
            "-Wall", "-Wextra"] + (["-fopenmp"] if mt else ["-Wno-unknown-pragmas"]) + ["-o", tmp, _SRC, "-lm"])
        os.replace(tmp, path)
    return path


def lib_mt():
    """The OpenMP build of the oracle (same arithmetic per row)."""
    global _lib_mt
    with _lock:
        if _lib_mt is None:
            _lib_mt = ctypes.CDLL(build(mt=True))
            _declare(_lib_mt)
    return _lib_mt


def lib():
    """The loaded oracle.  ``QBW_ORACLE_LIB`` points at another build of the
    same source (the mutation tests use it to load a deliberately broken copy)."""
    global _lib
    with _lock:
        if _lib is None:
            path = os.environ.get("QBW_ORACLE_LIB") or build()
            _lib = ctypes.CDLL(path)
            _declare(_lib)
    return _lib


def _declare(L):
    P = ctypes.c_void_p
    i64 = ctypes.c_int64
    L.oracle_fp16_to_f64.restype = ctypes.c_double
    L.oracle_fp16_to_f64.argtypes = [ctypes.c_uint16]
    L.oracle_bf16_to_f64.restype = ctypes.c_double
    L.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
    L.oracle_round_bf16.restype = ctypes.c_uint16
    L.oracle_round_bf16.argtypes = [ctypes.c_double]
    for name in ("oracle_round_bf16_array", "oracle_fp16_to_f64_array", "oracle_bf16_to_f64_array",
                 "oracle_gelu_tanh_array", "oracle_gelu_tanh_deriv_array"):
        getattr(L, name).restype = None
        getattr(L, name).argtypes = [P, i64, P]
    L.oracle_gelu_tanh.restype = ctypes.c_double
    L.oracle_gelu_tanh.argtypes = [ctypes.c_double]
    L.oracle_dequant.restype = ctypes.c_int
    L.oracle_dequant.argtypes = [ctypes.c_int, P, i64, i64, P]
    L.oracle_qmv.restype = ctypes.c_int
    L.oracle_qmv.argtypes = [ctypes.c_int, P, P, ctypes.c_int, i64, i64, P, P]
    L.oracle_qmv_rows.restype = ctypes.c_int
    L.oracle_qmv_rows.argtypes = [ctypes.c_int, P, P, ctypes.c_int, i64, i64, i64, P, P]
    L.oracle_gateup_q4_0.restype = ctypes.c_int
    L.oracle_gateup_q4_0.argtypes = [P, P, P, ctypes.c_int, i64, i64, P, P, P, P, P]
    L.oracle_qmm_q4_0.restype = ctypes.c_int
    L.oracle_qmm_q4_0.argtypes = [P, P, ctypes.c_int, i64, i64, i64, P, P]
    L.oracle_q4k_split_scale.restype = ctypes.c_int
    L.oracle_q4k_split_scale.argtypes = [P, P, ctypes.c_int, i64, i64, P]
    L.oracle_q4k_scale_min.restype = None
    L.oracle_q4k_scale_min.argtypes = [P, ctypes.c_int, P, P]
    L.oracle_mixbit_dequant.restype = ctypes.c_int
    L.oracle_mixbit_dequant.argtypes = [ctypes.c_int, P, P, P, i64, i64, i64, P]
    L.oracle_qmv_mixbit.restype = ctypes.c_int
    L.oracle_qmv_mixbit.argtypes = [ctypes.c_int, P, P, P, i64, P, ctypes.c_int, i64, i64, P, P, P]


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _act(x: np.ndarray):
    """Return (contiguous array, dtype code): float32 values or uint16 bf16 bits."""
    x = np.ascontiguousarray(x)
    if x.dtype == np.float32:
        return x, F32
    if x.dtype == np.uint16:
        return x, BF16
    raise TypeError(f"activations must be float32 or uint16 (bf16 bits), got {x.dtype}")


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"{what}: oracle returned {rc}")


# ---------------------------------------------------------------- scalars

def fp16_to_f64(bits) -> np.ndarray:
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(b.shape, dtype=np.float64)
    lib().oracle_fp16_to_f64_array(_ptr(b), b.size, _ptr(out))
    return out


def bf16_to_f64(bits) -> np.ndarray:
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(b.shape, dtype=np.float64)
    lib().oracle_bf16_to_f64_array(_ptr(b), b.size, _ptr(out))
    return out


def round_bf16(v) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.uint16)
    lib().oracle_round_bf16_array(_ptr(v), v.size, _ptr(out))
    return out


def gelu_tanh(v) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.float64)
    lib().oracle_gelu_tanh_array(_ptr(v), v.size, _ptr(out))
    return out


def gelu_tanh_deriv(v) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.float64)
    lib().oracle_gelu_tanh_deriv_array(_ptr(v), v.size, _ptr(out))
    return out


# ---------------------------------------------------------------- products

def _weights(w: np.ndarray) -> np.ndarray:
    w = np.ascontiguousarray(w)
    if w.dtype != np.uint8:
        raise TypeError("weights must be raw uint8 block bytes")
    return w


def dequant(fmt: str, w: np.ndarray, N: int, K: int) -> np.ndarray:
    w = _weights(w)
    out = np.empty((N, K), dtype=np.float32)
    _check(lib().oracle_dequant(_FMT[fmt], _ptr(w), N, K, _ptr(out)), "dequant")
    return out


def qmv(fmt: str, w: np.ndarray, x: np.ndarray, N: int, K: int):
    """y = W x and S = sum_k |w x| for every row (fp64)."""
    w = _weights(w)
    x, xt = _act(x)
    y = np.empty(N, dtype=np.float64)
    S = np.empty(N, dtype=np.float64)
    _check(lib().oracle_qmv(_FMT[fmt], _ptr(w), _ptr(x), xt, N, K, _ptr(y), _ptr(S)), "qmv")
    return y, S


def qmv_rows(fmt: str, w: np.ndarray, x: np.ndarray, n0: int, n1: int, K: int, threads: bool = False):
    """Rows [n0, n1) of y = W x, with S; ``w`` still holds the whole matrix.
    ``threads``: the OpenMP build (rows split over the host's cores)."""
    w = _weights(w)
    x, xt = _act(x)
    y = np.empty(n1 - n0, dtype=np.float64)
    S = np.empty(n1 - n0, dtype=np.float64)
    L = lib_mt() if threads else lib()
    _check(L.oracle_qmv_rows(_FMT[fmt], _ptr(w), _ptr(x), xt, n0, n1, K, _ptr(y), _ptr(S)), "qmv_rows")
    return y, S


def gateup_q4_0(wg: np.ndarray, wu: np.ndarray, x: np.ndarray, N: int, K: int, threads: bool = False):
    """Returns dict with g, u, out = gelu_tanh(g) * u, Sg, Su (all fp64)."""
    wg, wu = _weights(wg), _weights(wu)
    x, xt = _act(x)
    r = {k: np.empty(N, dtype=np.float64) for k in ("g", "u", "out", "Sg", "Su")}
    _check((lib_mt() if threads else lib()).oracle_gateup_q4_0(_ptr(wg), _ptr(wu), _ptr(x), xt, N, K, _ptr(r["g"]), _ptr(r["u"]),
                                    _ptr(r["out"]), _ptr(r["Sg"]), _ptr(r["Su"])), "gateup")
    return r


def qmm_q4_0(w: np.ndarray, X: np.ndarray, M: int, N: int, K: int, threads: bool = False):
    """Y[m, n] = sum_k X[m, k] W[n, k] and S[m, n] (fp64)."""
    w = _weights(w)
    X, xt = _act(X)
    Y = np.empty((M, N), dtype=np.float64)
    S = np.empty((M, N), dtype=np.float64)
    _check((lib_mt() if threads else lib()).oracle_qmm_q4_0(_ptr(w), _ptr(X), xt, M, N, K, _ptr(Y), _ptr(S)), "qmm")
    return Y, S


def q4k_split_scale(w: np.ndarray, x: np.ndarray, N: int, K: int) -> np.ndarray:
    """S2 = sum (|d_sub q| + |m_sub|) |x| per row of a Q4_K matrix (fp64): the
    error scale of the split d_sub * sum(q x) - m_sub * sum(x)."""
    w = _weights(w)
    x, xt = _act(x)
    S2 = np.empty(N, dtype=np.float64)
    _check(lib().oracle_q4k_split_scale(_ptr(w), _ptr(x), xt, N, K, _ptr(S2)), "q4k_split_scale")
    return S2


def q4k_scale_min(scale_bytes, j: int):
    """(sc, m) of sub-block j from a Q4_K super-block's 12 scale bytes."""
    sb = np.ascontiguousarray(scale_bytes, dtype=np.uint8)
    sc = ctypes.c_int()
    m = ctypes.c_int()
    lib().oracle_q4k_scale_min(_ptr(sb), j, ctypes.byref(sc), ctypes.byref(m))
    return sc.value, m.value


# ---------------------------------------------------------------- mixed-bit

def _mixbit_arrays(bits, qp, sc, bi):
    qp = np.ascontiguousarray(qp, dtype=np.uint32)
    sc = np.ascontiguousarray(sc, dtype=np.uint16)
    bi = np.ascontiguousarray(bi if bi is not None else np.zeros(1, np.uint16), dtype=np.uint16)
    return qp, sc, bi


def mixbit_dequant(bits: int, qp, sc, bi, group: int, N: int, K: int) -> np.ndarray:
    """W[n, k] as fp32 (the exact weight rounded once) for a mixed-bit matrix:
    words qp (uint32), fp16 scale bits sc and bias bits bi (int4 only)."""
    qp, sc, bi = _mixbit_arrays(bits, qp, sc, bi)
    out = np.empty((N, K), dtype=np.float32)
    _check(lib().oracle_mixbit_dequant(bits, _ptr(qp), _ptr(sc), _ptr(bi), group, N, K, _ptr(out)),
           "mixbit_dequant")
    return out


def qmv_mixbit(bits: int, qp, sc, bi, group: int, x: np.ndarray, N: int, K: int):
    """Returns (y, S, S2) in fp64: y = W x, S = sum |w x|, S2 the split's scale."""
    qp, sc, bi = _mixbit_arrays(bits, qp, sc, bi)
    x, xt = _act(x)
    y, S, S2 = (np.empty(N, dtype=np.float64) for _ in range(3))
    _check(lib().oracle_qmv_mixbit(bits, _ptr(qp), _ptr(sc), _ptr(bi), group, _ptr(x), xt, N, K,
                                   _ptr(y), _ptr(S), _ptr(S2)), "qmv_mixbit")
    return y, S, S2
