"""block_quantized_weight_gb300 -- Python binding of libqbw, the C ABI declared
in ``include/qbw.h`` (block-quantized GGUF Q8_0/Q4_0 matrix-vector products on
GB300).

This module only marshals arguments: it turns torch tensors into device
pointers, dtype codes and the current CUDA stream, calls the C function of the
same name and raises ``QbwError`` on a non-zero status.  Every step of the
computation runs in the library's CUDA kernels; there is no CPU fallback, and
importing a function whose library is missing raises immediately.
"""

from __future__ import annotations

import ctypes
import os
import threading

__all__ = [
    "QbwError", "load", "lib_path",
    "qmv_q8_0", "qmv_q4_0", "qmv_gateup_q4_0", "qmm_q4_0_smallM", "qmm_q4_0_smallM_workspace_bytes",
    "qmm_q4_0_smallM_noalloc", "NOALLOC_SCRATCH_BYTES", "qembed_q8_0", "qdequant_q8_0", "qdequant_q4_0", "qmv_q4_k", "qdequant_q4_k", "selftest_wait", "Chain", "fault_read", "status_str", "version",
    "F32", "BF16",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB = os.path.join(_HERE, "_build", "libqbw.so")
_lock = threading.Lock()
_lib = None

F32, BF16 = 0, 1
NOALLOC_SCRATCH_BYTES = 4 << 20  # QBW_QMM_NOALLOC_SCRATCH_BYTES
QBW_OK = 0


class QbwError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_str(status)}")


def lib_path() -> str:
    return _LIB


def load():
    """Load libqbw.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB):
                raise RuntimeError(f"libqbw.so is not built ({_LIB}); run "
                                   "`python -m block_quantized_weight_gb300.build`")
            L = ctypes.CDLL(_LIB)
            _declare(L)
            _lib = L
    return _lib


def _declare(L):
    P, i64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
    L.qbw_status_str.restype = ctypes.c_char_p
    L.qbw_status_str.argtypes = [i32]
    L.qbw_version.restype = ctypes.c_uint32
    L.qbw_version.argtypes = []
    for name in ("qmv_q8_0", "qmv_q4_0", "qmv_q4_k"):
        getattr(L, name).restype = i32
        getattr(L, name).argtypes = [P, P, i32, P, i32, i64, i64, i64, P]
    L.qmv_gateup_q4_0.restype = i32
    L.qmv_gateup_q4_0.argtypes = [P, P, P, i32, P, i32, i64, i64, i64, P]
    L.qmm_q4_0_smallM_workspace_bytes.restype = sz
    L.qmm_q4_0_smallM_workspace_bytes.argtypes = [i64, i64, i64]
    L.qmm_q4_0_smallM.restype = i32
    L.qmm_q4_0_smallM.argtypes = [P, P, i32, P, i32, i64, i64, i64, P, sz, P]
    L.qembed_q8_0.restype = i32
    L.qembed_q8_0.argtypes = [P, P, i64, P, i32, i64, i64, P]
    L.qmm_q4_0_smallM_noalloc.restype = i32
    L.qmm_q4_0_smallM_noalloc.argtypes = [P, P, i32, P, i32, i64, i64, i64, P]
    for name in ("qdequant_q8_0", "qdequant_q4_0", "qdequant_q4_k"):
        getattr(L, name).restype = i32
        getattr(L, name).argtypes = [P, P, i64, i64, P]
    L.qmv_mixbit.restype = i32
    L.qmv_mixbit.argtypes = [i32, P, P, P, i64, P, i32, P, i32, i64, i64, i64, P]
    L.qmv_mixbit_route.restype = i32
    L.qmv_mixbit_route.argtypes = [i32, P, P, P, i64, i32, i64, i64, ctypes.POINTER(ctypes.c_int)]
    L.qdequant_mixbit.restype = i32
    L.qdequant_mixbit.argtypes = [i32, P, P, P, i64, P, i64, i64, P]
    L.qbw_fault_read.restype = i32
    L.qbw_fault_read.argtypes = [ctypes.POINTER(ctypes.c_uint32), i32, P]
    L.qbw_selftest_wait.restype = i32
    L.qbw_selftest_wait.argtypes = [i32, ctypes.c_uint32, P]
    L.qbw_chain_create.restype = i32
    L.qbw_chain_create.argtypes = [ctypes.POINTER(_ChainStep), i32, ctypes.POINTER(P)]
    L.qbw_chain_run.restype = i32
    L.qbw_chain_run.argtypes = [P, P]
    L.qbw_chain_run_launches.restype = i32
    L.qbw_chain_run_launches.argtypes = [P, P]
    L.qbw_chain_destroy.restype = i32
    L.qbw_chain_destroy.argtypes = [P]


class _ChainStep(ctypes.Structure):
    """qbw_chain_step of include/qbw.h."""
    _fields_ = [("w", ctypes.c_void_p), ("w_up", ctypes.c_void_p), ("x", ctypes.c_void_p), ("y", ctypes.c_void_p),
                ("yt", ctypes.c_int), ("N", ctypes.c_int64), ("K", ctypes.c_int64)]


def status_str(status: int) -> str:
    return load().qbw_status_str(int(status)).decode()


def version() -> int:
    return int(load().qbw_version())


# ------------------------------------------------------------------ marshalling
def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    return 99  # rejected by the library with QBW_EDTYPE


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(int(getattr(stream, "cuda_stream", stream)))


def _check(status: int, where: str):
    if status != QBW_OK:
        raise QbwError(status, where)


def qmv_q8_0(w, x, y, M: int, N: int, K: int, stream=None):
    """y = W x for raw Q8_0 blocks ``w`` (uint8), activations ``x`` and outputs ``y`` (fp32/bf16)."""
    L = load()
    _check(L.qmv_q8_0(_ptr(w), _ptr(x), _dtype_code(x), _ptr(y), _dtype_code(y), M, N, K, _stream(stream)),
           "qmv_q8_0")
    return y


def qmv_q4_0(w, x, y, M: int, N: int, K: int, stream=None):
    """y = W x for raw Q4_0 blocks ``w`` (uint8)."""
    L = load()
    _check(L.qmv_q4_0(_ptr(w), _ptr(x), _dtype_code(x), _ptr(y), _dtype_code(y), M, N, K, _stream(stream)),
           "qmv_q4_0")
    return y


def qmv_q4_k(w, x, y, M: int, N: int, K: int, stream=None):
    """y = W x for raw Q4_K super-blocks ``w`` (uint8, 144 bytes per 256 weights)."""
    L = load()
    _check(L.qmv_q4_k(_ptr(w), _ptr(x), _dtype_code(x), _ptr(y), _dtype_code(y), M, N, K, _stream(stream)),
           "qmv_q4_k")
    return y


def qmv_mixbit(bits: int, qp, sc, bi, group: int, x, y, M: int, N: int, K: int, stream=None):
    """y = W x for a mixed-bit matrix: ``bits`` 2 (int2-symmetric), 4
    (int4-affine, ``bi`` required) or 8 (int8); words ``qp``, fp16 scale bits
    ``sc`` and bias bits ``bi`` (device tensors), one scale per ``group``
    weights of a row."""
    L = load()
    _check(L.qmv_mixbit(bits, _ptr(qp), _ptr(sc), _ptr(bi) if bi is not None else None, group, _ptr(x),
                        _dtype_code(x), _ptr(y), _dtype_code(y), M, N, K, _stream(stream)), "qmv_mixbit")
    return y


def qmv_mixbit_route(bits: int, qp, sc, bi, group: int, x, N: int, K: int) -> bool:
    """Whether qmv_mixbit with these arguments (activations like ``x``) takes
    the tensor-core form on the current device (test-only; launches nothing)."""
    L = load()
    tc = ctypes.c_int(-1)
    _check(L.qmv_mixbit_route(bits, _ptr(qp), _ptr(sc), _ptr(bi) if bi is not None else None, group, _dtype_code(x),
                              N, K, ctypes.byref(tc)), "qmv_mixbit_route")
    return tc.value == 1


def qdequant_mixbit(bits: int, qp, sc, bi, group: int, out, N: int, K: int, stream=None):
    """out[n, k] = w[n, k] (fp32) for a mixed-bit matrix (test-only)."""
    L = load()
    _check(L.qdequant_mixbit(bits, _ptr(qp), _ptr(sc), _ptr(bi) if bi is not None else None, group, _ptr(out),
                             N, K, _stream(stream)), "qdequant_mixbit")
    return out


def qmv_gateup_q4_0(w_gate, w_up, x, out, M: int, N: int, K: int, stream=None):
    """out = gelu_tanh(Wg x) * (Wu x) for two raw Q4_0 matrices."""
    L = load()
    _check(L.qmv_gateup_q4_0(_ptr(w_gate), _ptr(w_up), _ptr(x), _dtype_code(x), _ptr(out), _dtype_code(out),
                             M, N, K, _stream(stream)), "qmv_gateup_q4_0")
    return out


def qmm_q4_0_smallM_workspace_bytes(M: int, N: int, K: int) -> int:
    return int(load().qmm_q4_0_smallM_workspace_bytes(M, N, K))


def qmm_q4_0_smallM(w, X, Y, M: int, N: int, K: int, workspace=None, stream=None):
    """Y[M, N] = X[M, K] W^T for raw Q4_0 blocks ``w`` on the tensor cores.

    ``workspace`` is a uint8 device tensor of at least
    ``qmm_q4_0_smallM_workspace_bytes(M, N, K)`` bytes, zero-filled once when
    allocated (the library returns its counters to zero after every call).
    """
    L = load()
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(L.qmm_q4_0_smallM(_ptr(w), _ptr(X), _dtype_code(X), _ptr(Y), _dtype_code(Y), M, N, K,
                             _ptr(workspace), wbytes, _stream(stream)), "qmm_q4_0_smallM")
    return Y


def qmm_q4_0_smallM_noalloc(w, X, Y, M: int, N: int, K: int, stream=None):
    """qmm_q4_0_smallM with the library's static scratch instead of a caller
    workspace, for callers that cannot allocate device memory.  Calls on one
    device must not overlap in time; the first one does a one-time set-up."""
    _check(load().qmm_q4_0_smallM_noalloc(_ptr(w), _ptr(X), _dtype_code(X), _ptr(Y), _dtype_code(Y), M, N, K,
                                          _stream(stream)), "qmm_q4_0_smallM_noalloc")
    return Y


def qembed_q8_0(w, ids, out, N: int, K: int, stream=None):
    """out[i, :] = dequantized row ids[i] of the Q8_0 matrix ``w`` (N x K);
    ``ids`` an int32 device tensor, ``out`` fp32 or bf16 [len(ids), K]."""
    _check(load().qembed_q8_0(_ptr(w), _ptr(ids), ids.numel(), _ptr(out), _dtype_code(out), N, K, _stream(stream)),
           "qembed_q8_0")
    return out


def qdequant_q8_0(w, out, N: int, K: int, stream=None):
    L = load()
    _check(L.qdequant_q8_0(_ptr(w), _ptr(out), N, K, _stream(stream)), "qdequant_q8_0")
    return out


def qdequant_q4_0(w, out, N: int, K: int, stream=None):
    L = load()
    _check(L.qdequant_q4_0(_ptr(w), _ptr(out), N, K, _stream(stream)), "qdequant_q4_0")
    return out


def qdequant_q4_k(w, out, N: int, K: int, stream=None):
    L = load()
    _check(L.qdequant_q4_k(_ptr(w), _ptr(out), N, K, _stream(stream)), "qdequant_q4_k")
    return out


def selftest_wait(which: int, limit_us: int, stream=None):
    """Run a bounded wait that nothing completes (test-only; see qbw_selftest_wait)."""
    L = load()
    _check(L.qbw_selftest_wait(which, limit_us, _stream(stream)), "qbw_selftest_wait")


class Chain:
    """A chain of dependent Q4_0 products run as one launch (qbw_chain_create /
    qbw_chain_run / qbw_chain_destroy).  ``steps`` is a sequence of
    ``(w, w_up, x, y, N, K)``: ``w_up`` None for ``y = W x``, else the up
    matrix of a fused gate+up step; ``x`` bf16 [K]; ``y`` bf16 or fp32 [N].
    The tensors must stay alive and in place while the chain exists."""

    def __init__(self, steps):
        L = load()
        arr = (_ChainStep * len(steps))()
        self._keep = []
        for i, (w, w_up, x, y, N, K) in enumerate(steps):
            self._keep += [w, w_up, x, y]
            arr[i] = _ChainStep(w.data_ptr(), None if w_up is None else w_up.data_ptr(), x.data_ptr(),
                                y.data_ptr(), _dtype_code(y), int(N), int(K))
        h = ctypes.c_void_p()
        _check(L.qbw_chain_create(arr, len(steps), ctypes.byref(h)), "qbw_chain_create")
        self._h = h

    def run(self, stream=None):
        _check(load().qbw_chain_run(self._h, _stream(stream)), "qbw_chain_run")

    def run_launches(self, stream=None):
        """One launch per step, each prefetching the next step's first weight
        tiles into L2 (qbw_chain_run_launches)."""
        _check(load().qbw_chain_run_launches(self._h, _stream(stream)), "qbw_chain_run_launches")

    def close(self):
        if getattr(self, "_h", None):
            _check(load().qbw_chain_destroy(self._h), "qbw_chain_destroy")
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def fault_read(clear: bool = True, stream=None) -> int:
    """Synchronize ``stream`` and return (and optionally clear) the device fault word."""
    L = load()
    code = ctypes.c_uint32(0)
    _check(L.qbw_fault_read(ctypes.byref(code), 1 if clear else 0, _stream(stream)), "qbw_fault_read")
    return int(code.value)
