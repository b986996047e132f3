"""Seeded synthetic inputs laid out as raw GGUF block bytes.

This module is shared by both sides of every parity check: the CPU oracle
(``oracle/``) and the CUDA library (``block_quantized_weight_gb300``) are fed
the very same bytes from here.  It draws random numbers and arranges them in
memory; it holds none of the method's arithmetic (no block decoding, no dot
products, no GELU), so neither side can inherit a mistake from the other
through it.

Block layouts written here (the GGUF ``block_q8_0`` / ``block_q4_0`` records;
the gem architecture page, "M4 Max operating assumptions", names Q4_0 as the
"32-element/18-byte block" and Q8_0 as the token-table format):

* Q8_0, 34 bytes: little-endian fp16 scale ``d`` then 32 signed int8 codes.
* Q4_0, 18 bytes: little-endian fp16 scale ``d`` then 16 bytes ``qs``; code
  ``j`` (0..15) sits in the low nibble of ``qs[j]`` and code ``j + 16`` in its
  high nibble.

* Q4_K, 144 bytes per 256 weights (the GGUF ``block_q4_K`` record): fp16 ``d``,
  fp16 ``dmin``, 12 scale bytes (six-bit scale and min of each 32-weight
  sub-block), 128 bytes of nibbles.  The generator draws the 12 scale bytes
  and the 128 nibble bytes as uniform random bytes: every byte pattern is a
  valid block, so nothing here packs or interprets the six-bit fields.

A matrix with N rows and K columns (K a multiple of 32, of 256 for Q4_K) is
N rows of consecutive blocks, rows back to back, no padding.

Random streams.  Every matrix or activation owns one
``numpy.random.Generator(PCG64(SeedSequence([seed, stream, layer])))``.  A
weight matrix draws all of its scales first (row-major over blocks), then all
of its codes.  Activations use stream 99 unless told otherwise.

* Q8_0 scale: ``fp16(|N(0, 0.02)| / 127)``; codes uniform on -127..127.
* Q4_0 scale: ``fp16(|N(0, 0.02)| / 8)``; codes uniform on 0..15, drawn as
  uniform bytes (each byte is two independent uniform nibbles).
* Q4_K: ``d = fp16(|N(0, 0.02)| / 240)``, then ``dmin = fp16(|N(0, 0.02)| / 64)``
  for every super-block, then the scale bytes, then the nibble bytes.
* Activations: fp32 draws of N(0, 1); a bf16 activation is the fp32 draw
  rounded to nearest-even bf16.  bf16 arrays are returned as their uint16
  bit patterns.
* fp16 conversion of scales is numpy's float64 -> float16 cast, which rounds
  to nearest even and keeps subnormals.
"""

from __future__ import annotations

import concurrent.futures as _cf
import os

import numpy as np

QK = 32                     # weights per block
QK_K = 256                  # weights per Q4_K super-block
Q8_0_BLOCK_BYTES = 34       # 2 (fp16 d) + 32 (int8 q)
Q4_0_BLOCK_BYTES = 18       # 2 (fp16 d) + 16 (packed nibbles)
Q4_K_BLOCK_BYTES = 144      # 2 (fp16 d) + 2 (fp16 dmin) + 12 (scales) + 128 (nibbles)
ACT_STREAM = 99

_BLOCK_BYTES = {"q8_0": Q8_0_BLOCK_BYTES, "q4_0": Q4_0_BLOCK_BYTES, "q4_k": Q4_K_BLOCK_BYTES}
_BLOCK_ELEMS = {"q8_0": QK, "q4_0": QK, "q4_k": QK_K}


def block_bytes(fmt: str) -> int:
    return _BLOCK_BYTES[fmt]


def block_elems(fmt: str) -> int:
    return _BLOCK_ELEMS[fmt]


def row_bytes(fmt: str, K: int) -> int:
    be = _BLOCK_ELEMS[fmt]
    if K % be:
        raise ValueError(f"K={K} is not a multiple of {be}")
    return (K // be) * _BLOCK_BYTES[fmt]


def matrix_bytes(fmt: str, N: int, K: int) -> int:
    return N * row_bytes(fmt, K)


def rng(seed: int, stream: int, layer: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, stream, layer])))


def _assemble(d_bits: np.ndarray, payload: np.ndarray, bpb: int) -> np.ndarray:
    """Interleave fp16 scale bits and per-block payload bytes into block records."""
    nblk = d_bits.size
    out = np.empty((nblk, bpb), dtype=np.uint8)
    out[:, 0:2] = d_bits.astype("<u2").view(np.uint8).reshape(nblk, 2)
    out[:, 2:] = payload.reshape(nblk, bpb - 2)
    return out.reshape(-1)


def q8_0_weights(N: int, K: int, seed: int, stream: int = 0, layer: int = 0) -> np.ndarray:
    """Random Q8_0 matrix, returned as a flat uint8 array of N*K/32*34 bytes."""
    nb = N * (K // QK)
    if K % QK:
        raise ValueError("K must be a multiple of 32")
    g = rng(seed, stream, layer)
    d = (np.abs(g.standard_normal(nb)) * 0.02 / 127.0).astype(np.float16)
    q = g.integers(-127, 128, size=nb * QK, dtype=np.int8)
    return _assemble(d.view(np.uint16), q.view(np.uint8), Q8_0_BLOCK_BYTES)


def q4_0_weights(N: int, K: int, seed: int, stream: int = 0, layer: int = 0) -> np.ndarray:
    """Random Q4_0 matrix, returned as a flat uint8 array of N*K/32*18 bytes."""
    nb = N * (K // QK)
    if K % QK:
        raise ValueError("K must be a multiple of 32")
    g = rng(seed, stream, layer)
    d = (np.abs(g.standard_normal(nb)) * 0.02 / 8.0).astype(np.float16)
    qs = g.integers(0, 256, size=nb * 16, dtype=np.uint8)
    return _assemble(d.view(np.uint16), qs, Q4_0_BLOCK_BYTES)


def q4_k_weights(N: int, K: int, seed: int, stream: int = 0, layer: int = 0) -> np.ndarray:
    """Random Q4_K matrix, returned as a flat uint8 array of N*K/256*144 bytes."""
    if K % QK_K:
        raise ValueError("K must be a multiple of 256")
    nb = N * (K // QK_K)
    g = rng(seed, stream, layer)
    d = (np.abs(g.standard_normal(nb)) * 0.02 / 240.0).astype(np.float16)
    dmin = (np.abs(g.standard_normal(nb)) * 0.02 / 64.0).astype(np.float16)
    scales = g.integers(0, 256, size=nb * 12, dtype=np.uint8)
    qs = g.integers(0, 256, size=nb * 128, dtype=np.uint8)
    return q4_k_records(d.view(np.uint16), dmin.view(np.uint16), scales, qs)


def q4_k_records(d_bits, dmin_bits, scales, qs) -> np.ndarray:
    """Lay out Q4_K super-blocks from their fields: fp16 bits of d and dmin (one
    per block), 12 scale bytes and 128 nibble bytes per block."""
    d_bits = np.asarray(d_bits, dtype=np.uint16).reshape(-1)
    nb = d_bits.size
    out = np.empty((nb, Q4_K_BLOCK_BYTES), dtype=np.uint8)
    out[:, 0:2] = d_bits.astype("<u2").view(np.uint8).reshape(nb, 2)
    out[:, 2:4] = np.asarray(dmin_bits, dtype=np.uint16).reshape(-1).astype("<u2").view(np.uint8).reshape(nb, 2)
    out[:, 4:16] = np.asarray(scales, dtype=np.uint8).reshape(nb, 12)
    out[:, 16:] = np.asarray(qs, dtype=np.uint8).reshape(nb, 128)
    return out.reshape(-1)


def weights(fmt: str, N: int, K: int, seed: int, stream: int = 0, layer: int = 0) -> np.ndarray:
    if fmt == "q8_0":
        return q8_0_weights(N, K, seed, stream, layer)
    if fmt == "q4_0":
        return q4_0_weights(N, K, seed, stream, layer)
    if fmt == "q4_k":
        return q4_k_weights(N, K, seed, stream, layer)
    raise ValueError(fmt)


def many_weights(fmt: str, specs, threads: int | None = None):
    """Generate several matrices concurrently; ``specs`` holds (N, K, seed, stream, layer)."""
    threads = threads or min(16, os.cpu_count() or 1)
    with _cf.ThreadPoolExecutor(threads) as ex:
        return list(ex.map(lambda s: weights(fmt, *s), specs))


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 values to nearest-even bf16 and return the uint16 bit patterns.

    This is input preparation (the workload's activations *are* bf16); NaN is
    not produced by the generators and is not special-cased.
    """
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = u + 0x7FFF + ((u >> 16) & 1)
    return (u >> 16).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to fp32 values (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def activations(shape, seed: int, dtype: str = "f32", stream: int = ACT_STREAM, layer: int = 0) -> np.ndarray:
    """N(0,1) activations: float32 values, or uint16 bf16 bit patterns if dtype == 'bf16'."""
    g = rng(seed, stream, layer)
    a = g.standard_normal(shape, dtype=np.float32)
    if dtype == "f32":
        return a
    if dtype == "bf16":
        return f32_to_bf16_bits(a)
    raise ValueError(dtype)


def constant_blocks(fmt: str, N: int, K: int, d_bits: int, code: int) -> np.ndarray:
    """Every block has scale bits ``d_bits`` and every code equals ``code``.

    ``code`` is the stored code: -128..127 for Q8_0, 0..15 for Q4_0.
    """
    nb = N * (K // QK)
    d = np.full(nb, d_bits, dtype=np.uint16)
    if fmt == "q8_0":
        payload = np.full(nb * QK, code, dtype=np.int8).view(np.uint8)
        return _assemble(d, payload, Q8_0_BLOCK_BYTES)
    if fmt == "q4_0":
        payload = np.full(nb * 16, (code & 0xF) | ((code & 0xF) << 4), dtype=np.uint8)
        return _assemble(d, payload, Q4_0_BLOCK_BYTES)
    raise ValueError(fmt)


def random_with_scale_bits(fmt: str, N: int, K: int, seed: int, d_pool: np.ndarray) -> np.ndarray:
    """Random codes with scales drawn from a given pool of fp16 bit patterns.

    Used for edge cases (subnormal, maximal and zero scales).
    """
    nb = N * (K // QK)
    g = rng(seed, 7)
    d = np.asarray(d_pool, dtype=np.uint16)[g.integers(0, len(d_pool), size=nb)]
    if fmt == "q8_0":
        q = g.integers(-128, 128, size=nb * QK, dtype=np.int8)
        return _assemble(d, q.view(np.uint8), Q8_0_BLOCK_BYTES)
    qs = g.integers(0, 256, size=nb * 16, dtype=np.uint8)
    return _assemble(d, qs, Q4_0_BLOCK_BYTES)


# ------------------------------------------------------------ mixed-bit formats
# Quantized words qp (uint32), fp16 scales sc and (4-bit affine only) fp16
# biases bi, one scale/bias per group of `group` weights of a row.  Field k of
# a row occupies bits (k * b) % 32 .. of word (k * b) // 32 of that row,
# lowest bits first.  The generator draws raw field values uniformly over all
# 2^b patterns.

MIXBIT_BITS = (2, 4, 8)


def pack_fields(fields: np.ndarray, bits: int) -> np.ndarray:
    """Pack a [N, K] array of raw b-bit field values (0 .. 2^b - 1) into uint32
    words, row after row, lowest bits first."""
    f = np.asarray(fields, dtype=np.uint32)
    N, K = f.shape
    per = 32 // bits
    f = f.reshape(N, K // per, per)
    shifts = (np.arange(per, dtype=np.uint32) * bits)
    return np.bitwise_or.reduce(f << shifts, axis=2).astype(np.uint32).reshape(-1)


def mixbit_weights(bits: int, N: int, K: int, group: int, seed: int, stream: int = 0, layer: int = 0):
    """Random mixed-bit matrix: (qp words, sc bits, bi bits or None).  Scales are
    fp16(|N(0, 0.02)| / r) with r = 2, 8, 127 for 2, 4 and 8 bits; 4-bit biases
    are fp16(-z * scale) with z uniform in [6, 9] (a zero point near the middle
    of the code range)."""
    if bits not in MIXBIT_BITS or K % group or (K * bits) % 32:
        raise ValueError("unsupported mixed-bit shape")
    g = rng(seed, stream, layer)
    ng = N * (K // group)
    r = {2: 2.0, 4: 8.0, 8: 127.0}[bits]
    sc = (np.abs(g.standard_normal(ng)) * 0.02 / r).astype(np.float16)
    fields = g.integers(0, 1 << bits, size=(N, K), dtype=np.uint32)
    bi = None
    if bits == 4:
        z = g.uniform(6.0, 9.0, ng)
        bi = (-z * sc.astype(np.float64)).astype(np.float16).view(np.uint16)
    return pack_fields(fields, bits), sc.view(np.uint16), bi


def mixbit_bytes(bits: int, N: int, K: int, group: int) -> int:
    """Bytes of a mixed-bit matrix: words, scales and (4-bit) biases."""
    return N * K * bits // 8 + N * (K // group) * 2 * (2 if bits == 4 else 1)
