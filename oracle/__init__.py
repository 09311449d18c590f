"""CPU oracle for the packed Q4_K dequant-matmul -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
and reference legs may import this package. The GPU library never imports or links it, and it
shares no code with the GPU library.

The arithmetic lives in ``q4k_oracle.cpp`` (plain C++, compiled here with gcc
``-O2 -ffp-contract=off`` so that no multiply-add is fused). This module only
builds that file and marshals numpy arrays through ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "q4k_oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/liboracle.so`` (gcc, no GPU needed)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["g++", "-O2", "-ffp-contract=off", "-fno-fast-math", "-std=c++17",
           "-shared", "-fPIC", "-pthread", _SRC, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            u8p = ctypes.POINTER(ctypes.c_uint8)
            f32p = ctypes.POINTER(ctypes.c_float)
            f64p = ctypes.POINTER(ctypes.c_double)
            i64p = ctypes.POINTER(ctypes.c_int64)
            lib.oracle_f16_to_f32.argtypes = [ctypes.c_uint16]
            lib.oracle_f16_to_f32.restype = ctypes.c_float
            lib.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
            lib.oracle_bf16_to_f32.restype = ctypes.c_float
            lib.oracle_unpack_scales.argtypes = [u8p, u8p, u8p]
            lib.oracle_unpack_scales.restype = None
            lib.oracle_dequant_block.argtypes = [u8p, f32p]
            lib.oracle_dequant_block.restype = None
            lib.oracle_dequant.argtypes = [u8p, ctypes.c_int64, ctypes.c_int64, f32p]
            lib.oracle_dequant.restype = ctypes.c_int
            lib.oracle_matmul.argtypes = [u8p, ctypes.c_int64, ctypes.c_int64, f32p,
                                          ctypes.c_int64, i64p, ctypes.c_int64,
                                          f64p, f64p, ctypes.c_int]
            lib.oracle_matmul.restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def f16_to_f32(h: int) -> float:
    """IEEE binary16 bit pattern -> value (exact)."""
    return float(_load().oracle_f16_to_f32(int(h) & 0xFFFF))


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns (uint16 array) -> their exact fp32 values."""
    # bfloat16 is the upper half of a binary32 (the same definition as the C
    # oracle_bf16_to_f32, which a pin compares on all 65536 patterns).
    flat = np.ascontiguousarray(bits, dtype=np.uint16).reshape(-1)
    return (flat.astype(np.uint32) << 16).view(np.float32).reshape(np.shape(bits))


def bf16_to_f32_scalar(b: int) -> float:
    """One bfloat16 bit pattern -> value, through the C oracle."""
    return float(_load().oracle_bf16_to_f32(int(b) & 0xFFFF))


def unpack_scales(s12) -> tuple[list[int], list[int]]:
    """12 packed scale bytes -> (sc[8], m[8])."""
    s = np.ascontiguousarray(np.asarray(s12, dtype=np.uint8).reshape(12))
    sc = np.zeros(8, np.uint8)
    m = np.zeros(8, np.uint8)
    _load().oracle_unpack_scales(_ptr(s, ctypes.c_uint8), _ptr(sc, ctypes.c_uint8),
                                 _ptr(m, ctypes.c_uint8))
    return [int(v) for v in sc], [int(v) for v in m]


def dequant_block(blk) -> np.ndarray:
    """One 144-byte super-block -> 256 fp32 weights."""
    b = np.ascontiguousarray(np.asarray(blk, dtype=np.uint8).reshape(144))
    out = np.empty(256, np.float32)
    _load().oracle_dequant_block(_ptr(b, ctypes.c_uint8), _ptr(out, ctypes.c_float))
    return out


def dequant(W: np.ndarray, N: int, K: int) -> np.ndarray:
    """Packed W (uint8, N*K/256*144 bytes) -> fp32 [N, K]."""
    w = np.ascontiguousarray(W, dtype=np.uint8).reshape(-1)
    if w.size != N * (K // 256) * 144:
        raise ValueError("W size does not match N, K")
    out = np.empty((N, K), np.float32)
    rc = _load().oracle_dequant(_ptr(w, ctypes.c_uint8), N, K, _ptr(out, ctypes.c_float))
    if rc != 0:
        raise ValueError(f"oracle_dequant failed with status {rc}")
    return out


def matmul(W: np.ndarray, N: int, K: int, X: np.ndarray, rows=None, threads: int = 0):
    """Y[m, r] = sum_k X[m,k] * w(rows[r], k) and A = sum_k |X*w|, both float64.

    ``X`` is float32 [M, K] (pass bf16 inputs through :func:`bf16_to_f32`).
    ``rows`` selects rows of W (columns of Y); None means all N. To check a
    sample of a large matrix, pass just the sampled rows' bytes as a W of
    N = len(sample) rows.
    """
    w = np.ascontiguousarray(W, dtype=np.uint8).reshape(-1)
    x = np.ascontiguousarray(X, dtype=np.float32)
    if x.ndim != 2 or x.shape[1] != K:
        raise ValueError("X must be [M, K]")
    M = x.shape[0]
    if w.size != N * (K // 256) * 144:
        raise ValueError("W size does not match N, K")
    if rows is None:
        rr = None
        nrows = N
    else:
        rr = np.ascontiguousarray(rows, dtype=np.int64).reshape(-1)
        nrows = rr.size
    Y = np.empty((M, nrows), np.float64)
    A = np.empty((M, nrows), np.float64)
    rc = _load().oracle_matmul(_ptr(w, ctypes.c_uint8), N, K, _ptr(x, ctypes.c_float), M,
                               None if rr is None else _ptr(rr, ctypes.c_int64), nrows,
                               _ptr(Y, ctypes.c_double), _ptr(A, ctypes.c_double),
                               int(threads))
    if rc != 0:
        raise ValueError(f"oracle_matmul failed with status {rc}")
    return Y, A
