"""Python binding of libq4k, the GB300 packed Q4_K dequant-matmul library.

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI declared in ``include/q4k.h``. The functions mirror
the C names and take torch tensors (device memory, caller-owned) or raw device
pointers (ints). There is no fallback: if ``libq4k.so`` has not been built, or
a call fails, a ``Q4KError`` is raised.
"""
from __future__ import annotations

import ctypes
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libq4k.so")

Q4K_OK = 0
Q4K_ERR_NULL = -1
Q4K_ERR_BAD_DIM = -2
Q4K_ERR_CUDA = -3
Q4K_ERR_ALIGN = -4
Q4K_ERR_ARCH = -5
Q4K_ERR_TIMEOUT = -6

#: every symbol include/q4k.h declares
EXPORTS = ("q4k_status_string", "q4k_init", "q4k_dequant", "q4k_matmul", "q4k_matmul_bf16",
           "q4k_matmul_multi", "q4k_matmul_multi_bf16", "q4k_matmul_argmax",
           "q4k_matmul_argmax_bf16", "q4k_set_pdl", "q4k_device_error", "q4k_selftest_timeout")
MAX_GROUP = 8


_STATUS_NAMES = {Q4K_OK: "Q4K_OK", Q4K_ERR_NULL: "Q4K_ERR_NULL", Q4K_ERR_BAD_DIM: "Q4K_ERR_BAD_DIM",
                 Q4K_ERR_CUDA: "Q4K_ERR_CUDA", Q4K_ERR_ALIGN: "Q4K_ERR_ALIGN",
                 Q4K_ERR_ARCH: "Q4K_ERR_ARCH", Q4K_ERR_TIMEOUT: "Q4K_ERR_TIMEOUT"}


class Q4KError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {_STATUS_NAMES.get(status, 'unknown status')} ({status})")


_lock = threading.Lock()
_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libq4k.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise Q4KError(Q4K_ERR_CUDA, f"libq4k.so not built at {LIB_PATH} "
                               "(run gguf_q4_dequant_gb300.build.build())")
            L = ctypes.CDLL(LIB_PATH)
            vp, i64 = ctypes.c_void_p, ctypes.c_int64
            L.q4k_status_string.argtypes = [ctypes.c_int]
            L.q4k_status_string.restype = ctypes.c_char_p
            L.q4k_init.argtypes = []
            L.q4k_init.restype = ctypes.c_int
            L.q4k_dequant.argtypes = [vp, i64, i64, vp, vp]
            L.q4k_dequant.restype = ctypes.c_int
            L.q4k_matmul.argtypes = [vp, i64, i64, vp, i64, vp, vp]
            L.q4k_matmul.restype = ctypes.c_int
            L.q4k_matmul_bf16.argtypes = [vp, i64, i64, vp, i64, vp, vp]
            L.q4k_matmul_bf16.restype = ctypes.c_int
            vpp = ctypes.POINTER(ctypes.c_void_p)
            i64p = ctypes.POINTER(ctypes.c_int64)
            L.q4k_matmul_multi.argtypes = [ctypes.c_int, vpp, i64p, i64, vp, i64, vpp, vp]
            L.q4k_matmul_multi.restype = ctypes.c_int
            L.q4k_matmul_multi_bf16.argtypes = [ctypes.c_int, vpp, i64p, i64, vp, i64, vpp, vp]
            L.q4k_matmul_multi_bf16.restype = ctypes.c_int
            L.q4k_matmul_argmax.argtypes = [vp, i64, i64, vp, i64, vp, vp]
            L.q4k_matmul_argmax.restype = ctypes.c_int
            L.q4k_matmul_argmax_bf16.argtypes = [vp, i64, i64, vp, i64, vp, vp]
            L.q4k_matmul_argmax_bf16.restype = ctypes.c_int
            L.q4k_set_pdl.argtypes = [ctypes.c_int]
            L.q4k_set_pdl.restype = ctypes.c_int
            L.q4k_device_error.argtypes = [ctypes.c_int]
            L.q4k_device_error.restype = ctypes.c_int
            L.q4k_selftest_timeout.argtypes = [i64, vp]
            L.q4k_selftest_timeout.restype = ctypes.c_int
            _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().q4k_status_string(int(status)).decode()


def _ptr(t) -> int:
    if t is None:
        return 0
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise ValueError("tensor must live in CUDA device memory")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(rc: int, where: str):
    if rc != Q4K_OK:
        raise Q4KError(rc, where)


def _check_dtype(t, dtype, name):
    if not isinstance(t, int) and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")


def _dims_valid(N, K, M=1):
    return N >= 1 and M >= 1 and K >= 256 and K % 256 == 0


def _check_size(t, need: int, name: str):
    """A tensor (not a raw pointer) must hold at least `need` elements, so that
    no kernel reads or writes past it."""
    if t is not None and not isinstance(t, int) and t.numel() < need:
        raise ValueError(f"{name} holds {t.numel()} elements, the call needs {need}")


def _w_bytes(N, K):
    return N * (K // 256) * 144


def _check_matmul_sizes(W, N, K, X, M, Y):
    if not _dims_valid(N, K, M):
        return  # the C ABI rejects the dimensions themselves
    _check_size(W, _w_bytes(N, K), "W")
    _check_size(X, M * K, "X")
    _check_size(Y, M * N, "Y")


def q4k_init():
    _check(lib().q4k_init(), "q4k_init")


def q4k_dequant(W, N: int, K: int, out, stream=None):
    """out[n*K + k] = w(n, k): packed uint8 W -> fp32 out (both on the device)."""
    import torch
    _check_dtype(W, torch.uint8, "W")
    _check_dtype(out, torch.float32, "out")
    if _dims_valid(N, K):
        _check_size(W, _w_bytes(N, K), "W")
        _check_size(out, N * K, "out")
    _check(lib().q4k_dequant(_ptr(W), N, K, _ptr(out), _stream(stream)), "q4k_dequant")


def q4k_matmul(W, N: int, K: int, X, M: int, Y, stream=None):
    """Y[M, N] = X[M, K] (fp32) * W^T."""
    import torch
    _check_dtype(W, torch.uint8, "W")
    _check_dtype(X, torch.float32, "X")
    _check_dtype(Y, torch.float32, "Y")
    _check_matmul_sizes(W, N, K, X, M, Y)
    _check(lib().q4k_matmul(_ptr(W), N, K, _ptr(X), M, _ptr(Y), _stream(stream)), "q4k_matmul")


def q4k_matmul_bf16(W, N: int, K: int, X, M: int, Y, stream=None):
    """Y[M, N] = X[M, K] (bf16) * W^T."""
    import torch
    _check_dtype(W, torch.uint8, "W")
    _check_dtype(X, torch.bfloat16, "X")
    _check_dtype(Y, torch.float32, "Y")
    _check_matmul_sizes(W, N, K, X, M, Y)
    _check(lib().q4k_matmul_bf16(_ptr(W), N, K, _ptr(X), M, _ptr(Y), _stream(stream)),
           "q4k_matmul_bf16")


def q4k_matmul_multi(Ws, Ns, K: int, X, M: int, Ys, stream=None):
    """Y_i[M, N_i] = X[M, K] * W_i^T for matrices sharing K and X (fp32 or bf16 X)."""
    import torch
    count = len(Ws)
    if not (len(Ns) == len(Ys) == count):
        raise ValueError("Ws, Ns and Ys must have the same length")
    for W, Y in zip(Ws, Ys):
        _check_dtype(W, torch.uint8, "W")
        _check_dtype(Y, torch.float32, "Y")
    bf16 = not isinstance(X, int) and X.dtype == torch.bfloat16
    if not bf16:
        _check_dtype(X, torch.float32, "X")
    for W, N, Y in zip(Ws, Ns, Ys):
        _check_matmul_sizes(W, int(N), K, X, M, Y)
    w_arr = (ctypes.c_void_p * count)(*[_ptr(W) for W in Ws])
    n_arr = (ctypes.c_int64 * count)(*[int(n) for n in Ns])
    y_arr = (ctypes.c_void_p * count)(*[_ptr(Y) for Y in Ys])
    fn = lib().q4k_matmul_multi_bf16 if bf16 else lib().q4k_matmul_multi
    _check(fn(count, w_arr, n_arr, K, _ptr(X), M, y_arr, _stream(stream)), "q4k_matmul_multi")


def q4k_matmul_argmax(W, N: int, K: int, X, M: int, out, stream=None):
    """out[m] = argmax_n (X[M, K] * W^T)[m, n] (int64, lowest n on ties), fp32 or bf16 X, M <= 16."""
    import torch
    _check_dtype(W, torch.uint8, "W")
    _check_dtype(out, torch.int64, "out")
    bf16 = not isinstance(X, int) and X.dtype == torch.bfloat16
    if not bf16:
        _check_dtype(X, torch.float32, "X")
    _check_matmul_sizes(W, N, K, X, M, None)
    if M >= 1:
        _check_size(out, M, "out")
    fn = lib().q4k_matmul_argmax_bf16 if bf16 else lib().q4k_matmul_argmax
    _check(fn(_ptr(W), N, K, _ptr(X), M, _ptr(out), _stream(stream)), "q4k_matmul_argmax")


def argmax(W, N: int, K: int, X, out=None, stream=None):
    """Convenience: the fused argmax, allocating out with torch if not given."""
    import torch
    M = X.shape[0]
    if out is None:
        out = torch.empty(M, dtype=torch.int64, device=X.device)
    q4k_matmul_argmax(W, N, K, X, M, out, stream)
    return out


def q4k_selftest_timeout(limit_ns: int, stream=None):
    """Runs the one-thread kernel whose bounded wait runs out after limit_ns
    (the library's timeout path, without a fault); q4k_device_error() then
    reports Q4K_ERR_TIMEOUT."""
    _check(lib().q4k_selftest_timeout(int(limit_ns), _stream(stream)), "q4k_selftest_timeout")


def q4k_set_pdl(mode: int) -> int:
    """Programmatic-dependent-launch mode for later calls (0, 1 or 2); returns the old mode."""
    rc = lib().q4k_set_pdl(int(mode))
    if rc < 0:
        raise Q4KError(rc, "q4k_set_pdl")
    return rc


def q4k_device_error(clear: bool = True) -> int:
    """Status of the device error word (synchronous)."""
    return lib().q4k_device_error(1 if clear else 0)


def matmul(W, N: int, K: int, X, Y=None, stream=None):
    """Convenience: dispatch on X's dtype, allocating Y with torch if not given."""
    import torch
    M = X.shape[0]
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.float32, device=X.device)
    if X.dtype == torch.bfloat16:
        q4k_matmul_bf16(W, N, K, X, M, Y, stream)
    else:
        q4k_matmul(W, N, K, X, M, Y, stream)
    return Y
