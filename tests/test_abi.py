"""The C ABI without a GPU: the library builds for sm_103a, loads, exports every
symbol include/q4k.h declares, and rejects bad arguments on the host before any
CUDA call."""
import ctypes
import os
import re

import pytest

import gguf_q4_dequant_gb300 as q4k_pkg

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                      "include", "q4k.h")


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(q4k_\w+)\s*\(", text)))


def test_header_matches_binding_exports():
    assert _declared_functions() == sorted(q4k_pkg.EXPORTS)


def test_library_exports_every_declared_symbol(q4k):
    L = ctypes.CDLL(q4k.LIB_PATH)
    for name in _declared_functions():
        assert hasattr(L, name), name


def test_status_strings(q4k):
    for code in (0, -1, -2, -3, -4, -5, -6):
        s = q4k.status_string(code)
        assert s.startswith("Q4K_")
    assert q4k.status_string(7) == "unknown q4k status"


# Host-side checks happen before the library touches the device, so they run
# here without a GPU. Pointers are plain integers that are never dereferenced.
A16 = 1 << 20  # a 16-byte-aligned fake address


@pytest.mark.parametrize("call", ["dequant", "matmul", "matmul_bf16"])
def test_null_pointers_rejected(q4k, call):
    L = q4k.lib()
    if call == "dequant":
        assert L.q4k_dequant(None, 4, 256, A16, None) == q4k.Q4K_ERR_NULL
        assert L.q4k_dequant(A16, 4, 256, None, None) == q4k.Q4K_ERR_NULL
    else:
        f = L.q4k_matmul if call == "matmul" else L.q4k_matmul_bf16
        assert f(None, 4, 256, A16, 1, A16, None) == q4k.Q4K_ERR_NULL
        assert f(A16, 4, 256, None, 1, A16, None) == q4k.Q4K_ERR_NULL
        assert f(A16, 4, 256, A16, 1, None, None) == q4k.Q4K_ERR_NULL


@pytest.mark.parametrize("N,K,M", [(0, 256, 1), (-3, 256, 1), (4, 0, 1), (4, 255, 1), (4, 384, 1),
                                   (4, 128, 1), (4, 256, 0), (4, 256, -1), (1 << 31, 256, 1),
                                   (4, (1 << 24) + 256, 1), (4, 256, 1 << 31)])
def test_bad_dims_rejected(q4k, N, K, M):
    L = q4k.lib()
    assert L.q4k_matmul(A16, N, K, A16, M, A16, None) == q4k.Q4K_ERR_BAD_DIM
    assert L.q4k_matmul_bf16(A16, N, K, A16, M, A16, None) == q4k.Q4K_ERR_BAD_DIM
    if 1 <= M < (1 << 31):  # the dimension at fault is N or K
        assert L.q4k_dequant(A16, N, K, A16, None) == q4k.Q4K_ERR_BAD_DIM


def test_misaligned_pointers_rejected(q4k):
    L = q4k.lib()
    for off in (1, 4, 8):
        assert L.q4k_dequant(A16 + off, 4, 256, A16, None) == q4k.Q4K_ERR_ALIGN
        assert L.q4k_dequant(A16, 4, 256, A16 + off, None) == q4k.Q4K_ERR_ALIGN
        assert L.q4k_matmul(A16, 4, 256, A16 + off, 1, A16, None) == q4k.Q4K_ERR_ALIGN
        assert L.q4k_matmul_bf16(A16, 4, 256, A16, 1, A16 + off, None) == q4k.Q4K_ERR_ALIGN


def test_binding_rejects_wrong_dtypes(q4k):
    torch = pytest.importorskip("torch")
    W = torch.zeros(144, dtype=torch.int8)
    with pytest.raises(ValueError):
        q4k.q4k_matmul(W, 1, 256, 0, 1, 0, stream=0)


def test_missing_library_fails_loudly(monkeypatch):
    import gguf_q4_dequant_gb300 as m
    monkeypatch.setattr(m, "_lib", None)
    monkeypatch.setattr(m, "LIB_PATH", "/nonexistent/libq4k.so")
    with pytest.raises(m.Q4KError):
        m.lib()


def test_set_pdl_modes(q4k):
    L = q4k.lib()
    old = L.q4k_set_pdl(0)
    try:
        assert L.q4k_set_pdl(2) == 0
        assert L.q4k_set_pdl(1) == 2
        assert L.q4k_set_pdl(3) == q4k.Q4K_ERR_BAD_DIM
        assert L.q4k_set_pdl(-1) == q4k.Q4K_ERR_BAD_DIM
        assert L.q4k_set_pdl(0) == 1
    finally:
        L.q4k_set_pdl(old)


def test_grouped_call_host_checks(q4k):
    import ctypes as C
    L = q4k.lib()
    W = (C.c_void_p * 3)(A16, A16, A16)
    Y = (C.c_void_p * 3)(A16, A16, A16)
    N = (C.c_int64 * 3)(256, 128, 7)
    assert L.q4k_matmul_multi(0, W, N, 256, A16, 1, Y, None) == q4k.Q4K_ERR_BAD_DIM
    assert L.q4k_matmul_multi(9, W, N, 256, A16, 1, Y, None) == q4k.Q4K_ERR_BAD_DIM
    assert L.q4k_matmul_multi(3, None, N, 256, A16, 1, Y, None) == q4k.Q4K_ERR_NULL
    Wn = (C.c_void_p * 3)(A16, None, A16)
    assert L.q4k_matmul_multi(3, Wn, N, 256, A16, 1, Y, None) == q4k.Q4K_ERR_NULL
    Nb = (C.c_int64 * 3)(256, 0, 7)
    assert L.q4k_matmul_multi_bf16(3, W, Nb, 256, A16, 1, Y, None) == q4k.Q4K_ERR_BAD_DIM
    Ym = (C.c_void_p * 3)(A16, A16 + 4, A16)
    assert L.q4k_matmul_multi(3, W, N, 256, A16, 1, Ym, None) == q4k.Q4K_ERR_ALIGN
    assert L.q4k_matmul_multi(3, W, N, 300, A16, 1, Y, None) == q4k.Q4K_ERR_BAD_DIM


def test_argmax_host_checks(q4k):
    L = q4k.lib()
    for f in (L.q4k_matmul_argmax, L.q4k_matmul_argmax_bf16):
        assert f(None, 4, 256, A16, 1, A16, None) == q4k.Q4K_ERR_NULL
        assert f(A16, 4, 256, None, 1, A16, None) == q4k.Q4K_ERR_NULL
        assert f(A16, 4, 256, A16, 1, None, None) == q4k.Q4K_ERR_NULL
        assert f(A16, 4, 256, A16, 0, A16, None) == q4k.Q4K_ERR_BAD_DIM
        assert f(A16, 4, 256, A16, 17, A16, None) == q4k.Q4K_ERR_BAD_DIM   # decode only
        assert f(A16, 4, 300, A16, 1, A16, None) == q4k.Q4K_ERR_BAD_DIM
        assert f(A16, 4, 256, A16, 1, A16 + 4, None) == q4k.Q4K_ERR_ALIGN  # int64 out: 8-byte aligned
        assert f(A16, 4, 256, A16 + 8, 1, A16, None) == q4k.Q4K_ERR_ALIGN


def test_selftest_timeout_rejects_bad_limits(q4k):
    L = q4k.lib()
    for limit in (0, -5, 1_000_000_001):
        assert L.q4k_selftest_timeout(limit, None) == q4k.Q4K_ERR_BAD_DIM


def test_binding_checks_tensor_sizes(q4k):
    """A tensor shorter than the call needs is refused before the C ABI is
    reached (the kernels would read or write past it)."""
    torch = pytest.importorskip("torch")
    N, K, M = 4, 512, 3
    W = torch.zeros(N * (K // 256) * 144, dtype=torch.uint8)
    X = torch.zeros(M, K)
    Y = torch.zeros(M, N)
    cases = [
        lambda: q4k.q4k_matmul(W[:-16], N, K, X, M, Y),
        lambda: q4k.q4k_matmul(W, N, K, X[:2], M, Y),
        lambda: q4k.q4k_matmul(W, N, K, X, M, Y[:, :3].contiguous()),
        lambda: q4k.q4k_matmul_bf16(W, N, K, X.to(torch.bfloat16)[:1], M, Y),
        lambda: q4k.q4k_dequant(W, N, K, torch.zeros(N * K - 1)),
        lambda: q4k.q4k_dequant(W[:100], N, K, torch.zeros(N * K)),
        lambda: q4k.q4k_matmul_multi([W, W[:10]], [N, N], K, X, M, [Y, Y]),
        lambda: q4k.q4k_matmul_multi([W, W], [N, N], K, X, M, [Y, Y[:1]]),
        lambda: q4k.q4k_matmul_argmax(W, N, K, X, M, torch.zeros(M - 1, dtype=torch.int64)),
    ]
    for call in cases:
        with pytest.raises(ValueError, match="the call needs"):
            call()
    # right sizes pass the size checks and stop at the device check (host tensors)
    with pytest.raises(ValueError, match="CUDA device memory"):
        q4k.q4k_matmul(W, N, K, X, M, Y)
