"""The oracle pins must catch plausible mistakes.

Each case plants one mistake in a copy of the oracle's C++ source (a dropped
term, a wrong sign, index or shift, swapped nibbles, a wrong fp16 bias, a
transposed operand), compiles the copy with gcc into a temporary directory, and
checks that at least one pin fails on it. The real oracle is never modified.
"""
import ctypes
import os
import subprocess

import numpy as np
import pytest

import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "oracle", "q4k_oracle.cpp")

MUTANTS = {
    "m_low_wrong_byte": ("m[j] = s[j + 4] & 63;", "m[j] = s[j] & 63;"),
    "sc_high_shift": ("((s[j - 4] >> 6) << 4)", "((s[j - 4] >> 6) << 3)"),
    "m_high_wrong_byte": ("(s[j + 4] >> 4) | ((s[j] >> 6) << 4)",
                          "(s[j + 4] >> 4) | ((s[j - 4] >> 6) << 4)"),
    "sc_high_mask": ("(s[j + 4] & 15)", "(s[j + 4] & 31)"),
    "nibbles_swapped": ("q_lo = byte & 15, q_hi = byte >> 4", "q_lo = byte >> 4, q_hi = byte & 15"),
    "min_term_dropped": ("out[64 * c + l] = t_lo - u_lo;", "out[64 * c + l] = t_lo;"),
    "min_sign": ("out[64 * c + 32 + l] = t_hi - u_hi;", "out[64 * c + 32 + l] = t_hi + u_hi;"),
    "byte_index": ("qs[32 * c + l]", "qs[32 * c + (l ^ 1)]"),
    "chunk_stride": ("out[64 * c + 32 + l]", "out[64 * c + 16 + l]"),
    "dmin_for_d": ("const float t_lo = (d * (float)sc[j_lo])", "const float t_lo = (dmin * (float)sc[j_lo])"),
    "fp16_bias": ("expo - 25", "expo - 24"),
    "fp16_subnormal": ("std::ldexp((double)frac, -24)", "std::ldexp((double)frac, -23)"),
    "header_swap": ("oracle_f16_to_f32((uint16_t)(blk[0] | (blk[1] << 8)))",
                    "oracle_f16_to_f32((uint16_t)(blk[1] | (blk[0] << 8)))"),
    "x_transposed": ("const float* x = X + mi * K;", "const float* x = X + mi;"),
    "abs_dropped": ("aab += std::fabs(p);", "aab += p;"),
    "sc_low_mask": ("sc[j] = s[j] & 63;", "sc[j] = s[j] & 127;"),
    "high_nibble_sub_block": ("j_hi = 2 * c + 1", "j_hi = 2 * c"),
    "min_of_other_sub_block": ("const float u_lo = dmin * (float)m[j_lo];",
                               "const float u_lo = dmin * (float)m[j_hi];"),
    "inf_nan_swapped": ("frac == 0 ? INFINITY : NAN", "frac == 0 ? NAN : INFINITY"),
    "fp32_accumulator": ("acc += p;", "acc = (float)(acc + p);"),
    "row_subset_ignored": ("const int64_t n = rows ? rows[r] : r;", "const int64_t n = r;"),
    "last_thread_rows_dropped": ("r1 = std::min(nrows, r0 + per)", "r1 = std::min(nrows - 1, r0 + per)"),
    "row_layout": ("oracle_dequant_block(W + (n * KB + b) * 144, out + n * K + b * 256);",
                   "oracle_dequant_block(W + (b * N + n) * 144, out + n * K + b * 256);"),
}


class _Mutant:
    """Same call surface as the oracle module, backed by a mutated build."""

    def __init__(self, path):
        lib = ctypes.CDLL(path)
        u8p, f32p = ctypes.POINTER(ctypes.c_uint8), ctypes.POINTER(ctypes.c_float)
        f64p, i64p = ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int64)
        lib.oracle_f16_to_f32.argtypes = [ctypes.c_uint16]
        lib.oracle_f16_to_f32.restype = ctypes.c_float
        lib.oracle_unpack_scales.argtypes = [u8p, u8p, u8p]
        lib.oracle_dequant_block.argtypes = [u8p, f32p]
        lib.oracle_dequant.argtypes = [u8p, ctypes.c_int64, ctypes.c_int64, f32p]
        lib.oracle_matmul.argtypes = [u8p, ctypes.c_int64, ctypes.c_int64, f32p, ctypes.c_int64,
                                      i64p, ctypes.c_int64, f64p, f64p, ctypes.c_int]
        self.lib = lib

    @staticmethod
    def _p(a, t):
        return a.ctypes.data_as(ctypes.POINTER(t))

    def f16_to_f32(self, h):
        return float(self.lib.oracle_f16_to_f32(int(h) & 0xFFFF))

    def unpack_scales(self, s12):
        s = np.ascontiguousarray(np.asarray(s12, np.uint8).reshape(12))
        sc, m = np.zeros(8, np.uint8), np.zeros(8, np.uint8)
        self.lib.oracle_unpack_scales(self._p(s, ctypes.c_uint8), self._p(sc, ctypes.c_uint8),
                                      self._p(m, ctypes.c_uint8))
        return [int(v) for v in sc], [int(v) for v in m]

    def dequant_block(self, blk):
        b = np.ascontiguousarray(np.asarray(blk, np.uint8).reshape(144))
        out = np.empty(256, np.float32)
        self.lib.oracle_dequant_block(self._p(b, ctypes.c_uint8), self._p(out, ctypes.c_float))
        return out

    def dequant(self, W, N, K):
        w = np.ascontiguousarray(W, np.uint8).reshape(-1)
        out = np.empty((N, K), np.float32)
        self.lib.oracle_dequant(self._p(w, ctypes.c_uint8), N, K, self._p(out, ctypes.c_float))
        return out

    def matmul(self, W, N, K, X, rows=None, threads=0):
        w = np.ascontiguousarray(W, np.uint8).reshape(-1)
        x = np.ascontiguousarray(X, np.float32)
        M = x.shape[0]
        rr = None if rows is None else np.ascontiguousarray(rows, np.int64)
        nrows = N if rr is None else rr.size
        Y, A = np.empty((M, nrows)), np.empty((M, nrows))
        self.lib.oracle_matmul(self._p(w, ctypes.c_uint8), N, K, self._p(x, ctypes.c_float), M,
                               None if rr is None else self._p(rr, ctypes.c_int64), nrows,
                               self._p(Y, ctypes.c_double), self._p(A, ctypes.c_double), threads)
        return Y, A


def _pins_fail(mod):
    """Run the pin checks against ``mod``; True if any of them fails."""
    checks = [lambda: [pins.test_hand_worked_blocks(mod, c) for c in pins._golden_cases()],
              lambda: pins.test_fp16_spot_values(mod),
              lambda: pins.test_fp16_all_patterns_match_numpy(mod),
              lambda: pins.test_scale_bits_isolated(mod),
              lambda: pins.test_weights_are_the_exact_value_rounded_once(mod),
              lambda: pins.test_dequant_matrix_layout(mod),
              lambda: pins.test_matmul_brute_force(mod, 2, 512, 3),
              lambda: pins.test_matmul_invariants(mod)]
    for chk in checks:
        try:
            chk()
        except AssertionError:
            return True
    return False


def test_unmutated_copy_passes(tmp_path):
    so = tmp_path / "orig.so"
    subprocess.run(["g++", "-O2", "-ffp-contract=off", "-std=c++17", "-shared", "-fPIC",
                    "-pthread", SRC, "-o", str(so)], check=True)
    assert not _pins_fail(_Mutant(str(so)))


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    old, new = MUTANTS[name]
    text = open(SRC).read()
    assert text.count(old) == 1, f"mutation site for {name} not unique"
    src = tmp_path / f"{name}.cpp"
    src.write_text(text.replace(old, new, 1))
    so = tmp_path / f"{name}.so"
    subprocess.run(["g++", "-O2", "-ffp-contract=off", "-std=c++17", "-shared", "-fPIC",
                    "-pthread", str(src), "-o", str(so)], check=True)
    assert _pins_fail(_Mutant(str(so))), f"pins did not catch mutant {name}"
