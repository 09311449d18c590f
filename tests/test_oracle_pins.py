"""Pins of the CPU oracle against facts that do not come from the oracle itself.

- hand-worked super-blocks (tests/golden/q4k_hand_blocks.json, derived by hand
  from the Q4_K definition);
- IEEE binary16 / bfloat16 decoding against numpy's independent conversion on
  every bit pattern;
- per-bit isolation of all 96 scale bits, checked against a scatter table (which
  source bit lands in which destination field) that is the inverse view of the
  oracle's gather rule;
- pack -> unpack round trips through an independent packer;
- exactness: every Q4_K weight is d*sc*q - dmin*m rounded once to fp32 (the two
  products need at most 21 and 17 significant bits, so float64 evaluates the
  expression exactly and one float64 -> float32 conversion is the only rounding);
- brute force against numpy's float64 matmul on tiny shapes, and matmul
  invariants (one-hot rows, row sums, linearity, GEMM == stacked GEMVs).
"""
import json
import math
import os

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "q4k_hand_blocks.json")


# ---------------------------------------------------------------- packers ---
# Independent of the oracle: a scatter from fields to bytes.

def pack_scales(sc, m):
    s = [0] * 12
    for j in range(4):
        s[j] = (sc[j] & 63) | ((sc[j + 4] >> 4) << 6)
        s[j + 4] = (m[j] & 63) | ((m[j + 4] >> 4) << 6)
        s[j + 8] = (sc[j + 4] & 15) | ((m[j + 4] & 15) << 4)
    return s


def pack_qs(q):
    """q: 256 quants in weight order -> 128 qs bytes."""
    qs = [0] * 128
    for k, v in enumerate(q):
        c, r = divmod(k, 64)
        if r < 32:
            qs[32 * c + r] |= v & 15
        else:
            qs[32 * c + r - 32] |= (v & 15) << 4
    return qs


def make_block(d_bits, dmin_bits, scales, qs):
    b = [d_bits & 0xFF, d_bits >> 8, dmin_bits & 0xFF, dmin_bits >> 8]
    b += list(scales) + list(qs)
    assert len(b) == 144
    return np.array(b, dtype=np.uint8)


def f32_bits(a):
    return np.asarray(a, dtype=np.float32).view(np.uint32)


# ------------------------------------------------------------ golden file ---

def _golden_cases():
    with open(GOLDEN) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _golden_cases(), ids=lambda c: c["name"])
def test_hand_worked_blocks(oracle_mod, case):
    scales = [int(x, 16) for x in case["scales"].split()]
    if "sc" in case:
        # the hand-packed bytes agree with the independent packer
        assert pack_scales(case["sc"], case["m"]) == scales
        q = []
        for c in range(4):
            q += [(l + c) % 16 for l in range(32)]
            q += [(3 * l + c) % 16 for l in range(32)]
        qs = pack_qs(q)
    else:
        qs = [int(case["qs_fill"], 16)] * 128
        for pos, val in case.get("qs_set", {}).items():
            qs[int(pos)] = int(val, 16)
    blk = make_block(int(case["d"], 16), int(case["dmin"], 16), scales, qs)
    got = oracle_mod.dequant_block(blk)
    if "expect_per_subblock" in case:
        exp = np.repeat(np.array(case["expect_per_subblock"], np.float32), 32)
    elif "expect_all" in case:
        exp = np.full(256, case["expect_all"], np.float32)
    elif "expect_nonzero" in case:
        exp = np.zeros(256, np.float32)
        for k, v in case["expect_nonzero"].items():
            exp[int(k)] = v
    else:
        sc, m = case["sc"], case["m"]
        exp = np.array([0.25 * sc[k // 32] * q[k] - 0.125 * m[k // 32] for k in range(256)],
                       np.float32)
    # bitwise: the expected zeros are +0
    np.testing.assert_array_equal(f32_bits(got), f32_bits(exp))


# ------------------------------------------------------------ fp16 / bf16 ---

def test_fp16_spot_values(oracle_mod):
    assert oracle_mod.f16_to_f32(0x3C00) == 1.0
    assert oracle_mod.f16_to_f32(0x0001) == 2.0 ** -24
    assert oracle_mod.f16_to_f32(0x7BFF) == 65504.0
    z = oracle_mod.f16_to_f32(0x8000)
    assert z == 0.0 and math.copysign(1.0, z) == -1.0
    assert oracle_mod.f16_to_f32(0x3555) == 0.333251953125
    assert oracle_mod.f16_to_f32(0x7C00) == math.inf
    assert math.isnan(oracle_mod.f16_to_f32(0x7E00))


def test_fp16_all_patterns_match_numpy(oracle_mod):
    pats = np.arange(0, 1 << 16, dtype=np.uint32)
    ours = np.array([oracle_mod.f16_to_f32(int(h)) for h in pats], np.float32)
    ref = pats.astype(np.uint16).view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    np.testing.assert_array_equal(f32_bits(ours[~nan]), f32_bits(ref[~nan]))


def test_bf16_all_patterns(oracle_mod):
    pats = np.arange(0, 1 << 16, 97, dtype=np.uint32)
    scal = np.array([oracle_mod.bf16_to_f32_scalar(int(b)) for b in pats], np.float32)
    bulk = oracle_mod.bf16_to_f32(pats.astype(np.uint16))
    ok = ~np.isnan(scal)
    np.testing.assert_array_equal(f32_bits(scal[ok]), f32_bits(bulk[ok]))
    assert oracle_mod.bf16_to_f32_scalar(0x3F80) == 1.0
    assert oracle_mod.bf16_to_f32_scalar(0xC000) == -2.0


# ------------------------------------------------------ scale bit isolation ---

def _bit_destination(i, t):
    """Which field one set bit (byte i, bit t) of the 12 scale bytes feeds."""
    if i < 4:
        return ("sc", i, 1 << t) if t < 6 else ("sc", i + 4, 1 << (t - 2))
    if i < 8:
        return ("m", i - 4, 1 << t) if t < 6 else ("m", i, 1 << (t - 2))
    return ("sc", i - 4, 1 << t) if t < 4 else ("m", i - 4, 1 << (t - 4))


def test_scale_bits_isolated(oracle_mod):
    hit = set()
    for i in range(12):
        for t in range(8):
            s = [0] * 12
            s[i] = 1 << t
            sc, m = oracle_mod.unpack_scales(s)
            field, j, val = _bit_destination(i, t)
            exp_sc, exp_m = [0] * 8, [0] * 8
            (exp_sc if field == "sc" else exp_m)[j] = val
            assert (sc, m) == (exp_sc, exp_m), (i, t)
            hit.add((field, j, val))
    # the 96 bits cover every bit of the 16 six-bit fields exactly once
    assert len(hit) == 96


# ----------------------------------------------------------- round trips ---

def test_scale_pack_roundtrip_every_value(oracle_mod):
    rng = np.random.default_rng(1)
    for slot in range(16):
        for v in range(64):
            vals = rng.integers(0, 64, 16).tolist()
            vals[slot] = v
            sc, m = vals[:8], vals[8:]
            assert oracle_mod.unpack_scales(pack_scales(sc, m)) == (sc, m)


def test_scale_pack_roundtrip_random(oracle_mod):
    rng = np.random.default_rng(2)
    draws = rng.integers(0, 64, (20000, 16))
    for row in draws:
        sc, m = row[:8].tolist(), row[8:].tolist()
        assert oracle_mod.unpack_scales(pack_scales(sc, m)) == (sc, m)


def test_quant_pack_roundtrip(oracle_mod):
    rng = np.random.default_rng(3)
    ones = pack_scales([1] * 8, [0] * 8)
    for _ in range(50):
        q = rng.integers(0, 16, 256).tolist()
        blk = make_block(0x3C00, 0x0000, ones, pack_qs(q))
        np.testing.assert_array_equal(oracle_mod.dequant_block(blk), np.array(q, np.float32))


def _random_fp16_bits(rng, n):
    bits = rng.integers(0, 1 << 16, n).astype(np.uint16)
    finite = np.isfinite(bits.view(np.float16))
    return bits[finite]


def test_weights_are_the_exact_value_rounded_once(oracle_mod):
    rng = np.random.default_rng(4)
    dd = _random_fp16_bits(rng, 4000)
    for t in range(1500):
        d_bits, dmin_bits = int(dd[2 * t]), int(dd[2 * t + 1])
        sc = rng.integers(0, 64, 8).tolist()
        m = rng.integers(0, 64, 8).tolist()
        q = rng.integers(0, 16, 256).tolist()
        blk = make_block(d_bits, dmin_bits, pack_scales(sc, m), pack_qs(q))
        d = np.float64(np.uint16(d_bits).view(np.float16))
        dmin = np.float64(np.uint16(dmin_bits).view(np.float16))
        exact = np.array([d * sc[k // 32] * q[k] - dmin * m[k // 32] for k in range(256)],
                         np.float64)
        np.testing.assert_array_equal(f32_bits(oracle_mod.dequant_block(blk)),
                                      f32_bits(exact.astype(np.float32)))


def test_power_of_two_scales_exact(oracle_mod):
    # d = 2^-e, dmin = 2^-f: every weight is exactly sc*q*2^-e - m*2^-f
    rng = np.random.default_rng(5)
    for e in range(0, 14, 3):
        for f in range(0, 14, 4):
            d_bits = int(np.float16(2.0 ** -e).view(np.uint16))
            dmin_bits = int(np.float16(2.0 ** -f).view(np.uint16))
            sc = rng.integers(0, 64, 8).tolist()
            m = rng.integers(0, 64, 8).tolist()
            q = rng.integers(0, 16, 256).tolist()
            blk = make_block(d_bits, dmin_bits, pack_scales(sc, m), pack_qs(q))
            exp = [math.ldexp(sc[k // 32] * q[k], -e) - math.ldexp(m[k // 32], -f)
                   for k in range(256)]
            np.testing.assert_array_equal(oracle_mod.dequant_block(blk),
                                          np.array(exp, np.float32))


# ------------------------------------------------------- matrix and matmul ---

def _random_matrix(rng, N, K):
    return rng.integers(0, 256, N * (K // 256) * 144).astype(np.uint8)


def _finite_matrix(rng, N, K):
    W = _random_matrix(rng, N, K).reshape(N * K // 256, 144)
    for blk in W:  # d, dmin in [1e-3, 2e-2] like the workloads
        for off in (0, 2):
            v = np.float16(rng.uniform(1e-3, 2e-2)).view(np.uint16)
            blk[off], blk[off + 1] = int(v) & 0xFF, int(v) >> 8
    return W.reshape(-1)


def test_dequant_matrix_layout(oracle_mod):
    rng = np.random.default_rng(6)
    N, K = 3, 768
    W = _finite_matrix(rng, N, K)
    full = oracle_mod.dequant(W, N, K)
    blocks = W.reshape(N, K // 256, 144)
    for n in range(N):
        for b in range(K // 256):
            np.testing.assert_array_equal(full[n, 256 * b:256 * (b + 1)],
                                          oracle_mod.dequant_block(blocks[n, b]))


@pytest.mark.parametrize("N", [1, 2, 3])
@pytest.mark.parametrize("K", [256, 512])
@pytest.mark.parametrize("M", [1, 2, 3])
def test_matmul_brute_force(oracle_mod, N, K, M):
    rng = np.random.default_rng(100 * N + 10 * K + M)
    W = _finite_matrix(rng, N, K)
    X = rng.standard_normal((M, K)).astype(np.float32)
    Y, A = oracle_mod.matmul(W, N, K, X)
    w = oracle_mod.dequant(W, N, K).astype(np.float64)
    x = X.astype(np.float64)
    Yr = x @ w.T
    Ar = np.abs(x) @ np.abs(w).T
    np.testing.assert_allclose(Y, Yr, rtol=0, atol=1e-12 * Ar.max())
    np.testing.assert_allclose(A, Ar, rtol=1e-13)


def test_matmul_invariants(oracle_mod):
    rng = np.random.default_rng(7)
    N, K, M = 5, 512, 4
    W = _finite_matrix(rng, N, K)
    w = oracle_mod.dequant(W, N, K)
    # one-hot rows pick single weights exactly
    ks = [0, 31, 32, 255, 256, 300, 511]
    X = np.zeros((len(ks), K), np.float32)
    for i, k in enumerate(ks):
        X[i, k] = 1.0
    Y, _ = oracle_mod.matmul(W, N, K, X)
    np.testing.assert_array_equal(Y, w[:, ks].T.astype(np.float64))
    # all-ones row gives row sums
    Y1, _ = oracle_mod.matmul(W, N, K, np.ones((1, K), np.float32))
    np.testing.assert_allclose(Y1[0], [math.fsum(map(float, w[n])) for n in range(N)],
                               rtol=0, atol=1e-12 * np.abs(w).sum(axis=1).max())
    # linearity (small-integer activations keep 2*X1 - 0.5*X2 exact in fp32)
    X1 = rng.integers(-8, 9, (M, K)).astype(np.float32)
    X2 = rng.integers(-8, 9, (M, K)).astype(np.float32)
    Ya, Aa = oracle_mod.matmul(W, N, K, X1)
    Yb, Ab = oracle_mod.matmul(W, N, K, X2)
    Yc, _ = oracle_mod.matmul(W, N, K, (2.0 * X1 - 0.5 * X2).astype(np.float32))
    np.testing.assert_allclose(Yc, 2.0 * Ya - 0.5 * Yb, rtol=0, atol=1e-12 * (Aa + Ab).max())
    # a GEMM over M rows equals M separate GEMVs, bit for bit
    for m in range(M):
        Ym, Am = oracle_mod.matmul(W, N, K, X1[m:m + 1])
        np.testing.assert_array_equal(Ym[0], Ya[m])
        np.testing.assert_array_equal(Am[0], Aa[m])
    # row-subset mode and thread count do not change any output
    Ys, As = oracle_mod.matmul(W, N, K, X1, rows=[4, 0, 2], threads=3)
    np.testing.assert_array_equal(Ys, Ya[:, [4, 0, 2]])
    np.testing.assert_array_equal(As, Aa[:, [4, 0, 2]])


def test_oracle_rejects_bad_dims(oracle_mod):
    W = np.zeros(144, np.uint8)
    with pytest.raises(ValueError):
        oracle_mod.dequant(W, 1, 255)
    with pytest.raises(ValueError):
        oracle_mod.matmul(W, 1, 256, np.zeros((1, 256), np.float32), rows=[1])
