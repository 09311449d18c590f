"""The worst-case error bound of the factored GEMV is gamma_n * R * sum|w*x|,
where R = sum(|d*sc*q*x| + |dmin*m*x|) / sum|w*x| measures cancellation between the
two terms of each weight. These checks pin R on the workloads' weight
distribution. The bound (n <= 100 roundings for K <= 17408) then stays far
inside the 1e-4 bar of the decode path. The weight fields are unpacked here from
the Q4_K definition, and the weights they give are checked against the oracle."""
import numpy as np
import pytest

from gguf_q4_dequant_gb300 import synth

U = 2.0 ** -24


def _fields(Wr, K):
    blk = Wr.reshape(Wr.shape[0], K // 256, 144)
    d = blk[:, :, 0:2].copy().view(np.float16)[..., 0].astype(np.float64)
    dmin = blk[:, :, 2:4].copy().view(np.float16)[..., 0].astype(np.float64)
    s = blk[:, :, 4:16].astype(np.int64)
    sc = np.zeros(s.shape[:2] + (8,))
    m = np.zeros(s.shape[:2] + (8,))
    for j in range(8):
        if j < 4:
            sc[..., j], m[..., j] = s[..., j] & 63, s[..., j + 4] & 63
        else:
            sc[..., j] = (s[..., j + 4] & 15) | ((s[..., j - 4] >> 6) << 4)
            m[..., j] = (s[..., j + 4] >> 4) | ((s[..., j] >> 6) << 4)
    qs = blk[:, :, 16:].astype(np.int64)
    q = np.zeros(s.shape[:2] + (256,))
    for c in range(4):
        q[..., 64 * c:64 * c + 32] = qs[..., 32 * c:32 * c + 32] & 15
        q[..., 64 * c + 32:64 * c + 64] = qs[..., 32 * c:32 * c + 32] >> 4
    j = np.arange(256) // 32
    return d[..., None] * sc[..., j] * q, dmin[..., None] * m[..., j]


@pytest.mark.parametrize("wl", [1, 2, 3, 4])
def test_cancellation_ratio_keeps_the_gemv_bound_inside_the_bar(oracle_mod, wl):
    w = synth.WORKLOADS[wl]
    worst = 0.0
    for (layer, name, N, K) in w.matrices():
        if layer != 0 and name != "lm_head":
            continue
        rows = list(range(0, N, N // 16))[:16]
        Wr = synth.weight_sample_rows(synth.weight_seed(wl, layer, name), N, K, rows).numpy()
        t1, t2 = _fields(Wr, K)
        wv = t1 - t2
        ref = oracle_mod.dequant(Wr, len(rows), K).astype(np.float64)
        np.testing.assert_allclose(wv.reshape(len(rows), K), ref, rtol=0, atol=2.0 ** -20 * np.abs(ref).max())
        x = synth.activations(synth.x_seed(wl, K, 1), 1, K).numpy()[0].astype(np.float64)
        xb = x.reshape(K // 256, 256)[None]
        R = (np.abs(t1 * xb).sum((1, 2)) + np.abs(t2 * xb).sum((1, 2))) / np.abs(wv * xb).sum((1, 2))
        worst = max(worst, float(R.max()))
        n = 27 + K // 256  # roundings per product, at most
        assert n * U / (1 - n * U) * R.max() < 1e-4 / 4
    assert worst < 2.0
