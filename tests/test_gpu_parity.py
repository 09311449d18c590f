"""GPU parity: libq4k (through its C ABI) against the CPU oracle, element by element.

Bars: dequant bit-exact; GEMV (M <= 16, fp32 or bf16 activations) within
1e-4 * sum_k |x*w| per output; tcgen05 GEMM (bf16 activations, M >= 17) within
5e-3 * sum_k |x*w| per output. Inputs are drawn on the host by the seeded
generator and copied to the device; expected values come from the oracle only.
"""
import numpy as np
import pytest
import torch

from gguf_q4_dequant_gb300 import synth

pytestmark = pytest.mark.gpu

TOL_GEMV = 1e-4
TOL_GEMM = 5e-3
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _cuda(q4k):
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    torch.cuda.set_device(0)
    q4k.q4k_init()
    yield
    torch.cuda.synchronize()
    assert q4k.q4k_device_error() == 0


def _x_for_oracle(oracle_mod, X):
    if X.dtype == torch.bfloat16:
        return oracle_mod.bf16_to_f32(X.view(torch.int16).numpy().view(np.uint16))
    return X.numpy()


def _check_matmul(q4k, oracle_mod, Wh, Wd, N, K, X, tol, rows=None, W_rows=None):
    """Runs the library on (Wd, X) and compares the columns `rows` (all if None)."""
    M = X.shape[0]
    Y = torch.full((M, N), float("nan"), device=DEV)
    q4k.matmul(Wd, N, K, X.to(DEV), Y)
    torch.cuda.synchronize()
    Xo = _x_for_oracle(oracle_mod, X)
    if rows is None:
        Yref, A = oracle_mod.matmul(Wh.numpy(), N, K, Xo)
        got = Y.cpu().double().numpy()
    else:
        Yref, A = oracle_mod.matmul(W_rows.numpy(), len(rows), K, Xo)
        got = Y[:, torch.as_tensor(rows, device=DEV)].cpu().double().numpy()
    assert np.all(np.isfinite(got)), "unwritten or non-finite outputs"
    err = np.abs(got - Yref)
    bound = tol * A + 1e-30
    worst = float(np.max(err / bound))
    assert worst <= 1.0, f"max |err| / ({tol} * sum|wx|) = {worst:.3f}"
    return worst


# ------------------------------------------------------------------ dequant ---

def _dequant_check(q4k, oracle_mod, Wh, N, K):
    out = torch.full((N, K), float("nan"), device=DEV)
    q4k.q4k_dequant(Wh.to(DEV), N, K, out)
    torch.cuda.synchronize()
    ref = oracle_mod.dequant(Wh.numpy(), N, K)
    got = out.cpu().numpy()
    np.testing.assert_array_equal(got.view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("N,K", [(1, 256), (3, 512), (256, 512), (257, 1280), (64, 17408)])
def test_dequant_bit_exact(q4k, oracle_mod, N, K):
    _dequant_check(q4k, oracle_mod, synth.weight_rows(1000 + N, N, K), N, K)


def test_dequant_arbitrary_fp16_scales(q4k, oracle_mod):
    # d and dmin over (almost) all finite fp16 bit patterns, incl. subnormals and negatives
    rng = np.random.default_rng(11)
    N, K = 512, 1024
    Wh = synth.weight_rows(77, N, K).numpy().reshape(-1, 144).copy()
    bits = rng.integers(0, 1 << 16, (Wh.shape[0], 2)).astype(np.uint16)
    bits[~np.isfinite(bits.view(np.float16))] = 0x3C00
    Wh[:, 0:4] = bits.view(np.uint8).reshape(-1, 4)
    _dequant_check(q4k, oracle_mod, torch.from_numpy(Wh.reshape(N, -1)), N, K)


def test_dequant_golden_blocks(q4k, oracle_mod):
    import test_oracle_pins as pins
    blocks = []
    for case in pins._golden_cases():
        scales = [int(x, 16) for x in case["scales"].split()]
        qs = [int(case.get("qs_fill", "00"), 16)] * 128
        for pos, val in case.get("qs_set", {}).items():
            qs[int(pos)] = int(val, 16)
        blocks.append(pins.make_block(int(case["d"], 16), int(case["dmin"], 16), scales, qs))
    Wh = torch.from_numpy(np.stack(blocks))
    _dequant_check(q4k, oracle_mod, Wh, len(blocks), 256)


@pytest.mark.parametrize("wl", [1, 2, 3, 4])
def test_dequant_layer0_full_size(q4k, oracle_mod, wl):
    w = synth.WORKLOADS[wl]
    shapes = {(n, k): m for (layer, m, n, k) in w.matrices() if layer == 0 or m == "lm_head"}
    for (N, K), name in shapes.items():
        Wh = synth.weight_rows(synth.weight_seed(wl, 0, name), N, K)
        _dequant_check(q4k, oracle_mod, Wh, N, K)


# --------------------------------------------------------------------- GEMV ---

@pytest.mark.parametrize("N", [1, 7, 32, 33, 100, 300])
@pytest.mark.parametrize("K", [256, 768, 2048])
@pytest.mark.parametrize("xdt", ["f32", "bf16"])
def test_gemv_ragged(q4k, oracle_mod, N, K, xdt):
    Wh = synth.weight_rows(2000 + N + K, N, K)
    Wd = Wh.to(DEV)
    dt = torch.bfloat16 if xdt == "bf16" else torch.float32
    for M in (1, 2, 3, 4, 5, 8, 9, 13, 16):
        X = synth.activations(3000 + M + K, M, K, dt)
        _check_matmul(q4k, oracle_mod, Wh, Wd, N, K, X, TOL_GEMV)


@pytest.mark.parametrize("N", [1, 128, 300])
@pytest.mark.parametrize("KB", [64, 37])
@pytest.mark.parametrize("M,xdt", [(1, "f32"), (2, "f32"), (3, "bf16"), (16, "f32")])
def test_gemv_split_k_widths(q4k, oracle_mod, N, KB, M, xdt):
    """Few tiles and a long K: the launch splits K across clusters of up to 16
    CTAs (8 for M > 2), with K-slices that do not divide K evenly (37 super-blocks);
    the ranks' partial sums meet in rank 0's shared memory."""
    K = 256 * KB
    Wh = synth.weight_rows(7000 + N + KB, N, K)
    dt = torch.bfloat16 if xdt == "bf16" else torch.float32
    X = synth.activations(7100 + M + KB, M, K, dt)
    _check_matmul(q4k, oracle_mod, Wh, Wh.to(DEV), N, K, X, TOL_GEMV)


@pytest.mark.parametrize("M", [1, 4])
def test_gemv_tiny_workload(q4k, oracle_mod, M):
    w = synth.WORKLOADS[0]
    (_, name, N, K), = w.matrices()
    Wh = synth.weight_rows(synth.weight_seed(0, 0, name), N, K)
    X = synth.activations(synth.x_seed(0, K, M), M, K)
    _check_matmul(q4k, oracle_mod, Wh, Wh.to(DEV), N, K, X, TOL_GEMV)


def test_gemv_activation_scales(q4k, oracle_mod):
    # per-block exponent handling: huge, tiny, zero and mixed-magnitude blocks
    N, K = 96, 2048
    Wh = synth.weight_rows(5, N, K)
    Wd = Wh.to(DEV)
    base = synth.activations(6, 4, K)
    scale = torch.ones(4, K)
    scale[0, :256] = 1e30
    scale[0, 256:512] = 1e-30
    scale[1, :] = 1e-38
    scale[2, 512:768] = 0.0
    scale[3, ::7] = 3e4
    X = (base * scale).float()
    _check_matmul(q4k, oracle_mod, Wh, Wd, N, K, X, TOL_GEMV)
    _check_matmul(q4k, oracle_mod, Wh, Wd, N, K, torch.zeros(2, K), TOL_GEMV)


@pytest.mark.parametrize("N,K", [(96, 2048), (300, 256), (40960, 1024)])
def test_gemv_activation_scales_one_and_two_rows(q4k, oracle_mod, N, K):
    """The CUDA-core decode kernel (M <= 2) on the same extreme activation rows.
    96 x 2048 splits K across a cluster; with one super-block per row (K = 256)
    or at least as many tiles as CTA slots (40960 rows) the launch does not
    split K, and the one-row fp32 kernel then unpacks the codes of bits 20..31
    of each qs word on the FMA pipe (activations pre-scaled for that layout)."""
    Wh = synth.weight_rows(11 + N, N, K)
    Wd = Wh.to(DEV)
    base = synth.activations(12, 6, K)
    scale = torch.ones(6, K)
    scale[0, :256] = 1e30
    scale[0, 256:512] = 1e-30
    scale[1, :] = 1e-38
    scale[2, 512:768] = 0.0
    scale[3, ::7] = 3e4
    scale[4, :] = 0.0
    X = (base * scale).float()
    for r in range(6):
        _check_matmul(q4k, oracle_mod, Wh, Wd, N, K, X[r:r + 1].contiguous(), TOL_GEMV)
    for r in range(0, 6, 2):
        _check_matmul(q4k, oracle_mod, Wh, Wd, N, K, X[r:r + 2].contiguous(), TOL_GEMV)
        Xb = X[r:r + 2].clamp(-3e38, 3e38).to(torch.bfloat16)
        _check_matmul(q4k, oracle_mod, Wh, Wd, N, K, Xb[:1].contiguous(), TOL_GEMV)


def test_fp32_large_m_runs_in_16_row_slices(q4k, oracle_mod):
    N, K = 200, 1024
    Wh = synth.weight_rows(9, N, K)
    Wd = Wh.to(DEV)
    for M in (17, 33):
        X = synth.activations(10 + M, M, K)
        _check_matmul(q4k, oracle_mod, Wh, Wd, N, K, X, TOL_GEMV)
        Y = q4k.matmul(Wd, N, K, X.to(DEV))
        Y16 = torch.cat([q4k.matmul(Wd, N, K, X[i:i + 16].contiguous().to(DEV))
                         for i in range(0, M, 16)])
        assert torch.equal(Y, Y16)


# --------------------------------------------------------------------- GEMM ---

@pytest.mark.parametrize("M", [17, 31, 32, 33, 64, 65, 100, 128, 129, 255, 256, 257, 512])
def test_gemm_ragged(q4k, oracle_mod, M):
    for (N, K) in ((128, 256), (200, 1024), (384, 512)):
        Wh = synth.weight_rows(4000 + N + K, N, K)
        X = synth.activations(5000 + M + K, M, K, torch.bfloat16)
        _check_matmul(q4k, oracle_mod, Wh, Wh.to(DEV), N, K, X, TOL_GEMM)


@pytest.mark.parametrize("M", [40, 64, 100, 128, 200])
def test_gemm_tile_widths(q4k, oracle_mod, M):
    """Every tile width's ring configuration: 64-token tiles (X ring of two 4-step
    copies), 128-token tiles (X ring as deep as the A ring), 256-token tiles (one
    X step per copy, 4 X stages), over several weight tiles and a K of 8 super-blocks."""
    N, K = 300, 2048
    Wh = synth.weight_rows(6500 + M, N, K)
    X = synth.activations(6600 + M, M, K, torch.bfloat16)
    _check_matmul(q4k, oracle_mod, Wh, Wh.to(DEV), N, K, X, TOL_GEMM)


@pytest.mark.parametrize("M", [32, 512])
def test_gemm_partial_wave_as_two_launches(q4k, oracle_mod, M):
    """A matrix whose unsplit CTAs end in a partial wave: the plan runs the full
    waves' tiles unsplit and the rest of the tiles as a second, K-split launch.
    Sampled output rows cover both launches' tiles (and the boundary)."""
    N, K = 200 * 128, 1024
    Wd = synth.weight_rows(6700 + M, N, K, device=DEV)
    rows = sorted(set(_sample_rows(N, n=192, seed=M)) | {151 * 128 + 127, 152 * 128, N - 1})
    W_rows = synth.weight_sample_rows(6700 + M, N, K, rows)
    X = synth.activations(6800 + M, M, K, torch.bfloat16)
    _check_matmul(q4k, oracle_mod, None, Wd, N, K, X, TOL_GEMM, rows=rows, W_rows=W_rows)


def test_gemm_long_k(q4k, oracle_mod):
    N, K, M = 256, 12288, 300
    Wh = synth.weight_rows(6000, N, K)
    X = synth.activations(6001, M, K, torch.bfloat16)
    _check_matmul(q4k, oracle_mod, Wh, Wh.to(DEV), N, K, X, TOL_GEMM)


def test_gemm_rows_beyond_one_launch(q4k, oracle_mod):
    """More activation rows than one launch covers (65535 grid rows of the
    narrowest 32-token tile): the call runs in row chunks, the last 5 rows long.
    X repeats a block of P rows, P prime, so a chunk that read or wrote at the
    wrong row offset would not line up with the expected rows."""
    N, K, P = 130, 256, 4099
    b = 65535 * 32  # first row of the second chunk
    M = b + 5
    Wh = synth.weight_rows(8100, N, K)
    Xp = synth.activations(8101, P, K, torch.bfloat16)
    X = Xp.to(DEV).repeat((M + P - 1) // P, 1)[:M].contiguous()
    Y = torch.full((M, N), float("nan"), device=DEV)
    q4k.matmul(Wh.to(DEV), N, K, X, Y)
    torch.cuda.synchronize()
    del X
    assert bool(torch.isfinite(Y).all()), "unwritten or non-finite outputs"
    Yref, A = oracle_mod.matmul(Wh.numpy(), N, K, _x_for_oracle(oracle_mod, Xp))
    rng = np.random.default_rng(8102)
    rows = sorted(set(range(40)) | set(range(b - 40, M)) | set(rng.integers(0, M, 200).tolist()))
    got = Y[torch.as_tensor(rows, device=DEV)].cpu().double().numpy()
    src = np.asarray(rows) % P
    worst = float(np.max(np.abs(got - Yref[src]) / (TOL_GEMM * A[src] + 1e-30)))
    assert worst <= 1.0, f"max |err| / ({TOL_GEMM} * sum|wx|) = {worst:.3f}"


def test_dispatch_boundaries(q4k, oracle_mod):
    """Rows 1..2: CUDA-core GEMV; 3..16: the tensor-core decode kernel, both
    held to the GEMV bar; 17 up: the GEMM."""
    N, K = 160, 512
    Wh = synth.weight_rows(7000, N, K)
    Wd = Wh.to(DEV)
    for M, tol in ((2, TOL_GEMV), (3, TOL_GEMV), (16, TOL_GEMV), (17, TOL_GEMM), (32, TOL_GEMM),
                   (33, TOL_GEMM)):
        X = synth.activations(7001 + M, M, K, torch.bfloat16)
        _check_matmul(q4k, oracle_mod, Wh, Wd, N, K, X, tol)


# ------------------------------------------------------------- full sizes ---

def _sample_rows(N, n=256, seed=0):
    rng = np.random.default_rng(seed + N)
    pick = set(rng.choice(N, size=min(N, n), replace=False).tolist())
    pick |= {0, 1, N - 2, N - 1}
    return sorted(pick)


@pytest.mark.parametrize("wl", [1, 2, 3, 4])
def test_full_size_sampled(q4k, oracle_mod, parity_record, wl):
    """Layer-0 matrices (and the lm_head) at full size, in the launch
    configuration the benchmark times; sampled output columns are compared with
    the oracle, and the device-drawn weights are checked against the host draw."""
    w = synth.WORKLOADS[wl]
    mats = [(m, n, k) for (layer, m, n, k) in w.matrices() if layer == 0 or m == "lm_head"]
    cases = [(M, "f32") for M in w.decode_m if "f32" in w.x_dtypes]
    cases += [(M, "bf16") for M in w.decode_m if "bf16" in w.x_dtypes]
    cases += [(M, "bf16") for M in w.prefill_m]
    for name, N, K in mats:
        seed = synth.weight_seed(wl, 0, name)
        Wd = synth.weight_rows(seed, N, K, device=DEV)
        rows = _sample_rows(N)
        W_rows = synth.weight_sample_rows(seed, N, K, rows)
        assert torch.equal(Wd[torch.as_tensor(rows, device=DEV)].cpu(), W_rows)
        for M, xdt in cases:
            dt = torch.bfloat16 if xdt == "bf16" else torch.float32
            X = synth.activations(synth.x_seed(wl, K, M), M, K, dt)
            tol = TOL_GEMM if (dt == torch.bfloat16 and M > 16) else TOL_GEMV
            worst = _check_matmul(q4k, oracle_mod, None, Wd, N, K, X, tol, rows=rows, W_rows=W_rows)
            key = (wl, M, xdt)
            parity_record[key] = max(parity_record.get(key, 0.0), worst)
        del Wd
        torch.cuda.empty_cache()


@pytest.mark.parametrize("wl,M,xdt", [(1, 1, "f32"), (3, 512, "bf16")])
def test_benchmark_launches_layer0(q4k, oracle_mod, parity_record, wl, M, xdt):
    """Layer 0 of the two benchmark sweeps, launched as bench.py times them:
    q/k/v and gate/up as grouped calls built by the benchmark's own helper,
    all calls of the layer in one CUDA graph on a side stream with programmatic
    dependent launch (mode 2). Sampled output rows of every matrix are compared
    with the oracle. Each group writes its own output buffer here, so no
    group's outputs are overwritten by the next."""
    import bench
    bf16 = xdt == "bf16"
    dt = torch.bfloat16 if bf16 else torch.float32
    tol = TOL_GEMM if (bf16 and M > 16) else TOL_GEMV
    _, mats, names = bench._weights(wl, DEV, 1, with_names=True)
    Ks = sorted({K for (_, _, K) in mats})
    xh = {K: synth.activations(synth.x_seed(wl, K, M), M, K, dt) for K in Ks}
    xd = {K: xh[K].to(DEV) for K in Ks}
    stream = torch.cuda.Stream()
    groups = bench._group_spans(names)
    ys, calls = [], []
    for grp in groups:
        sub = [mats[j] for j in grp]
        yg = torch.empty(M * sum(N for (_, N, _) in sub), device=DEV)
        cg = bench._grouped_calls(q4k, sub, [names[j] for j in grp], xd, yg, stream.cuda_stream,
                                  M=M, bf16=bf16)
        assert len(cg) == 1
        ys.append(yg)
        calls += cg
    old = q4k.q4k_set_pdl(2)
    try:
        g = bench._capture(torch, calls, stream)
        with torch.cuda.stream(stream):
            for yg in ys:
                yg.fill_(float("nan"))
            g.replay()
        torch.cuda.synchronize()
    finally:
        q4k.q4k_set_pdl(old)
    for grp, yg in zip(groups, ys):
        off = 0
        for j in grp:
            _, N, K = mats[j]
            rows = _sample_rows(N, n=64)
            W_rows = synth.weight_sample_rows(synth.weight_seed(wl, 0, names[j][1]), N, K, rows)
            Yref, A = oracle_mod.matmul(W_rows.numpy(), len(rows), K, _x_for_oracle(oracle_mod, xh[K]))
            got = yg[off:off + M * N].view(M, N)[:, torch.as_tensor(rows, device=DEV)]
            got = got.cpu().double().numpy()
            assert np.all(np.isfinite(got)), f"{names[j][1]}: unwritten outputs"
            worst = float(np.max(np.abs(got - Yref) / (tol * A + 1e-30)))
            assert worst <= 1.0, f"{names[j][1]}: max |err| / ({tol} * sum|wx|) = {worst:.3f}"
            key = (wl, M, xdt)
            parity_record[key] = max(parity_record.get(key, 0.0), worst)
            off += M * N
    del g, calls, ys, mats
    torch.cuda.empty_cache()


# ------------------------------------------------------------ plumbing ---

def test_outputs_stay_inside_y(q4k):
    N, K = 100, 512
    Wd = synth.weight_rows(8, N, K).to(DEV)
    for M, dt in ((3, torch.float32), (40, torch.bfloat16)):
        X = synth.activations(9, M, K, dt).to(DEV)
        guard = 64
        buf = torch.full((guard + M * N + guard,), float("nan"), device=DEV)
        Y = buf[guard:guard + M * N].view(M, N)
        q4k.matmul(Wd, N, K, X, Y)
        torch.cuda.synchronize()
        assert torch.isnan(buf[:guard]).all() and torch.isnan(buf[-guard:]).all()
        assert torch.isfinite(Y).all()


def test_side_stream_and_graph_capture(q4k):
    N, K = 512, 2048
    Wd = synth.weight_rows(12, N, K).to(DEV)
    X1 = synth.activations(13, 1, K).to(DEV)
    Xp = synth.activations(14, 64, K, torch.bfloat16).to(DEV)
    ref1 = q4k.matmul(Wd, N, K, X1)
    refp = q4k.matmul(Wd, N, K, Xp)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    Y1 = torch.empty(1, N, device=DEV)
    Yp = torch.empty(64, N, device=DEV)
    with torch.cuda.stream(s):
        q4k.matmul(Wd, N, K, X1, Y1)
        q4k.matmul(Wd, N, K, Xp, Yp)
    s.synchronize()
    assert torch.equal(Y1, ref1) and torch.equal(Yp, refp)
    g = torch.cuda.CUDAGraph()
    Y1.zero_()
    Yp.zero_()
    with torch.cuda.graph(g):
        q4k.matmul(Wd, N, K, X1, Y1)
        q4k.matmul(Wd, N, K, Xp, Yp)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(Y1, ref1) and torch.equal(Yp, refp)


def test_repeat_calls_are_deterministic(q4k):
    N, K = 300, 4096
    Wd = synth.weight_rows(15, N, K).to(DEV)
    for M, dt in ((1, torch.float32), (8, torch.bfloat16), (200, torch.bfloat16)):
        X = synth.activations(16, M, K, dt).to(DEV)
        a = q4k.matmul(Wd, N, K, X)
        b = q4k.matmul(Wd, N, K, X)
        torch.cuda.synchronize()
        assert torch.equal(a, b)


@pytest.mark.parametrize("mode", [1, 2])
def test_pdl_dependent_chain(q4k, mode):
    """With programmatic dependent launch, a call whose activations are the
    previous call's output must still see that output (eager and in a graph)."""
    K = 2048
    Ws = [synth.weight_rows(20 + i, K, K).to(DEV) for i in range(4)]
    Wp = synth.weight_rows(30, 512, K).to(DEV)
    x0 = synth.activations(31, 1, K).to(DEV)

    def chain():
        x = x0
        for W in Ws:  # M=1 GEMV chain: each output is directly the next input
            x = q4k.matmul(W, K, K, x)
        xb = x.expand(40, K).to(torch.bfloat16).contiguous()
        return x, q4k.matmul(Wp, 512, K, xb)  # tcgen05 GEMM after the GEMV chain

    old = q4k.q4k_set_pdl(0)
    try:
        ref_x, ref_y = chain()
        torch.cuda.synchronize()
        q4k.q4k_set_pdl(mode)
        for _ in range(3):
            x, y = chain()
            torch.cuda.synchronize()
            assert torch.equal(x, ref_x) and torch.equal(y, ref_y)
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            chain()  # warm the allocator on this stream
            s.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                gx, gy = chain()
            g.replay()
            s.synchronize()
        assert torch.equal(gx, ref_x) and torch.equal(gy, ref_y)
    finally:
        q4k.q4k_set_pdl(old)


@pytest.mark.parametrize("xdt", ["f32", "bf16"])
def test_grouped_matmul(q4k, oracle_mod, xdt):
    """q4k_matmul_multi: several matrices sharing K and X in one call (ragged N,
    including sizes that split K across a cluster and ones that do not)."""
    K = 1536
    Ns = [384, 128, 96, 3000, 1]
    Whs = [synth.weight_rows(8000 + i, n, K) for i, n in enumerate(Ns)]
    Wds = [w.to(DEV) for w in Whs]
    dt = torch.bfloat16 if xdt == "bf16" else torch.float32
    Ms = (1, 3, 16, 40, 300) if xdt == "bf16" else (1, 3, 16, 20)
    for M in Ms:
        X = synth.activations(8100 + M, M, K, dt)
        Ys = [torch.full((M, n), float("nan"), device=DEV) for n in Ns]
        q4k.q4k_matmul_multi(Wds, Ns, K, X.to(DEV), M, Ys)
        torch.cuda.synchronize()
        tol = TOL_GEMM if (dt == torch.bfloat16 and M > 16) else TOL_GEMV
        Xo = _x_for_oracle(oracle_mod, X)
        for Wh, n, Y in zip(Whs, Ns, Ys):
            Yref, A = oracle_mod.matmul(Wh.numpy(), n, K, Xo)
            got = Y.cpu().double().numpy()
            assert np.all(np.isfinite(got))
            assert float(np.max(np.abs(got - Yref) / (tol * A + 1e-30))) <= 1.0


def test_grouped_gemm_eight_matrices(q4k, oracle_mod):
    """The largest group through the tensor-core GEMM (one launch, global tile
    index -> matrix), twice in a row: results within the GEMM bar and identical."""
    K = 768
    Ns = [128, 1, 129, 640, 255, 384, 16, 1000]
    Whs = [synth.weight_rows(8400 + i, n, K) for i, n in enumerate(Ns)]
    Wds = [w.to(DEV) for w in Whs]
    M = 200
    X = synth.activations(8500, M, K, torch.bfloat16)
    Xd = X.to(DEV)
    runs = []
    for _ in range(2):
        Ys = [torch.full((M, n), float("nan"), device=DEV) for n in Ns]
        q4k.q4k_matmul_multi(Wds, Ns, K, Xd, M, Ys)
        torch.cuda.synchronize()
        runs.append([y.cpu() for y in Ys])
    Xo = _x_for_oracle(oracle_mod, X)
    for Wh, n, a, b in zip(Whs, Ns, runs[0], runs[1]):
        assert torch.equal(a, b)
        Yref, A = oracle_mod.matmul(Wh.numpy(), n, K, Xo)
        got = a.double().numpy()
        assert np.all(np.isfinite(got))
        assert float(np.max(np.abs(got - Yref) / (TOL_GEMM * A + 1e-30))) <= 1.0


def test_grouped_matmul_in_graph_with_pdl(q4k):
    K = 2048
    Ns = [2048, 512, 512]
    Wds = [synth.weight_rows(8200 + i, n, K).to(DEV) for i, n in enumerate(Ns)]
    X = synth.activations(8300, 1, K).to(DEV)
    ref = [q4k.matmul(W, n, K, X) for W, n in zip(Wds, Ns)]
    torch.cuda.synchronize()
    old = q4k.q4k_set_pdl(2)
    try:
        s = torch.cuda.Stream()
        Ys = [torch.zeros(1, n, device=DEV) for n in Ns]
        with torch.cuda.stream(s):
            q4k.q4k_matmul_multi(Wds, Ns, K, X, 1, Ys)
            s.synchronize()
            first = [y.clone() for y in Ys]
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                q4k.q4k_matmul_multi(Wds, Ns, K, X, 1, Ys)
            for y in Ys:
                y.zero_()
            g.replay()
            s.synchronize()
        for a, b, r in zip(first, Ys, ref):
            assert torch.equal(a, b)
            assert torch.allclose(a, r, rtol=0, atol=1e-3)
    finally:
        q4k.q4k_set_pdl(old)


# ---------------------------------------------------------- fused argmax ---

def _argmax_valid(oracle_mod, Wh, N, K, X, got):
    """got[m] is a correct argmax of row m under the oracle: within the GEMV
    bar of the exact maximum (rows whose leaders differ by less than that may
    pick either)."""
    Yref, A = oracle_mod.matmul(Wh.numpy(), N, K, _x_for_oracle(oracle_mod, X))
    for m, n in enumerate(got):
        best = int(np.argmax(Yref[m]))
        slack = TOL_GEMV * (A[m, n] + A[m, best])
        assert Yref[m, n] >= Yref[m, best] - slack, (m, n, best)


@pytest.mark.parametrize("N,K", [(300, 512), (1000, 2048), (4097, 768)])
@pytest.mark.parametrize("M,xdt", [(1, "f32"), (4, "bf16"), (16, "f32")])
def test_argmax_matches_gemv_and_oracle(q4k, oracle_mod, N, K, M, xdt):
    """The fused argmax equals the argmax (first maximum) of the library's own
    GEMV outputs -- the same kernel computes the same values -- and is a correct
    argmax of the exact product."""
    Wh = synth.weight_rows(9000 + N + K, N, K)
    Wd = Wh.to(DEV)
    dt = torch.bfloat16 if xdt == "bf16" else torch.float32
    X = synth.activations(9100 + M, M, K, dt)
    Xd = X.to(DEV)
    out = torch.full((M,), -7, dtype=torch.int64, device=DEV)
    q4k.q4k_matmul_argmax(Wd, N, K, Xd, M, out)
    Y = q4k.matmul(Wd, N, K, Xd)
    torch.cuda.synchronize()
    got = out.cpu().tolist()
    assert got == torch.argmax(Y, dim=1).cpu().tolist()
    _argmax_valid(oracle_mod, Wh, N, K, X, got)


def test_argmax_ties_go_to_the_lowest_index(q4k):
    """Rows with identical bytes give identical outputs; when they hold the
    maximum, the lowest of them is returned."""
    N, K, M = 2000, 1024, 3
    W = synth.weight_rows(9200, N, K)
    X = synth.activations(9201, M, K).to(DEV)
    Wd = W.to(DEV)
    first = q4k.argmax(Wd, N, K, X).cpu().tolist()
    for m in range(M):
        top = first[m]
        W2 = W.clone()
        for dst in (top // 3, top // 3 + 1, N - 1):  # copies below and above it
            W2[dst] = W[top]
        got = q4k.argmax(W2.to(DEV), N, K, X).cpu().tolist()
        assert got[m] == min(top // 3, top), (m, got[m], top)


def test_argmax_lm_head_full_size(q4k, oracle_mod):
    """The tied lm_head of the Llama-3.2-3B shape (128256 x 3072), M = 1, at full
    size: equal to the GEMV's argmax and valid under the oracle."""
    N, K = 128256, 3072
    seed = synth.weight_seed(2, 28, "lm_head")
    Wd = synth.weight_rows(seed, N, K, device=DEV)
    X = synth.activations(synth.x_seed(2, K, 1), 1, K)
    Xd = X.to(DEV)
    got = q4k.argmax(Wd, N, K, Xd).cpu().tolist()
    Y = q4k.matmul(Wd, N, K, Xd)
    assert got == torch.argmax(Y, dim=1).cpu().tolist()
    Wh = Wd.cpu()
    del Wd
    torch.cuda.empty_cache()
    _argmax_valid(oracle_mod, Wh, N, K, X, got)


def test_argmax_in_graph_with_pdl(q4k):
    N, K = 5000, 2048
    Wd = synth.weight_rows(9300, N, K).to(DEV)
    X = synth.activations(9301, 2, K).to(DEV)
    ref = q4k.argmax(Wd, N, K, X).clone()
    old = q4k.q4k_set_pdl(2)
    try:
        s = torch.cuda.Stream()
        out = torch.full((2,), -1, dtype=torch.int64, device=DEV)
        with torch.cuda.stream(s):
            q4k.q4k_matmul_argmax(Wd, N, K, X, 2, out)
            s.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                q4k.q4k_matmul_argmax(Wd, N, K, X, 2, out)
            out.fill_(-1)
            g.replay()
            s.synchronize()
        assert torch.equal(out, ref)
    finally:
        q4k.q4k_set_pdl(old)
