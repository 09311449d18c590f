"""Host-side logic of bench.py that decides what the timed sweeps launch: which
matrices form a grouped call, and where each matrix's outputs go."""
import bench
from gguf_q4_dequant_gb300 import synth


def _names(wl):
    return [(layer, m) for (layer, m, _, _) in synth.WORKLOADS[wl].matrices()]


def test_groups_follow_shared_inputs():
    names = _names(1)
    groups = bench._group_spans(names)
    assert [j for g in groups for j in g] == list(range(len(names)))  # a partition, in order
    assert len(groups) == 4 * 16  # q/k/v, o, gate/up, down per layer
    for g in groups:
        ms = [names[j][1] for j in g]
        assert ms in (["q_proj", "k_proj", "v_proj"], ["o_proj"], ["gate_proj", "up_proj"],
                      ["down_proj"])
        assert len({names[j][0] for j in g}) == 1  # never across layers


def test_lm_head_is_its_own_call():
    names = _names(2)
    groups = bench._group_spans(names)
    assert [names[j][1] for j in groups[-1]] == ["lm_head"]


class _FakeLib:
    def __init__(self):
        self.calls = []

    def q4k_matmul_multi(self, n, Ws, Ns, K, x, M, Ys, stream):
        self.calls.append((M, [Ns[i] for i in range(n)], [Ys[i] for i in range(n)]))
        return 0

    q4k_matmul_multi_bf16 = q4k_matmul_multi


class _FakeQ4K:
    Q4KError = RuntimeError

    def __init__(self):
        self._lib = _FakeLib()

    def lib(self):
        return self._lib


class _T:
    """Stands in for a device tensor: only data_ptr() is used."""
    def __init__(self, ptr):
        self.ptr = ptr

    def data_ptr(self):
        return self.ptr


def _outputs(wl, M):
    w = synth.WORKLOADS[wl]
    mats = [(_T(1 << 30), N, K) for (_, _, N, K) in w.matrices()]
    names = _names(wl)
    x = {K: _T(1 << 20) for (_, _, K) in mats}
    base = 1 << 40
    q4k = _FakeQ4K()
    calls = bench._grouped_calls(q4k, mats, names, x, _T(base), 0, M=M, bf16=M > 16)
    for c in calls:
        c()
    return q4k.lib().calls, base


def test_decode_outputs_are_disjoint_slices():
    """At M = 1 every matrix of the sweep writes its own slice of one buffer."""
    calls, base = _outputs(1, 1)
    spans = sorted((y - base, y - base + 4 * n) for (_, ns, ys) in calls for n, y in zip(ns, ys))
    assert spans[0][0] == 0
    for (a0, a1), (b0, b1) in zip(spans, spans[1:]):
        assert a1 == b0  # contiguous, no overlap
    assert spans[-1][1] == 4 * sum(n for (_, _, n, _) in synth.WORKLOADS[1].matrices())


def test_prefill_group_members_do_not_overlap():
    """At M > 1 the matrices of one grouped call write disjoint M x N blocks that
    fit the buffer _group_y_floats sizes; the groups reuse them."""
    M = 512
    calls, base = _outputs(3, M)
    w = synth.WORKLOADS[3]
    mats = [(None, N, K) for (_, _, N, K) in w.matrices()]
    limit = 4 * bench._group_y_floats(mats, _names(3), M)
    for (m, ns, ys) in calls:
        assert m == M
        spans = sorted((y - base, y - base + 4 * M * n) for n, y in zip(ns, ys))
        for (a0, a1), (b0, b1) in zip(spans, spans[1:]):
            assert a1 <= b0
        assert spans[0][0] >= 0 and spans[-1][1] <= limit


def test_clock_samples_are_summarised(tmp_path, monkeypatch):
    """The clock record in the JSON line: median SM clock of the busy samples,
    the maximum clock, and every throttle reason seen active (a stand-in
    nvidia-smi on PATH prints fixed samples)."""
    import os
    import time
    lines = [
        "0, 345, 2070, 120.0, 0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "0, 1800, 2070, 1100.5, 100, 0x4, Not Active, Not Active, Not Active, Active",
        "0, 2000, 2070, 1000.0, 97, 0x0, Not Active, Not Active, Not Active, Not Active",
        "0, 1900, 2070, 1050.0, 100, 0x4, Not Active, Not Active, Not Active, Active",
    ]
    fake = tmp_path / "nvidia-smi"
    fake.write_text("#!/bin/sh\ncat <<'X'\n" + "\n".join(lines) + "\nX\nexec sleep 30\n")
    fake.chmod(0o755)
    monkeypatch.setenv("PATH", f"{tmp_path}{os.pathsep}{os.environ['PATH']}")
    keep = tmp_path / "clocks.csv"
    s = bench.ClockSampler(0, str(keep))
    s.start()
    for _ in range(100):  # until the stand-in has printed its samples
        if keep.exists() and keep.read_text().count("\n") >= len(lines):
            break
        time.sleep(0.05)
    rec = s.stop()
    assert rec == {"sm_mhz": 1900.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}
    assert keep.exists()  # a path given by the caller is kept
    t = bench.ClockSampler(0)
    t.start()
    t.stop()
    assert not os.path.exists(t.path)  # the default temporary file is removed


def test_prefill_oracle_sample_is_extrapolated_consistently():
    """The prefill CPU baseline: a rate from sampled rows, and the full sweep
    time implied by that rate over all 2*M*N*K of the workload."""
    rec = bench.cpu_oracle_prefill(0.2, 2, rows_per_matrix=2)
    ns = rec["ns_per_weight_token"]
    assert ns > 0 and rec["cores"] == 2
    w = synth.WORKLOADS[bench.PREFILL_WL]
    full = sum(N * K for (_, _, N, K) in w.matrices()) * bench.PREFILL_M
    assert abs(rec["extrapolated_s_per_sweep"] - ns * full * 1e-9) <= 0.051
    assert "extrapolated" in rec["sample"]
