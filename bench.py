"""Benchmark of the packed Q4_K dequant-matmul (libq4k) on one GB300 per rank.

Metric: Q4_K dequant-matmul -- GEMV packed-weight GB/s (M=1); GEMM TFLOP/s (M=512).

A step is one pass of the hot path over one batch:
  * decode (the headline `value`): the Qwen3-14B-shaped sweep, 40 layers x 7
    Q4_K matrices (7.43 GB packed, the largest weight set), M = 1 fp32
    activation row, q/k/v and gate/up as grouped calls (160 GEMV launches),
    replayed from a CUDA graph; value = packed weight bytes per step / step
    time. Beside it: the same sweep with one call per matrix, end to end from
    host buffers (graph replay, and eager call-by-call through the C ABI), a
    warm per-shape table (each distinct launch shape timed on its own), and
    the Llama-3.2-1B / -3B-shaped sweeps as keyed sub-results.
  * prefill (`gemm`): the Qwen3-8B-shaped sweep, 36 layers x 7 matrices (3.9 GB
    packed), M = 512 bf16 token rows, grouped the same way (144 tcgen05 GEMM
    launches); value = 2*M*N*K flops per step / step time. Beside it: one call
    per matrix, and the Qwen3-14B sweep at M = 2048 and the Qwen3-8B sweep at
    M = 32 and 1024 (`gemm_workloads`).
  * `dequant`: the standalone dequantisation of the 128256 x 3072 lm_head.
Every weight set is larger than L2, so every step streams weights from HBM.
Inputs are synthetic (seeded generator), resident in HBM before timing.

`--impl reference` times the CPU oracle (the plain C++ reference the library
is checked against) on a bounded sample of the same decode workload; the
`cpu_baseline` of the GPU line is the same measurement, taken in a separate
process so that both run under the same conditions.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "Q4_K dequant-matmul: GEMV packed-weight GB/s (M=1); GEMM TFLOP/s (M=512)"
DECODE_WL = 4                     # headline: the largest weight set, M = 1
DECODE_EXTRA_WLS = (1, 2)         # keyed sub-results at M = 1
DECODE_EXTRA_M = (4, 16)          # the headline weight set at more activation rows (tensor-core kernel)
PREFILL_WL, PREFILL_M = 3, 512    # the GEMM metric
GEMM_EXTRA = ((4, 2048), (3, 32), (3, 1024))
LM_HEAD = (2, 128256, 3072)       # (workload, N, K) of the lm_head used by the argmax and dequant legs


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d["hbm_gbs"], d["bf16_tflops"], d.get("bf16_tflops_sustained"), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


KERNEL_SOURCES = {
    "q4k_gemv_kernel<1,f32>": ["gguf_q4_dequant_gb300/csrc/q4k_gemv.cu",
                               "gguf_q4_dequant_gb300/csrc/q4k_device.cuh",
                               "gguf_q4_dequant_gb300/csrc/q4k_internal.h"],
    "q4k_gemm_kernel": ["gguf_q4_dequant_gb300/csrc/q4k_gemm.cu",
                        "gguf_q4_dequant_gb300/csrc/q4k_device.cuh",
                        "gguf_q4_dequant_gb300/csrc/q4k_internal.h"],
    "q4k_dequant_kernel": ["gguf_q4_dequant_gb300/csrc/q4k_dequant.cu",
                           "gguf_q4_dequant_gb300/csrc/q4k_device.cuh"],
}


def sources_sha256(kernel):
    import hashlib
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def measured_traffic(kernel, workload=None):
    """DRAM bytes per launch from the committed ncu summary, or None when the
    kernel's sources changed after the counters were taken (or none exist for
    this workload)."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        rec = json.load(f).get(kernel)
    if not rec or rec.get("sources_sha256") != sources_sha256(kernel):
        return None
    if workload is not None and rec.get("workload") != workload:
        return None
    return rec["dram_bytes_per_launch"]


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def _host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# ------------------------------------------------------------- CPU oracle ---

_HOST_DECODE = None


def _host_decode_set():
    """Host copies of the first layer of the decode sweep (every layer has the
    same shapes) and its activation rows, drawn once."""
    global _HOST_DECODE
    if _HOST_DECODE is None:
        from gguf_q4_dequant_gb300 import synth
        w = synth.WORKLOADS[DECODE_WL]
        mats = [(synth.weight_rows(synth.weight_seed(DECODE_WL, layer, name), N, K).numpy(), N, K)
                for (layer, name, N, K) in w.matrices() if layer == 0]
        xs = {K: synth.activations(synth.x_seed(DECODE_WL, K, 1), 1, K).numpy()
              for K in {K for (_, _, K) in mats}}
        _HOST_DECODE = (w, mats, xs)
    return _HOST_DECODE


def cpu_oracle_decode(budget_s: float, threads: int):
    """Times the oracle (as it stands) over the first layer of the decode sweep,
    matrix by matrix in sweep order and round again, until `budget_s` seconds
    of oracle time have elapsed."""
    import oracle
    oracle.build()
    w, mats, xs = _host_decode_set()
    total_bytes, elapsed, done = 0, 0.0, 0
    while elapsed < budget_s:
        Wh, N, K = mats[done % len(mats)]
        t0 = time.perf_counter()
        oracle.matmul(Wh, N, K, xs[K], threads=threads)
        elapsed += time.perf_counter() - t0
        total_bytes += Wh.size
        done += 1
    return {"value": total_bytes / elapsed / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"oracle matmul over the {len(mats)} matrices of layer 0 of the {w.name} "
                      f"(every layer has these shapes), in sweep order, {done} calls "
                      f"({total_bytes / 1e6:.0f} MB packed, M=1 fp32), {elapsed:.1f} s of CPU time"}


def cpu_oracle_prefill(budget_s: float, threads: int, rows_per_matrix: int = 8):
    """Times the oracle on the prefill workload (M = 512 bf16 token rows) over a
    seeded subset of each matrix's output rows, in sweep order, until `budget_s`
    seconds of oracle time; reports ns per (weight x token) and the full sweep
    time that rate implies (labelled as extrapolated)."""
    import numpy as np
    import torch
    import oracle
    from gguf_q4_dequant_gb300 import synth
    oracle.build()
    w = synth.WORKLOADS[PREFILL_WL]
    mats = w.matrices()
    xs = {}
    rng = np.random.default_rng(PREFILL_WL)
    elapsed, done, wt = 0.0, 0, 0
    while elapsed < budget_s and done < len(mats):
        layer, name, N, K = mats[done]
        if K not in xs:
            xb = synth.activations(synth.x_seed(PREFILL_WL, K, PREFILL_M), PREFILL_M, K, torch.bfloat16)
            xs[K] = oracle.bf16_to_f32(xb.view(torch.int16).numpy().view(np.uint16))
        rows = sorted(rng.choice(N, size=rows_per_matrix, replace=False).tolist())
        Wr = synth.weight_sample_rows(synth.weight_seed(PREFILL_WL, layer, name), N, K, rows).numpy()
        t0 = time.perf_counter()
        oracle.matmul(Wr, len(rows), K, xs[K], threads=threads)
        elapsed += time.perf_counter() - t0
        wt += len(rows) * K * PREFILL_M
        done += 1
    ns = float(f"{elapsed / wt * 1e9:.6g}")
    full = sum(N * K for (_, _, N, K) in mats) * PREFILL_M
    return {"ns_per_weight_token": ns, "cores": threads,
            "extrapolated_s_per_sweep": round(ns * full * 1e-9, 1),
            "extrapolated_tflops": round(2.0 / ns * 1e-3, 6),
            "sample": f"oracle matmul over {rows_per_matrix} seeded output rows of each of the first "
                      f"{done} matrices of the prefill sweep ({w.name}, M={PREFILL_M} bf16), "
                      f"{elapsed:.1f} s of CPU time; the full-sweep time is extrapolated"}


def check_dequant_sample(path):
    """The oracle's dequantisation of the sampled rows saved by the GPU run,
    compared bit for bit with the library's output for those rows."""
    import numpy as np
    import oracle
    oracle.build()
    d = np.load(path)
    rows, packed, got = d["rows"], d["packed"], d["got"]
    N, K = len(rows), int(d["K"])
    ref = oracle.dequant(packed, N, K)
    same = bool(np.array_equal(ref.view(np.uint32), got.view(np.uint32)))
    return {"rows_checked": int(N), "bit_exact": same,
            "sample": f"{N} seeded rows of the {int(d['N_full'])} x {K} matrix, all {N * K} weights"}


def cpu_baselines(budget_s: float, dequant_sample: str = ""):
    """The oracle as it stands: the decode sample on all host cores (the
    reported value), the same on one thread, and a row sample of the prefill
    workload on all host cores."""
    cores = _host_cores()
    for _ in range(3):  # the same warm-up as the reference arm's default
        cpu_oracle_decode(0.5, cores)
    cb = cpu_oracle_decode(budget_s, cores)
    one = cpu_oracle_decode(max(1.0, budget_s / 4), 1)
    cb["single_thread"] = {"value": one["value"], "unit": one["unit"], "sample": one["sample"]}
    cb["prefill"] = cpu_oracle_prefill(max(1.0, budget_s / 2), cores)
    if dequant_sample:
        cb["dequant_check"] = check_dequant_sample(dequant_sample)
    cb["process"] = "a separate CPU-only process (no CUDA context), as the reference arm"
    return cb


def cpu_baselines_subprocess(budget_s: float, dequant_sample: str = ""):
    """cpu_baselines() in a fresh interpreter without CUDA, so that the timing
    sees the same conditions as `--impl reference`."""
    cmd = [sys.executable, os.path.abspath(__file__), "--cpu-baseline-only",
           "--cpu-budget", str(budget_s)]
    if dequant_sample:
        cmd += ["--dequant-sample", dequant_sample]
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run(cmd, capture_output=True, text=True, env=env, check=True)
    return json.loads(r.stdout.strip().splitlines()[-1])


def max_over_ranks(times, ws, device="cpu"):
    """Every timing as its maximum over the job's ranks (called by all ranks)."""
    import torch
    keys = sorted(times)
    t = torch.tensor([times[k] for k in keys], device=device, dtype=torch.float64)
    if ws > 1:
        import torch.distributed as dist
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return dict(zip(keys, t.tolist()))


def _decode_config_name():
    from gguf_q4_dequant_gb300 import synth
    w = synth.WORKLOADS[DECODE_WL]
    return (f"{w.name}: {len(w.matrices())} Q4_K matrices, {w.packed_bytes() / 1e6:.1f} MB packed, "
            f"M=1 fp32 activations")


def run_reference(args):
    ws, rank, _ = _dist()
    if rank != 0:
        return
    threads = _host_cores()
    samples = []
    for _ in range(args.warmup):
        cpu_oracle_decode(0.5, threads)
    for _ in range(args.steps):
        samples.append(cpu_oracle_decode(args.ref_budget, threads))
    value = statistics.median(s["value"] for s in samples)
    cb = dict(samples[-1])
    cb["value"] = value
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": _decode_config_name() + " (bounded sample: layer 0's matrices)",
                   "parallelism": "host threads"},
        "cpu_baseline": cb,
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


# ------------------------------------------------------------------ clocks ---

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,utilization.gpu,"
             "clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, path: str = ""):
        self.proc = None
        self.temporary = not path
        if self.temporary:
            fd, path = tempfile.mkstemp(prefix=f"q4k_clocks_rank{gpu_index}_", suffix=".csv")
            os.close(fd)
        self.path = path
        self.gpu = gpu_index

    def start(self):
        try:
            os.makedirs(os.path.dirname(os.path.abspath(self.path)), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            if self.temporary and os.path.exists(self.path):
                os.remove(self.path)
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    rows.append((float(parts[1]), float(parts[2]), float(parts[4]), parts[6:10]))
                except ValueError:
                    continue
        if self.temporary:
            os.remove(self.path)
        if not rows:
            return None
        busy = [r for r in rows if r[2] > 0] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in busy for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in busy), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(busy)}


# ------------------------------------------------------------------ GPU arm ---

def _weights(wl, dev, layers, with_names=False):
    from gguf_q4_dequant_gb300 import synth
    w = synth.WORKLOADS[wl]
    sel = [(layer, name, N, K) for (layer, name, N, K) in w.matrices() if not layers or layer < layers]
    mats = [(synth.weight_rows(synth.weight_seed(wl, layer, name), N, K, device=dev), N, K)
            for (layer, name, N, K) in sel]
    if with_names:
        return w, mats, [(layer, name) for (layer, name, _, _) in sel]
    return w, mats


# Matrices of a layer that take the same input: one grouped call each.
SHARED_INPUT = (("q_proj", "k_proj", "v_proj"), ("gate_proj", "up_proj"))


def _group_spans(names):
    """Index lists of consecutive matrices that share their input (SHARED_INPUT)."""
    groups, i = [], 0
    while i < len(names):
        layer, name = names[i]
        span = 1
        for g in SHARED_INPUT:
            if name == g[0] and [n for (_, n) in names[i:i + len(g)]] == list(g):
                span = len(g)
        groups.append(list(range(i, i + span)))
        i += span
    return groups


def _grouped_calls(q4k, mats, names, x_dev, y, stream_ptr, M=1, bf16=False, groups=None):
    """A sweep with q/k/v and gate/up as grouped calls (one launch each). At
    M = 1 every matrix writes its own slice of `y`; at larger M the matrices of
    one group write disjoint slices and the groups reuse them. `groups` picks a
    subset of _group_spans(names) (default: all, in sweep order)."""
    import ctypes
    lib = q4k.lib()
    fn = lib.q4k_matmul_multi_bf16 if bf16 else lib.q4k_matmul_multi
    all_groups = _group_spans(names)
    offs = [0] * len(mats)
    o = 0
    for grp in all_groups:
        if M > 1:
            o = 0
        for j in grp:
            offs[j] = o
            o += M * mats[j][1]
    calls = []
    for grp in (all_groups if groups is None else groups):
        K = mats[grp[0]][2]
        Ws = (ctypes.c_void_p * len(grp))(*[mats[j][0].data_ptr() for j in grp])
        Ns = (ctypes.c_int64 * len(grp))(*[mats[j][1] for j in grp])
        Ys = (ctypes.c_void_p * len(grp))(*[y.data_ptr() + 4 * offs[j] for j in grp])

        def call(Ws=Ws, Ns=Ns, Ys=Ys, K=K, n=len(grp)):
            rc = fn(n, Ws, Ns, K, x_dev[K].data_ptr(), M, Ys, stream_ptr)
            if rc != 0:
                raise q4k.Q4KError(rc, "grouped sweep")
        calls.append(call)
    return calls


def _group_y_floats(mats, names, M):
    """Output floats _grouped_calls needs for M > 1: the largest group."""
    return max(M * sum(mats[j][1] for j in grp) for grp in _group_spans(names))


def _shape_classes(mats, names):
    """Groups of the sweep keyed by their launch shape: (matrix names, row
    counts, K) -> list of groups in sweep order."""
    classes = {}
    for grp in _group_spans(names):
        key = (tuple(names[j][1] for j in grp), tuple(mats[j][1] for j in grp), mats[grp[0]][2])
        classes.setdefault(key, []).append(grp)
    return classes


def _sweep_calls(q4k, mats, x_dev, y, M, bf16, stream_ptr):
    """One closure per matrix, each issuing one public-API call on `stream_ptr`.
    At M = 1 every matrix writes its own slice of `y`; at larger M they share it."""
    lib = q4k.lib()
    fn = lib.q4k_matmul_bf16 if bf16 else lib.q4k_matmul
    calls, off = [], 0
    for (Wd, N, K) in mats:
        args = (Wd.data_ptr(), N, K, x_dev[K].data_ptr(), M, y.data_ptr() + 4 * off, stream_ptr)

        def call(a=args):
            rc = fn(*a)
            if rc != 0:
                raise q4k.Q4KError(rc, "sweep")
        calls.append(call)
        if M == 1:
            off += N
    return calls


def _capture(torch, calls, stream):
    for c in calls:  # first use outside capture
        c()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for c in calls:
            c()
    torch.cuda.synchronize()
    return g


def _time_graph(torch, graph, stream, steps, warmup, barrier):
    """ms per replay, CUDA events on the stream the graph is replayed on."""
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            graph.replay()
        torch.cuda.synchronize()
        barrier()
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for _ in range(steps):
            graph.replay()
        end.record(stream)
        torch.cuda.synchronize()
        barrier()
    return start.elapsed_time(end) / steps


def _gpu_setup(args):
    import torch
    import gguf_q4_dequant_gb300 as q4k
    from gguf_q4_dequant_gb300 import build as q4k_build
    q4k_build.build()
    _, _, local = _dist()
    torch.cuda.set_device(local)
    q4k.q4k_init()
    q4k.q4k_set_pdl(args.pdl)
    return torch, q4k, f"cuda:{local}"


def run_profile_shape(args):
    """Microbenchmark of one matrix shape: a CUDA graph of back-to-back calls over
    enough distinct weight copies to exceed L2; prints per-launch time."""
    import math
    torch, q4k, dev = _gpu_setup(args)
    from gguf_q4_dequant_gb300 import synth
    N, K, M = (int(v) for v in args.profile_shape.split(","))
    wb = N * K // 256 * 144
    R = min(64, max(2, math.ceil(args.profile_bytes / wb)))
    Ws = [synth.weight_rows(0x5eed + i, N, K, device=dev) for i in range(R)]
    bf16 = M > 16 or args.x_bf16
    X = synth.activations(0x5eed, M, K, torch.bfloat16 if bf16 else torch.float32).to(dev)
    Y = torch.empty(M, N, device=dev)
    lib = q4k.lib()
    fn = lib.q4k_matmul_bf16 if bf16 else lib.q4k_matmul
    stream = torch.cuda.Stream()
    calls = [(lambda W=W: fn(W.data_ptr(), N, K, X.data_ptr(), M, Y.data_ptr(), stream.cuda_stream))
             for W in Ws]
    g = _capture(torch, calls, stream)
    ms = _time_graph(torch, g, stream, args.steps, args.warmup, lambda: None)
    us = ms * 1e3 / R
    print(json.dumps({"shape": {"N": N, "K": K, "M": M}, "x_dtype": "bf16" if bf16 else "f32",
                      "pdl": args.pdl, "copies": R, "us_per_launch": round(us, 3),
                      "packed_GBps": round(wb / us / 1e3, 1),
                      "TFLOPs": round(2 * M * N * K / us / 1e6, 2),
                      "device_error": q4k.q4k_device_error()}))


def _sweep_record(torch, q4k, wl, mats, names, M, xdt, stream, steps, warmup, hbm, bf16_peak,
                  barrier=lambda: None):
    """One grouped sweep of workload `wl` at M rows (fp32 or bf16), in a CUDA
    graph: ms per sweep, packed GB/s and TFLOP/s with their roofline fractions."""
    from gguf_q4_dequant_gb300 import synth
    dev = mats[0][0].device
    bf16 = xdt == "bf16"
    dt = torch.bfloat16 if bf16 else torch.float32
    xs = {K: synth.activations(synth.x_seed(wl, K, M), M, K, dt).to(dev)
          for K in sorted({K for (_, _, K) in mats})}
    ny = sum(N for (_, N, _) in mats) if M == 1 else _group_y_floats(mats, names, M)
    y = torch.empty(ny, device=dev)
    calls = _grouped_calls(q4k, mats, names, xs, y, stream.cuda_stream, M=M, bf16=bf16)
    g = _capture(torch, calls, stream)
    ms = _time_graph(torch, g, stream, steps, warmup, barrier)
    wbytes = sum(Wd.numel() for (Wd, _, _) in mats)
    flops = sum(2 * M * N * K for (_, N, K) in mats)
    gbps = wbytes / (ms * 1e-3) / 1e9
    tf = flops / (ms * 1e-3) / 1e12
    rec = {"workload": synth.WORKLOADS[wl].name, "M": M, "x_dtype": xdt,
           "kernel": ("q4k_gemv_kernel" if M <= 2 else "q4k_tcgemv_kernel") if M <= 16 else "q4k_gemm_kernel",
           "launches_per_step": len(calls), "steps": steps, "ms_per_step": round(ms, 5),
           "packed_GBps": round(gbps, 1), "frac_of_hbm": round(gbps / hbm, 4),
           "TFLOPs": round(tf, 2), "frac_of_bf16": round(tf / bf16_peak, 4)}
    del g
    return rec, len(calls) * steps


def run_all_configs(args):
    """Every workload of synth.WORKLOADS at every M and activation dtype it
    names, each as full sweeps with q/k/v and gate/up grouped, in a CUDA graph;
    one JSON line per case, plus the standalone dequant kernel."""
    torch, q4k, dev = _gpu_setup(args)
    from gguf_q4_dequant_gb300 import synth
    stream = torch.cuda.Stream()
    hbm, bf16_peak, _, _ = _peaks()
    steps = max(3, min(args.steps, 20))
    for wl in (1, 2, 3, 4):
        w, mats, names = _weights(wl, dev, 0, with_names=True)
        cases = [(M, x) for x in w.x_dtypes for M in w.decode_m]
        cases += [(M, "bf16") for M in w.prefill_m]
        for M, xdt in cases:
            rec, _ = _sweep_record(torch, q4k, wl, mats, names, M, xdt, stream, steps, args.warmup,
                                   hbm, bf16_peak)
            rec["device_error"] = q4k.q4k_device_error()
            print(json.dumps(rec), flush=True)
        del mats
        torch.cuda.empty_cache()
    print(json.dumps(_dequant_leg(torch, q4k, dev, stream, steps, args.warmup, hbm)[0]), flush=True)


def _dequant_leg(torch, q4k, dev, stream, steps, warmup, hbm, barrier=lambda: None, sample_path=""):
    """K1 on the lm_head: read + write GB/s. Optionally saves a seeded sample of
    output rows (with their packed bytes) for the bit-exactness check that the
    CPU-baseline process runs against the oracle."""
    from gguf_q4_dequant_gb300 import synth
    wl, N, K = LM_HEAD
    Wd = synth.weight_rows(synth.weight_seed(wl, 28, "lm_head"), N, K, device=dev)
    out = torch.empty(N, K, device=dev)
    g = _capture(torch, [lambda: q4k.q4k_dequant(Wd, N, K, out, stream=stream.cuda_stream)], stream)
    ms = _time_graph(torch, g, stream, steps, warmup, barrier)
    moved = Wd.numel() + out.numel() * 4
    gbps = moved / (ms * 1e-3) / 1e9
    rec = {"kernel": "q4k_dequant_kernel", "workload": f"lm_head {N} x {K} -> fp32",
           "us": round(ms * 1e3, 2), "read_plus_write_GBps": round(gbps, 1),
           "frac_of_hbm": round(gbps / hbm, 4), "algorithmic_bytes": moved,
           "roofline": {"bound": "hbm", "achieved": round(gbps, 1), "peak": hbm, "unit": "GB/s",
                        "frac": round(gbps / hbm, 4),
                        "traffic": measured_traffic("q4k_dequant_kernel")}}
    if sample_path:
        import numpy as np
        gen = np.random.default_rng(12345)
        rows = np.sort(gen.choice(N, size=64, replace=False))
        idx = torch.as_tensor(rows, device=dev)
        torch.cuda.synchronize()
        np.savez(sample_path, rows=rows, K=K, N_full=N,
                 packed=Wd[idx].cpu().numpy(), got=out[idx].cpu().numpy())
    del g, out, Wd
    torch.cuda.empty_cache()
    return rec, steps


def run_sweep_only(args):
    """Profiling aid: only the headline decode sweep (weights, the grouped calls,
    one CUDA graph, timing); `--only dequant`: only the standalone dequant leg."""
    torch, q4k, dev = _gpu_setup(args)
    stream = torch.cuda.Stream()
    hbm, _, _, _ = _peaks()
    if args.only == "dequant":
        rec, _ = _dequant_leg(torch, q4k, dev, stream, args.steps, args.warmup, hbm)
        rec["device_error"] = q4k.q4k_device_error()
        print(json.dumps(rec))
        return
    from gguf_q4_dequant_gb300 import synth
    w, mats, names = _weights(DECODE_WL, dev, args.layers, with_names=True)
    xs = {K: synth.activations(synth.x_seed(DECODE_WL, K, 1), 1, K).to(dev)
          for K in sorted({K for (_, _, K) in mats})}
    y = torch.empty(sum(N for (_, N, _) in mats), device=dev)
    calls = _grouped_calls(q4k, mats, names, xs, y, stream.cuda_stream)
    g = _capture(torch, calls, stream)
    ms = _time_graph(torch, g, stream, args.steps, args.warmup, lambda: None)
    wb = sum(Wd.numel() for (Wd, _, _) in mats)
    print(json.dumps({"workload": w.name, "layers": args.layers or w.layers, "launches_per_step": len(calls),
                      "ms_per_step": round(ms, 5), "packed_GBps": round(wb / ms / 1e6, 1),
                      "frac_of_hbm": round(wb / ms / 1e6 / hbm, 4), "device_error": q4k.q4k_device_error()}))


def run_gpu(args):
    import torch
    ws, rank, local = _dist()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device(f"cuda:{local}"))

        def barrier():
            dist.barrier()
    else:
        def barrier():
            pass
    torch, q4k, dev = _gpu_setup(args)
    from gguf_q4_dequant_gb300 import synth
    hbm, bf16_peak, bf16_sust, peak_kind = _peaks()
    stream = torch.cuda.Stream()
    sp = stream.cuda_stream
    out = {"metric": METRIC, "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
           "data": "synthetic (seeded Q4_K weights, N(0,1) activations)"}
    sampler = ClockSampler(local, args.clocks_csv.replace("{rank}", str(rank)))
    sampler.start()
    launches = 0
    times = {}
    dq_sample = ""
    resident = {}  # workload -> (mats, names) kept for a later leg

    if args.only in ("all", "decode"):
        # ------------------------------------------- headline decode sweep ---
        w4, mats4, names4 = _weights(DECODE_WL, dev, args.layers, with_names=True)
        resident[DECODE_WL] = (mats4, names4)
        Ks = sorted({K for (_, _, K) in mats4})
        x_host = {K: synth.activations(synth.x_seed(DECODE_WL, K, 1), 1, K).pin_memory() for K in Ks}
        x_dev = {K: x_host[K].to(dev) for K in Ks}
        y4 = torch.empty(sum(N for (_, N, _) in mats4), device=dev)
        calls4 = _grouped_calls(q4k, mats4, names4, x_dev, y4, sp)
        g4 = _capture(torch, calls4, stream)
        bytes4 = sum(Wd.numel() for (Wd, _, _) in mats4)
        # the same sweep with one call per matrix
        calls4u = _sweep_calls(q4k, mats4, x_dev, y4, 1, False, sp)
        g4u = _capture(torch, calls4u, stream)
        times["decode_per_matrix"] = _time_graph(torch, g4u, stream, args.steps, args.warmup, barrier)
        launches += args.steps * len(calls4u)
        del g4u
        # steady load for ~1.5 s so that the clock samples see the working clock
        with torch.cuda.stream(stream):
            t_end = time.time() + 1.5
            while time.time() < t_end:
                for _ in range(20):
                    g4.replay()
                torch.cuda.synchronize()
        times["decode"] = _time_graph(torch, g4, stream, args.steps, args.warmup, barrier)
        launches += args.steps * len(calls4)
        # warm per-shape table: every launch of one shape back to back in a graph
        # (the 40 layers' copies exceed L2), one graph per distinct shape
        per_shape = []
        for key, groups in _shape_classes(mats4, names4).items():
            cs = _grouped_calls(q4k, mats4, names4, x_dev, y4, sp, groups=groups)
            gs = _capture(torch, cs, stream)
            tkey = "shape:" + "+".join(key[0])
            times[tkey] = _time_graph(torch, gs, stream, args.steps, args.warmup, barrier)
            launches += args.steps * len(cs)
            nbytes = sum(mats4[j][0].numel() for grp in groups for j in grp) // len(groups)
            per_shape.append({"call": "+".join(key[0]), "rows": list(key[1]), "K": key[2],
                              "launches_per_step": len(groups), "_tkey": tkey,
                              "algorithmic_bytes_per_launch": nbytes + 4 * key[2] + 4 * sum(key[1])})
            del gs
        # end to end through the public API with host buffers: (a) the captured
        # graph, (b) eager, call by call through the C ABI. Each step copies
        # the activation rows in from pinned memory and every output back.
        y_host = torch.empty(y4.numel(), pin_memory=True)
        h2d = sum(x.numel() * 4 for x in x_host.values())
        d2h = y4.numel() * 4
        with torch.cuda.stream(stream):
            def e2e_graph():
                for K, xh in x_host.items():
                    x_dev[K].copy_(xh, non_blocking=True)
                g4.replay()
                y_host.copy_(y4, non_blocking=True)
                stream.synchronize()

            def e2e_eager():
                for K, xh in x_host.items():
                    x_dev[K].copy_(xh, non_blocking=True)
                for c in calls4:
                    c()
                y_host.copy_(y4, non_blocking=True)
                stream.synchronize()
            for name, step in (("e2e", e2e_graph), ("e2e_eager", e2e_eager)):
                for _ in range(args.warmup):
                    step()
                barrier()
                t0 = time.perf_counter()
                for _ in range(args.steps):
                    step()
                times[name] = (time.perf_counter() - t0) * 1e3 / args.steps
                launches += args.steps * len(calls4)
                barrier()
            # host cost of issuing the sweep's calls (no synchronisation inside)
            stream.synchronize()
            t0 = time.perf_counter()
            for c in calls4:
                c()
            host_issue_ms = (time.perf_counter() - t0) * 1e3
            launches += len(calls4)
            stream.synchronize()
        avg_launch_ms = times["decode"] / len(calls4)
        achieved = bytes4 / len(calls4) / (avg_launch_ms * 1e-3) / 1e9
        out.update({
            "unit": "GB/s",
            "config": {"workload": _decode_config_name() if not args.layers else
                       f"{w4.name} (first {args.layers} layers)",
                       "l2": "inputs larger than L2 (every step streams all weights from HBM)",
                       "launch": f"one CUDA graph per sweep, q4k_set_pdl({args.pdl}); q/k/v and "
                                 f"gate/up as grouped calls ({len(calls4)} launches per step)",
                       "parallelism": f"replicas x{ws}"},
            "roofline": {"bound": "hbm", "kernel": "q4k_gemv_kernel<1,f32>",
                         "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                         "frac": round(achieved / hbm, 4),
                         "peak_source": f"{peak_kind} hbm_gbs (copy, burst)",
                         "traffic": measured_traffic("q4k_gemv_kernel<1,f32>", w4.name),
                         "avg_launch_us": round(avg_launch_ms * 1e3, 3),
                         "avg_launch_basis": "CUDA-graph sweep time / launches (gaps included)",
                         "algorithmic_bytes_per_launch": round(bytes4 / len(calls4)),
                         "per_shape": per_shape},
            "e2e": {"unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "how": "pinned host -> device activations, the captured sweep, all outputs "
                           "device -> host, per step"},
            "e2e_eager": {"unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                          "how": "as e2e, with the sweep issued call by call through the C ABI "
                                 "(q4k_matmul_multi via ctypes, no graph)",
                          "host_issue_us_per_call": round(host_issue_ms * 1e3 / len(calls4), 2)},
        })
        out["_bytes4"] = bytes4
        out["_calls4"] = len(calls4)
        out["_calls4u"] = len(calls4u)
        del g4, calls4, calls4u
        torch.cuda.empty_cache()

        # -------------------- the same weights at 4 and 16 activation rows ---
        out["decode_rows"] = []
        for M in DECODE_EXTRA_M:
            rec, n = _sweep_record(torch, q4k, DECODE_WL, mats4, names4, M, "f32", stream, args.steps,
                                   args.warmup, hbm, bf16_peak, barrier)
            rec["kernel"] = "q4k_tcgemv_kernel"
            launches += n
            out["decode_rows"].append(rec)
        # ------------------------------------------- other decode sweeps ---
        out["decode_workloads"] = []
        for wl in DECODE_EXTRA_WLS:
            w, mats, names = _weights(wl, dev, args.layers, with_names=True)
            rec, n = _sweep_record(torch, q4k, wl, mats, names, 1, "f32", stream, args.steps,
                                   args.warmup, hbm, bf16_peak, barrier)
            launches += n
            out["decode_workloads"].append(rec)
            if wl != LM_HEAD[0]:
                del mats
                continue
            # the lm_head as a greedy pick: the fused GEMV + argmax call
            # against the GEMV followed by torch's argmax
            lib = q4k.lib()
            _, Nl, Kl = LM_HEAD
            Wl = mats[-1][0]
            xl = synth.activations(synth.x_seed(wl, Kl, 1), 1, Kl).to(dev)
            yl = torch.empty(1, Nl, device=dev)
            idx = torch.empty(1, dtype=torch.int64, device=dev)
            idx2 = torch.empty(1, dtype=torch.int64, device=dev)

            def fused():
                rc = lib.q4k_matmul_argmax(Wl.data_ptr(), Nl, Kl, xl.data_ptr(), 1, idx.data_ptr(), sp)
                if rc != 0:
                    raise q4k.Q4KError(rc, "lm_head argmax")

            def two_step():
                rc = lib.q4k_matmul(Wl.data_ptr(), Nl, Kl, xl.data_ptr(), 1, yl.data_ptr(), sp)
                if rc != 0:
                    raise q4k.Q4KError(rc, "lm_head gemv")
                torch.argmax(yl, dim=1, out=idx2)
            gf = _capture(torch, [fused], stream)
            times["lm_head_argmax"] = _time_graph(torch, gf, stream, args.steps, args.warmup, barrier)
            launches += args.steps * 3
            gt = _capture(torch, [two_step], stream)
            times["lm_head_gemv_then_argmax"] = _time_graph(torch, gt, stream, args.steps, args.warmup,
                                                            barrier)
            launches += args.steps
            torch.cuda.synchronize()
            if not torch.equal(idx, idx2):
                raise RuntimeError("fused argmax differs from the GEMV's argmax")
            out["_lm_head_bytes"] = Wl.numel()
            del gf, gt, Wl, mats
            torch.cuda.empty_cache()

        # ------------------------------------------------ standalone dequant ---
        if ws == 1 and rank == 0 and not args.no_cpu_baseline:
            dq_sample = os.path.join(tempfile.mkdtemp(prefix="q4k_dq_"), "rows.npz")
        rec, n = _dequant_leg(torch, q4k, dev, stream, args.steps, args.warmup, hbm, barrier,
                              sample_path=dq_sample)
        launches += n
        out["dequant"] = rec

    if args.only in ("all", "prefill"):
        w3, mats3, names3 = _weights(PREFILL_WL, dev, args.layers, with_names=True)
        Ks = sorted({K for (_, _, K) in mats3})
        x3 = {K: synth.activations(synth.x_seed(PREFILL_WL, K, PREFILL_M), PREFILL_M, K,
                                   torch.bfloat16).to(dev) for K in Ks}
        y3 = torch.empty(_group_y_floats(mats3, names3, PREFILL_M), device=dev)
        calls3 = _grouped_calls(q4k, mats3, names3, x3, y3, sp, M=PREFILL_M, bf16=True)
        g3 = _capture(torch, calls3, stream)
        flops3 = sum(2 * PREFILL_M * N * K for (_, N, K) in mats3)
        bytes3 = sum(Wd.numel() for (Wd, _, _) in mats3)
        steps3 = max(3, args.steps // 4)
        times["prefill"] = _time_graph(torch, g3, stream, steps3, args.warmup, barrier)
        launches += steps3 * len(calls3)
        del g3
        # the same sweep with one call per matrix
        calls3u = _sweep_calls(q4k, mats3, x3, y3, PREFILL_M, True, sp)
        g3u = _capture(torch, calls3u, stream)
        times["prefill_per_matrix"] = _time_graph(torch, g3u, stream, steps3, args.warmup, barrier)
        launches += steps3 * len(calls3u)
        del g3u, x3, y3
        gemm_ms = times["prefill"] / len(calls3)  # in-graph, gaps between launches included
        achieved3 = flops3 / len(calls3) / (gemm_ms * 1e-3) / 1e12
        out["gemm"] = {
            "metric": "GEMM TFLOP/s (M=512)", "unit": "TFLOP/s", "steps": steps3,
            "workload": f"{w3.name}: {len(mats3)} Q4_K matrices, {bytes3 / 1e9:.2f} GB packed, "
                        f"M={PREFILL_M} bf16 activations",
            "launch": f"one CUDA graph per sweep; q/k/v and gate/up as grouped calls "
                      f"({len(calls3)} launches per step)",
            "launches_per_step": len(calls3),
            "roofline": {"bound": "tensor", "kernel": "q4k_gemm_kernel<BN> (BN, split per launch plan)",
                         "achieved": round(achieved3, 1), "peak": bf16_peak, "unit": "TFLOP/s",
                         "frac": round(achieved3 / bf16_peak, 4),
                         "frac_of_sustained": round(achieved3 / bf16_sust, 4) if bf16_sust else None,
                         "peak_source": f"{peak_kind} bf16_tflops (cuBLAS burst)",
                         "traffic": measured_traffic("q4k_gemm_kernel"),
                         "avg_launch_us": round(gemm_ms * 1e3, 2),
                         "avg_launch_basis": "CUDA-graph sweep time / launches (gaps included)"}}
        out["_flops3"] = flops3
        # the other prefill sizes: 32 and 1024 rows on this set, 2048 on the largest
        out["gemm_workloads"] = []
        for wl, M in GEMM_EXTRA:
            if wl == PREFILL_WL:
                mats, names = mats3, names3
            else:
                if wl not in resident:
                    _, m_, n_ = _weights(wl, dev, args.layers, with_names=True)
                    resident[wl] = (m_, n_)
                mats, names = resident[wl]
            rec, n = _sweep_record(torch, q4k, wl, mats, names, M, "bf16", stream, steps3,
                                   args.warmup, hbm, bf16_peak, barrier)
            rec["frac_of_bf16_sustained"] = round(rec["TFLOPs"] / bf16_sust, 4) if bf16_sust else None
            launches += n
            out["gemm_workloads"].append(rec)
        del mats3

    out["clocks"] = sampler.stop()
    tkeys = {k: v for k, v in times.items()}
    times = max_over_ranks(tkeys, ws, dev)
    out["device_error"] = q4k.q4k_device_error()
    out["gpu_launches"] = launches
    if rank != 0:
        return
    if "decode" in times:
        b4 = out.pop("_bytes4")
        out.pop("_calls4")
        out["value"] = round(ws * b4 / (times["decode"] * 1e-3) / 1e9, 2)
        out["ms_per_step"] = round(times["decode"], 5)
        total_ms = 0.0
        for rec in out["roofline"]["per_shape"]:
            ms = times[rec.pop("_tkey")]
            us = ms * 1e3 / rec["launches_per_step"]
            total_ms += us * rec["launches_per_step"] / 1e3
            gb = rec["algorithmic_bytes_per_launch"] / (us * 1e-6) / 1e9
            rec.update({"us_per_launch": round(us, 3), "achieved_GBps": round(gb, 1),
                        "frac": round(gb / hbm, 4)})
        out["roofline"]["per_shape_sum_ms"] = round(total_ms, 5)
        out["roofline"]["per_shape_basis"] = (
            "each distinct launch shape of the sweep timed alone: a CUDA graph of its launches "
            "(one per layer, back to back, > L2 of weights), CUDA events; sum of count x us "
            "against ms_per_step")
        out["decode_one_call_per_matrix"] = {
            "value": round(ws * b4 / (times["decode_per_matrix"] * 1e-3) / 1e9, 2), "unit": "GB/s",
            "ms_per_step": round(times["decode_per_matrix"], 5),
            "launches_per_step": out.pop("_calls4u")}
        for key in ("e2e", "e2e_eager"):
            out[key]["value"] = round(ws * b4 / (times[key] * 1e-3) / 1e9, 2)
            out[key]["ms_per_step"] = round(times[key], 4)
        lb = out.pop("_lm_head_bytes")
        out["lm_head_argmax"] = {
            "workload": "lm_head 128256 x 3072 (Llama-3.2-3B shape), M=1 fp32, greedy pick",
            "fused_us": round(times["lm_head_argmax"] * 1e3, 2),
            "fused_packed_GBps": round(lb / (times["lm_head_argmax"] * 1e-3) / 1e9, 1),
            "gemv_then_torch_argmax_us": round(times["lm_head_gemv_then_argmax"] * 1e3, 2),
            "same_index": True}
    if "prefill" in times:
        f3 = out.pop("_flops3")
        out["gemm"]["value"] = round(ws * f3 / (times["prefill"] * 1e-3) / 1e12, 2)
        out["gemm"]["ms_per_step"] = round(times["prefill"], 4)
        out["gemm"]["one_call_per_matrix"] = {
            "value": round(ws * f3 / (times["prefill_per_matrix"] * 1e-3) / 1e12, 2),
            "unit": "TFLOP/s", "ms_per_step": round(times["prefill_per_matrix"], 4),
            "frac": round(f3 / (times["prefill_per_matrix"] * 1e-3) / 1e12 / bf16_peak, 4)}
    if args.layers:
        out["config"] = dict(out.get("config", {}), profiling_subset=f"first {args.layers} layers")
    if ws == 1 and not args.no_cpu_baseline and args.only == "all":
        out["cpu_baseline"] = cpu_baselines_subprocess(args.cpu_budget, dq_sample)
        dc = out["cpu_baseline"].pop("dequant_check", None)
        if dc is not None:
            out["dequant"]["bit_exact_check"] = dc
    print(json.dumps(out))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="libq4k", choices=["libq4k", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=10.0,
                    help="seconds of oracle CPU time for cpu_baseline")
    ap.add_argument("--ref-budget", type=float, default=5.0,
                    help="seconds of oracle CPU time per reference step")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-baseline-only", action="store_true",
                    help="(internal) print cpu_baselines() as JSON; run in a CPU-only process")
    ap.add_argument("--dequant-sample", default="", help="(internal) rows saved by the GPU run")
    ap.add_argument("--pdl", type=int, default=2, choices=[0, 1, 2],
                    help="q4k_set_pdl mode for the sweeps (2: weights may stream early)")
    ap.add_argument("--only", default="all", choices=["all", "decode", "prefill", "sweep", "dequant"],
                    help="profiling aid: run one leg only (sweep: the headline decode sweep alone; "
                         "dequant: the standalone dequant leg alone)")
    ap.add_argument("--layers", type=int, default=0,
                    help="profiling aid: use only the first L layers of each weight set")
    ap.add_argument("--profile-shape", default="",
                    help="microbenchmark one shape 'N,K,M' (bf16 activations when M > 16)")
    ap.add_argument("--x-bf16", action="store_true", help="--profile-shape with bf16 activations")
    ap.add_argument("--all-configs", action="store_true",
                    help="time every workload at every M / X dtype (one JSON line each)")
    ap.add_argument("--profile-bytes", type=float, default=300e6,
                    help="weight bytes to rotate through in --profile-shape (> L2)")
    ap.add_argument("--clocks-csv", default="",
                    help="keep the nvidia-smi clock samples in this file ('{rank}' is replaced "
                         "by the rank; default: a temporary file)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.cpu_baseline_only:
        print(json.dumps(cpu_baselines(args.cpu_budget, args.dequant_sample)))
    elif args.impl == "reference":
        run_reference(args)
    elif args.profile_shape:
        run_profile_shape(args)
    elif args.all_configs:
        run_all_configs(args)
    elif args.only in ("sweep", "dequant"):
        run_sweep_only(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
