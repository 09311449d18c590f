"""Benchmark of the packed Q4_K dequant-matmul (libq4k) on one GB300 per rank.

Metric: Q4_K dequant-matmul -- GEMV packed-weight GB/s (M=1); GEMM TFLOP/s (M=512).

A step is one pass of the hot path over one batch:
  * decode leg (the headline `value`): the Llama-3.2-1B-shaped sweep, 16
    layers x 7 Q4_K matrices (547 MB packed), M = 1 fp32 activation row,
    q/k/v and gate/up as grouped calls (64 GEMV launches), replayed from a
    CUDA graph; value = packed weight bytes per step / step time. The same
    sweep with one call per matrix (112 launches) and end to end from host
    buffers are reported beside it, with the fused lm_head greedy pick.
  * prefill leg (`gemm`): the Qwen3-8B-shaped sweep, 36 layers x 7 matrices
    (3.9 GB packed), M = 512 bf16 token rows, grouped the same way (144
    tcgen05 GEMM launches; 252 with one call per matrix); value = 2*M*N*K
    flops per step / step time.
Both weight sets are larger than L2, so every step streams weights from HBM.
Inputs are synthetic (seeded generator), resident in HBM before timing.

`--impl reference` times the CPU oracle (the plain C++ reference the library
is checked against) on a bounded sample of the same decode workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "Q4_K dequant-matmul: GEMV packed-weight GB/s (M=1); GEMM TFLOP/s (M=512)"
DECODE_WL, PREFILL_WL, PREFILL_M = 1, 3, 512


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d["hbm_gbs"], d["bf16_tflops"], d.get("bf16_tflops_sustained"), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


KERNEL_SOURCES = {
    "gemv_kernel<1,f32>": ["gguf_q4_dequant_gb300/csrc/q4k_gemv.cu", "gguf_q4_dequant_gb300/csrc/q4k_device.cuh",
                           "gguf_q4_dequant_gb300/csrc/q4k_internal.h"],
    "gemm_kernel": ["gguf_q4_dequant_gb300/csrc/q4k_gemm.cu", "gguf_q4_dequant_gb300/csrc/q4k_device.cuh",
                    "gguf_q4_dequant_gb300/csrc/q4k_internal.h"],
}


def sources_sha256(kernel):
    import hashlib
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def measured_traffic(kernel):
    """DRAM bytes per launch from the committed ncu summary, or None when the
    kernel's sources changed after the counters were taken."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        rec = json.load(f).get(kernel)
    if not rec or rec.get("sources_sha256") != sources_sha256(kernel):
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
    """Host copies of the decode sweep's weights and activation rows (drawn once)."""
    global _HOST_DECODE
    if _HOST_DECODE is None:
        from gguf_q4_dequant_gb300 import synth
        w = synth.WORKLOADS[DECODE_WL]
        mats = [(synth.weight_rows(synth.weight_seed(DECODE_WL, layer, name), N, K).numpy(), N, K)
                for (layer, name, N, K) in w.matrices()]
        xs = {K: synth.activations(synth.x_seed(DECODE_WL, K, 1), 1, K).numpy()
              for K in {K for (_, _, K) in mats}}
        _HOST_DECODE = (w, mats, xs)
    return _HOST_DECODE


def cpu_oracle_decode(budget_s: float, threads: int):
    """Times the oracle (as it stands) over the decode sweep, matrix by matrix in
    sweep order, until `budget_s` seconds of oracle time have elapsed."""
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
            "sample": f"oracle matmul over {done} matrices of the decode sweep in sweep order "
                      f"({done / len(mats):.2f} sweeps, {total_bytes / 1e6:.0f} MB packed, M=1), "
                      f"{elapsed:.1f} s of CPU time"}


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


def cpu_baselines(budget_s: float):
    """The oracle as it stands: the decode sweep on all host cores (the
    reported value), the same on one thread, and a row sample of the prefill
    workload on all host cores."""
    cores = _host_cores()
    cb = cpu_oracle_decode(budget_s, cores)
    one = cpu_oracle_decode(max(1.0, budget_s / 4), 1)
    cb["single_thread"] = {"value": one["value"], "unit": one["unit"], "sample": one["sample"]}
    cb["prefill"] = cpu_oracle_prefill(max(1.0, budget_s / 2), cores)
    return cb


def max_over_ranks(times, ws, device="cpu"):
    """Every timing as its maximum over the job's ranks (called by all ranks)."""
    import torch
    keys = sorted(times)
    t = torch.tensor([times[k] for k in keys], device=device, dtype=torch.float64)
    if ws > 1:
        import torch.distributed as dist
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return dict(zip(keys, t.tolist()))


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
        "config": {"workload": "llama-3.2-1b-shaped decode sweep, M=1 fp32 (bounded sample)",
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
            import tempfile
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


def _grouped_calls(q4k, mats, names, x_dev, y, stream_ptr, M=1, bf16=False):
    """A sweep with q/k/v and gate/up as grouped calls (one launch each). At
    M = 1 every matrix writes its own slice of `y`; at larger M the matrices of
    one group write disjoint slices and the groups reuse them."""
    import ctypes
    lib = q4k.lib()
    fn = lib.q4k_matmul_multi_bf16 if bf16 else lib.q4k_matmul_multi
    groups = _group_spans(names)
    offs = [0] * len(mats)
    o = 0
    for grp in groups:
        if M > 1:
            o = 0
        for j in grp:
            offs[j] = o
            o += M * mats[j][1]
    calls = []
    for grp in groups:
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


def run_profile_shape(args):
    """Microbenchmark of one matrix shape: a CUDA graph of back-to-back calls over
    enough distinct weight copies to exceed L2; prints per-launch time."""
    import math
    import torch
    import gguf_q4_dequant_gb300 as q4k
    from gguf_q4_dequant_gb300 import build as q4k_build
    from gguf_q4_dequant_gb300 import synth
    N, K, M = (int(v) for v in args.profile_shape.split(","))
    q4k_build.build()
    torch.cuda.set_device(0)
    q4k.q4k_init()
    q4k.q4k_set_pdl(args.pdl)
    dev = "cuda:0"
    wb = N * K // 256 * 144
    R = min(64, max(2, math.ceil(args.profile_bytes / wb)))
    Ws = [synth.weight_rows(0x5eed + i, N, K, device=dev) for i in range(R)]
    bf16 = M > 16
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


def run_all_configs(args):
    """Every workload of synth.WORKLOADS at every M and activation dtype it
    names, each as full sweeps with q/k/v and gate/up grouped, in a CUDA graph;
    one JSON line per case, plus the standalone dequant kernel."""
    import torch
    import gguf_q4_dequant_gb300 as q4k
    from gguf_q4_dequant_gb300 import build as q4k_build
    from gguf_q4_dequant_gb300 import synth
    q4k_build.build()
    torch.cuda.set_device(0)
    q4k.q4k_init()
    q4k.q4k_set_pdl(args.pdl)
    dev = "cuda:0"
    stream = torch.cuda.Stream()
    sp = stream.cuda_stream
    hbm, bf16_peak, _, _ = _peaks()
    steps = max(3, min(args.steps, 20))
    for wl in (1, 2, 3, 4):
        w, mats, names = _weights(wl, dev, 0, with_names=True)
        Ks = sorted({K for (_, _, K) in mats})
        wbytes = sum(Wd.numel() for (Wd, _, _) in mats)
        nk = sum(N * K for (_, N, K) in mats)
        cases = [(M, x) for x in w.x_dtypes for M in w.decode_m]
        cases += [(M, "bf16") for M in w.prefill_m]
        for M, xdt in cases:
            bf16 = xdt == "bf16"
            dt = torch.bfloat16 if bf16 else torch.float32
            xs = {K: synth.activations(synth.x_seed(wl, K, M), M, K, dt).to(dev) for K in Ks}
            ny = sum(N for (_, N, _) in mats) if M == 1 else _group_y_floats(mats, names, M)
            y = torch.empty(ny, device=dev)
            calls = _grouped_calls(q4k, mats, names, xs, y, sp, M=M, bf16=bf16)
            g = _capture(torch, calls, stream)
            ms = _time_graph(torch, g, stream, steps, args.warmup, lambda: None)
            gbps = wbytes / (ms * 1e-3) / 1e9
            tf = 2 * M * nk / (ms * 1e-3) / 1e12
            print(json.dumps({"workload": wl, "name": w.name, "M": M, "x_dtype": xdt,
                              "kernel": "gemv_kernel" if M <= 16 else "gemm_kernel",
                              "launches_per_sweep": len(calls), "steps": steps,
                              "ms_per_sweep": round(ms, 4), "packed_GBps": round(gbps, 1),
                              "frac_of_hbm": round(gbps / hbm, 4), "TFLOPs": round(tf, 2),
                              "frac_of_bf16": round(tf / bf16_peak, 4),
                              "device_error": q4k.q4k_device_error()}), flush=True)
            del g, calls, xs, y
        del mats
        torch.cuda.empty_cache()
    # K1: the lm_head of the Llama-3.2-3B shape expanded to fp32
    N, K = 128256, 3072
    Wd = synth.weight_rows(synth.weight_seed(2, 28, "lm_head"), N, K, device=dev)
    out = torch.empty(N, K, device=dev)
    g = _capture(torch, [lambda: q4k.q4k_dequant(Wd, N, K, out, stream=stream.cuda_stream)], stream)
    ms = _time_graph(torch, g, stream, steps, args.warmup, lambda: None)
    moved = Wd.numel() + out.numel() * 4
    print(json.dumps({"kernel": "dequant_kernel", "shape": {"N": N, "K": K}, "ms": round(ms, 4),
                      "read_plus_write_GBps": round(moved / (ms * 1e-3) / 1e9, 1),
                      "frac_of_hbm": round(moved / (ms * 1e-3) / 1e9 / hbm, 4),
                      "device_error": q4k.q4k_device_error()}), flush=True)


def run_gpu(args):
    import torch
    import gguf_q4_dequant_gb300 as q4k
    from gguf_q4_dequant_gb300 import build as q4k_build
    from gguf_q4_dequant_gb300 import synth
    ws, rank, local = _dist()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device(f"cuda:{local}"))

        def barrier():
            dist.barrier()
    else:
        def barrier():
            pass
    q4k_build.build()
    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    q4k.q4k_init()
    q4k.q4k_set_pdl(args.pdl)
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

    if args.only in ("all", "decode"):
        w1, mats1, names1 = _weights(DECODE_WL, dev, args.layers, with_names=True)
        Ks = sorted({K for (_, _, K) in mats1})
        x_host = {K: synth.activations(synth.x_seed(DECODE_WL, K, 1), 1, K).pin_memory() for K in Ks}
        x_dev = {K: x_host[K].to(dev) for K in Ks}
        y1 = torch.empty(sum(N for (_, N, _) in mats1), device=dev)
        calls1 = _grouped_calls(q4k, mats1, names1, x_dev, y1, sp)
        g1 = _capture(torch, calls1, stream)
        bytes1 = sum(Wd.numel() for (Wd, _, _) in mats1)
        # the same sweep with one call per matrix
        calls1u = _sweep_calls(q4k, mats1, x_dev, y1, 1, False, sp)
        g1u = _capture(torch, calls1u, stream)
        times["decode_per_matrix"] = _time_graph(torch, g1u, stream, args.steps, args.warmup, barrier)
        launches += args.steps * len(calls1u)
        del g1u
        # steady load for ~1.5 s so that the clock samples see the working clock
        with torch.cuda.stream(stream):
            t_end = time.time() + 1.5
            while time.time() < t_end:
                for _ in range(50):
                    g1.replay()
                torch.cuda.synchronize()
        times["decode"] = _time_graph(torch, g1, stream, args.steps, args.warmup, barrier)
        launches += args.steps * len(calls1)
        # e2e through the public API with host buffers: copy the activation rows
        # in from pinned memory, run the captured q4k_matmul calls, read every
        # output row back.
        y_host = torch.empty(y1.numel(), pin_memory=True)
        h2d = sum(x.numel() * 4 for x in x_host.values())
        d2h = y1.numel() * 4
        with torch.cuda.stream(stream):
            def e2e_step():
                for K, xh in x_host.items():
                    x_dev[K].copy_(xh, non_blocking=True)
                g1.replay()
                y_host.copy_(y1, non_blocking=True)
                stream.synchronize()
            for _ in range(args.warmup):
                e2e_step()
            barrier()
            t0 = time.perf_counter()
            for _ in range(args.steps):
                e2e_step()
            times["e2e"] = (time.perf_counter() - t0) * 1e3 / args.steps
            barrier()
        launches += args.steps * len(calls1)
        bpl = bytes1 / len(calls1)
        gemv_ms = times["decode"] / len(calls1)  # in-graph, gaps between launches included
        achieved = bpl / (gemv_ms * 1e-3) / 1e9
        out.update({
            "unit": "GB/s",
            "config": {"workload": f"{w1.name}: {len(mats1)} Q4_K matrices, "
                                   f"{bytes1 / 1e6:.1f} MB packed, M=1 fp32 activations",
                       "l2": "inputs larger than L2 (every step streams all weights from HBM)",
                       "launch": f"one CUDA graph per sweep, q4k_set_pdl({args.pdl}); q/k/v and "
                                 f"gate/up as grouped calls ({len(calls1)} launches per step)",
                       "parallelism": f"replicas x{ws}"},
            "roofline": {"bound": "hbm", "kernel": "gemv_kernel<1,f32>", "achieved": round(achieved, 1),
                         "peak": hbm, "unit": "GB/s", "frac": round(achieved / hbm, 4),
                         "peak_source": f"{peak_kind} hbm_gbs (copy, burst)",
                         "traffic": measured_traffic("gemv_kernel<1,f32>"),
                         "avg_launch_us": round(gemv_ms * 1e3, 3),
                         "avg_launch_basis": "CUDA-graph sweep time / launches (gaps included)",
                         "algorithmic_bytes_per_launch": round(bpl)},
            "e2e": {"unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        })
        del g1
        out["_bytes1"] = bytes1
        out["_names1"] = names1
        for (Wd, _, _) in mats1:
            del Wd
        del mats1, calls1
        torch.cuda.empty_cache()

        # the lm_head of the Llama-3.2-3B shape as a greedy pick: the fused
        # GEMV + argmax call against the GEMV followed by torch's argmax
        import ctypes
        lib = q4k.lib()
        Nl, Kl = 128256, 3072
        Wl = synth.weight_rows(synth.weight_seed(2, 28, "lm_head"), Nl, Kl, device=dev)
        xl = synth.activations(synth.x_seed(2, Kl, 1), 1, Kl).to(dev)
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
        times["lm_head_gemv_then_argmax"] = _time_graph(torch, gt, stream, args.steps, args.warmup, barrier)
        launches += args.steps
        torch.cuda.synchronize()
        if not torch.equal(idx, idx2):
            raise RuntimeError("fused argmax differs from the GEMV's argmax")
        out["_lm_head_bytes"] = Wl.numel()
        del gf, gt, Wl
        torch.cuda.empty_cache()

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
        del g3u
        gemm_ms = times["prefill"] / len(calls3)  # in-graph, gaps between launches included
        achieved3 = flops3 / len(calls3) / (gemm_ms * 1e-3) / 1e12
        out["gemm"] = {
            "metric": "GEMM TFLOP/s (M=512)", "unit": "TFLOP/s", "steps": steps3,
            "workload": f"{w3.name}: {len(mats3)} Q4_K matrices, {bytes3 / 1e9:.2f} GB packed, "
                        f"M={PREFILL_M} bf16 activations",
            "launch": f"one CUDA graph per sweep; q/k/v and gate/up as grouped calls "
                      f"({len(calls3)} launches per step)",
            "launches_per_step": len(calls3),
            "roofline": {"bound": "tensor", "kernel": "gemm_kernel<BN> (BN, split per launch plan)",
                         "achieved": round(achieved3, 1), "peak": bf16_peak, "unit": "TFLOP/s",
                         "frac": round(achieved3 / bf16_peak, 4),
                         "frac_of_sustained": round(achieved3 / bf16_sust, 4) if bf16_sust else None,
                         "peak_source": f"{peak_kind} bf16_tflops (cuBLAS burst)",
                         "traffic": measured_traffic("gemm_kernel"),
                         "avg_launch_us": round(gemm_ms * 1e3, 2),
                         "avg_launch_basis": "CUDA-graph sweep time / launches (gaps included)"}}
        out["_flops3"] = flops3

    out["clocks"] = sampler.stop()
    times = max_over_ranks(times, ws, dev)
    out["device_error"] = q4k.q4k_device_error()
    out["gpu_launches"] = launches
    if rank != 0:
        return
    if "decode" in times:
        b1 = out.pop("_bytes1")
        out["value"] = round(ws * b1 / (times["decode"] * 1e-3) / 1e9, 2)
        out["ms_per_step"] = round(times["decode"], 5)
        out["decode_one_call_per_matrix"] = {
            "value": round(ws * b1 / (times["decode_per_matrix"] * 1e-3) / 1e9, 2), "unit": "GB/s",
            "ms_per_step": round(times["decode_per_matrix"], 5),
            "launches_per_step": len(out.pop("_names1"))}
        out["e2e"]["value"] = round(ws * b1 / (times["e2e"] * 1e-3) / 1e9, 2)
        out["e2e"]["ms_per_step"] = round(times["e2e"], 4)
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
            "unit": "TFLOP/s", "ms_per_step": round(times["prefill_per_matrix"], 4)}
    if args.layers:
        out["config"] = dict(out.get("config", {}), profiling_subset=f"first {args.layers} layers")
    if ws == 1 and not args.no_cpu_baseline and args.only == "all":
        out["cpu_baseline"] = cpu_baselines(args.cpu_budget)
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
    ap.add_argument("--pdl", type=int, default=2, choices=[0, 1, 2],
                    help="q4k_set_pdl mode for the sweeps (2: weights may stream early)")
    ap.add_argument("--only", default="all", choices=["all", "decode", "prefill"],
                    help="profiling aid: run one leg only")
    ap.add_argument("--layers", type=int, default=0,
                    help="profiling aid: use only the first L layers of each weight set")
    ap.add_argument("--profile-shape", default="",
                    help="microbenchmark one shape 'N,K,M' (bf16 activations when M > 16)")
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
    if args.impl == "reference":
        run_reference(args)
    elif args.profile_shape:
        run_profile_shape(args)
    elif args.all_configs:
        run_all_configs(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
