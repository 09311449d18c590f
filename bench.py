"""Benchmark of the packed Q4_K dequant-matmul (libq4k) on one GB300 per rank.

Metric: Q4_K dequant-matmul -- GEMV packed-weight GB/s (M=1); GEMM TFLOP/s (M=512).

A step is one pass of the hot path over one batch:
  * decode leg (the headline `value`): the Llama-3.2-1B-shaped sweep, 16
    layers x 7 Q4_K matrices (547 MB packed), M = 1 fp32 activation row,
    112 GEMV launches replayed from a CUDA graph; value = packed weight bytes
    per step / step time.
  * prefill leg (`gemm`): the Qwen3-8B-shaped sweep, 36 layers x 7 matrices
    (3.9 GB packed), M = 512 bf16 token rows, 252 tcgen05 GEMM launches;
    value = 2*M*N*K flops per step / step time.
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

def cpu_oracle_decode(budget_s: float, threads: int):
    """Times the oracle on whole layers of the decode sweep until `budget_s`."""
    import numpy as np
    import oracle
    from gguf_q4_dequant_gb300 import synth
    oracle.build()
    w = synth.WORKLOADS[DECODE_WL]
    total_bytes, elapsed, layers = 0, 0.0, 0
    xs = {}
    for layer in range(w.layers):
        for (name, N, K) in w.layer_shapes:
            Wh = synth.weight_rows(synth.weight_seed(DECODE_WL, layer, name), N, K).numpy()
            if K not in xs:
                xs[K] = synth.activations(synth.x_seed(DECODE_WL, K, 1), 1, K).numpy()
            t0 = time.perf_counter()
            oracle.matmul(Wh, N, K, xs[K], threads=threads)
            elapsed += time.perf_counter() - t0
            total_bytes += Wh.size
        layers += 1
        if elapsed >= budget_s:
            break
    return {"value": total_bytes / elapsed / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"oracle matmul over {layers} of {w.layers} layers of the decode sweep "
                      f"({total_bytes / 1e6:.0f} MB packed, M=1), {elapsed:.1f} s of CPU time"}


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

    def __init__(self, gpu_index: int):
        self.proc = None
        self.path = os.path.join(ROOT, "gpurun_out", f"clocks_rank{gpu_index}.csv")
        self.gpu = gpu_index

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
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
        if not rows:
            return None
        busy = [r for r in rows if r[2] > 0] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in busy for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in busy), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(busy)}


# ------------------------------------------------------------------ GPU arm ---

def _build_decode(dev):
    import torch
    from gguf_q4_dequant_gb300 import synth
    w = synth.WORKLOADS[DECODE_WL]
    mats = []
    for (layer, name, N, K) in w.matrices():
        mats.append((synth.weight_rows(synth.weight_seed(DECODE_WL, layer, name), N, K, device=dev),
                     N, K))
    Ks = sorted({K for (_, _, K) in mats})
    x_host = {K: synth.activations(synth.x_seed(DECODE_WL, K, 1), 1, K).pin_memory() for K in Ks}
    x_dev = {K: x_host[K].to(dev) for K in Ks}
    y_total = sum(N for (_, N, _) in mats)
    y = torch.empty(y_total, device=dev)
    return w, mats, x_host, x_dev, y


def _build_prefill(dev):
    import torch
    from gguf_q4_dequant_gb300 import synth
    w = synth.WORKLOADS[PREFILL_WL]
    mats = []
    for (layer, name, N, K) in w.matrices():
        mats.append((synth.weight_rows(synth.weight_seed(PREFILL_WL, layer, name), N, K, device=dev),
                     N, K))
    Ks = sorted({K for (_, _, K) in mats})
    x_dev = {K: synth.activations(synth.x_seed(PREFILL_WL, K, PREFILL_M), PREFILL_M, K,
                                  torch.bfloat16).to(dev) for K in Ks}
    y = torch.empty(PREFILL_M * max(N for (_, N, _) in mats), device=dev)
    return w, mats, x_dev, y


def _sweep_fn(q4k, mats, x_dev, y, M, bf16):
    """Returns a callable issuing one sweep (one launch per matrix) on the current stream."""
    lib = q4k.lib()
    calls = []
    off = 0
    for (Wd, N, K) in mats:
        yp = y.data_ptr() + (off * 4 if M == 1 else 0)
        calls.append((Wd.data_ptr(), N, K, x_dev[K].data_ptr(), yp))
        if M == 1:
            off += N
    fn = lib.q4k_matmul_bf16 if bf16 else lib.q4k_matmul

    def run(stream_ptr):
        for (wp, N, K, xp, yp) in calls:
            rc = fn(wp, N, K, xp, M, yp, stream_ptr)
            if rc != 0:
                raise q4k.Q4KError(rc, "sweep")
    return run


def _time_graph(torch, graph, stream, steps, warmup, barrier):
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
    return start.elapsed_time(end) / steps  # ms per step


def _per_launch_ms(torch, run_calls, stream, reps=3):
    """Average kernel duration with CUDA events around every launch of a sweep."""
    durs = []
    for _ in range(reps):
        evs = []
        for call in run_calls:
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            call()
            b.record(stream)
            evs.append((a, b))
        torch.cuda.synchronize()
        durs.extend(a.elapsed_time(b) for a, b in evs)
    return statistics.mean(durs)


def run_gpu(args):
    import torch
    import gguf_q4_dequant_gb300 as q4k
    from gguf_q4_dequant_gb300 import build as q4k_build
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
    hbm, bf16_peak, bf16_sust, peak_kind = _peaks()

    # ---------------------------------------------------------- decode leg ---
    w1, mats1, x_host1, x_dev1, y1 = _build_decode(dev)
    bytes1 = sum(Wd.numel() for (Wd, _, _) in mats1)
    launches1 = len(mats1)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        sweep1 = _sweep_fn(q4k, mats1, x_dev1, y1, 1, False)
        sweep1(stream.cuda_stream)  # first use outside capture
        torch.cuda.synchronize()
        g1 = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g1, stream=stream):
            sweep1(torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()

    sampler = ClockSampler(local)
    sampler.start()
    # keep the GPU busy ~1.5 s so the clock samples reflect steady load
    t_end = time.time() + 1.5
    while time.time() < t_end:
        for _ in range(50):
            g1.replay()
        torch.cuda.synchronize()
    ms1 = _time_graph(torch, g1, stream, args.steps, args.warmup, barrier)

    # ---------------------------------------------------------- prefill leg ---
    w3, mats3, x_dev3, y3 = _build_prefill(dev)
    flops3 = sum(2 * PREFILL_M * N * K for (_, N, K) in mats3)
    bytes3 = sum(Wd.numel() for (Wd, _, _) in mats3)
    launches3 = len(mats3)
    with torch.cuda.stream(stream):
        sweep3 = _sweep_fn(q4k, mats3, x_dev3, y3, PREFILL_M, True)
        sweep3(stream.cuda_stream)
        torch.cuda.synchronize()
        g3 = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g3, stream=stream):
            sweep3(torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    ms3 = _time_graph(torch, g3, stream, max(1, args.steps // 4), args.warmup, barrier)
    clocks = sampler.stop()

    # ------------------------------------------- per-launch kernel durations ---
    lib = q4k.lib()
    with torch.cuda.stream(stream):
        sp = stream.cuda_stream
        calls1 = [(lambda Wd=Wd, N=N, K=K, o=o: lib.q4k_matmul(Wd.data_ptr(), N, K,
                                                               x_dev1[K].data_ptr(), 1,
                                                               y1.data_ptr() + 4 * o, sp))
                  for (Wd, N, K), o in zip(mats1, _offsets(mats1))]
        gemv_ms = _per_launch_ms(torch, calls1, stream)
        calls3 = [(lambda Wd=Wd, N=N, K=K: lib.q4k_matmul_bf16(Wd.data_ptr(), N, K,
                                                               x_dev3[K].data_ptr(), PREFILL_M,
                                                               y3.data_ptr(), sp))
                  for (Wd, N, K) in mats3]
        gemm_ms = _per_launch_ms(torch, calls3, stream, reps=1)

    # ------------------------------------------------------------------ e2e ---
    # the public C ABI with host buffers: per step, copy the activation rows
    # from pinned host memory, run the sweep, read all outputs back.
    y_host = torch.empty(y1.numel(), pin_memory=True)
    h2d = sum(x.numel() * 4 for x in x_host1.values())
    d2h = y1.numel() * 4
    with torch.cuda.stream(stream):
        def e2e_step():
            for K, xh in x_host1.items():
                x_dev1[K].copy_(xh, non_blocking=True)
            sweep1(stream.cuda_stream)
            y_host.copy_(y1, non_blocking=True)
        for _ in range(args.warmup):
            e2e_step()
        torch.cuda.synchronize()
        barrier()
        t0 = time.perf_counter()
        for _ in range(args.steps):
            e2e_step()
        torch.cuda.synchronize()
        e2e_ms = (time.perf_counter() - t0) * 1e3 / args.steps
        barrier()

    # ------------------------------------------------------- max over ranks ---
    times = torch.tensor([ms1, ms3, e2e_ms], device=dev, dtype=torch.float64)
    if ws > 1:
        import torch.distributed as dist
        dist.all_reduce(times, op=dist.ReduceOp.MAX)
    ms1, ms3, e2e_ms = times.tolist()
    err = q4k.q4k_device_error()
    if rank != 0:
        return
    value = ws * bytes1 / (ms1 * 1e-3) / 1e9
    gemm_tflops = ws * flops3 / (ms3 * 1e-3) / 1e12
    gemv_bytes_per_launch = bytes1 / launches1
    gemv_achieved = gemv_bytes_per_launch / (gemv_ms * 1e-3) / 1e9
    gemm_achieved = flops3 / launches3 / (gemm_ms * 1e-3) / 1e12
    out = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms1, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded Q4_K weights, N(0,1) activations)",
        "config": {"workload": f"{w1.name}: {launches1} Q4_K matrices, "
                               f"{bytes1 / 1e6:.1f} MB packed, M=1 fp32 activations",
                   "l2": "inputs larger than L2 (every step streams all weights from HBM)",
                   "launch": "one CUDA graph per sweep", "parallelism": f"replicas x{ws}"},
        "roofline": {"bound": "hbm", "kernel": "gemv_kernel<1,f32>",
                     "achieved": round(gemv_achieved, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(gemv_achieved / hbm, 4), "peak_source": f"{peak_kind} hbm_gbs",
                     "traffic": None,
                     "avg_launch_us": round(gemv_ms * 1e3, 3),
                     "algorithmic_bytes_per_launch": round(gemv_bytes_per_launch)},
        "gemm": {"metric": "GEMM TFLOP/s (M=512)", "value": round(gemm_tflops, 2), "unit": "TFLOP/s",
                 "workload": f"{w3.name}: {launches3} Q4_K matrices, {bytes3 / 1e9:.2f} GB packed, "
                             f"M={PREFILL_M} bf16 activations",
                 "ms_per_step": round(ms3, 4), "steps": max(1, args.steps // 4),
                 "roofline": {"bound": "tensor", "kernel": "gemm_kernel<256>",
                              "achieved": round(gemm_achieved, 1), "peak": bf16_peak,
                              "unit": "TFLOP/s", "frac": round(gemm_achieved / bf16_peak, 4),
                              "frac_of_sustained": (round(gemm_achieved / bf16_sust, 4)
                                                    if bf16_sust else None),
                              "peak_source": f"{peak_kind} bf16_tflops", "traffic": None,
                              "avg_launch_us": round(gemm_ms * 1e3, 2)}},
        "e2e": {"value": round(ws * bytes1 / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_ms, 4)},
        "gpu_launches": args.steps * launches1 + max(1, args.steps // 4) * launches3,
        "clocks": clocks,
        "device_error": err,
    }
    if ws == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_oracle_decode(args.cpu_budget, _host_cores())
    print(json.dumps(out))


def _offsets(mats):
    o, offs = 0, []
    for (_, N, _) in mats:
        offs.append(o)
        o += N
    return offs


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
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
