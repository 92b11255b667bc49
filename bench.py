"""Benchmark of the fine-grained FP8 hot path on GB300.

One step = 1x128 quantisation of the activation X (bf16 -> E4M3 + FP32
scales) followed by the block-scaled FP8 GEMM Y = X W^T (bf16 out), on the
dense projection workload: M = 4096 tokens, K = N = 7168, X with log-normal
per-channel magnitudes, W ~ N(0, 0.02) quantised once in 128x128 blocks
before timing (weights change once per optimiser step, not per GEMM). The
metric is whole-job TFLOP/s (2*M*N*K per step) on the device with inputs
resident in HBM; ``e2e`` adds the host->device copy of X and the
device->host copy of Y (pinned host buffers) inside the timed region.

Usage:
    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun (N > 1) every rank runs its own replica of the workload
(weak scaling, no data-path collective); the step time is the max over ranks.
``--impl reference`` times the CPU oracle on a bounded sample of the same
workload (rank 0 only).
"""
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

METRIC = "block-scaled FP8 GEMM TFLOP/s (% FP8 peak); quantize GB/s (% HBM)"
M, K, N = 4096, 7168, 7168
WORKLOAD = "dense projection fprop: quant 1x128 + block-scaled GEMM, M=4096 K=7168 N=7168, bf16 out"
L2_FLUSH_BYTES = 512 << 20
QUANT_BYTES_PER_ELEM = 2 + 1 + 4.0 / 128      # read bf16, write E4M3, write one FP32 scale per 128


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, 1900.0, 1700.0, "fallback"


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


class ClockSampler:
    """nvidia-smi clock/throttle sampling during the timed region."""

    def __init__(self, index, out_path):
        self.index = index
        self.out_path = out_path
        self.proc = None

    def __enter__(self):
        try:
            self.f = open(self.out_path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index),
                 "--query-gpu=clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                 "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                 "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        self.f.close()

    def summary(self):
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        try:
            for line in open(self.out_path):
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 8:
                    continue
                try:
                    sm.append(float(parts[0]))
                    mx = max(mx, float(parts[1]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[4:8]):
                    if v.lower() == "active":
                        reasons.add(n)
        except OSError:
            pass
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        loaded = [v for v in sm if v > 0.5 * mx] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def run_ours(args):
    import torch

    import fp8_fine_grained_gb300 as fg
    from fp8_fine_grained_gb300 import synth

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
        pg = dist

    x, w = synth.dense(seed=rank, device=dev, M=M, K=K, N=N)
    wq, sw = fg.fp8_quant_128x128(w)
    del w
    xq = torch.empty((M, K), dtype=torch.uint8, device=dev)
    sx = torch.empty((K // 128, M), dtype=torch.float32, device=dev)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        fg.fp8_quant_1x128(x, q=xq, scales=sx)
        fg.fprop(xq, sx, wq, sw, c=y)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if fg.device_status() != 0:
        raise RuntimeError("device status after warm-up")

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    hbm, bf16_burst, bf16_sust, peak_kind = peaks()
    clocks = ClockSampler(local, os.path.join(ROOT, "gpurun_out", "bench_clocks_rank%d.csv" % rank)
                          if os.path.isdir(os.path.join(ROOT, "gpurun_out")) else "/tmp/fp8fg_clocks_%d.csv" % rank)
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    with clocks:
        for i in range(args.steps):
            flush.zero_()                       # evict L2 between steps (outside the events)
            ev[i][0].record(stream)
            fg.fp8_quant_1x128(x, q=xq, scales=sx)
            ev[i][1].record(stream)
            fg.fprop(xq, sx, wq, sw, c=y)
            ev[i][2].record(stream)
        torch.cuda.synchronize()
    if pg:
        pg.barrier()
    if fg.device_status() != 0:
        raise RuntimeError("device status after timing")
    t_quant = [ev[i][0].elapsed_time(ev[i][1]) for i in range(args.steps)]
    t_gemm = [ev[i][1].elapsed_time(ev[i][2]) for i in range(args.steps)]
    t_step = [a + b for a, b in zip(t_quant, t_gemm)]
    ms_step = sum(t_step) / len(t_step)
    ms_quant = sum(t_quant) / len(t_quant)
    ms_gemm = sum(t_gemm) / len(t_gemm)

    # end to end through the public API: pinned host X in, pinned host Y out
    xh = x.cpu().pin_memory()
    yh = torch.empty((M, N), dtype=torch.bfloat16).pin_memory()
    xd = torch.empty_like(x)

    def e2e_step():
        xd.copy_(xh, non_blocking=True)
        fg.fp8_quant_1x128(xd, q=xq, scales=sx)
        fg.fprop(xq, sx, wq, sw, c=y)
        yh.copy_(y, non_blocking=True)

    for _ in range(max(1, args.warmup)):
        e2e_step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if pg:
        pg.barrier()
    e0.record(stream)
    for _ in range(args.steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    ms_e2e = e0.elapsed_time(e1) / args.steps

    if pg:
        t = torch.tensor([ms_step, ms_e2e, ms_gemm, ms_quant], dtype=torch.float64, device=dev)
        pg.all_reduce(t, op=pg.ReduceOp.MAX)
        ms_step, ms_e2e, ms_gemm, ms_quant = [float(v) for v in t.tolist()]

    flops = 2.0 * M * N * K
    fp8_peak = 2.0 * bf16_burst           # nominal FP8/BF16 dense ratio 4.5/2.25 on the measured BF16 burst
    gemm_tflops = flops / (ms_gemm * 1e-3) / 1e12
    quant_gbs = QUANT_BYTES_PER_ELEM * M * K / (ms_quant * 1e-3) / 1e9
    value = world * flops / (ms_step * 1e-3) / 1e12
    e2e_value = world * flops / (ms_e2e * 1e-3) / 1e12

    if rank != 0:
        if pg:
            pg.destroy_process_group()
        return None

    traffic = load_traffic()
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "e4m3 x e4m3 -> f32 accumulate, bf16 out",
        "data": "synthetic (seeded: X log-normal channels, W ~ N(0,0.02))",
        "config": {"workload": WORKLOAD, "M": M, "K": K, "N": N, "l2": "flushed between steps (512 MiB write)",
                   "weights": "pre-quantised 128x128 outside the timed region",
                   "parallelism": "replica per GPU" if world > 1 else "single GPU"},
        "roofline": {"bound": "tensor", "kernel": "gemm_kernel<FPROP,bf16>",
                     "achieved": round(gemm_tflops, 1), "peak": round(fp8_peak, 1), "unit": "TFLOP/s",
                     "frac": round(gemm_tflops / fp8_peak, 4),
                     "peak_source": "%s bf16 burst %.0f TFLOP/s x 2 (nominal FP8/BF16 ratio)" % (peak_kind, bf16_burst),
                     "traffic": traffic.get("gemm")},
        "quant": {"kernel": "quant_rows_kernel", "ms": round(ms_quant, 4), "achieved": round(quant_gbs, 1),
                  "peak": hbm, "unit": "GB/s", "frac": round(quant_gbs / hbm, 4), "bound": "hbm",
                  "bytes_per_elem": QUANT_BYTES_PER_ELEM, "peak_source": peak_kind, "traffic": traffic.get("quant")},
        "gemm_ms": round(ms_gemm, 4),
        "clocks": clocks.summary(),
        "e2e": {"value": round(e2e_value, 2), "unit": "TFLOP/s", "h2d_bytes_per_step": M * K * 2,
                "d2h_bytes_per_step": M * N * 2, "ms_per_step": round(ms_e2e, 4)},
        "gpu_launches": 2 * args.steps,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(budget_s=args.cpu_seconds)
    print(json.dumps(line), flush=True)
    if pg:
        pg.destroy_process_group()
    return line


def kernel_source_sha():
    import hashlib
    h = hashlib.sha256()
    for f in ("gemm.cu", "quant.cu", "ptx.cuh"):
        with open(os.path.join(ROOT, "fp8_fine_grained_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def load_traffic():
    """DRAM bytes per launch from the committed ncu capture, or {} when the
    kernel sources changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return {}
    return d if d.get("source_sha") == kernel_source_sha() else {}


def cpu_sample(rows, seed=0):
    """Oracle on a bounded sample of the workload: 1x128 quantisation of
    ``rows`` rows of X and their GEMM rows against the full pre-quantised W.
    Returns (seconds, flops, threads)."""
    import numpy as np
    import torch

    import oracle
    from fp8_fine_grained_gb300 import synth

    g = torch.Generator()
    g.manual_seed(seed)
    c = torch.exp(torch.randn(K, generator=g))
    xs = (torch.randn(rows, K, generator=g) * c).to(torch.bfloat16)
    w = (torch.randn(N, K, generator=g) * 0.02).to(torch.bfloat16)
    wq, sw = oracle.quant_128x128(synth.bf16_bits(w))
    xb = synth.bf16_bits(xs)
    t0 = time.perf_counter()
    xq, sx = oracle.quant_1x128(xb)
    oracle.fprop(xq, sx, wq, sw, want_exact=False)
    dt = time.perf_counter() - t0
    return dt, 2.0 * rows * N * K, oracle.num_threads()


def cpu_baseline(budget_s=15.0):
    dt, fl, th = cpu_sample(8)
    rows = max(8, min(4096, int(8 * budget_s / max(dt, 1e-3))))
    dt, fl, th = cpu_sample(rows)
    return {"value": round(fl / dt / 1e12, 6), "unit": "TFLOP/s", "cores": th, "kind": "oracle",
            "sample": "%d of %d rows of X quantised 1x128 and multiplied by the full 7168x7168 W "
                      "(W quantised outside the timing); %.1f s" % (rows, M, dt)}


def run_reference(args):
    world, rank, local = dist_env()
    if rank != 0:
        return None
    budget = max(1.0, min(20.0, args.cpu_seconds))
    # size one step so that warmup + steps stay within a few minutes
    dt, fl, th = cpu_sample(4)
    rows = max(4, min(4096, int(4 * budget / max(dt, 1e-3))))
    for _ in range(args.warmup):
        cpu_sample(min(rows, 8))
    times = []
    for i in range(args.steps):
        dt, fl, th = cpu_sample(rows, seed=i)
        times.append(dt)
    ms = 1e3 * sum(times) / len(times)
    value = fl / (ms * 1e-3) / 1e12
    line = {
        "metric": METRIC, "impl": "reference", "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e4m3 x e4m3 -> f64 block sums, f32 accumulate",
        "data": "synthetic (seeded)",
        "config": {"workload": WORKLOAD, "M": M, "K": K, "N": N},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": th, "kind": "oracle",
                         "sample": "per step %d of %d rows of X, quantised and multiplied by the full W" % (rows, M)},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return line


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
