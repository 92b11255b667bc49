"""Benchmark of the fine-grained FP8 hot path on GB300.

Default workload (``--workload dense``): one step = 1x128 quantisation of the
activation X (bf16 -> E4M3 + FP32 scales) followed by the block-scaled FP8
GEMM Y = X W^T (bf16 out) for a dense projection with M = 4096 tokens and
K = N = 7168. X has log-normal per-channel magnitudes, W ~ N(0, 0.02) is
quantised once in 128x128 blocks before timing (weights change once per
optimiser step, not per GEMM). The metric is whole-job TFLOP/s (2*M*N*K per
step) on the device with inputs resident in HBM; ``e2e`` adds the
host->device copy of X and the device->host copy of Y (pinned host buffers)
inside the timed region, every step, with the copies and kernels of
consecutive steps overlapped on three streams.

Other workloads, one JSON line each, for the remaining kernels:
    trio      linear layer 7168 -> 18432 at M = 8192: weight quantise, X and
              dY quantised row-wise and transposed (both from one read),
              fprop, dgrad, wgrad
    moe       4096 tokens, 256 experts (2048 x 7168), top-8 with a Zipf(1.1)
              expert bias: X quantised 1x128 once per token and written to
              its 8 routed rows in expert order + grouped expert GEMM
    outliers  M = 16384 fprop with outlier channels and weight blocks
    tiny      128 x 256 x 128 fprop, FP32 out (latency)
    dense_e4m3  the dense step with the GEMM's output quantised 1x128 in its
              epilogue
    dense_mx, trio_mx, moe_mx  the dense, trio and MoE steps in the microscaling variant:
              power-of-two group scales, GEMMs on the tensor cores'
              block-scaled MMA (no per-block promotion)

Every kernel of a step is timed with CUDA events on the launching stream; L2
is flushed between steps (a 512 MiB write, then a 256 MiB read so that no
dirty lines are written back inside the next step), outside the events.

Usage:
    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload dense|trio|moe|moe_layer|outliers|tiny|dense_e4m3|dense_mx|trio_mx|moe_mx]
Under torchrun (N > 1) every rank runs its own replica of the workload
(weak scaling, no data-path collective); times are the max over ranks.
``--impl reference`` times the CPU oracle on a bounded sample of the same
workload (rank 0 only).
"""
import argparse
import hashlib
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

METRIC = "block-scaled FP8 GEMM TFLOP/s (% FP8 peak); quantize GB/s (% HBM)"
L2_FLUSH_BYTES = 512 << 20
L2_CLEAN_BYTES = 256 << 20
Q1X128_B = 2 + 1 + 4.0 / 128       # bytes per element: read bf16, write E4M3, one FP32 scale per 128
QDUAL_B = 2 + 2 * (1 + 4.0 / 128)  # one bf16 read, both layouts written
Q128X128_B = 2 + 1 + 4.0 / 16384   # one FP32 scale per 128x128 block

WORKLOADS = {
    "dense": "dense projection fprop: quant 1x128 + block-scaled GEMM, M=4096 K=7168 N=7168, bf16 out",
    "trio": "linear 7168->18432 at M=8192: quant W 128x128, X/dY 1x128 and transposed; fprop, dgrad, wgrad",
    "moe": "MoE experts: 4096 tokens, 256 experts 2048x7168, top-8 with Zipf(1.1) bias; quant X + grouped GEMM",
    "outliers": "outlier-heavy fprop: quant 1x128 + block-scaled GEMM, M=16384 K=7168 N=7168, bf16 out",
    "tiny": "tiny fprop: quant X 1x128 + quant W 128x128 + GEMM, 128x256x128, FP32 out",
    "dense_e4m3": "dense projection fprop, output quantised 1x128 in the GEMM epilogue (E4M3 + scales, the "
                  "next layer's input): quant X 1x128 + GEMM, M=4096 K=7168 N=7168",
    "dense_mx": "dense projection fprop, microscaling variant (power-of-two scales, tensor-core block "
                "scaling): quant 1x128 + GEMM, M=4096 K=7168 N=7168, bf16 out",
    "moe_layer": "MoE layer forward on one GPU: 4096 tokens, 256 experts 2048x7168, top-8 with Zipf(1.1) bias; "
                 "FP8 dispatch (each token quantised once into its 8 expert-order rows) + grouped GEMM + "
                 "gate-weighted combine of the 8 bf16 expert rows",
    "moe_mx": "MoE experts, microscaling variant (power-of-two scales, tensor-core block scaling): 4096 tokens, "
              "256 experts 2048x7168, top-8 with Zipf(1.1) bias; quant X into expert order + grouped GEMM",
    "trio_mx": "linear 7168->18432 at M=8192, microscaling variant (power-of-two scales, tensor-core block "
               "scaling): quant W 128x128, X/dY 1x128 and transposed; fprop, dgrad, wgrad",
}


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, 1900.0, "fallback"


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def reduce_max(values, pg):
    """Element-wise max of a list of floats over all ranks (identity without a group)."""
    if pg is None:
        return list(values)
    import torch
    backend = pg.get_backend()
    dev = torch.device("cuda", torch.cuda.current_device()) if backend == "nccl" else torch.device("cpu")
    t = torch.tensor(list(values), dtype=torch.float64, device=dev)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


class _NvmlClocks:
    """Read-only NVML queries through the driver's library (ctypes): the SM
    clock, its maximum, the power draw and the clock event reasons of one
    GPU. Unavailable (ok False) where the library cannot be loaded."""

    SM = 1  # NVML_CLOCK_SM
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown"}

    def __init__(self, index):
        import ctypes
        self.ct = ctypes
        self.ok = False
        try:
            self.lib = ctypes.CDLL("libnvidia-ml.so.1")
            if self.lib.nvmlInit_v2() != 0:
                return
            self.h = ctypes.c_void_p()
            if self.lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(self.h)) != 0:
                return
            self.reasons_fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
            mx = ctypes.c_uint()
            if self.lib.nvmlDeviceGetMaxClockInfo(self.h, self.SM, ctypes.byref(mx)) != 0:
                return
            self.max_mhz = mx.value
            self.ok = self.sample() is not None
        except (OSError, AttributeError):
            self.ok = False

    def sample(self):
        ct = self.ct
        clk, mw, rs = ct.c_uint(), ct.c_uint(), ct.c_ulonglong()
        if self.lib.nvmlDeviceGetClockInfo(self.h, self.SM, ct.byref(clk)) != 0:
            return None
        if self.reasons_fn(self.h, ct.byref(rs)) != 0:
            return None
        if self.lib.nvmlDeviceGetPowerUsage(self.h, ct.byref(mw)) != 0:
            mw.value = 0
        return clk.value, mw.value / 1000.0, rs.value

    def close(self):
        try:
            self.lib.nvmlShutdown()
        except (OSError, AttributeError):
            pass


class ClockSampler:
    """Clock and throttle-reason sampling around the timed region, each
    sample with its timestamp; the summary keeps only the samples taken
    inside it. Samples come from NVML every millisecond (a thread of this
    process, read-only queries), or, where NVML cannot be loaded, from
    nvidia-smi every 50 ms. Both write the same CSV rows."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NVML_PERIOD_S = 0.001

    def __init__(self, index, out_path=None):
        self.index = index
        if out_path is None:
            fd, out_path = tempfile.mkstemp(prefix="fp8fg_clocks_", suffix=".csv")
            os.close(fd)
            self.tmp = True
        else:
            self.tmp = False
        self.out_path = out_path
        self.proc = None
        self.f = None
        self.thread = None
        self.stop = None
        self.source = "unsampled"
        self.regions = []

    def _nvml_loop(self, nv):
        import datetime
        order = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        while not self.stop.is_set():
            t = time.time()
            r = nv.sample()
            if r is not None:
                clk, watts, mask = r
                seen = {name for bit, name in nv.REASONS.items() if mask & bit}
                stamp = datetime.datetime.fromtimestamp(t).strftime("%Y/%m/%d %H:%M:%S.%f")
                self.f.write("%s, %d, %d, %.2f, 0x%x, %s\n" % (
                    stamp, clk, nv.max_mhz, watts, mask,
                    ", ".join("Active" if n in seen else "Not Active" for n in order)))
            time.sleep(self.NVML_PERIOD_S)
        nv.close()

    def __enter__(self):
        import threading
        try:
            self.f = open(self.out_path, "w")
        except OSError:
            self.f = None
            return self
        nv = _NvmlClocks(self.index)
        if nv.ok:
            self.stop = threading.Event()
            self.thread = threading.Thread(target=self._nvml_loop, args=(nv,), daemon=True)
            self.thread.start()
            self.source = "NVML, every 1 ms"
        else:
            try:
                self.proc = subprocess.Popen(
                    ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                     "--format=csv,noheader,nounits", "-lms", "50"],
                    stdout=self.f, stderr=subprocess.DEVNULL)
                self.source = "nvidia-smi, every 50 ms"
            except OSError:
                self.proc = None
        time.sleep(0.3)
        return self

    def mark(self, t0, t1):
        """Host wall-clock bounds of one timed region."""
        self.regions.append((t0, t1))

    def __exit__(self, *a):
        if self.thread is not None:
            self.stop.set()
            self.thread.join(timeout=5)
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.f is not None:
            self.f.close()

    def summary(self, region=None):
        out = summarize_clocks(self.out_path, [region] if region else self.regions)
        out["source"] = self.source
        return out

    def cleanup(self):
        if self.tmp:
            try:
                os.unlink(self.out_path)
            except OSError:
                pass


def _stamp(text):
    """nvidia-smi timestamp (local time) -> seconds since the epoch."""
    import datetime
    for fmt in ("%Y/%m/%d %H:%M:%S.%f", "%Y/%m/%d %H:%M:%S"):
        try:
            return datetime.datetime.strptime(text.strip(), fmt).timestamp()
        except ValueError:
            continue
    return None


def summarize_clocks(path, regions):
    """Median SM clock, the maximum and every throttle reason seen, over the
    samples whose timestamp falls inside one of the timed regions. With no
    sample inside (a region shorter than the sampling interval), the clock
    is reported as None and the nearest samples (within 0.25 s of a region)
    are summarised separately, labelled as such."""
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    rows = []
    try:
        for line in open(path):
            parts = [q.strip() for q in line.split(",")]
            if len(parts) < 9:
                continue
            ts = _stamp(parts[0])
            try:
                sm, mx = float(parts[1]), float(parts[2])
            except ValueError:
                continue
            rows.append((ts, sm, mx, {n for n, v in zip(names, parts[5:9]) if v.lower() == "active"}))
    except OSError:
        pass

    def pick(slack):
        return [r for r in rows if r[0] is not None and any(a - slack <= r[0] <= b + slack for a, b in regions)]

    def summ(sel):
        return {"sm_mhz": statistics.median(r[1] for r in sel), "sm_max_mhz": max(r[2] for r in sel),
                "reasons": sorted(set().union(*(r[3] for r in sel))), "samples": len(sel)}

    if not rows:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
    inside = pick(0.0)
    timed_s = round(sum(b - a for a, b in regions), 4)
    if inside:
        out = summ(inside)
        out["timed_region_s"] = timed_s
        return out
    near = pick(0.25)
    out = {"sm_mhz": None, "sm_max_mhz": max(r[2] for r in rows), "reasons": [], "samples": 0,
           "timed_region_s": timed_s,
           "note": "no clock sample fell inside the timed region"}
    if near:
        out["within_0.25s_of_timed_region"] = summ(near)
    return out


# --------------------------------------------------------------- workloads ----

class Part:
    """One kernel of a step: a launch, its bound and its algorithmic units
    (bytes for HBM-bound kernels, flops for tensor-bound ones)."""

    def __init__(self, name, kernel, fn, bound, units, extra_bytes=None):
        self.name, self.kernel, self.fn, self.bound, self.units = name, kernel, fn, bound, units
        self.extra_bytes = extra_bytes   # grouped GEMM: bytes moved, reported beside the flops


def build(workload, dev, seed, fg, synth):
    """Device tensors, the step's parts, the metric's flops per step and the
    host copies of e2e (inputs to upload, outputs to download)."""
    import torch
    W = {}
    mx = workload.endswith("_mx")           # power-of-two scales, block-scaled MMA
    if mx:
        workload = workload[:-3]
    if workload in ("dense", "outliers", "tiny", "dense_e4m3"):
        if workload in ("dense", "dense_e4m3"):
            x, w = synth.dense(seed=seed, device=dev)
        elif workload == "outliers":
            x, w, _, _ = synth.outliers(seed=seed, device=dev)
        else:
            x, w = synth.tiny(seed=seed, device=dev)
        Mx, Kx = x.shape
        Nw = w.shape[0]
        out_dt = torch.float32 if workload == "tiny" else torch.bfloat16
        xq = torch.empty((Mx, Kx), dtype=torch.uint8, device=dev)
        sx = torch.empty((Kx // 128, (Mx + 3) // 4 * 4), dtype=torch.float32, device=dev)
        wq = torch.empty((Nw, Kx), dtype=torch.uint8, device=dev)
        sw = torch.empty((Nw // 128, Kx // 128), dtype=torch.float32, device=dev)
        y = torch.empty((Mx, Nw), dtype=out_dt, device=dev)
        parts = [Part("quant_x_1x128", "quant_rows_kernel",
                      lambda: fg.fp8_quant_1x128(x, q=xq, scales=sx, pow2=mx), "hbm", Q1X128_B * Mx * Kx)]
        if workload == "tiny":
            parts.append(Part("quant_w_128x128", "quant_blocks_kernel",
                              lambda: fg.fp8_quant_128x128(w, q=wq, scales=sw), "hbm", Q128X128_B * Nw * Kx))
        else:
            fg.fp8_quant_128x128(w, q=wq, scales=sw, pow2=mx)
        if workload == "dense_e4m3":
            yq = torch.empty((Mx, Nw), dtype=torch.uint8, device=dev)
            sy = torch.empty((Nw // 128, (Mx + 3) // 4 * 4), dtype=torch.float32, device=dev)
            parts.append(Part("fprop_e4m3", "gemm_kernel<FPROP, E4M3 out>",
                              lambda: fg.fp8_gemm_blockscaled_e4m3(fg.FPROP, xq, sx, wq, sw, c=yq, scales=sy),
                              "tensor", 2.0 * Mx * Nw * Kx))
            outs = [yq, sy]
        elif mx:
            parts.append(Part("fprop", "gemm_mx_kernel<FPROP>",
                              lambda: fg.fp8_gemm_mx(fg.FPROP, xq, sx, wq, sw, c=y), "tensor", 2.0 * Mx * Nw * Kx))
            outs = [y]
        else:
            parts.append(Part("fprop", "gemm_kernel<FPROP>", lambda: fg.fprop(xq, sx, wq, sw, c=y), "tensor",
                              2.0 * Mx * Nw * Kx))
            outs = [y]
        W.update(inputs=[x], outputs=outs, flops=2.0 * Mx * Nw * Kx,
                 dims={"M": Mx, "K": Kx, "N": Nw})
    elif workload == "trio":
        x, w, dy = synth.trio(seed=seed, device=dev)
        Mx, Kx = x.shape
        Nw = w.shape[0]
        wq = torch.empty((Nw, Kx), dtype=torch.uint8, device=dev)
        sw = torch.empty((Nw // 128, Kx // 128), dtype=torch.float32, device=dev)
        xq = torch.empty((Mx, Kx), dtype=torch.uint8, device=dev)
        sx = torch.empty((Kx // 128, Mx), dtype=torch.float32, device=dev)
        xqT = torch.empty((Kx, Mx), dtype=torch.uint8, device=dev)
        sxT = torch.empty((Mx // 128, Kx), dtype=torch.float32, device=dev)
        dyq = torch.empty((Mx, Nw), dtype=torch.uint8, device=dev)
        sdy = torch.empty((Nw // 128, Mx), dtype=torch.float32, device=dev)
        dyqT = torch.empty((Nw, Mx), dtype=torch.uint8, device=dev)
        sdyT = torch.empty((Mx // 128, Nw), dtype=torch.float32, device=dev)
        y = torch.empty((Mx, Nw), dtype=torch.bfloat16, device=dev)
        dx = torch.empty((Mx, Kx), dtype=torch.bfloat16, device=dev)
        dw = torch.empty((Nw, Kx), dtype=torch.float32, device=dev)
        f = 2.0 * Mx * Nw * Kx
        gemm = (lambda mode, *a, c: fg.fp8_gemm_mx(mode, *a, c=c)) if mx else \
            (lambda mode, *a, c: fg.fp8_gemm_blockscaled(mode, *a, c=c))
        gk = "gemm_mx_kernel" if mx else "gemm_kernel"
        parts = [
            Part("quant_w_128x128", "quant_blocks_kernel",
                 lambda: fg.fp8_quant_128x128(w, q=wq, scales=sw, pow2=mx), "hbm", Q128X128_B * Nw * Kx),
            # X and dY each read once for both layouts (1x128 rows for
            # fprop/dgrad, 128x1 transposed for wgrad)
            Part("quant_x_dual", "quant_dual_kernel",
                 lambda: fg.fp8_quant_1x128_dual(x, q=xq, scales=sx, qT=xqT, scalesT=sxT, pow2=mx), "hbm",
                 QDUAL_B * Mx * Kx),
            Part("quant_dy_dual", "quant_dual_kernel",
                 lambda: fg.fp8_quant_1x128_dual(dy, q=dyq, scales=sdy, qT=dyqT, scalesT=sdyT, pow2=mx), "hbm",
                 QDUAL_B * Mx * Nw),
            Part("fprop", gk + "<FPROP>", lambda: gemm(fg.FPROP, xq, sx, wq, sw, c=y), "tensor", f),
            Part("dgrad", gk + "<DGRAD>", lambda: gemm(fg.DGRAD, dyq, sdy, wq, sw, c=dx), "tensor", f),
            Part("wgrad", gk + "<WGRAD>", lambda: gemm(fg.WGRAD, dyqT, sdyT, xqT, sxT, c=dw), "tensor", f),
        ]
        W.update(inputs=[x, dy], outputs=[y, dx, dw], flops=3 * f, dims={"M": Mx, "K": Kx, "N": Nw})
    elif workload == "moe_layer":
        from fp8_fine_grained_gb300 import ep
        mo = synth.moe(seed=seed, device=dev, make_weights=False)
        E, Nw, Kx = 256, 2048, mo.x.shape[1]
        wq = torch.empty((E, Nw, Kx), dtype=torch.uint8, device=dev)
        sw = torch.empty((E, Nw // 128, Kx // 128), dtype=torch.float32, device=dev)
        g = torch.Generator(device=dev)
        g.manual_seed(seed + 1)
        for e in range(E):
            we = (torch.randn(Nw, Kx, generator=g, device=dev) * 0.02).to(torch.bfloat16)
            fg.fp8_quant_128x128(we, q=wq[e], scales=sw[e])
        T, topk = mo.topk_ids.shape
        plan = ep.plan_dispatch(mo.topk_ids, E, 1)      # rows by (expert, token): the routing's row order
        R = plan.n_send
        off = torch.zeros(E + 1, dtype=torch.int32, device=dev)
        off[1:] = torch.cumsum(plan.send_counts[0], 0).to(torch.int32)
        dest, gates = plan.dest, mo.gates
        xg = torch.empty((R, Kx), dtype=torch.uint8, device=dev)
        sxg = torch.empty((Kx // 128, R), dtype=torch.float32, device=dev)
        y = torch.empty((R, Nw), dtype=torch.bfloat16, device=dev)
        out = torch.empty((T, Nw), dtype=torch.bfloat16, device=dev)
        nonempty = int((plan.send_counts[0] > 0).sum().item())
        moved = nonempty * Nw * Kx + R * Kx + R * Nw * 2 + sw.numel() * 4 + R * (Kx // 128) * 4
        f = 2.0 * R * Nw * Kx
        parts = [
            Part("quant_x_scatter", "quant_rows_scatter_kernel",
                 lambda: fg.fp8_quant_1x128_scatter(mo.x, dest, R, q=xg, scales=sxg), "hbm",
                 2 * T * Kx + (Q1X128_B - 2) * R * Kx + 4 * R),
            Part("grouped", "gemm_kernel<GROUPED_C>",
                 lambda: fg.fp8_grouped_gemm(xg, sxg, None, off, wq, sw, R, y=y), "tensor", f, extra_bytes=moved),
            Part("combine", "moe_combine_kernel",
                 lambda: fg.fp8_moe_combine(y, dest, gates, out=out), "hbm", 2 * R * Nw + 2 * T * Nw + 8 * T * topk),
        ]
        W.update(inputs=[mo.x, dest, gates], outputs=[out], flops=f,
                 dims={"tokens": T, "experts": E, "N": Nw, "K": Kx, "rows": R, "nonempty_experts": nonempty})
    elif workload == "moe":
        mo = synth.moe(seed=seed, device=dev, make_weights=False)
        E, Nw, Kx = 256, 2048, mo.x.shape[1]
        # weights one expert at a time (bf16 for all 256 would be 7.5 GB)
        wq = torch.empty((E, Nw, Kx), dtype=torch.uint8, device=dev)
        sw = torch.empty((E, Nw // 128, Kx // 128), dtype=torch.float32, device=dev)
        g = torch.Generator(device=dev)
        g.manual_seed(seed + 1)
        for e in range(E):
            we = (torch.randn(Nw, Kx, generator=g, device=dev) * 0.02).to(torch.bfloat16)
            fg.fp8_quant_128x128(we, q=wq[e], scales=sw[e], pow2=mx)
        T = mo.x.shape[0]
        R = int(mo.expert_offsets[-1].item())
        # the routed rows are quantised straight into expert order (the
        # dispatch, in token order: each token read once and written to its
        # 8 rows), then each expert's GEMM reads contiguous 128-row tiles
        topk = R // T
        dest = torch.argsort(mo.row_index.long(), stable=True).to(torch.int32).reshape(T, topk).contiguous()
        xg = torch.empty((R, Kx), dtype=torch.uint8, device=dev)
        sxg = torch.empty((Kx // 128, R), dtype=torch.float32, device=dev)
        y = torch.empty((R, Nw), dtype=torch.bfloat16, device=dev)
        nonempty = int((mo.counts > 0).sum().item())
        moved = nonempty * Nw * Kx + R * Kx + R * Nw * 2 + sw.numel() * 4 + R * (Kx // 128) * 4
        f = 2.0 * R * Nw * Kx
        parts = [
            Part("quant_x_scatter", "quant_rows_scatter_kernel",
                 lambda: fg.fp8_quant_1x128_scatter(mo.x, dest, R, q=xg, scales=sxg, pow2=mx), "hbm",
                 2 * T * Kx + (Q1X128_B - 2) * R * Kx + 4 * R),
            Part("grouped", "gemm_mx_kernel<GROUPED_C>" if mx else "gemm_kernel<GROUPED_C>",
                 (lambda: fg.fp8_grouped_gemm_mx(xg, sxg, mo.expert_offsets, wq, sw, R, y=y)) if mx else
                 (lambda: fg.fp8_grouped_gemm(xg, sxg, None, mo.expert_offsets, wq, sw, R, y=y)), "tensor",
                 f, extra_bytes=moved),
        ]
        cnt = mo.counts.cpu()
        W.update(inputs=[mo.x, dest, mo.expert_offsets], outputs=[y], flops=f,
                 dims={"tokens": T, "experts": E, "N": Nw, "K": Kx, "rows": R, "nonempty_experts": nonempty,
                       "rows_per_expert_max": int(cnt.max()), "rows_per_expert_median": float(cnt.float().median())})
    else:
        raise ValueError(workload)
    W["parts"] = parts
    return W


# ------------------------------------------------------------------ timing ----

def kernel_source_sha():
    """Hash of every kernel and host source of the library (file names and
    contents, in name order)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "fp8_fine_grained_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f.endswith((".cu", ".cuh", ".h", ".cpp")):
            h.update(f.encode())
            with open(os.path.join(csrc, f), "rb") as fh:
                h.update(fh.read())
    return h.hexdigest()[:16]


def load_traffic(workload):
    """DRAM bytes per launch from the committed ncu capture, or {} when the
    kernel sources changed since the counters were taken."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return {}
    if d.get("source_sha") != kernel_source_sha():
        return {}
    return d.get(workload, {})


def time_parts(W, args, pg, clocks, stream, flush_l2):
    """W untimed warm-up steps, then exactly K timed steps of the workload
    with one CUDA event pair around each whole step (the parts back to
    back, as an application runs them: consecutive kernels may overlap
    their launch and set-up), L2 flushed before every step outside the
    events. Then K more steps with an event after every part, for the
    per-kernel breakdown (events between kernels add about 2 us each and
    stop that overlap). Returns the mean ms of every part and of the whole
    step (max over ranks) and the host bounds of the first timed region."""
    import torch

    import fp8_fine_grained_gb300 as fg
    parts = W["parts"]
    n = len(parts)
    # warm-up right before the timed loop (after the clock sampler started),
    # so that clocks and memory are at their working state when timing starts
    for _ in range(args.warmup):
        flush_l2()
        for p_ in parts:
            p_.fn()
    torch.cuda.synchronize()
    if fg.device_status() != 0:
        raise RuntimeError("device status after warm-up")
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    whole = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    t0 = time.time()
    for i in range(args.steps):
        flush_l2()                           # outside the events
        whole[i][0].record(stream)
        for p_ in parts:
            p_.fn()
        whole[i][1].record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    clocks.mark(t0, t1)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(n + 1)] for _ in range(args.steps)]
    for i in range(args.steps):
        flush_l2()
        ev[i][0].record(stream)
        for j, p_ in enumerate(parts):
            p_.fn()
            ev[i][j + 1].record(stream)
    torch.cuda.synchronize()
    clocks.mark(t1, time.time())
    if pg:
        pg.barrier()
    if fg.device_status() != 0:
        raise RuntimeError("device status after timing")
    step_ms = sum(whole[i][0].elapsed_time(whole[i][1]) for i in range(args.steps)) / args.steps
    part_ms = [sum(ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(args.steps)) / args.steps
               for j in range(n)]
    vals = reduce_max(part_ms + [step_ms], pg)
    return vals[:n], vals[n], (t0, t1)


def kernel_entries(parts, part_ms, traffic, hbm, fp8_peak):
    """Per part: time, achieved rate against its roofline, DRAM traffic."""
    kernels = []
    for p_, ms in zip(parts, part_ms):
        if p_.bound == "hbm":
            ach, peak, unit = p_.units / (ms * 1e-3) / 1e9, hbm, "GB/s"
        else:
            ach, peak, unit = p_.units / (ms * 1e-3) / 1e12, fp8_peak, "TFLOP/s"
        k = {"part": p_.name, "kernel": p_.kernel, "ms": round(ms, 4), "bound": p_.bound,
             "achieved": round(ach, 1), "peak": round(peak, 1), "unit": unit, "frac": round(ach / peak, 4),
             "traffic": traffic.get(p_.name)}
        if p_.extra_bytes:
            gbs = p_.extra_bytes / (ms * 1e-3) / 1e9
            k["bytes"] = int(p_.extra_bytes)
            k["achieved_gbs"] = round(gbs, 1)
            k["frac_hbm"] = round(gbs / hbm, 4)
        kernels.append(k)
    return kernels


def e2e_run(W, args, dev, rank, fg, synth, pg):
    """End to end through the public API: every step uploads its inputs from
    pinned host memory, runs the step and reads its outputs back into
    pinned host memory. Two copies of the workload's device buffers and
    three streams let step i's upload, step i-1's kernels and step i-2's
    read-back run at the same time (as a data loader feeding a training or
    serving loop does); each step still moves all of its bytes."""
    import torch
    sets = [W, build(args.workload, dev, rank, fg, synth)]
    hin = [t.cpu().pin_memory() for t in W["inputs"]]
    hout = [[torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in S["outputs"]] for S in sets]
    s_in, s_cmp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    in_done = [torch.cuda.Event() for _ in sets]
    cmp_done = [torch.cuda.Event() for _ in sets]
    out_done = [torch.cuda.Event() for _ in sets]
    for k in range(len(sets)):      # all slots start free
        cmp_done[k].record(s_cmp)
        out_done[k].record(s_out)

    def e2e_step(i):
        k = i % len(sets)
        S = sets[k]
        s_in.wait_event(cmp_done[k])            # the slot's inputs are no longer read
        with torch.cuda.stream(s_in):
            for d, h in zip(S["inputs"], hin):
                d.copy_(h, non_blocking=True)
            in_done[k].record(s_in)
        s_cmp.wait_event(in_done[k])
        s_cmp.wait_event(out_done[k])           # the slot's outputs have been read back
        with torch.cuda.stream(s_cmp):
            for p_ in S["parts"]:
                p_.fn()
            cmp_done[k].record(s_cmp)
        s_out.wait_event(cmp_done[k])
        with torch.cuda.stream(s_out):
            for d, h in zip(S["outputs"], hout[k]):
                h.copy_(d, non_blocking=True)
            out_done[k].record(s_out)

    for i in range(max(2, args.warmup)):
        e2e_step(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_steps = max(2, min(args.steps, 200))
    if pg:
        pg.barrier()
    e0.record(s_in)
    for i in range(e2e_steps):
        e2e_step(i)
    s_out.wait_stream(s_in)
    s_out.wait_stream(s_cmp)
    e1.record(s_out)
    torch.cuda.synchronize()
    if fg.device_status() != 0:
        raise RuntimeError("device status after the end-to-end steps")
    ms = reduce_max([e0.elapsed_time(e1) / e2e_steps], pg)[0]
    del sets
    return {"ms": ms, "h2d": sum(t.numel() * t.element_size() for t in W["inputs"]),
            "d2h": sum(t.numel() * t.element_size() for t in W["outputs"])}


# the five workloads of the measurement plan; the headline is one of them,
# the others are reported under "configs" on the same line
CONFIG_SET = ("tiny", "dense", "trio", "moe", "moe_layer", "outliers")


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
        dist.init_process_group("nccl")
        pg = dist

    hbm, bf16, peak_kind = peaks()
    fp8_peak = 2.0 * bf16   # nominal FP8/BF16 dense ratio 4.5/2.25 on the measured BF16 burst
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    clean = torch.ones(L2_CLEAN_BYTES // 4, dtype=torch.float32, device=dev)
    sink = torch.empty((), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def flush_l2():
        flush.zero_()
        torch.sum(clean, dim=0, out=sink)

    clocks = ClockSampler(local, args.clock_log)
    W = build(args.workload, dev, rank, fg, synth)
    parts = W["parts"]
    flops, dims = W["flops"], W["dims"]
    n = len(parts)
    with clocks:
        part_ms, ms_step, region = time_parts(W, args, pg, clocks, stream, flush_l2)
    clk = clocks.summary(region)

    e2e = e2e_run(W, args, dev, rank, fg, synth, pg) if args.workload in WORKLOADS else None
    value = world * flops / (ms_step * 1e-3) / 1e12

    # the other workloads of the measurement plan, each timed the same way
    configs = {}
    if not args.headline_only and args.workload in CONFIG_SET:
        del W
        torch.cuda.empty_cache()
        for name in CONFIG_SET:
            if name == args.workload:
                continue
            Wc = build(name, dev, rank, fg, synth)
            cclk = ClockSampler(local)
            with cclk:
                cms, cstep, creg = time_parts(Wc, args, pg, cclk, stream, flush_l2)
            kern = kernel_entries(Wc["parts"], cms, load_traffic(name), hbm, fp8_peak)
            dom = max(range(len(cms)), key=lambda j: cms[j])
            configs[name] = {"workload": WORKLOADS[name], "ms_per_step": round(cstep, 4),
                             "sum_of_parts_ms": round(sum(cms), 4),
                             "value": round(world * Wc["flops"] / (cstep * 1e-3) / 1e12, 2),
                             "unit": "TFLOP/s", "dims": Wc["dims"],
                             "roofline": {k: kern[dom][k] for k in ("kernel", "bound", "achieved", "peak", "unit",
                                                                    "frac", "traffic")},
                             "kernels": kern, "clocks": cclk.summary(creg),
                             "gpu_launches": len(Wc["parts"]) * args.steps}
            cclk.cleanup()
            del Wc
            torch.cuda.empty_cache()
    clocks.cleanup()

    if rank != 0:
        if pg:
            pg.destroy_process_group()
        return None

    traffic = load_traffic(args.workload)
    kernels = kernel_entries(parts, part_ms, traffic, hbm, fp8_peak)
    dom = max(range(n), key=lambda j: part_ms[j])
    dk = kernels[dom]
    roofline = {"bound": dk["bound"], "kernel": dk["kernel"], "achieved": dk["achieved"], "peak": dk["peak"],
                "unit": dk["unit"], "frac": dk["frac"], "traffic": dk["traffic"],
                "peak_source": ("%s HBM copy" % peak_kind) if dk["bound"] == "hbm" else
                ("%s bf16 burst %.0f TFLOP/s x 2 (nominal FP8/BF16 ratio)" % (peak_kind, bf16))}
    if "frac_hbm" in dk:
        roofline.update(achieved_gbs=dk["achieved_gbs"], frac_hbm=dk["frac_hbm"], hbm_peak=hbm)
    quant = next((k for k in kernels if k["part"].startswith("quant_x")), None)
    if quant is not None and n == 2:
        # quantise + one GEMM: what the quantiser adds to the step beyond the
        # GEMM's own time (the GEMM is launched under the quantiser's tail)
        gemm_ms = part_ms[1 - parts.index(next(p_ for p_ in parts if p_.name.startswith("quant_x")))]
        quant = dict(quant, step_minus_gemm_us=round((ms_step - gemm_ms) * 1e3, 1),
                     step_minus_gemm_note="whole-step time minus the GEMM's own event time: the quantiser "
                                          "and the launch gap; the GEMM sets itself up under the quantiser's "
                                          "last wave (programmatic dependent launch)")
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 4),
        "timing": "value and ms_per_step: one CUDA event pair around each of the K whole steps; "
                  "kernels: K further steps with an event after every part (sum_of_parts_ms)",
        "sum_of_parts_ms": round(sum(part_ms), 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "e4m3 x e4m3 -> f32 accumulate",
        "data": "synthetic (seeded torch Philox; shapes and distributions of the workload)",
        "config": config_of(args.workload, world),
        "dims": dims,
        "roofline": roofline,
        "quant": quant,
        "kernels": kernels,
        "clocks": clk,
        "gpu_launches": n * args.steps,
        "gpu_launches_breakdown_pass": n * args.steps,
    }
    if e2e:
        line["e2e"] = {"value": round(world * flops / (e2e["ms"] * 1e-3) / 1e12, 2),
                       "unit": "TFLOP/s", "h2d_bytes_per_step": e2e["h2d"], "d2h_bytes_per_step": e2e["d2h"],
                       "ms_per_step": round(e2e["ms"], 4),
                       "pipeline": "upload, kernels and read-back of consecutive steps overlap "
                                   "(two buffer sets, three streams)"}
    if configs:
        line["configs"] = configs
    if args.workload in ("dense", "dense_mx", "dense_e4m3"):
        ref = cublas_fp8_reference(dev)
        line["fp8_cublas_reference"] = ref
        if ref.get("tflops"):
            line["fp8_cublas_reference"]["gemm_vs_cublas"] = round(dk["achieved"] / ref["tflops"], 4)
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.workload, budget_s=args.cpu_seconds)
    print(json.dumps(line), flush=True)
    if pg:
        pg.destroy_process_group()
    return line


def cublas_fp8_reference(dev, M=4096, N=7168, K=7168, steps=20):
    """Context for the FP8 peak: cuBLAS's per-tensor-scaled FP8 GEMM
    (torch._scaled_mm, E4M3 x E4M3 -> bf16, no block scales and no
    promotion) on the dense shape, TFLOP/s from CUDA events, L2 flushed
    between calls. None where the call is unavailable."""
    import torch
    try:
        g = torch.Generator(device=dev)
        g.manual_seed(0)
        a = torch.randn(M, K, generator=g, device=dev).to(torch.float8_e4m3fn)
        b = torch.randn(N, K, generator=g, device=dev).to(torch.float8_e4m3fn).t()
        one = torch.ones((), dtype=torch.float32, device=dev)
        flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

        def call():
            return torch._scaled_mm(a, b, scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
        for _ in range(3):
            call()
        ts = []
        for _ in range(steps):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            call()
            e1.record()
            ts.append((e0, e1))
        torch.cuda.synchronize()
        ms = sum(x.elapsed_time(y) for x, y in ts) / steps
        return {"tflops": round(2.0 * M * N * K / (ms * 1e-3) / 1e12, 1), "ms": round(ms, 4),
                "what": "torch._scaled_mm (cuBLAS), per-tensor scales, %dx%dx%d, bf16 out; context only, "
                        "not the roofline denominator" % (M, N, K)}
    except Exception as e:  # the call is missing or unsupported on this build
        return {"tflops": None, "why": type(e).__name__}


def config_of(workload, world):
    """The workload's config object, printed identically by both arms."""
    M, K, N = oracle_dims(workload)
    return {"workload": WORKLOADS[workload],
            "l2": "flushed between steps (512 MiB write + 256 MiB read, outside the timed region)",
            "parallelism": "replica per GPU" if world > 1 else "single GPU", "M": M, "K": K, "N": N}


# -------------------------------------------------------------- CPU oracle ----

def oracle_dims(workload):
    """(M, K, N) of the workload's first GEMM, the one the CPU sample runs."""
    return {"dense": (4096, 7168, 7168), "dense_e4m3": (4096, 7168, 7168), "outliers": (16384, 7168, 7168),
            "trio": (8192, 7168, 18432), "moe": (32768, 7168, 2048), "moe_layer": (32768, 7168, 2048),
            "tiny": (128, 256, 128),
            "dense_mx": (4096, 7168, 7168), "trio_mx": (8192, 7168, 18432), "moe_mx": (32768, 7168, 2048)}[workload]


def cpu_sample(workload, rows, seed=0):
    """Oracle on a bounded sample of the workload: 1x128 quantisation of
    ``rows`` activation rows and their rows of the first GEMM against the
    full pre-quantised weight. Returns (seconds, flops, threads)."""
    import torch

    import oracle
    from fp8_fine_grained_gb300 import synth

    M, K, N = oracle_dims(workload)
    pow2 = workload.endswith("_mx")
    rows = min(rows, M)
    g = torch.Generator()
    g.manual_seed(seed)
    c = torch.exp(torch.randn(K, generator=g))
    xs = (torch.randn(rows, K, generator=g) * c).to(torch.bfloat16)
    w = (torch.randn(N, K, generator=g) * 0.02).to(torch.bfloat16)
    wq, sw = oracle.quant_128x128(synth.bf16_bits(w), pow2=pow2)
    xb = synth.bf16_bits(xs)
    t0 = time.perf_counter()
    xq, sx = oracle.quant_1x128(xb, pow2=pow2)
    oracle.fprop(xq, sx, wq, sw, want_exact=False)
    dt = time.perf_counter() - t0
    return dt, 2.0 * rows * N * K, oracle.num_threads()


def cpu_baseline(workload, budget_s=15.0, single_s=None):
    """The oracle on a bounded sample of the workload, on all host cores,
    and (``single_thread``) on one core over a smaller sample."""
    import oracle

    M, K, N = oracle_dims(workload)
    dt, fl, th = cpu_sample(workload, 8)
    rows = max(8, min(M, int(8 * budget_s / max(dt, 1e-3))))
    dt, fl, th = cpu_sample(workload, rows)
    out = {"value": round(fl / dt / 1e12, 6), "unit": "TFLOP/s", "cores": th, "kind": "oracle",
           "sample": "%d of %d rows of X quantised 1x128 and multiplied by the full %dx%d W "
                     "(W quantised outside the timing); %.1f s" % (rows, M, N, K, dt)}
    single_s = budget_s / 3 if single_s is None else single_s
    per_row = dt / rows * th  # one core, if the oracle scales with its threads
    rows1 = max(1, min(M, int(single_s / max(per_row, 1e-6))))
    oracle.set_num_threads(1)
    try:
        dt1, fl1, th1 = cpu_sample(workload, rows1)
    finally:
        oracle.set_num_threads(th)
    out["single_thread"] = {"value": round(fl1 / dt1 / 1e12, 6), "cores": th1,
                            "sample": "%d rows; %.1f s" % (rows1, dt1)}
    return out


def run_reference(args):
    world, rank, local = dist_env()
    if rank != 0:
        return None
    # keep the whole run (warm-up and timed steps) to about two minutes
    budget = max(0.5, min(20.0, args.cpu_seconds, 120.0 / max(1, args.steps + args.warmup)))
    M, K, N = oracle_dims(args.workload)
    dt, fl, th = cpu_sample(args.workload, 4)
    rows = max(4, min(M, int(4 * budget / max(dt, 1e-3))))
    for _ in range(args.warmup):
        cpu_sample(args.workload, min(rows, 8))
    times = []
    for i in range(args.steps):
        dt, fl, th = cpu_sample(args.workload, rows, seed=i)
        times.append(dt)
    ms = 1e3 * sum(times) / len(times)
    value = fl / (ms * 1e-3) / 1e12
    line = {
        "metric": METRIC, "impl": "reference", "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e4m3 x e4m3 -> f64 block sums, f32 accumulate",
        "data": "synthetic (seeded)",
        "config": config_of(args.workload, world),
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": th, "kind": "oracle",
                         "sample": "per step %d of %d rows of X, quantised and multiplied by the full W" % (rows, M)},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return line


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=None)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="dense")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--headline-only", action="store_true",
                    help="time only --workload (skip the other workloads under \"configs\")")
    ap.add_argument("--clock-log", default=None,
                    help="keep the nvidia-smi clock samples in this file (default: a temporary file)")
    args = ap.parse_args()
    if args.impl == "reference":
        args.steps = 3 if args.steps is None else args.steps
        args.warmup = 1 if args.warmup is None else args.warmup
        run_reference(args)
        return
    # the default timed region lasts about a second so that clock samples land in it
    args.steps = 2000 if args.steps is None else args.steps
    args.warmup = 20 if args.warmup is None else args.warmup
    if args.warmup < 3:
        args.warmup = 3
    run_ours(args)


if __name__ == "__main__":
    main()
