"""Host-side logic of bench.py (no GPU): clock-log parsing, the traffic
lookup keyed by the kernel sources, and the max-over-ranks reduction run as
two gloo ranks on the CPU."""
import json
import os

import pytest
import torch.multiprocessing as mp

import bench


def _clock_lines():
    return "\n".join([
        "2026/12/02 10:00:00.000, 1995, 2070, 180.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "2026/12/02 10:00:00.050, 2070, 2070, 900.5, 0x0, Not Active, Not Active, Not Active, Not Active",
        "2026/12/02 10:00:00.100, 1950, 2070, 1390.0, 0x4, Not Active, Not Active, Not Active, Active",
        "2026/12/02 10:00:00.150, 1995, 2070, 200.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "garbage line",
    ])


def test_clock_summary_keeps_only_samples_inside_the_timed_region(tmp_path):
    p = tmp_path / "c.csv"
    p.write_text(_clock_lines())
    t = bench._stamp("2026/12/02 10:00:00.000")
    s = bench.summarize_clocks(str(p), [(t + 0.04, t + 0.11)])
    assert s["samples"] == 2              # the idle samples before and after are left out
    assert s["sm_max_mhz"] == 2070
    assert s["sm_mhz"] == 2010.0          # median of the two samples inside
    assert s["reasons"] == ["sw_power_cap"]


def test_clock_summary_says_so_when_no_sample_is_inside(tmp_path):
    p = tmp_path / "c.csv"
    p.write_text(_clock_lines())
    t = bench._stamp("2026/12/02 10:00:00.000")
    s = bench.summarize_clocks(str(p), [(t + 0.06, t + 0.08)])   # 20 ms, between two samples
    assert s["samples"] == 0 and s["sm_mhz"] is None and "no clock sample" in s["note"]
    assert s["within_0.25s_of_timed_region"]["samples"] == 4


def test_clock_summary_without_samples(tmp_path):
    s = bench.summarize_clocks(str(tmp_path / "missing.csv"), [(0.0, 1.0)])
    assert s["samples"] == 0 and s["reasons"] == ["unsampled"]


def test_both_arms_print_the_same_config():
    for w in bench.WORKLOADS:
        assert bench.config_of(w, 1) == bench.config_of(w, 1)
    src = open(bench.__file__).read()
    assert src.count('"config": config_of(args.workload, world)') == 2


def test_traffic_lookup_follows_kernel_sources(tmp_path, monkeypatch):
    prof = tmp_path / "profiles"
    prof.mkdir()
    (tmp_path / "fp8_fine_grained_gb300").mkdir()
    (tmp_path / "fp8_fine_grained_gb300" / "csrc").symlink_to(os.path.join(bench.ROOT, "fp8_fine_grained_gb300", "csrc"))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    sha = bench.kernel_source_sha()
    (prof / "traffic.json").write_text(json.dumps({"source_sha": sha, "dense": {"fprop": 123}}))
    assert bench.load_traffic("dense") == {"fprop": 123}
    (prof / "traffic.json").write_text(json.dumps({"source_sha": "0" * 16, "dense": {"fprop": 123}}))
    assert bench.load_traffic("dense") == {}


def test_workload_catalogue_matches_oracle_dims():
    for w in bench.WORKLOADS:
        M, K, N = bench.oracle_dims(w)
        assert K % 128 == 0 and N % 128 == 0 and M > 0


def _rank(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    vals = bench.reduce_max([1.0 + rank, 10.0 - rank, 0.5 * rank], dist)
    out[rank] = vals
    dist.destroy_process_group()


def test_reduce_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert out[0] == out[1] == [2.0, 10.0, 0.5]


def test_reduce_max_single_process_is_identity():
    assert bench.reduce_max([3.0, 1.0], None) == [3.0, 1.0]


def test_cpu_baseline_reports_all_cores_and_one_core():
    cb = bench.cpu_baseline("tiny", budget_s=0.3, single_s=0.1)
    assert cb["kind"] == "oracle" and cb["unit"] == "TFLOP/s"
    assert cb["value"] > 0 and cb["cores"] >= 1
    st = cb["single_thread"]
    assert st["cores"] == 1 and st["value"] > 0
    import oracle
    assert oracle.num_threads() == cb["cores"]  # restored afterwards


def test_nvml_sampler_rows_parse_like_nvidia_smi_rows(tmp_path):
    """The 1 ms sampler's rows (written from a stand-in for the NVML queries)
    go through the same summary: clock, maximum and the reasons' bits."""
    import threading
    import time

    class FakeNvml:
        REASONS = bench._NvmlClocks.REASONS
        max_mhz = 2070

        def __init__(self):
            self.closed = False

        def sample(self):
            return 1980, 912.5, 0x4 | 0x1   # power cap, and an idle bit that is not reported

        def close(self):
            self.closed = True

    cs = bench.ClockSampler(0, str(tmp_path / "c.csv"))
    cs.f = open(cs.out_path, "w")
    cs.stop = threading.Event()
    nv = FakeNvml()
    th = threading.Thread(target=cs._nvml_loop, args=(nv,))
    t0 = time.time()
    th.start()
    time.sleep(0.05)
    t1 = time.time()
    cs.stop.set()
    th.join()
    cs.f.close()
    s = bench.summarize_clocks(cs.out_path, [(t0, t1)])
    assert s["samples"] >= 5
    assert s["sm_mhz"] == 1980 and s["sm_max_mhz"] == 2070 and s["reasons"] == ["sw_power_cap"]
    assert nv.closed
