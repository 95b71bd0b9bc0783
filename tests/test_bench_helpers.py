"""bench.py's measurement plumbing on the CPU: nvidia-smi parsing, the clock
summary of the timed window, and when stored ncu traffic may be reported."""
import io
import json
import math
import os
from types import SimpleNamespace

import bench


def _sampler(samples=None, lines=None):
    s = bench.ClockSampler.__new__(bench.ClockSampler)  # no nvidia-smi process
    s.samples = list(samples or [])
    s.thread = None
    s.proc = SimpleNamespace(stdout=io.StringIO(lines or ""), poll=lambda: 0)
    return s


def test_reader_parses_hex_and_decimal_masks_and_skips_junk():
    lines = ("0, 2070, 2070, 441.50, 0x0000000000000004, Not Active, Not Active, Not Active, Active\n"
             "0, 1980, 2070, [N/A], 12, Active, Not Active, Not Active, Active\n"
             "garbage line\n"
             "0, notanumber, 2070, 400, 0x0\n")
    s = _sampler(lines=lines)
    s._reader()
    assert len(s.samples) == 2
    _, sm, mx, pw, act = s.samples[0]
    assert (sm, mx, pw, act) == (2070.0, 2070.0, 441.5, 0x4)
    _, sm, mx, pw, act = s.samples[1]
    assert (sm, mx, act) == (1980.0, 2070.0, 12) and math.isnan(pw)


def test_summary_keeps_the_timed_window_and_names_the_reasons():
    samples = [(0.5, 1000.0, 2070.0, 100.0, 0x8),     # before the window: ignored
               (1.0, 2070.0, 2070.0, 900.0, 0x4),
               (1.5, 2000.0, 2070.0, float("nan"), 0x0),
               (2.0, 2065.0, 2070.0, 1200.0, 0x4),
               (3.5, 500.0, 2070.0, 50.0, 0x40)]      # after: ignored
    out = _sampler(samples).summary(1.0, 2.0)
    assert out["window"] == "timed" and out["samples"] == 3
    assert out["sm_mhz"] == 2065.0 and out["sm_max_mhz"] == 2070.0
    assert out["reasons"] == ["sw_power_cap"]
    assert out["power_w_max"] == 1200.0


def test_summary_reports_slowdowns_seen_inside_the_window():
    samples = [(1.0, 1500.0, 2070.0, 1000.0, 0x8 | 0x20), (1.1, 1600.0, 2070.0, 1000.0, 0x40)]
    out = _sampler(samples).summary(0.9, 1.2)
    assert set(out["reasons"]) == {"hw_slowdown", "sw_thermal_slowdown", "hw_thermal_slowdown"}


def test_summary_falls_back_to_the_nearest_samples_or_none():
    samples = [(0.0, 2000.0, 2070.0, 10.0, 0), (10.0, 2010.0, 2070.0, 10.0, 0), (20.0, 2020.0, 2070.0, 10.0, 0),
               (30.0, 2030.0, 2070.0, 10.0, 0)]
    out = _sampler(samples).summary(10.4, 10.5)  # shorter than the sampling period
    assert out["window"] == "nearest" and out["samples"] == 3
    empty = _sampler([]).summary(0.0, 1.0)
    assert empty["window"] == "none" and empty["sm_mhz"] is None and empty["samples"] == 0


def test_stop_is_safe_without_a_process():
    s = _sampler()
    s.proc = None
    s.stop()
    s.stop()


def _stored():
    with open(os.path.join(bench.ROOT, "profiles", "traffic.json")) as f:
        return {k: v for k, v in json.load(f).items() if not k.startswith("_")}


def test_traffic_is_reported_only_for_the_captured_kernel_and_plan():
    stored = _stored()
    assert stored, "the committed ncu summaries record traffic"
    for key, e in stored.items():
        workload, variant = key.rsplit("/", 1)
        kernel = "splitk" if int(variant) == 4 else "dense"
        plan = SimpleNamespace(**e["plan"])
        got = bench.load_traffic(workload, int(variant), plan)
        if e["kernel_hash"] == bench.kernel_source_hash(kernel):
            assert got == e["dram_bytes_per_launch"]
        else:
            assert got is None  # the kernel changed since the capture
        other = SimpleNamespace(**dict(e["plan"], grid=e["plan"]["grid"] + 2))
        assert bench.load_traffic(workload, int(variant), other) is None  # another launch plan
    assert bench.load_traffic("no_such_workload", 3, None) is None


def test_kernel_hash_covers_every_source_it_names():
    for kernel, files in bench.KERNEL_SOURCES.items():
        for rel in files:
            assert os.path.exists(os.path.join(bench.ROOT, "tensor_core_half_gb300", "csrc", rel)), rel
        h = bench.kernel_source_hash(kernel)
        assert len(h) == 16 and h == bench.kernel_source_hash(kernel)


def test_reference_arm_prints_the_contract_line():
    # The reference arm times the oracle on the host cores and prints one JSON
    # line with the same metric and config as the CUDA arm, marked as such.
    import subprocess
    import sys
    r = subprocess.run([sys.executable, os.path.join(bench.ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], capture_output=True, text=True, timeout=600, cwd=bench.ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 1 and d["steps"] == 1 and d["warmup"] == 3
    assert d["metric"].startswith("TFLOPS") and d["unit"] == "TFLOPS" and d["higher_is_better"] is True
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["vs_baseline"] is None
    assert d["data"] == "synthetic" and d["config"]["workload"] == "square4096_bf16"
    # the same problem config the CUDA arm prints (sizes, layout and all three dtypes)
    from tensor_core_half_gb300 import workloads
    assert d["config"] == bench.problem_config(workloads.WORKLOADS["square4096_bf16"], 1)
    assert (d["config"]["in"], d["config"]["acc"], d["config"]["out"]) == ("bf16", "f32", "bf16")
    cpu = d["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["cores"] >= 1 and cpu["value"] == d["value"] and cpu["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_roofline_object_uses_the_peak_of_its_bound():
    from tensor_core_half_gb300 import workloads
    peaks = {"hbm_gbs": 6000.0, "bf16_tflops": 2000.0, "bf16_tflops_sustained": 1600.0}
    w = workloads.WORKLOADS["square4096_bf16"]
    ms = 0.08
    r = bench.roofline_for(w, "tensor", ms, peaks, "measured", False)
    assert r["bound"] == "tensor" and r["peak"] == 2000.0 and r["unit"] == "TFLOP/s"
    assert math.isclose(r["achieved"], round(w.flops / 1e12 / (ms / 1e3), 2))
    assert math.isclose(r["frac"], round(r["achieved"] / 2000.0, 4), abs_tol=1e-4)
    assert bench.roofline_for(w, "tensor", ms, peaks, "measured", True)["peak"] == 1600.0
    s = workloads.WORKLOADS["skinny16x16384x8192_bf16"]
    r = bench.roofline_for(s, "hbm", 0.045, peaks, "measured", False)
    assert r["bound"] == "hbm" and r["peak"] == 6000.0 and r["unit"] == "GB/s"
    assert math.isclose(r["achieved"], round(s.compulsory_bytes / 1e9 / 45e-6, 1))


def test_secondary_workloads_cover_the_targets():
    # 8192^3 bf16 and the skinny product are targets of their own; the other
    # two are the shapes with less than one wave of tiles
    from tensor_core_half_gb300 import workloads
    assert set(bench.SECONDARY) <= set(workloads.WORKLOADS)
    assert "square8192_bf16" in bench.SECONDARY and "skinny16x16384x8192_bf16" in bench.SECONDARY
    assert bench.workload_metric(workloads.WORKLOADS["skinny16x16384x8192_bf16"])[3] == "hbm"
    assert bench.workload_metric(workloads.WORKLOADS["square8192_bf16"])[3] == "tensor"


def test_in_kernel_clocks_pair_each_ctas_begin_and_end():
    """Two CTAs, three launches: each (begin, end) pair in time order gives
    cycles / ns; the 31-bit cycle counter may wrap between the two."""
    rows = []
    t = 1_000_000
    for launch in range(3):
        for cta, mhz in ((0, 1800.0), (1, 2000.0)):
            c0 = (2**31 - 50_000) if (launch == 1 and cta == 0) else 1_000 * (launch + 1)  # wraps in launch 1
            dt = 80_000  # ns
            rows.append((t, cta, 0, 1, -1, c0))
            rows.append((t + dt, cta, 0, 2, -1, (c0 + int(mhz * dt / 1e3)) % 2**31))
            rows.append((t + 10, cta, 3, 3, 5, 0))  # an item record is ignored
        t += 100_000
    rows.reverse()  # append order is not time order
    c = bench.in_kernel_clocks(rows, len(rows), 12)
    assert c["cta_launches"] == 6 and c["stamps"] == 18
    assert c["sm_mhz_min"] == 1800.0 and c["sm_mhz_max"] == 2000.0
    assert c["sm_mhz_median"] in (1800.0, 2000.0)
