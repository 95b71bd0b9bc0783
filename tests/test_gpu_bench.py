"""bench.py's own arm on the GPU, end to end: one short run of the headline
workload and one of the skinny workload, each printing the single JSON line
the benchmark contract asks for.  Checks the keys and their internal
consistency (value against ms_per_step, roofline against the peaks file, the
end-to-end byte counts against the workload, the in-kernel clock stamps
against the plan's CTA count)."""
import json
import math
import os
import subprocess
import sys

import pytest
import torch

from tensor_core_half_gb300 import hgemm, workloads

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
STEPS, WARMUP = 6, 3


def _run(*extra):
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--steps", str(STEPS), "--warmup", str(WARMUP),
           "--no-cpu-baseline", "--e2e-steps", "3", "--no-secondary", "--wake-seconds", "0.2",
           "--rest-seconds", "0.3", "--sustained-seconds", "0", *extra]
    out = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, out.stdout[-2000:]
    return json.loads(lines[0])


def _plan_grid(w):
    st, p = hgemm.hgemm_plan(w.M, w.N, w.K, hgemm.LAYOUTS[w.layout], hgemm.DTYPES[w.in_dtype],
                             hgemm.DTYPES[w.acc_dtype], hgemm.DTYPES[w.out_dtype],
                             torch.cuda.get_device_properties(0).multi_processor_count)
    assert st == hgemm.HGEMM_OK
    return p.grid


@pytest.mark.timeout(900)
@pytest.mark.parametrize("workload", [None, "skinny16x16384x8192_bf16"])
def test_bench_line_keeps_the_contract(workload):
    d = _run(*(["--workload", workload] if workload else []))
    w = workloads.WORKLOADS[workload or workloads.HEADLINE]
    flops = 2.0 * w.M * w.N * w.K
    assert d["n_gpus"] == 1 and d["steps"] == STEPS and d["warmup"] == WARMUP
    assert d["data"] == "synthetic" and d["scaling"] == "weak" and d["higher_is_better"] is True
    assert d["vs_baseline"] is None and d["gpu_launches"] == STEPS
    assert d["config"]["workload"] == w.name
    # value is the metric over the device-timed launches
    if d["unit"] == "TFLOPS":
        assert math.isclose(d["value"], flops / (d["ms_per_step"] * 1e-3) / 1e12, rel_tol=1e-3)
        assert d["roofline"]["bound"] == "tensor" and d["roofline"]["unit"] == "TFLOP/s"
    else:
        assert d["unit"] == "GB/s" and d["roofline"]["bound"] == "hbm" and d["roofline"]["unit"] == "GB/s"
        assert math.isclose(d["value"], w.compulsory_bytes / (d["ms_per_step"] * 1e-3) / 1e9, rel_tol=1e-3)
    r = d["roofline"]
    assert r["achieved"] > 0 and r["peak"] > 0
    assert math.isclose(r["frac"], r["achieved"] / r["peak"], rel_tol=2e-3)
    assert r["traffic"] is None or r["traffic"] > 0
    # end to end: the step's inputs up and its result down, counted from the tensors
    e = d["e2e"]
    assert e["h2d_bytes_per_step"] == (w.M * w.K + w.N * w.K) * 2
    assert e["d2h_bytes_per_step"] == w.M * w.N * 2
    assert 0 < e["value"] <= d["value"] * 1.05
    # the SM clock inside the timed launches, from every CTA's begin/end stamps
    k = d["clocks"]["in_kernel"]
    grid = _plan_grid(w)
    assert k["stamps"] == k["stamps_expected"] == 2 * grid * STEPS
    assert k["cta_launches"] == grid * STEPS
    assert 300.0 < k["sm_mhz_min"] <= k["sm_mhz_median"] <= k["sm_mhz_max"] < 3000.0
