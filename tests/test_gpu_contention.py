"""The dense kernels on a GPU that other work shares.

A background kernel holds some SMs while the GEMM runs on another stream, so
not every cluster of the GEMM's grid can be resident at once.  Both schedules
must stay correct (a stream-K contributor that has not started must not block
the others); the dynamic schedule (cluster launch control) must also keep most
of its speed, where the static one runs its left-over clusters as a second
wave.  Run with -s to see the measured rates.
"""
import ctypes
import os
import subprocess
import tempfile
import time

import numpy as np
import pytest
import torch

from tests import parity
from tensor_core_half_gb300 import hgemm, workloads

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def load():
    out = os.path.join(tempfile.mkdtemp(prefix="hgemm_load_"), "gpu_load.so")
    subprocess.check_call(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-shared", "-Xcompiler",
                           "-fPIC", os.path.join(HERE, "gpu_load.cu"), "-o", out])
    lib = ctypes.CDLL(out)
    lib.hold_sms.argtypes = [ctypes.c_int, ctypes.c_ulonglong, ctypes.c_void_p]
    lib.hold_sms.restype = ctypes.c_int
    return lib


def _timed(h, A, B, C, launches, load, busy, bg):
    for _ in range(3):
        h.run(A, B, C)
    torch.cuda.synchronize()
    if busy:
        assert load.hold_sms(busy, 300_000_000, ctypes.c_void_p(bg.cuda_stream)) == 0
        time.sleep(0.02)  # the background CTAs are resident before the GEMMs start
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(launches):
        h.run(A, B, C)
    e1.record()
    e1.synchronize()
    ms = e0.elapsed_time(e1) / launches
    torch.cuda.synchronize()
    st, detail = h.sync_status()
    assert st == hgemm.HGEMM_OK, (st, hex(detail))
    return ms


@pytest.mark.parametrize("schedule", ["static", "dynamic"])
def test_splitk_parity_with_busy_sms(load, schedule):
    M, N, K = 16, 16384, 4096
    a, b, ab, bb = parity.inputs(M, N, K, "TN", "bf16", ("normal", 1.0), 92)
    A, B = a.cuda(), b.cuda()
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    bg = torch.cuda.Stream()
    with hgemm.Handle() as h:
        h.set_option(hgemm.HGEMM_OPT_SCHEDULE, hgemm.SCHEDULES[schedule])
        _timed(h, A, B, C, 5, load, 24, bg)
    parity.check(workloads.bits(C.cpu()), ab, bb, M, N, K, "TN", "bf16", "f32", "bf16")


def test_splitk_rates_with_busy_sms(load):
    # Reported (run with -s).  The static split over every SM runs the CTAs
    # that find no free SM as a second wave; the dynamic schedule must not
    # lose to it once SMs are busy.  The whole-tile layout the planner picks
    # here (128 CTAs for 128 tiles) leaves 24 SMs spare and is reported too.
    M, N, K = 16, 16384, 8192
    A = torch.randn((M, K), device="cuda").bfloat16()
    B = torch.randn((N, K), device="cuda").bfloat16()
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    bg = torch.cuda.Stream()
    rate = {}
    layouts = {"whole": ("static", 1), "split": ("static", 2), "dynamic": ("dynamic", 1)}
    for busy in (0, 16):
        for name, (schedule, sk) in layouts.items():
            with hgemm.Handle() as h:
                h.set_option(hgemm.HGEMM_OPT_SCHEDULE, hgemm.SCHEDULES[schedule])
                h.set_option(hgemm.HGEMM_OPT_STREAM_K, sk)
                ms = _timed(h, A, B, C, 50, load, busy, bg)
            rate[(busy, name)] = (M * K + N * K + M * N) * 2 / ms / 1e6
            print("16x16384x8192 bf16 split-K, %2d SMs held by other work, %-7s layout: %.0f GB/s" % (
                busy, name, rate[(busy, name)]))
    assert rate[(16, "dynamic")] > rate[(16, "split")]


@pytest.mark.parametrize("schedule", ["static", "dynamic"])
@pytest.mark.parametrize("sk", [1, 0])
def test_parity_with_busy_sms(load, schedule, sk):
    M, N, K = 2048, 4096, 1024
    a, b, ab, bb = parity.inputs(M, N, K, "TN", "bf16", ("normal", 1.0), 91)
    A, B = a.cuda(), b.cuda()
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    bg = torch.cuda.Stream()
    with hgemm.Handle() as h:
        h.set_option(hgemm.HGEMM_OPT_SCHEDULE, hgemm.SCHEDULES[schedule])
        h.set_option(hgemm.HGEMM_OPT_STREAM_K, sk)
        _timed(h, A, B, C, 5, load, 24, bg)
    parity.check(workloads.bits(C.cpu()), ab, bb, M, N, K, "TN", "bf16", "f32", "bf16")


def test_dynamic_schedule_keeps_speed_with_busy_sms(load):
    M = N = K = 8192
    A = torch.randn((M, K), device="cuda").bfloat16()
    B = torch.randn((N, K), device="cuda").bfloat16()
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    bg = torch.cuda.Stream()
    rate = {}
    for busy in (0, 16):
        for schedule in ("static", "dynamic"):
            with hgemm.Handle() as h:
                h.set_option(hgemm.HGEMM_OPT_SCHEDULE, hgemm.SCHEDULES[schedule])
                ms = _timed(h, A, B, C, 10, load, busy, bg)
            rate[(busy, schedule)] = 2.0 * M * N * K / ms / 1e9
            print("8192^3 bf16, %2d SMs held by other work, %-7s schedule: %.0f TFLOPS" % (busy, schedule,
                                                                                          rate[(busy, schedule)]))
    # The static plan leaves clusters for a second wave; cluster launch control
    # hands their work to the clusters that run.
    assert rate[(16, "dynamic")] > 1.25 * rate[(16, "static")]
    assert rate[(16, "dynamic")] > 0.7 * rate[(0, "dynamic")]
