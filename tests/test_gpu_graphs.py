"""CUDA graph capture of hgemm_run, and independent handles on concurrent streams."""
import numpy as np
import pytest
import torch

from tests import parity
from tensor_core_half_gb300 import hgemm, workloads

pytestmark = pytest.mark.gpu

CASES = [(4096, 4096, 1024, "2sm256"), (16, 16384, 4096, "splitk"), (1000, 3000, 4104, "auto")]


def _inputs(M, N, K, seed):
    a, b, ab, bb = parity.inputs(M, N, K, "TN", "bf16", ("normal", 1.0), seed)
    return a.cuda(), b.cuda(), ab, bb


def test_graph_capture_and_replay():
    # Warm up outside the capture (workspace allocation), capture one launch of
    # each case in one graph, replay it twice and check every result.
    data = []
    with hgemm.Handle() as h:
        h.set_option(hgemm.HGEMM_OPT_STREAM_K, 2)  # stream-K partials inside the graph too
        for i, (M, N, K, variant) in enumerate(CASES):
            A, B, ab, bb = _inputs(M, N, K, 121 + i)
            C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
            data.append((M, N, K, variant, A, B, C, ab, bb))
        for M, N, K, variant, A, B, C, _, _ in data:
            h.set_option(hgemm.HGEMM_OPT_FORCE_VARIANT, hgemm.VARIANTS[variant])
            h.run(A, B, C)
        assert h.sync_status()[0] == hgemm.HGEMM_OK
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for M, N, K, variant, A, B, C, _, _ in data:
                h.set_option(hgemm.HGEMM_OPT_FORCE_VARIANT, hgemm.VARIANTS[variant])
                assert h.run(A, B, C, check=False) == hgemm.HGEMM_OK
        for _, _, _, _, _, _, C, _, _ in data:
            C.fill_(0)
        for _ in range(2):
            g.replay()
        torch.cuda.synchronize()
        assert h.sync_status()[0] == hgemm.HGEMM_OK
        first = [workloads.bits(d[6].cpu()) for d in data]
        for (M, N, K, variant, A, B, C, ab, bb), got in zip(data, first):
            parity.check(got, ab, bb, M, N, K, "TN", "bf16", "f32", "bf16")
        g.replay()
        torch.cuda.synchronize()
        for (*_, C, _, _), got in zip(data, first):
            assert np.array_equal(workloads.bits(C.cpu()), got)  # replays repeat bit for bit


@pytest.mark.filterwarnings("ignore:The CUDA Graph is empty")
def test_capture_refuses_to_allocate():
    # A fresh handle has no workspace: inside a capture a split-K launch that
    # needs one (the K split, forced here) must refuse (UNSUPPORTED, nothing
    # enqueued) instead of calling cudaMalloc.
    M, N, K = 16, 16384, 4096
    A, B, ab, bb = _inputs(M, N, K, 131)
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    with hgemm.Handle() as h:
        h.set_option(hgemm.HGEMM_OPT_STREAM_K, 2)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            st = h.run(A, B, C, check=False)
        assert st == hgemm.HGEMM_ERR_UNSUPPORTED
        assert h.run(A, B, C, check=False) == hgemm.HGEMM_OK  # outside a capture it allocates and runs
        assert h.sync_status()[0] == hgemm.HGEMM_OK
    # Whole tiles (the planner's layout here) use no workspace: a fresh
    # handle's launch can be captured directly.
    with hgemm.Handle() as h:
        st, p = hgemm.hgemm_plan(M, N, K, num_sms=torch.cuda.get_device_properties(0).multi_processor_count)
        assert p.splitk_align == p.k_blocks and p.workspace_bytes == 0
        C.fill_(0)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            assert h.run(A, B, C, check=False) == hgemm.HGEMM_OK
        g.replay()
        torch.cuda.synchronize()
        assert h.sync_status()[0] == hgemm.HGEMM_OK
    parity.check(workloads.bits(C.cpu()), ab, bb, M, N, K, "TN", "bf16", "f32", "bf16")


def test_handles_on_concurrent_streams():
    # Two handles, two streams, stream-K and split-K launches interleaved: the
    # workspaces are per handle, so the results must be those of serial runs.
    cases = [(4096, 4096, 1024, "2sm256", 141), (16, 16384, 4096, "splitk", 142)]
    ins = [_inputs(M, N, K, seed) for M, N, K, _, seed in cases]
    handles = [hgemm.Handle(), hgemm.Handle()]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = []
    try:
        for i, ((M, N, K, variant, _), (A, B, ab, bb)) in enumerate(zip(cases, ins)):
            handles[i].set_option(hgemm.HGEMM_OPT_FORCE_VARIANT, hgemm.VARIANTS[variant])
            handles[i].set_option(hgemm.HGEMM_OPT_STREAM_K, 2)
            outs.append([torch.empty((M, N), dtype=torch.bfloat16, device="cuda") for _ in range(4)])
        torch.cuda.synchronize()
        for rep in range(4):
            for i, ((M, N, K, variant, _), (A, B, ab, bb)) in enumerate(zip(cases, ins)):
                with torch.cuda.stream(streams[i]):
                    handles[i].run(A, B, outs[i][rep])
        torch.cuda.synchronize()
        for i, ((M, N, K, variant, _), (A, B, ab, bb)) in enumerate(zip(cases, ins)):
            assert handles[i].sync_status()[0] == hgemm.HGEMM_OK
            ref = workloads.bits(outs[i][0].cpu())
            parity.check(ref, ab, bb, M, N, K, "TN", "bf16", "f32", "bf16")
            for rep in range(1, 4):
                assert np.array_equal(workloads.bits(outs[i][rep].cpu()), ref)
    finally:
        for h in handles:
            h.close()
