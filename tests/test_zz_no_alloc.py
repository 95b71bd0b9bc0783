"""The allocation-free skinny-M entry point (hgemm_run_splitk_noalloc).

For callers that cannot call cudaMalloc while they multiply -- code inside a
caching allocator or an out-of-memory handler, a process whose device memory
is all held by its own pool, loops that cannot take cudaMalloc's implicit
synchronisation.  The entry point keeps its scratch in a fixed array in the
library's device image instead of a handle-owned workspace.

The test calls it twice in a row through the C ABI (the second call finds the
first call's leftovers in the shared array) and checks each output against the
existing entry point, hgemm_run with its split-K variant, within the
tolerance the parity tests use: |x - y| <= ulp_out(ref) + 2^-20 * sum|ab|,
ref being the oracle's exact result.  This file is collected last so that a
run that stops at the first failure has run every other test first.
"""
import numpy as np
import pytest
import torch

import oracle
from tests import parity
from tensor_core_half_gb300 import hgemm, workloads

pytestmark = pytest.mark.gpu

TD = {"f16": torch.float16, "bf16": torch.bfloat16}


@pytest.mark.parametrize("M,N,K,fin,fout", [(16, 16384, 8192, "bf16", "bf16"), (1, 1000, 72, "f16", "f16"),
                                            (40, 4096, 1024, "bf16", "f16"), (64, 264, 8200, "f16", "bf16")])
def test_noalloc_matches_hgemm_run_on_two_calls(M, N, K, fin, fout):
    a, b, ab, bb = parity.inputs(M, N, K, "TN", fin, ("normal", 0.02), 4)
    A, B = a.cuda(), b.cuda()
    stream = torch.cuda.current_stream().cuda_stream

    # the existing entry point, split-K variant
    with hgemm.Handle() as h:
        h.set_option(hgemm.HGEMM_OPT_FORCE_VARIANT, hgemm.HGEMM_VARIANT_SPLITK)
        C_ref = torch.empty((M, N), dtype=TD[fout], device="cuda")
        h.run(A, B, C_ref, layout="TN", acc="f32")
        st, detail = h.sync_status()
        assert st == hgemm.HGEMM_OK, hex(detail)
    existing = oracle.decode(workloads.bits(C_ref.cpu()).ravel(), fout)

    _, exact, absdot = oracle.gemm(ab, bb, M, N, K, "TN", fin, fout, want_exact=True, want_abs=True)
    tol = parity.bound(exact.ravel(), absdot.ravel(), "f32", fout)

    for call in range(2):
        C = torch.full((M, N), float("nan"), dtype=TD[fout], device="cuda")
        st = hgemm.hgemm_run_splitk_noalloc(A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K,
                                            hgemm.DTYPES[fin], hgemm.DTYPES[fout], stream)
        assert st == hgemm.HGEMM_OK, hgemm.hgemm_status_string(st)
        torch.cuda.synchronize()
        got = oracle.decode(workloads.bits(C.cpu()).ravel(), fout)
        diff = np.abs(got - existing)
        assert np.all(diff <= tol), "call %d: %d entries differ beyond tolerance, max %g" % (
            call, int((~(diff <= tol)).sum()), float(np.nanmax(diff)))
        parity.check(workloads.bits(C.cpu()), ab, bb, M, N, K, "TN", fin, "f32", fout)


def test_noalloc_rejects_sizes_beyond_its_maximum():
    A = torch.zeros((128, 64), dtype=torch.bfloat16, device="cuda")
    B = torch.zeros((64, 64), dtype=torch.bfloat16, device="cuda")
    C = torch.zeros((128, 64), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    R = hgemm.hgemm_run_splitk_noalloc
    bf = hgemm.HGEMM_BF16
    assert R(A.data_ptr(), B.data_ptr(), C.data_ptr(), 65, 64, 64, bf, bf, s) == hgemm.HGEMM_ERR_UNSUPPORTED
    assert R(A.data_ptr(), B.data_ptr(), C.data_ptr(), 16, 1 << 30, 64, bf, bf, s) == hgemm.HGEMM_ERR_UNSUPPORTED
    # one arrival counter per 128-column tile fits 2 MiB up to N = 67,108,864
    assert R(A.data_ptr(), B.data_ptr(), C.data_ptr(), 16, 67108864 + 8, 64, bf, bf, s) == \
        hgemm.HGEMM_ERR_UNSUPPORTED
    assert R(A.data_ptr(), B.data_ptr(), C.data_ptr(), 16, 60, 64, bf, bf, s) == hgemm.HGEMM_ERR_MISALIGNED
    assert R(A.data_ptr(), B.data_ptr(), A.data_ptr(), 16, 64, 64, bf, bf, s) == hgemm.HGEMM_ERR_ALIAS
    assert R(0, B.data_ptr(), C.data_ptr(), 16, 64, 64, bf, bf, s) == hgemm.HGEMM_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert torch.all(C == 0)
