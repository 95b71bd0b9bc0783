"""Outputs with more than 2^31 entries and very large tile counts.

The operands are drawn on the device (seeded torch generator, standard
normal, rounded to bf16) and never leave it; the sampled entries and the rows
of A and B they need are gathered to the host, where the oracle computes
those dot products (tests/parity.py: check_gathered)."""
import pytest
import torch

from tests import parity
from tensor_core_half_gb300 import hgemm

pytestmark = pytest.mark.gpu


def _normal(shape, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    return torch.randn(shape, generator=g, device="cuda").bfloat16()


@pytest.fixture(scope="module")
def dense_operands():
    M = N = 49152  # M * N = 2.4e9 > 2^31 output entries
    K = 64
    A = _normal((M, K), 101)
    B = _normal((N, K), 102)
    yield M, N, K, A, B
    del A, B
    torch.cuda.empty_cache()


@pytest.mark.parametrize("schedule,epilogue", [("static", "tma"), ("dynamic", "direct")])
def test_dense_more_than_2_31_outputs(dense_operands, schedule, epilogue):
    M, N, K, A, B = dense_operands
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    with hgemm.Handle() as h:
        h.set_option(hgemm.HGEMM_OPT_SCHEDULE, hgemm.SCHEDULES[schedule])
        h.set_option(hgemm.HGEMM_OPT_EPILOGUE, hgemm.EPILOGUES[epilogue])
        h.run(A, B, C, layout="TN", acc="f32")
        st, detail = h.sync_status()
        assert st == hgemm.HGEMM_OK, hex(detail)
    parity.check_gathered(C, A, B, M, N, K, "TN", "bf16", "f32", "bf16", seed=7)
    del C
    torch.cuda.empty_cache()


def test_dense_nn_more_than_2_31_outputs():
    M, N, K = 40960, 57344, 72  # ragged K; 2.3e9 outputs
    A = _normal((M, K), 103)
    B = _normal((K, N), 104)
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    with hgemm.Handle() as h:
        h.run(A, B, C, layout="NN", acc="f32")
        st, detail = h.sync_status()
        assert st == hgemm.HGEMM_OK, hex(detail)
    parity.check_gathered(C, A, B, M, N, K, "NN", "bf16", "f32", "bf16", seed=8)
    del A, B, C
    torch.cuda.empty_cache()


@pytest.mark.parametrize("schedule", ["static", "dynamic"])
def test_splitk_huge_n(schedule):
    M, N, K = 16, 1 << 28, 8  # 2^21 tiles of 128 rows of N; M * N = 2^32 outputs
    A = _normal((M, K), 105)
    B = _normal((N, K), 106)
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    with hgemm.Handle() as h:
        h.set_option(hgemm.HGEMM_OPT_SCHEDULE, hgemm.SCHEDULES[schedule])
        st, p = hgemm.hgemm_plan(M, N, K, num_sms=torch.cuda.get_device_properties(0).multi_processor_count,
                                 schedule=hgemm.SCHEDULES[schedule])
        assert st == 0 and p.variant == hgemm.HGEMM_VARIANT_SPLITK and p.num_tiles == 1 << 21
        h.run(A, B, C, layout="TN", acc="f32")
        st, detail = h.sync_status()
        assert st == hgemm.HGEMM_OK, hex(detail)
    parity.check_gathered(C, A, B, M, N, K, "TN", "bf16", "f32", "bf16", seed=9)
    del A, B, C
    torch.cuda.empty_cache()
