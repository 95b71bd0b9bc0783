"""GPU parity on every workload of the table at its full size, in the launch
configuration the benchmark times (automatic variant choice).

Outputs up to 2048 on every side, and the ragged and skinny workloads, are
checked in full; larger ones on 8192 seeded entries plus every entry of the
rows and columns at tile boundaries."""
import pytest
import torch

from tests import parity
from tensor_core_half_gb300 import hgemm, workloads

pytestmark = pytest.mark.gpu

TORCH_DT = {"f16": torch.float16, "bf16": torch.bfloat16}


@pytest.fixture(scope="module")
def h():
    handle = hgemm.Handle()
    yield handle
    handle.close()


_cache = {}


def _inputs(w):
    key = (w.M, w.N, w.K, w.layout, w.in_dtype, w.dist, w.seed, w.scale_inv_sqrt_k)
    if key not in _cache:
        _cache.clear()
        _cache[key] = parity.inputs(w.M, w.N, w.K, w.layout, w.in_dtype, w.dist, w.seed, w.scale_inv_sqrt_k)
    return _cache[key]


def _check(h, w, variant="auto", schedule="static"):
    a, b, ab, bb = _inputs(w)
    A, B = a.cuda(), b.cuda()
    C = torch.empty((w.M, w.N), dtype=TORCH_DT[w.out_dtype], device="cuda")
    h.set_option(hgemm.HGEMM_OPT_FORCE_VARIANT, hgemm.VARIANTS[variant])
    h.set_option(hgemm.HGEMM_OPT_SCHEDULE, hgemm.SCHEDULES[schedule])
    try:
        h.run(A, B, C, layout=w.layout, acc=w.acc_dtype)
        st, detail = h.sync_status()
    finally:
        h.set_option(hgemm.HGEMM_OPT_FORCE_VARIANT, hgemm.HGEMM_VARIANT_AUTO)
        h.set_option(hgemm.HGEMM_OPT_SCHEDULE, hgemm.HGEMM_SCHEDULE_STATIC)
    assert st == hgemm.HGEMM_OK, hex(detail)
    got = workloads.bits(C.cpu())
    del A, B, C
    full = max(w.M, w.N, w.K) <= 2048 or w.name.startswith(("ragged", "skinny"))
    return parity.check(got, ab, bb, w.M, w.N, w.K, w.layout, w.in_dtype, w.acc_dtype, w.out_dtype,
                        sampled=not full, n_random=8192, seed=w.seed)


ORDER = sorted(workloads.WORKLOADS, key=lambda n: (workloads.WORKLOADS[n].M * workloads.WORKLOADS[n].N *
                                                   workloads.WORKLOADS[n].K, n))


@pytest.mark.parametrize("name", ORDER)
def test_workload(h, name):
    _check(h, workloads.WORKLOADS[name])


@pytest.mark.parametrize("name", ["skinny16x16384x8192_bf16", "ragged1000x3000x4104_bf16", "square4096_bf16"])
def test_workload_dynamic_schedule(h, name):
    _check(h, workloads.WORKLOADS[name], schedule="dynamic")


@pytest.mark.parametrize("variant", ["1sm128", "1sm256"])
def test_headline_other_variants(h, variant):
    _check(h, workloads.WORKLOADS["square4096_bf16"], variant)

