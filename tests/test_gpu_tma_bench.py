"""The TMA micro-benchmark copies the right bytes in every copy form."""
import pytest
import torch

from tensor_core_half_gb300 import hgemm, tma_bench

pytestmark = pytest.mark.gpu

MODES = list(hgemm.TMA_MODES.values())


@pytest.fixture(scope="module")
def src():
    return tma_bench.source(1024, 2048)


@pytest.mark.parametrize("walk", list(hgemm.TMA_WALKS.values()), ids=list(hgemm.TMA_WALKS))
@pytest.mark.parametrize("mode", MODES, ids=list(hgemm.TMA_MODES))
@pytest.mark.parametrize("rows,cols", [(128, 64), (64, 128), (256, 128), (8, 64)])
def test_every_cta_holds_its_tiles(src, mode, rows, cols, walk):
    depth = max(1, min(6, (96 * 1024) // (rows * cols * 2)))
    res = tma_bench.run_checked(src, mode, rows, cols, depth, 40, check_ctas=1 << 20, walk=walk)
    assert res.ctas == torch.cuda.get_device_properties(0).multi_processor_count
    assert res.tile_bytes == rows * cols * 2 and res.bytes == res.ctas * 40 * res.tile_bytes
    assert res.bytes_per_clk_sm > 0 and res.gbs > 0 and res.sm_mhz > 0


@pytest.mark.parametrize("mode,issuers", [(hgemm.HGEMM_TMA_2D_128B, 2), (hgemm.HGEMM_TMA_2D_16B, 2)])
def test_two_issuing_warps(src, mode, issuers):
    tma_bench.run_checked(src, mode, 128, 128, 4, 33, issuers=issuers, check_ctas=1 << 20)


def test_fewer_rounds_than_slots_and_few_ctas(src):
    res = tma_bench.run_checked(src, hgemm.HGEMM_TMA_3D_128B, 128, 128, 6, 3, ctas=5, check_ctas=1 << 20)
    assert res.ctas == 5


def test_a_wrong_tile_is_detected():
    # the check itself must be able to fail: sums of a neighbouring tile differ
    a = tma_bench.expected_sums(1024, 2048, hgemm.HGEMM_TMA_2D_128B, 128, 64, [5])
    b = tma_bench.expected_sums(1024, 2048, hgemm.HGEMM_TMA_2D_128B, 128, 64, [6])
    assert a != b


def test_rejects_bad_shapes(src):
    h, w = src.shape
    bad = [(hgemm.HGEMM_TMA_2D_128B, 128, 96, 2, 8, 1),   # 128-byte modes need 64-column multiples
           (hgemm.HGEMM_TMA_2D_16B, 100, 64, 2, 8, 1),    # rows multiple of 8
           (hgemm.HGEMM_TMA_3D_16B, 128, 64, 2, 8, 2),    # one copy per tile: one issuer
           (hgemm.HGEMM_TMA_2D_128B, 128, 64, 17, 8, 1),  # depth <= 16
           (7, 128, 64, 2, 8, 1)]
    st = hgemm.hgemm_tma_bench(src.data_ptr(), h, w, hgemm.HGEMM_TMA_BULK, 128, 64, 2, 8, walk=2)[0]
    assert st == hgemm.HGEMM_ERR_INVALID_ARG
    for mode, r, c, depth, iters, iss in bad:
        st = hgemm.hgemm_tma_bench(src.data_ptr(), h, w, mode, r, c, depth, iters, iss)[0]
        assert st == hgemm.HGEMM_ERR_INVALID_ARG, (mode, r, c, depth, iss)
    st = hgemm.hgemm_tma_bench(src.data_ptr(), h, w, hgemm.HGEMM_TMA_2D_128B, 256, 256, 8, 8)[0]
    assert st == hgemm.HGEMM_ERR_UNSUPPORTED  # 8 x 128 KiB slots do not fit in shared memory
