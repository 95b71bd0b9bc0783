"""GPU parity of the CUDA path (through the C ABI) against the CPU oracle.

Sizes here finish in seconds on the oracle and still span several tiles and
ragged tails; the full workload table is covered in test_gpu_workloads.py.
"""
import numpy as np
import pytest
import torch

import oracle
from tests import parity
from tensor_core_half_gb300 import hgemm, workloads

pytestmark = pytest.mark.gpu

TORCH_DT = {"f16": torch.float16, "bf16": torch.bfloat16}
DENSE_VARIANTS = ["1sm128", "1sm256", "2sm256", "2sm192"]
NN_UNSUPPORTED = {"2sm192"}  # 192-column tiles split B into 96-column halves: TN only


@pytest.fixture(scope="module")
def h():
    handle = hgemm.Handle()
    yield handle
    handle.close()


def run(h, a, b, M, N, K, layout, acc, out, variant="auto", C=None, stream_k=1, schedule="static", epilogue="tma"):
    h.set_option(hgemm.HGEMM_OPT_FORCE_VARIANT, hgemm.VARIANTS[variant])
    h.set_option(hgemm.HGEMM_OPT_STREAM_K, stream_k)
    h.set_option(hgemm.HGEMM_OPT_SCHEDULE, hgemm.SCHEDULES[schedule])
    h.set_option(hgemm.HGEMM_OPT_EPILOGUE, hgemm.EPILOGUES[epilogue])
    try:
        if layout == "NN" and variant in NN_UNSUPPORTED:
            A, B = a.cuda(), b.cuda()
            C = torch.empty((M, N), dtype=TORCH_DT[out], device="cuda")
            assert h.run(A, B, C, layout=layout, acc=acc, check=False) == hgemm.HGEMM_ERR_UNSUPPORTED
            pytest.skip("variant %s does not take the NN layout" % variant)
        A, B = a.cuda(), b.cuda()
        if C is None:
            C = torch.empty((M, N), dtype=TORCH_DT[out], device="cuda")
        h.run(A, B, C, layout=layout, acc=acc)
        st, detail = h.sync_status()
        assert st == hgemm.HGEMM_OK, (hgemm.hgemm_status_string(st), hex(detail))
        return workloads.bits(C.cpu())
    finally:
        h.set_option(hgemm.HGEMM_OPT_FORCE_VARIANT, hgemm.HGEMM_VARIANT_AUTO)
        h.set_option(hgemm.HGEMM_OPT_STREAM_K, 1)
        h.set_option(hgemm.HGEMM_OPT_SCHEDULE, hgemm.HGEMM_SCHEDULE_STATIC)
        h.set_option(hgemm.HGEMM_OPT_EPILOGUE, hgemm.HGEMM_EPILOGUE_TMA_STORE)


@pytest.mark.parametrize("variant", ["auto"] + DENSE_VARIANTS)
def test_square256_f16(h, variant):
    w = workloads.WORKLOADS["square256_f16"]
    a, b, ab, bb = parity.inputs(w.M, w.N, w.K, w.layout, w.in_dtype, w.dist, w.seed)
    got = run(h, a, b, w.M, w.N, w.K, w.layout, w.acc_dtype, w.out_dtype, variant)
    parity.check(got, ab, bb, w.M, w.N, w.K, w.layout, w.in_dtype, w.acc_dtype, w.out_dtype)


DTYPE_COMBOS = [("f16", "f32", "f16"), ("f16", "f32", "bf16"), ("bf16", "f32", "bf16"), ("bf16", "f32", "f16"),
                ("f16", "f16", "f16"), ("f16", "f16", "bf16")]


@pytest.mark.parametrize("variant", DENSE_VARIANTS)
@pytest.mark.parametrize("layout", ["TN", "NN"])
@pytest.mark.parametrize("combo", DTYPE_COMBOS, ids=["-".join(c) for c in DTYPE_COMBOS])
def test_dtype_layout_variant_matrix(h, combo, layout, variant):
    fin, acc, out = combo
    M, N, K = 384, 520, 200  # ragged in M (for 256-row tiles), N and K
    a, b, ab, bb = parity.inputs(M, N, K, layout, fin, ("uniform", -1.0, 1.0), 11)
    got = run(h, a, b, M, N, K, layout, acc, out, variant)
    parity.check(got, ab, bb, M, N, K, layout, fin, acc, out)


RAGGED_M = [1, 8, 120, 128, 129, 257, 1000]
RAGGED_N = [8, 120, 136, 264, 1000]


@pytest.mark.parametrize("layout", ["TN", "NN"])
@pytest.mark.parametrize("K", [8, 72, 640])
@pytest.mark.parametrize("N", RAGGED_N)
@pytest.mark.parametrize("M", RAGGED_M)
def test_ragged_sweep(h, M, N, K, layout):
    a, b, ab, bb = parity.inputs(M, N, K, layout, "bf16", ("normal", 1.0), M * 7 + N * 3 + K)
    got = run(h, a, b, M, N, K, layout, "f32", "bf16")
    parity.check(got, ab, bb, M, N, K, layout, "bf16", "f32", "bf16")


@pytest.mark.parametrize("layout", ["TN", "NN"])
@pytest.mark.parametrize("M,N", [(129, 1000), (1000, 264), (16, 1000)])
def test_ragged_long_k(h, M, N, layout):
    K = 4104
    a, b, ab, bb = parity.inputs(M, N, K, layout, "f16", ("uniform", -1.0, 1.0), 5)
    got = run(h, a, b, M, N, K, layout, "f32", "f16")
    parity.check(got, ab, bb, M, N, K, layout, "f16", "f32", "f16")


@pytest.mark.parametrize("variant", ["auto"] + DENSE_VARIANTS)
@pytest.mark.parametrize("layout", ["TN", "NN"])
def test_small_integers_bit_exact_f32_acc(h, layout, variant):
    # |C| <= 16 * 4096 = 65536 < 2^24: every partial sum is exact in fp32, so the
    # device result is RNE(exact) whatever the accumulation order.
    M, N, K = 320, 384, 4096
    a, b, ab, bb = parity.inputs(M, N, K, layout, "bf16", ("int", -4, 4), 21)
    got = run(h, a, b, M, N, K, layout, "f32", "bf16", variant)
    ref, _, _ = oracle.gemm(ab, bb, M, N, K, layout, "bf16", "bf16")
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("variant", DENSE_VARIANTS)
def test_small_integers_bit_exact_f16_acc(h, variant):
    # {-1,0,1} with K <= 2048: every partial sum is an integer of magnitude <= 2048,
    # exactly representable in fp16.
    M, N, K = 256, 256, 2048
    a, b, ab, bb = parity.inputs(M, N, K, "TN", "f16", ("int", -1, 1), 22)
    got = run(h, a, b, M, N, K, "TN", "f16", "f16", variant)
    ref, _, _ = oracle.gemm(ab, bb, M, N, K, "TN", "f16", "f16")
    assert np.array_equal(got, ref)


def _overflow_operands(M, N, K, layout):
    # C[i, j] = s_j * (A[i, 0] + A[i, 1]) with s_j = +1 for even j, -1 for odd:
    # A[i, 0] runs over fp16's largest values, A[i, 1] over small integers, so
    # the sums cross fp16's overflow threshold (halfway between 65504 and 2^16:
    # 65519 rounds to 65504, 65520 to infinity) on both signs.  Every partial
    # sum is an integer below 2^24, exact in fp32 in any order.
    big = np.array([65504.0, 65472.0, 65440.0, 32768.0], np.float32)
    a = torch.zeros((M, K), dtype=torch.float32)
    a[:, 0] = torch.from_numpy(big[np.arange(M) % big.size])
    a[:, 1] = torch.from_numpy(((np.arange(M) * 7) % 81 - 40).astype(np.float32))
    sign = torch.from_numpy(np.where(np.arange(N) % 2 == 0, 1.0, -1.0).astype(np.float32))
    bt = torch.zeros((N, K), dtype=torch.float32)  # [N, K]
    bt[:, 0] = sign
    bt[:, 1] = sign
    b = bt if layout == "TN" else bt.t().contiguous()
    a, b = a.half(), b.half()
    return a, b, workloads.bits(a), workloads.bits(b)


@pytest.mark.parametrize("epilogue", ["tma", "direct"])
@pytest.mark.parametrize("layout", ["TN", "NN"])
@pytest.mark.parametrize("variant,M", [("auto", 300)] + [(v, 300) for v in DENSE_VARIANTS] + [("splitk", 48)])
def test_output_overflow_rounds_like_the_oracle(h, variant, M, layout, epilogue):
    # Rounding to fp16 output at its overflow threshold: bit-exact against the
    # oracle's round-to-nearest-even, infinities included.
    if variant == "splitk" and layout == "NN":
        pytest.skip("split-K takes the TN layout")
    if variant == "splitk" and epilogue == "direct":
        pytest.skip("the epilogue option applies to the dense kernels")
    N, K = 520, 64
    a, b, ab, bb = _overflow_operands(M, N, K, layout)
    got = run(h, a, b, M, N, K, layout, "f32", "f16", variant, epilogue=epilogue)
    ref, _, _ = oracle.gemm(ab, bb, M, N, K, layout, "f16", "f16")
    assert np.isinf(oracle.decode(ref.ravel(), "f16")).sum() > 0  # the threshold is crossed
    assert np.array_equal(got, ref)


def _nonfinite_operands(M, N, K, seed):
    # Normal data with a +inf in row 7 of A (k = 13), whose B entries are 0, +1
    # and -1 by column (inf * 0 = NaN, +-inf otherwise), a NaN in row M-2 of A
    # and a -inf in column 400 of B (k = 77), which meets the +inf of row 7.
    a, bt, _, _ = parity.inputs(M, N, K, "TN", "bf16", ("normal", 1.0), seed)
    a, bt = a.float(), bt.float()
    a[7, 13] = float("inf")
    bt[:, 13] = torch.from_numpy(np.array([0.0, 1.0, -1.0], np.float32)[np.arange(N) % 3])
    a[M - 2, 50] = float("nan")
    bt[400, 77] = float("-inf")
    a, bt = a.bfloat16(), bt.bfloat16()
    return a, bt, workloads.bits(a), workloads.bits(bt)


@pytest.mark.parametrize("variant,M,stream_k", [("auto", 300, 1), ("2sm256", 300, 2), ("1sm128", 300, 1),
                                                ("splitk", 48, 0), ("splitk", 48, 2)])
def test_nonfinite_inputs_propagate_like_the_oracle(h, variant, M, stream_k):
    # Inputs are unspecified beyond finite values, but IEEE arithmetic fixes
    # where infinities and NaNs land: NaN and inf positions and signs must be
    # those of the oracle's double-precision sum; every finite entry is still
    # within tolerance.  Split tiles (stream-K, the K split) add partials that
    # hold infinities.
    N, K = 520, 200
    a, b, ab, bb = _nonfinite_operands(M, N, K, 23)
    got = oracle.decode(run(h, a, b, M, N, K, "TN", "f32", "bf16", variant, stream_k=stream_k).ravel(), "bf16")
    ref_bits, ref, absdot = oracle.gemm(ab, bb, M, N, K, "TN", "bf16", "bf16", want_exact=True, want_abs=True)
    ref_out = oracle.decode(ref_bits.ravel(), "bf16")
    assert np.array_equal(np.isnan(got), np.isnan(ref_out))
    assert np.isnan(ref_out).sum() >= N and np.isinf(ref_out).sum() > 0
    inf = np.isinf(ref_out)
    assert np.array_equal(got[inf], ref_out[inf])
    fin = np.isfinite(ref_out)
    assert np.array_equal(np.isfinite(got), fin)
    ref, absdot = ref.ravel()[fin], absdot.ravel()[fin]
    assert (np.abs(got[fin] - ref) <= parity.bound(ref, absdot, "f32", "bf16")).all()


@pytest.mark.parametrize("M", [1, 5, 16, 17, 33, 48, 64])
@pytest.mark.parametrize("N,K", [(8, 64), (1000, 72), (4096, 1024), (384, 8192)])
def test_splitk_shapes(h, M, N, K):
    a, b, ab, bb = parity.inputs(M, N, K, "TN", "bf16", ("normal", 0.02), 4)
    got = run(h, a, b, M, N, K, "TN", "f32", "bf16", "splitk")
    parity.check(got, ab, bb, M, N, K, "TN", "bf16", "f32", "bf16")


@pytest.mark.parametrize("stream_k", [0, 1, 2], ids=["whole", "auto", "split"])
@pytest.mark.parametrize("M,N,K", [(16, 16384, 2048), (33, 12288, 1024), (64, 20480, 520), (1, 8, 64),
                                   (5, 1000, 72), (48, 2048, 4104)])
def test_splitk_layouts(h, M, N, K, stream_k):
    # Whole tiles per CTA (no tile's K range split: no partials, no fix-up)
    # and the balanced K split give the same products up to fp32 summation
    # order; HGEMM_OPT_STREAM_K 0 / 2 force one or the other.
    a, b, ab, bb = parity.inputs(M, N, K, "TN", "bf16", ("normal", 1.0), 91)
    got = run(h, a, b, M, N, K, "TN", "f32", "bf16", "splitk", stream_k=stream_k)
    parity.check(got, ab, bb, M, N, K, "TN", "bf16", "f32", "bf16")
    again = run(h, a, b, M, N, K, "TN", "f32", "bf16", "splitk", stream_k=stream_k)
    assert np.array_equal(got, again)


@pytest.mark.parametrize("stream_k", [0, 2], ids=["whole", "split"])
def test_splitk_layouts_small_integers_bit_exact(h, stream_k):
    M, N, K = 24, 16384, 4096
    a, b, ab, bb = parity.inputs(M, N, K, "TN", "bf16", ("int", -4, 4), 92)
    got = run(h, a, b, M, N, K, "TN", "f32", "bf16", "splitk", stream_k=stream_k)
    ref, _, _ = oracle.gemm(ab, bb, M, N, K, "TN", "bf16", "bf16")
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("M", [1, 16, 33, 64])
@pytest.mark.parametrize("N,K", [(4096, 1024), (384, 8192), (16384, 2048), (1000, 4104)])
def test_splitk_dynamic_parity(h, M, N, K):
    # Dynamic split-K: big chunks on the SMs that start, small chunks taken
    # over by those that finish first; fixed summation order per tile.
    a, b, ab, bb = parity.inputs(M, N, K, "TN", "bf16", ("normal", 1.0), 86)
    got = run(h, a, b, M, N, K, "TN", "f32", "bf16", "splitk", schedule="dynamic")
    parity.check(got, ab, bb, M, N, K, "TN", "bf16", "f32", "bf16")
    again = run(h, a, b, M, N, K, "TN", "f32", "bf16", "splitk", schedule="dynamic")
    assert np.array_equal(got, again)


def test_splitk_dynamic_small_integers_bit_exact(h):
    M, N, K = 40, 8192, 4096
    a, b, ab, bb = parity.inputs(M, N, K, "TN", "bf16", ("int", -4, 4), 87)
    got = run(h, a, b, M, N, K, "TN", "f32", "bf16", "splitk", schedule="dynamic")
    ref, _, _ = oracle.gemm(ab, bb, M, N, K, "TN", "bf16", "bf16")
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("M,K", [(16, 1032), (33, 4104), (5, 520)])
def test_splitk_whole_tiles_ragged_k_from_every_offset(h, M, K):
    # Whole tiles walk K from (tile mod 8)/8 of their k-blocks and wrap, so with
    # a ragged K the short last k-block (zero-filled past K) falls in the middle
    # of most tiles' walks; 128 tiles cover all eight offsets.
    N = 16384
    st, p = hgemm.hgemm_plan(M, N, K, num_sms=torch.cuda.get_device_properties(0).multi_processor_count, stream_k=0)
    assert p.variant == hgemm.HGEMM_VARIANT_SPLITK and p.splitk_align == p.k_blocks and K % 128 != 0
    a, b, ab, bb = parity.inputs(M, N, K, "TN", "bf16", ("normal", 1.0), 94)
    got = run(h, a, b, M, N, K, "TN", "f32", "bf16", "splitk", stream_k=0)
    parity.check(got, ab, bb, M, N, K, "TN", "bf16", "f32", "bf16")
    a, b, ab, bb = parity.inputs(M, N, K, "TN", "bf16", ("int", -4, 4), 95)
    got = run(h, a, b, M, N, K, "TN", "f32", "bf16", "splitk", stream_k=0)
    ref, _, _ = oracle.gemm(ab, bb, M, N, K, "TN", "bf16", "bf16")
    assert np.array_equal(got, ref)


def test_splitk_small_integers_bit_exact(h):
    M, N, K = 16, 2048, 4096
    a, b, ab, bb = parity.inputs(M, N, K, "TN", "f16", ("int", -4, 4), 23)
    got = run(h, a, b, M, N, K, "TN", "f32", "f16", "splitk")
    ref, _, _ = oracle.gemm(ab, bb, M, N, K, "TN", "f16", "f16")
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("variant,M", [("2sm256", 640), ("1sm256", 640), ("1sm128", 640), ("splitk", 40)])
def test_run_to_run_determinism(h, variant, M):
    N, K = 1024, 2048
    a, b, _, _ = parity.inputs(M, N, K, "TN", "bf16", ("normal", 1.0), 31)
    first = run(h, a, b, M, N, K, "TN", "f32", "bf16", variant)
    for _ in range(3):
        assert np.array_equal(run(h, a, b, M, N, K, "TN", "f32", "bf16", variant), first)


@pytest.mark.parametrize("layout", ["TN", "NN"])
def test_variants_agree_bitwise(h, layout):
    # The dense variants differ only in data movement and tile shape; each output
    # is one tensor-core accumulation over K in the same order.
    M, N, K = 512, 512, 1024
    a, b, _, _ = parity.inputs(M, N, K, layout, "f16", ("uniform", -1.0, 1.0), 32)
    outs = [run(h, a, b, M, N, K, layout, "f32", "f16", v, stream_k=0) for v in DENSE_VARIANTS
            if not (layout == "NN" and v in NN_UNSUPPORTED)]
    for o in outs[1:]:
        assert np.array_equal(o, outs[0])


@pytest.mark.parametrize("stream_k", [1, 3], ids=["auto", "pieces"])
@pytest.mark.parametrize("variant", DENSE_VARIANTS)
@pytest.mark.parametrize("layout", ["TN", "NN"])
@pytest.mark.parametrize("combo", [("bf16", "f32", "bf16"), ("f16", "f16", "f16")], ids=["bf16", "f16acc"])
@pytest.mark.parametrize("M,N,K", [(1024, 1280, 1024), (768, 520, 4104), (256, 264, 200)])
def test_stream_k_parity(h, M, N, K, combo, layout, variant, stream_k):
    # Tile counts that leave a partial last wave, so stream-K splits tiles
    # (the estimate's choice, or every leftover tile cut into equal K pieces).
    fin, acc, out = combo
    st, p = hgemm.hgemm_plan(M, N, K, hgemm.LAYOUTS[layout], hgemm.DTYPES[fin], hgemm.DTYPES[acc], hgemm.DTYPES[out],
                             torch.cuda.get_device_properties(0).multi_processor_count, hgemm.VARIANTS[variant], 0,
                             stream_k)
    if layout == "NN" and variant in NN_UNSUPPORTED:
        assert st == hgemm.HGEMM_ERR_UNSUPPORTED
        pytest.skip("variant %s does not take the NN layout" % variant)
    assert st == 0
    if stream_k == 3:
        assert p.stream_k and p.sk_pieces >= 2
    a, b, ab, bb = parity.inputs(M, N, K, layout, fin, ("uniform", -1.0, 1.0), 61)
    got = run(h, a, b, M, N, K, layout, acc, out, variant, stream_k=stream_k)
    parity.check(got, ab, bb, M, N, K, layout, fin, acc, out)
    again = run(h, a, b, M, N, K, layout, acc, out, variant, stream_k=stream_k)
    assert np.array_equal(got, again)  # the fix-up order is fixed: run-to-run identical


@pytest.mark.parametrize("stream_k", [1, 2, 3], ids=["auto", "ranges", "pieces"])
@pytest.mark.parametrize("variant", DENSE_VARIANTS)
def test_stream_k_small_integers_bit_exact(h, variant, stream_k):
    M, N, K = 640, 640, 4096
    a, b, ab, bb = parity.inputs(M, N, K, "TN", "bf16", ("int", -4, 4), 62)
    got = run(h, a, b, M, N, K, "TN", "f32", "bf16", variant, stream_k=stream_k)
    ref, _, _ = oracle.gemm(ab, bb, M, N, K, "TN", "bf16", "bf16")
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("M,N,K", [(4096, 4096, 2048), (4096, 5120, 1024), (2560, 9984, 768)])
def test_stream_k_pieces_at_wave_scale(h, M, N, K):
    """Shapes with whole waves plus leftover tiles, planned the way the
    headline is (whole waves of 256 x 256 tiles, each leftover tile cut into
    2 to 4 equal K pieces): sampled parity against the oracle and run-to-run
    identity, for the estimate's plan and for equal ranges per cluster."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    st, p = hgemm.hgemm_plan(M, N, K, num_sms=sms)
    assert st == 0 and p.stream_k and p.sk_pieces >= 2 and p.dp_tiles > 0
    a, b, ab, bb = parity.inputs(M, N, K, "TN", "bf16", ("normal", 1.0), 63)
    for sk in (1, 2):
        got = run(h, a, b, M, N, K, "TN", "f32", "bf16", stream_k=sk)
        parity.check(got, ab, bb, M, N, K, "TN", "bf16", "f32", "bf16", sampled=True)
        assert np.array_equal(got, run(h, a, b, M, N, K, "TN", "f32", "bf16", stream_k=sk))


@pytest.mark.parametrize("M,N,K,layout,combo", [(4096, 4096, 1032, "NN", ("f16", "f16", "f16")),
                                                 (4096, 5120, 1080, "TN", ("bf16", "f32", "bf16")),
                                                 (2560, 9984, 776, "NN", ("bf16", "f32", "f16"))])
def test_stream_k_pieces_odd_k_blocks(h, M, N, K, layout, combo):
    """K pieces forced (stream-K 3) where the k-block count is odd, so a
    tile's pieces differ by one k-block, on NN and fp16-accumulate plans at
    wave scale: sampled parity and run-to-run identity."""
    fin, acc, out = combo
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    st, p = hgemm.hgemm_plan(M, N, K, hgemm.LAYOUTS[layout], hgemm.DTYPES[fin], hgemm.DTYPES[acc], hgemm.DTYPES[out],
                             sms, hgemm.HGEMM_VARIANT_AUTO, 0, 3)
    assert st == 0 and p.stream_k and p.sk_pieces >= 2 and p.dp_tiles > 0 and p.k_blocks % 2 == 1
    a, b, ab, bb = parity.inputs(M, N, K, layout, fin, ("uniform", -1.0, 1.0), 64)
    got = run(h, a, b, M, N, K, layout, acc, out, stream_k=3)
    parity.check(got, ab, bb, M, N, K, layout, fin, acc, out, sampled=True)
    assert np.array_equal(got, run(h, a, b, M, N, K, layout, acc, out, stream_k=3))


# Dynamic schedule (cluster launch control).  Shapes with more work ids than
# resident clusters, so that running clusters cancel pending ones and take
# their ids, with and without stream-K ranges; plus a ragged shape.
DYNAMIC_CASES = [("2sm256", 4096, 4096, 128, 1), ("2sm256", 4096, 4096, 128, 0), ("1sm128", 2048, 2048, 256, 0),
                 ("1sm256", 2048, 4096, 192, 1), ("2sm192", 2048, 3072, 136, 1), ("2sm256", 1000, 3000, 4104, 1),
                 ("1sm128", 130, 136, 72, 1), ("2sm256", 4096, 4096, 1024, 3), ("2sm256", 4096, 4096, 256, 2),
                 ("1sm128", 1000, 3000, 520, 3)]


@pytest.mark.parametrize("variant,M,N,K,sk", DYNAMIC_CASES)
def test_dynamic_schedule_parity(h, variant, M, N, K, sk):
    a, b, ab, bb = parity.inputs(M, N, K, "TN", "bf16", ("normal", 1.0), 81)
    got = run(h, a, b, M, N, K, "TN", "f32", "bf16", variant, stream_k=sk, schedule="dynamic")
    parity.check(got, ab, bb, M, N, K, "TN", "bf16", "f32", "bf16")
    # the same ids with the same contents: bitwise equal to the static schedule
    ref = run(h, a, b, M, N, K, "TN", "f32", "bf16", variant, stream_k=sk, schedule="static")
    assert np.array_equal(got, ref)
    again = run(h, a, b, M, N, K, "TN", "f32", "bf16", variant, stream_k=sk, schedule="dynamic")
    assert np.array_equal(got, again)


@pytest.mark.parametrize("variant", ["2sm256", "1sm128"])
def test_dynamic_schedule_nn_f16_acc_and_integers(h, variant):
    M, N, K = 2048, 2560, 1024
    a, b, ab, bb = parity.inputs(M, N, K, "NN", "f16", ("uniform", -1.0, 1.0), 82)
    got = run(h, a, b, M, N, K, "NN", "f16", "f16", variant, schedule="dynamic")
    parity.check(got, ab, bb, M, N, K, "NN", "f16", "f16", "f16")
    M, N, K = 2048, 2048, 1024
    a, b, ab, bb = parity.inputs(M, N, K, "TN", "bf16", ("int", -4, 4), 83)
    got = run(h, a, b, M, N, K, "TN", "f32", "bf16", variant, schedule="dynamic")
    ref, _, _ = oracle.gemm(ab, bb, M, N, K, "TN", "bf16", "bf16")
    assert np.array_equal(got, ref)


# Direct-store epilogue: same bits as the TMA-store epilogue, ragged edges
# clipped by the stores' own bounds checks.
DIRECT_CASES = [("1sm128", "TN", 1000, 1000, 1024, ("bf16", "f32", "bf16")),
                ("1sm256", "NN", 129, 264, 640, ("f16", "f32", "f16")),
                ("2sm256", "TN", 1024, 1280, 1024, ("bf16", "f32", "bf16")),
                ("2sm256", "NN", 768, 520, 4104, ("f16", "f16", "f16")),
                ("2sm192", "TN", 1000, 3000, 4104, ("bf16", "f32", "f16")),
                ("2sm256", "TN", 1, 8, 8, ("bf16", "f32", "bf16"))]


@pytest.mark.parametrize("variant,layout,M,N,K,combo", DIRECT_CASES)
def test_direct_epilogue_parity(h, variant, layout, M, N, K, combo):
    fin, acc, out = combo
    a, b, ab, bb = parity.inputs(M, N, K, layout, fin, ("uniform", -1.0, 1.0), 84)
    got = run(h, a, b, M, N, K, layout, acc, out, variant, epilogue="direct")
    parity.check(got, ab, bb, M, N, K, layout, fin, acc, out)
    ref = run(h, a, b, M, N, K, layout, acc, out, variant, epilogue="tma")
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("variant,M,N,K", [("2sm256", 300, 264, 200), ("1sm128", 130, 136, 72),
                                           ("2sm192", 257, 392, 136), ("splitk", 17, 1000, 8192)])
def test_direct_epilogue_guard_bands_untouched(h, variant, M, N, K):
    a, b, ab, bb = parity.inputs(M, N, K, "TN", "bf16", ("normal", 1.0), 85)
    pad = 4096
    buf = torch.full((pad + M * N + pad,), 0x7E7E, dtype=torch.int16, device="cuda")
    C = buf[pad:pad + M * N].view(torch.bfloat16).view(M, N)
    got = run(h, a, b, M, N, K, "TN", "f32", "bf16", variant, C=C, epilogue="direct", schedule="dynamic")
    parity.check(got, ab, bb, M, N, K, "TN", "bf16", "f32", "bf16")
    host = buf.cpu().numpy()
    assert np.all(host[:pad] == 0x7E7E) and np.all(host[pad + M * N:] == 0x7E7E)


@pytest.mark.parametrize("variant,M,N,K", [("2sm256", 300, 264, 200), ("1sm128", 130, 136, 72),
                                           ("splitk", 17, 520, 200), ("1sm256", 1, 8, 8)])
def test_guard_bands_untouched(h, variant, M, N, K):
    a, b, ab, bb = parity.inputs(M, N, K, "TN", "bf16", ("normal", 1.0), 41)
    pad = 4096
    buf = torch.full((pad + M * N + pad,), 0x7E7E, dtype=torch.int16, device="cuda")
    C = buf[pad:pad + M * N].view(torch.bfloat16).view(M, N)
    got = run(h, a, b, M, N, K, "TN", "f32", "bf16", variant, C=C)
    parity.check(got, ab, bb, M, N, K, "TN", "bf16", "f32", "bf16")
    host = buf.cpu().numpy()
    assert np.all(host[:pad] == 0x7E7E) and np.all(host[pad + M * N:] == 0x7E7E)


def test_k_zero_fills_zero(h):
    M, N = 100, 72
    C = torch.full((M, N), 3.0, dtype=torch.float16, device="cuda")
    A = torch.empty((M, 0), dtype=torch.float16, device="cuda")
    B = torch.empty((N, 0), dtype=torch.float16, device="cuda")
    st = hgemm.hgemm_run(h.h, A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, 0, hgemm.HGEMM_LAYOUT_TN,
                         hgemm.HGEMM_F16, hgemm.HGEMM_F32, hgemm.HGEMM_F16, torch.cuda.current_stream().cuda_stream)
    assert st == hgemm.HGEMM_OK
    assert h.sync_status()[0] == hgemm.HGEMM_OK
    bits = workloads.bits(C.cpu())
    assert np.all(bits == 0)  # +0, not -0


def test_empty_m_or_n_is_noop(h):
    C = torch.full((4, 8), 1.0, dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    for M, N in [(0, 8), (4, 0)]:
        assert hgemm.hgemm_run(h.h, 0, 0, C.data_ptr(), M, N, 64, 0, 1, 2, 1, s) == hgemm.HGEMM_OK
    assert h.sync_status()[0] == hgemm.HGEMM_OK
    assert torch.all(C == 1.0)


def test_argument_validation(h):
    s = torch.cuda.current_stream().cuda_stream
    A = torch.zeros((64, 64), dtype=torch.float16, device="cuda")
    B = torch.zeros((64, 64), dtype=torch.float16, device="cuda")
    C = torch.zeros((64, 64), dtype=torch.float16, device="cuda")
    a, b, c = A.data_ptr(), B.data_ptr(), C.data_ptr()
    F16, BF16, F32 = hgemm.HGEMM_F16, hgemm.HGEMM_BF16, hgemm.HGEMM_F32
    R = hgemm.hgemm_run
    assert R(0, a, b, c, 64, 64, 64, 0, F16, F32, F16, s) == hgemm.HGEMM_ERR_INVALID_ARG
    assert R(h.h, 0, b, c, 64, 64, 64, 0, F16, F32, F16, s) == hgemm.HGEMM_ERR_INVALID_ARG
    assert R(h.h, a, 0, c, 64, 64, 64, 0, F16, F32, F16, s) == hgemm.HGEMM_ERR_INVALID_ARG
    assert R(h.h, a, b, 0, 64, 64, 64, 0, F16, F32, F16, s) == hgemm.HGEMM_ERR_INVALID_ARG
    assert R(h.h, a, b, c, -1, 64, 64, 0, F16, F32, F16, s) == hgemm.HGEMM_ERR_INVALID_ARG
    assert R(h.h, a, b, c, 64, 64, 1 << 31, 0, F16, F32, F16, s) == hgemm.HGEMM_ERR_INVALID_ARG
    assert R(h.h, a, b, c, 64, 64, 64, 2, F16, F32, F16, s) == hgemm.HGEMM_ERR_INVALID_ARG
    assert R(h.h, a, b, c, 64, 64, 64, 0, 7, F32, F16, s) == hgemm.HGEMM_ERR_INVALID_ARG
    assert R(h.h, a, b, c, 64, 64, 64, 0, BF16, F16, F16, s) == hgemm.HGEMM_ERR_UNSUPPORTED
    assert R(h.h, a, b, c, 64, 64, 64, 0, F32, F32, F16, s) == hgemm.HGEMM_ERR_UNSUPPORTED
    assert R(h.h, a, b, c, 64, 64, 64, 0, F16, F32, F32, s) == hgemm.HGEMM_ERR_UNSUPPORTED
    assert R(h.h, a + 2, b, c, 64, 64, 64, 0, F16, F32, F16, s) == hgemm.HGEMM_ERR_MISALIGNED
    assert R(h.h, a, b + 8, c, 64, 64, 56, 0, F16, F32, F16, s) == hgemm.HGEMM_ERR_MISALIGNED
    assert R(h.h, a, b, c + 2, 64, 56, 64, 0, F16, F32, F16, s) == hgemm.HGEMM_ERR_MISALIGNED
    assert R(h.h, a, b, c, 64, 60, 64, 0, F16, F32, F16, s) == hgemm.HGEMM_ERR_MISALIGNED   # N % 8
    assert R(h.h, a, b, c, 64, 64, 60, 0, F16, F32, F16, s) == hgemm.HGEMM_ERR_MISALIGNED   # K % 8
    assert R(h.h, a, b, a, 64, 64, 64, 0, F16, F32, F16, s) == hgemm.HGEMM_ERR_ALIAS
    assert R(h.h, a, b, b + 128, 8, 8, 64, 0, F16, F32, F16, s) == hgemm.HGEMM_ERR_ALIAS
    assert h.sync_status()[0] == hgemm.HGEMM_OK
    assert torch.all(C == 0)  # nothing was launched


@pytest.mark.parametrize("variant,M,schedule", [("1sm128", 512, "static"), ("2sm256", 512, "static"),
                                                ("splitk", 16, "static"), ("1sm128", 4096, "dynamic"),
                                                ("2sm256", 4096, "dynamic"), ("splitk", 16, "dynamic")])
def test_bounded_wait_gives_up_and_recovers(h, variant, M, schedule):
    # The first CTA's producer drops its first stage; the MMA warp's wait on that
    # stage can never succeed, gives up after the limit, and every role exits.
    N, K = 1024, 1024
    a, b, ab, bb = parity.inputs(M, N, K, "TN", "bf16", ("normal", 1.0), 51)
    A, B = a.cuda(), b.cuda()
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    h.set_option(hgemm.HGEMM_OPT_FORCE_VARIANT, hgemm.VARIANTS[variant])
    h.set_option(hgemm.HGEMM_OPT_TIMEOUT_NS, 20_000_000)
    h.set_option(hgemm.HGEMM_OPT_INJECT_FAULT, 1)
    h.set_option(hgemm.HGEMM_OPT_SCHEDULE, hgemm.SCHEDULES[schedule])
    try:
        h.run(A, B, C, layout="TN", acc="f32")
        st, detail = h.sync_status()
        assert st == hgemm.HGEMM_ERR_TIMEOUT, (st, hex(detail))
        assert (detail & 0xFF) == hgemm.HGEMM_ERR_TIMEOUT and ((detail >> 8) & 0xFF) in (1, 2, 3, 4)
    finally:
        h.set_option(hgemm.HGEMM_OPT_INJECT_FAULT, 0)
        h.set_option(hgemm.HGEMM_OPT_TIMEOUT_NS, 2_000_000_000)
        h.set_option(hgemm.HGEMM_OPT_FORCE_VARIANT, hgemm.HGEMM_VARIANT_AUTO)
        h.set_option(hgemm.HGEMM_OPT_SCHEDULE, hgemm.HGEMM_SCHEDULE_STATIC)
        h.set_option(hgemm.HGEMM_OPT_EPILOGUE, hgemm.HGEMM_EPILOGUE_TMA_STORE)
    # the context is still usable and the next launch is correct
    got = run(h, a, b, M, N, K, "TN", "f32", "bf16", variant, schedule=schedule)
    parity.check(got, ab, bb, M, N, K, "TN", "bf16", "f32", "bf16")


# Checked mode (HGEMM_OPT_CHECKS): valid runs of every kind report nothing.
CHECKED_CASES = [("2sm256", "TN", 4096, 4096, 256, 2, "static"), ("2sm256", "TN", 4096, 4096, 256, 2, "dynamic"),
                 ("1sm128", "NN", 1000, 3000, 520, 1, "dynamic"), ("2sm192", "TN", 1000, 3000, 4104, 1, "static"),
                 ("1sm256", "TN", 2048, 4096, 192, 1, "dynamic"), ("2sm256", "NN", 768, 520, 4104, 1, "static"),
                 ("splitk", "TN", 16, 16384, 4096, 1, "static"), ("splitk", "TN", 16, 16384, 4096, 2, "static"),
                 ("splitk", "TN", 40, 8192, 8192, 1, "dynamic"),
                 ("2sm256", "TN", 4096, 4096, 1024, 3, "static"), ("2sm256", "NN", 4096, 4096, 1024, 3, "dynamic"),
                 ("1sm128", "TN", 1000, 3000, 520, 3, "static")]


@pytest.mark.parametrize("variant,layout,M,N,K,sk,schedule", CHECKED_CASES)
def test_checked_runs_report_nothing(h, variant, layout, M, N, K, sk, schedule):
    a, b, ab, bb = parity.inputs(M, N, K, layout, "bf16", ("normal", 1.0), 88)
    h.set_option(hgemm.HGEMM_OPT_CHECKS, 1)
    try:
        got = run(h, a, b, M, N, K, layout, "f32", "bf16", variant, stream_k=sk, schedule=schedule)
    finally:
        h.set_option(hgemm.HGEMM_OPT_CHECKS, 0)
    parity.check(got, ab, bb, M, N, K, layout, "bf16", "f32", "bf16")


@pytest.mark.parametrize("sk", [2, 3], ids=["ranges", "pieces"])
@pytest.mark.parametrize("variant,M,N,K,schedule", [("2sm256", 4096, 4096, 256, "static"),
                                                    ("2sm256", 4096, 4096, 256, "dynamic"),
                                                    ("splitk", 16, 16384, 4096, "static"),
                                                    ("splitk", 16, 16384, 4096, "dynamic")])
def test_checks_catch_corrupted_tickets(h, variant, M, N, K, schedule, sk):
    # The host fills the fix-up ticket counters with 0x01 bytes before the
    # launch: every ticket is then far past its tile's contributor count.  The
    # kernels only compare tickets (no access depends on them, no wait), so the
    # launch ends; the checks must report it.  The next launch is correct.
    a, b, ab, bb = parity.inputs(M, N, K, "TN", "bf16", ("normal", 1.0), 89)
    A, B = a.cuda(), b.cuda()
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    h.set_option(hgemm.HGEMM_OPT_FORCE_VARIANT, hgemm.VARIANTS[variant])
    h.set_option(hgemm.HGEMM_OPT_SCHEDULE, hgemm.SCHEDULES[schedule])
    h.set_option(hgemm.HGEMM_OPT_STREAM_K, sk)  # split the dense tiles even where the estimate would not
    h.set_option(hgemm.HGEMM_OPT_CHECKS, 1)
    h.set_option(hgemm.HGEMM_OPT_INJECT_FAULT, 2)
    try:
        h.run(A, B, C, layout="TN", acc="f32")
        st, detail = h.sync_status()
        assert st == hgemm.HGEMM_ERR_CHECK, (st, hex(detail))
        assert (detail & 0xFF) == hgemm.HGEMM_ERR_CHECK and ((detail >> 8) & 0xFF) == hgemm.HGEMM_CHECK_TICKET
    finally:
        h.set_option(hgemm.HGEMM_OPT_INJECT_FAULT, 0)
        h.set_option(hgemm.HGEMM_OPT_CHECKS, 0)
        h.set_option(hgemm.HGEMM_OPT_STREAM_K, 1)
        h.set_option(hgemm.HGEMM_OPT_SCHEDULE, hgemm.HGEMM_SCHEDULE_STATIC)
        h.set_option(hgemm.HGEMM_OPT_FORCE_VARIANT, hgemm.HGEMM_VARIANT_AUTO)
    got = run(h, a, b, M, N, K, "TN", "f32", "bf16", variant, stream_k=2, schedule=schedule)
    parity.check(got, ab, bb, M, N, K, "TN", "bf16", "f32", "bf16")


@pytest.mark.parametrize("pinned", [True, False], ids=["pinned", "pageable"])
@pytest.mark.parametrize("layout", ["TN", "NN"])
@pytest.mark.parametrize("M,N,K", [(1000, 1000, 1024), (3000, 520, 200), (16, 2048, 4096), (5, 8, 0)])
def test_run_host_end_to_end(h, M, N, K, layout, pinned):
    a, b, ab, bb = parity.inputs(M, N, K, layout, "bf16", ("normal", 1.0), 81)
    if pinned:
        a, b = a.pin_memory(), b.pin_memory()
    C = torch.full((M, N), float("nan"), dtype=torch.bfloat16)
    if pinned:
        C = C.pin_memory()
    h.run_host(a, b, C, layout=layout, acc="f32")
    st, detail = h.sync_status()
    assert st == hgemm.HGEMM_OK, hex(detail)
    parity.check(workloads.bits(C), ab, bb, M, N, K, layout, "bf16", "f32", "bf16")


def test_run_host_back_to_back_calls(h):
    # Consecutive calls alternate between two staging sets and overlap on the
    # device; every output must still be the product of its own inputs.
    M, N, K = 1536, 1024, 512
    sets = [parity.inputs(M, N, K, "TN", "f16", ("uniform", -1.0, 1.0), 90 + i) for i in range(4)]
    # The pinned copies stay referenced until the copies have run: the host
    # allocator may hand a freed block to the next pin_memory() at once.
    pinned = [(a.pin_memory(), b.pin_memory()) for a, b, _, _ in sets]
    outs = []
    for ap, bp in pinned:
        C = torch.empty((M, N), dtype=torch.float16).pin_memory()
        h.run_host(ap, bp, C, layout="TN", acc="f32")
        outs.append(C)
    assert h.sync_status()[0] == hgemm.HGEMM_OK
    for (a, b, ab, bb), C in zip(sets, outs):
        parity.check(workloads.bits(C), ab, bb, M, N, K, "TN", "f16", "f32", "f16")


def test_run_host_alternating_streams(h):
    # The benchmark's end-to-end loop: consecutive calls alternate between two
    # caller streams, so one call's uploads overlap the previous call's GEMM
    # and download.  Six calls reuse each staging set three times; every output
    # must be the product of its own inputs.
    M, N, K = 2048, 1536, 1024
    sets = [parity.inputs(M, N, K, "TN", "bf16", ("normal", 1.0), 95 + i) for i in range(6)]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    pinned = [(a.pin_memory(), b.pin_memory()) for a, b, _, _ in sets]
    outs = []
    for i, (ap, bp) in enumerate(pinned):
        C = torch.full((M, N), float("nan"), dtype=torch.bfloat16).pin_memory()
        h.run_host(ap, bp, C, layout="TN", acc="f32", stream=streams[i % 2])
        outs.append(C)
    torch.cuda.synchronize()
    assert h.sync_status()[0] == hgemm.HGEMM_OK
    for (a, b, ab, bb), C in zip(sets, outs):
        parity.check(workloads.bits(C), ab, bb, M, N, K, "TN", "bf16", "f32", "bf16")


def test_tensor_maps_follow_shape_and_type(h):
    # One allocation per operand, reused with other shapes, element types and
    # kernels (dense and split-K), then with the first again: every result
    # must be the product of its own operands.
    buf_a = torch.empty(1 << 20, dtype=torch.int16, device="cuda")
    buf_b = torch.empty(1 << 21, dtype=torch.int16, device="cuda")
    buf_c = torch.empty(1 << 20, dtype=torch.int16, device="cuda")
    cases = [(512, 768, 1024, "bf16"), (768, 512, 1024, "bf16"), (512, 768, 512, "f16"), (16, 2048, 1024, "bf16"),
             (16, 1024, 2048, "bf16"), (512, 768, 1024, "bf16")]
    for i, (M, N, K, dt) in enumerate(cases):
        a, b, ab, bb = parity.inputs(M, N, K, "TN", dt, ("normal", 1.0), 140 + i)
        A = buf_a[:M * K].view(TORCH_DT[dt]).view(M, K)
        B = buf_b[:N * K].view(TORCH_DT[dt]).view(N, K)
        C = buf_c[:M * N].view(TORCH_DT[dt]).view(M, N)
        A.copy_(a.cuda())
        B.copy_(b.cuda())
        C.fill_(float("nan"))
        h.run(A, B, C, layout="TN", acc="f32")
        st, detail = h.sync_status()
        assert st == hgemm.HGEMM_OK, hex(detail)
        parity.check(workloads.bits(C.cpu()), ab, bb, M, N, K, "TN", dt, "f32", dt)


def test_env_force_variant(monkeypatch):
    # HGEMM_FORCE_VARIANT pins the variant of the handles created while it is
    # set: forced split-K refuses M > 64; a forced 1-SM tile computes as usual.
    M, N, K = 128, 256, 256
    a, b, ab, bb = parity.inputs(M, N, K, "TN", "bf16", ("normal", 1.0), 93)
    A, B = a.cuda(), b.cuda()
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    monkeypatch.setenv("HGEMM_FORCE_VARIANT", "splitk")
    with hgemm.Handle() as h:
        assert h.run(A, B, C, layout="TN", acc="f32", check=False) == hgemm.HGEMM_ERR_UNSUPPORTED
    monkeypatch.setenv("HGEMM_FORCE_VARIANT", "1sm128")
    with hgemm.Handle() as h:
        h.run(A, B, C, layout="TN", acc="f32")
        assert h.sync_status()[0] == hgemm.HGEMM_OK
    parity.check(workloads.bits(C.cpu()), ab, bb, M, N, K, "TN", "bf16", "f32", "bf16")
    monkeypatch.delenv("HGEMM_FORCE_VARIANT")
    with hgemm.Handle() as h:  # unset: automatic again
        assert h.run(A, B, C, layout="TN", acc="f32", check=False) == hgemm.HGEMM_OK
