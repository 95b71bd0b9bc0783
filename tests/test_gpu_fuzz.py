"""Seeded random crossings of shape and every option of the dense and split-K
paths, each checked against the oracle (all entries of the small products,
sampled entries plus tile-boundary rows and columns of the others).

The feature tests pin each option on its own; these draws cross them --
variant x layout x dtypes x stream-K mode x schedule x epilogue x
rasterisation height x ragged M, N, K -- where an interaction between two
options would otherwise go unseen.  A forced variant that cannot take the
drawn problem must say so (HGEMM_ERR_UNSUPPORTED) and launch nothing."""
import numpy as np
import pytest
import torch

from tests import parity
from tensor_core_half_gb300 import hgemm, workloads

pytestmark = pytest.mark.gpu

TORCH_DT = {"f16": torch.float16, "bf16": torch.bfloat16}
COMBOS = [("bf16", "f32", "bf16"), ("f16", "f32", "f16"), ("f16", "f32", "bf16"), ("bf16", "f32", "f16"),
          ("f16", "f16", "f16"), ("f16", "f16", "bf16")]
VARIANTS = ["auto", "1sm128", "1sm256", "2sm256", "2sm192", "splitk"]
FULL_CHECK_MACS = 3e8  # products up to this size are compared entry by entry


def _draws(n, seed):
    r = np.random.default_rng(seed)
    out = []
    for i in range(n):
        variant = VARIANTS[int(r.integers(len(VARIANTS)))]
        if variant == "splitk":
            M = int(r.integers(1, 65))
            layout = "TN"
            combo = COMBOS[int(r.integers(4))]  # fp32 accumulation
        else:
            M = int(r.choice([1, 7, 100, 128, 255, 256, 257, 600, 1000, 1500, 2100]))
            layout = str(r.choice(["TN", "NN"]))
            combo = COMBOS[int(r.integers(len(COMBOS)))]
        N = 8 * int(r.integers(1, 420))
        K = 8 * int(r.integers(1, 320))
        out.append(dict(case=i, seed=seed, M=M, N=N, K=K, layout=layout, combo=combo, variant=variant,
                        stream_k=int(r.integers(0, 4)), schedule=str(r.choice(["static", "dynamic"])),
                        epilogue=str(r.choice(["tma", "direct"])), group_m=int(r.choice([0, 1, 3, 8, 16]))))
    return out


CASES = _draws(32, 901) + _draws(32, 902) + _draws(32, 903)


@pytest.fixture(scope="module")
def h():
    handle = hgemm.Handle()
    yield handle
    handle.close()


@pytest.mark.parametrize("d", CASES, ids=lambda d: "s%d-%d-%s-%dx%dx%d" % (d["seed"], d["case"], d["variant"],
                                                                            d["M"], d["N"], d["K"]))
def test_random_crossing_matches_the_oracle(h, d):
    M, N, K, layout = d["M"], d["N"], d["K"], d["layout"]
    fin, acc, out = d["combo"]
    a, b, ab, bb = parity.inputs(M, N, K, layout, fin, ("normal", 1.0), 1000 * d["seed"] + d["case"])
    A, B = a.cuda(), b.cuda()
    C = torch.empty((M, N), dtype=TORCH_DT[out], device="cuda")
    h.set_option(hgemm.HGEMM_OPT_FORCE_VARIANT, hgemm.VARIANTS[d["variant"]])
    h.set_option(hgemm.HGEMM_OPT_STREAM_K, d["stream_k"])
    h.set_option(hgemm.HGEMM_OPT_SCHEDULE, hgemm.SCHEDULES[d["schedule"]])
    h.set_option(hgemm.HGEMM_OPT_EPILOGUE, hgemm.EPILOGUES[d["epilogue"]])
    h.set_option(hgemm.HGEMM_OPT_GROUP_M, d["group_m"])
    try:
        st = h.run(A, B, C, layout=layout, acc=acc, check=False)
        nn_192 = d["variant"] == "2sm192" and layout == "NN"
        if nn_192:  # 192-column tiles split B into 96-column halves: TN only
            assert st == hgemm.HGEMM_ERR_UNSUPPORTED
            return
        assert st == hgemm.HGEMM_OK, hgemm.hgemm_status_string(st)
        st, detail = h.sync_status()
        assert st == hgemm.HGEMM_OK, (hgemm.hgemm_status_string(st), hex(detail))
    finally:
        h.set_option(hgemm.HGEMM_OPT_FORCE_VARIANT, hgemm.HGEMM_VARIANT_AUTO)
        h.set_option(hgemm.HGEMM_OPT_STREAM_K, 1)
        h.set_option(hgemm.HGEMM_OPT_SCHEDULE, hgemm.HGEMM_SCHEDULE_STATIC)
        h.set_option(hgemm.HGEMM_OPT_EPILOGUE, hgemm.HGEMM_EPILOGUE_TMA_STORE)
        h.set_option(hgemm.HGEMM_OPT_GROUP_M, 0)
    got = workloads.bits(C.cpu())
    full = float(M) * N * K <= FULL_CHECK_MACS
    parity.check(got, ab, bb, M, N, K, layout, fin, acc, out, sampled=not full, n_random=4096, seed=d["case"])
