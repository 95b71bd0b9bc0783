"""The intra-kernel tracer records exactly the schedule the planner describes,
and a traced launch still computes the right C: tracing adds global stores to
every role of both kernels (producer, MMA issuer, epilogue, stream-K and
split-K fix-ups), so every traced result is checked against the oracle."""
import collections

import pytest
import torch

from tests import parity
from tensor_core_half_gb300 import hgemm, trace

pytestmark = pytest.mark.gpu


def _traced_run(h, M, N, K, seed, capacity):
    """Runs one traced bf16 TN product, checks C against the oracle (in full:
    every shape here is small enough) and returns the trace records."""
    a, b, ab, bb = parity.inputs(M, N, K, "TN", "bf16", ("normal", 1.0), seed)
    A, B = a.cuda(), b.cuda()
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    h.run(A, B, C, layout="TN", acc="f32")
    st, detail = h.sync_status()
    assert st == hgemm.HGEMM_OK, (st, hex(detail))
    st, n, rows = hgemm.hgemm_trace_read(h.h, capacity)
    assert st == hgemm.HGEMM_OK and n == len(rows) > 0
    got = C.view(torch.int16).cpu().numpy().view("uint16")
    parity.check(got, ab, bb, M, N, K, "TN", "bf16", "f32", "bf16")
    return rows


# Stream-K 2 splits every tile of a partial wave between clusters, so the
# traced fix-up path (partials published, the last contributor's reduction)
# runs on every tile; 3 cuts the tiles left after whole waves into equal K
# pieces; the split-K cases run the whole-tile and the balanced split layouts.
TRACE_CASES = [("2sm256", 1024, 1280, 1024, 1), ("1sm128", 640, 1000, 4104, 1), ("splitk", 16, 4096, 4096, 1),
               ("2sm256", 1000, 3000, 4104, 2), ("2sm192", 768, 520, 4104, 2), ("1sm256", 640, 1000, 1032, 2),
               ("1sm128", 256, 264, 200, 2), ("splitk", 48, 3000, 2000, 2), ("splitk", 16, 16384, 2048, 0),
               ("2sm256", 4096, 2560, 512, 3), ("1sm128", 1000, 3000, 520, 3)]


@pytest.mark.parametrize("variant,M,N,K,sk", TRACE_CASES)
def test_trace_matches_plan(variant, M, N, K, sk):
    with hgemm.Handle() as h:
        h.set_option(hgemm.HGEMM_OPT_FORCE_VARIANT, hgemm.VARIANTS[variant])
        h.set_option(hgemm.HGEMM_OPT_STREAM_K, sk)
        h.set_option(hgemm.HGEMM_OPT_TRACE, 1 << 16)
        rows = _traced_run(h, M, N, K, 71, 1 << 16)
        st2, n2, _ = hgemm.hgemm_trace_read(h.h, 16)
        assert st2 == hgemm.HGEMM_OK and n2 == 0  # reading empties the buffer
        # The same handle with tracing off gives the same bits: the trace
        # records add stores but change neither the schedule nor the sums.
        h.set_option(hgemm.HGEMM_OPT_TRACE, 0)
        a, b, _, _ = parity.inputs(M, N, K, "TN", "bf16", ("normal", 1.0), 71)
        A, B = a.cuda(), b.cuda()
        C0 = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        C1 = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        h.run(A, B, C0, layout="TN", acc="f32")
        h.set_option(hgemm.HGEMM_OPT_TRACE, 1 << 16)
        h.run(A, B, C1, layout="TN", acc="f32")
        assert h.sync_status()[0] == hgemm.HGEMM_OK
        assert torch.equal(C0.view(torch.int16), C1.view(torch.int16))
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    st, p = hgemm.hgemm_plan(M, N, K, 0, hgemm.HGEMM_BF16, hgemm.HGEMM_F32, hgemm.HGEMM_BF16, sms,
                             hgemm.VARIANTS[variant], 0, sk)
    kinds = collections.Counter((r[2], r[3]) for r in rows)
    assert kinds[(0, 1)] == p.grid and kinds[(0, 2)] == p.grid  # every CTA begins and ends
    if variant == "splitk":
        return
    if sk == 2:
        assert p.stream_k and p.dp_tiles == 0  # every tile is split
    if sk == 3:
        assert p.stream_k and p.sk_pieces >= 2 and p.dp_tiles > 0  # whole waves, then equal K pieces
    clusters = p.grid // p.cta_group
    items, partials = 0, 0
    for c in range(clusters):
        i = 0
        while True:
            s, t, a0, b0, slot = hgemm.hgemm_plan_work_item(p, c, i)
            if s != 0:
                break
            items += 1
            partials += slot >= 0
            i += 1
    # producer and epilogue run in every CTA; the MMA issuer in one CTA per cluster
    assert kinds[(1, 3)] == kinds[(1, 4)] == items * p.cta_group
    assert kinds[(2, 3)] == kinds[(2, 4)] == items
    assert kinds[(3, 3)] == kinds[(3, 4)] == items * p.cta_group
    # every partial item either publishes its partial or, arriving last, reduces the tile
    assert kinds[(3, 5)] + kinds[(3, 6)] == partials * p.cta_group
    # each split tile is reduced once per CTA of the pair, by its last contributor
    split_tiles = len({t for c in range(clusters) for t in _partial_tiles(p, c)})
    assert kinds[(3, 6)] == split_tiles * p.cta_group
    s = trace.summary(rows)
    assert s["items"] == items * (1 + 2 * p.cta_group)


def _partial_tiles(p, c):
    i, out = 0, []
    while True:
        s, t, a0, b0, slot = hgemm.hgemm_plan_work_item(p, c, i)
        if s != 0:
            return out
        if slot >= 0:
            out.append(t)
        i += 1


@pytest.mark.parametrize("variant,M,N,K,sk", [("2sm256", 4096, 4096, 256, 1), ("1sm128", 2048, 4096, 128, 0)])
def test_dynamic_schedule_takes_over_pending_clusters(variant, M, N, K, sk):
    """Under the dynamic schedule one cluster is launched per work id, but the
    clusters that start first cancel the launch of the others and run their
    ids: fewer CTAs begin than were launched, and every id's items appear
    exactly once."""
    with hgemm.Handle() as h:
        h.set_option(hgemm.HGEMM_OPT_FORCE_VARIANT, hgemm.VARIANTS[variant])
        h.set_option(hgemm.HGEMM_OPT_STREAM_K, sk)
        h.set_option(hgemm.HGEMM_OPT_SCHEDULE, hgemm.HGEMM_SCHEDULE_DYNAMIC)
        h.set_option(hgemm.HGEMM_OPT_TRACE, 1 << 18)
        rows = _traced_run(h, M, N, K, 72, 1 << 18)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    st, p = hgemm.hgemm_plan(M, N, K, 0, hgemm.HGEMM_BF16, hgemm.HGEMM_F32, hgemm.HGEMM_BF16, sms,
                             hgemm.VARIANTS[variant], 0, sk)
    launched = p.work_ids * p.cta_group
    began = collections.Counter(r[1] for r in rows if r[2] == 0 and r[3] == 1)
    assert p.work_ids > p.grid // p.cta_group  # more ids than resident clusters
    assert 0 < len(began) <= p.grid < launched  # only resident CTAs ran; the rest were cancelled
    expect = collections.Counter()
    for i in range(p.work_ids):
        j = 0
        while True:
            s, t, a0, b0, slot = hgemm.hgemm_plan_id_item(p, i, j)
            if s != 0:
                break
            expect[(t, a0, b0)] += 1
            j += 1
    # MMA issuer items (one per cluster): item_begin carries (tile, kb0), item_end (tile, kb1)
    got = collections.Counter()
    for sp in trace.spans(rows):
        if sp["role"] == "mma":
            got[(sp["tile"], sp["begin_value"], sp["end_value"])] += 1
    assert got == expect


def test_dynamic_splitk_takes_over_small_chunks():
    """Dynamic split-K: one CTA is launched per chunk, the CTAs that run
    first take over the small chunks, and every (tile, k-block) unit is
    multiplied exactly once."""
    M, N, K = 16, 16384, 4096
    with hgemm.Handle() as h:
        h.set_option(hgemm.HGEMM_OPT_SCHEDULE, hgemm.HGEMM_SCHEDULE_DYNAMIC)
        h.set_option(hgemm.HGEMM_OPT_TRACE, 1 << 18)
        rows = _traced_run(h, M, N, K, 73, 1 << 18)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    st, p = hgemm.hgemm_plan(M, N, K, num_sms=sms, schedule=hgemm.HGEMM_SCHEDULE_DYNAMIC)
    assert p.variant == hgemm.HGEMM_VARIANT_SPLITK and p.splitk_chunks > p.grid
    began = {r[1] for r in rows if r[2] == 0 and r[3] == 1}
    assert 0 < len(began) <= p.grid < p.splitk_chunks
    covered = collections.Counter()
    for sp in trace.spans(rows):
        if sp["role"] == "mma":
            for kb in range(sp["begin_value"], sp["end_value"]):
                covered[(sp["tile"], kb)] += 1
    assert len(covered) == p.num_tiles * p.k_blocks and set(covered.values()) == {1}


@pytest.mark.parametrize("M,N,K", [(16, 16384, 8192), (16, 4096, 4096), (48, 3000, 2000)])
def test_splitk_segments_in_plan_order(M, N, K):
    """Static split-K: every CTA's MMA issuer works through its chunk's
    segments in the order the planner gives (longest last)."""
    with hgemm.Handle() as h:
        h.set_option(hgemm.HGEMM_OPT_TRACE, 1 << 18)
        rows = _traced_run(h, M, N, K, 75, 1 << 18)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    st, p = hgemm.hgemm_plan(M, N, K, num_sms=sms)
    assert p.variant == hgemm.HGEMM_VARIANT_SPLITK
    seen = collections.defaultdict(list)
    for t, cta, role, kind, item, value in sorted(rows):
        if role == 2 and kind == 3:
            seen[cta].append((item, value))
    assert len(seen) == p.grid
    for c in range(p.grid):
        expect, i = [], 0
        while True:
            s, tile, kb0, kb1, first = hgemm.hgemm_plan_splitk_segment(p, c, i)
            if s != hgemm.HGEMM_OK:
                break
            expect.append((tile, kb0))
            i += 1
        assert seen[c] == expect, c


@pytest.mark.parametrize("variant,M,N,K,sk", [("2sm256", 4096, 2560, 4096, 3), ("1sm128", 1000, 3000, 2056, 2),
                                              ("splitk", 16, 16384, 8192, 0)])
def test_launch_stamps_only(variant, M, N, K, sk):
    """HGEMM_OPT_TRACE_ITEMS = 0: every CTA of every launch records only its
    kernel begin and end, whose cycle-counter and timer values give the SM
    clock each CTA ran at; the launches compute the same bits as an untraced
    one, which matches the oracle on sampled entries."""
    launches = 3
    a, b, ab, bb = parity.inputs(M, N, K, "TN", "bf16", ("normal", 1.0), 76)
    A, B = a.cuda(), b.cuda()
    C0 = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    Cs = [torch.empty_like(C0) for _ in range(launches)]
    with hgemm.Handle() as h:
        h.set_option(hgemm.HGEMM_OPT_FORCE_VARIANT, hgemm.VARIANTS[variant])
        h.set_option(hgemm.HGEMM_OPT_STREAM_K, sk)
        h.run(A, B, C0, layout="TN", acc="f32")
        h.set_option(hgemm.HGEMM_OPT_TRACE, 1 << 16)
        h.set_option(hgemm.HGEMM_OPT_TRACE_ITEMS, 0)
        for C in Cs:
            h.run(A, B, C, layout="TN", acc="f32")
        st, detail = h.sync_status()
        assert st == hgemm.HGEMM_OK, (st, hex(detail))
        st, n, rows = hgemm.hgemm_trace_read(h.h, 1 << 16)
        assert st == hgemm.HGEMM_OK and n == len(rows)
        assert hgemm.hgemm_set_option(h.h, hgemm.HGEMM_OPT_TRACE_ITEMS, 2) == hgemm.HGEMM_ERR_INVALID_ARG
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    st, p = hgemm.hgemm_plan(M, N, K, 0, hgemm.HGEMM_BF16, hgemm.HGEMM_F32, hgemm.HGEMM_BF16, sms,
                             hgemm.VARIANTS[variant], 0, sk)
    assert n == 2 * p.grid * launches
    assert all(r[2] == 0 and r[3] in (1, 2) for r in rows)
    per_cta = collections.Counter((r[1], r[3]) for r in rows)
    assert len(per_cta) == 2 * p.grid and set(per_cta.values()) == {launches}
    mhz = trace.launch_clocks(rows)
    assert len(mhz) == p.grid * launches
    assert 200.0 < sorted(mhz)[len(mhz) // 2] < 4000.0
    for C in Cs:
        assert torch.equal(C.view(torch.int16), C0.view(torch.int16))
    got = C0.view(torch.int16).cpu().numpy().view("uint16")
    parity.check(got, ab, bb, M, N, K, "TN", "bf16", "f32", "bf16", sampled=True, n_random=4096, seed=3)
