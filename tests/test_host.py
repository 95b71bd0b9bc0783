"""Host-side tests of the C ABI (no GPU): symbols, validation, planning,
the persistent scheduler's tile map, the split-K partition and the tcgen05
descriptor encodings."""
import ctypes

import pytest
import torch

from tensor_core_half_gb300 import hgemm

H = hgemm
ST_OK, ST_INV, ST_UNS, ST_MIS = H.HGEMM_OK, H.HGEMM_ERR_INVALID_ARG, H.HGEMM_ERR_UNSUPPORTED, H.HGEMM_ERR_MISALIGNED


def test_library_exports_every_declared_symbol():
    names = H.declared_functions()
    assert len(names) >= 12
    lib = H.lib()
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_constants_match_the_header():
    """Every enumerator include/hgemm.h declares has a binding constant of the
    same name and value (the binding restates them; a stale copy would pass
    the wrong option or status to the library)."""
    import pathlib
    import re

    text = (pathlib.Path(__file__).resolve().parents[1] / "include" / "hgemm.h").read_text()
    declared = re.findall(r"(?m)^\s*(HGEMM_[A-Za-z0-9_]+)\s*=\s*(-?\d+)", text)
    assert len(declared) >= 39 and any(n == "HGEMM_OPT_TRACE_ITEMS" for n, _ in declared)
    wrong = [(n, v, getattr(H, n, None)) for n, v in declared if getattr(H, n, None) != int(v)]
    assert not wrong, wrong


def test_status_strings():
    for s in range(0, 10):
        assert H.hgemm_status_string(s).startswith("HGEMM_")
    assert "unknown" in H.hgemm_status_string(99)
    assert H.hgemm_version() >= 100


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device path")
def test_create_without_device_reports_no_device():
    with pytest.raises(H.HgemmError) as e:
        H.hgemm_create()
    assert e.value.status == H.HGEMM_ERR_NO_DEVICE


def test_null_handle_is_rejected():
    assert H.hgemm_run(None, 16, 16, 16, 8, 8, 8, 0, 0, 2, 0, None) == ST_INV
    assert H.hgemm_sync_status(None)[0] == ST_INV
    assert H.hgemm_set_option(None, H.HGEMM_OPT_GROUP_M, 4) == ST_INV
    assert H.hgemm_destroy(None) == ST_OK


def plan(M, N, K, layout=0, fin=1, acc=2, out=1, sms=152, variant=0, group_m=0, stream_k=1):
    return H.hgemm_plan(M, N, K, layout, fin, acc, out, sms, variant, group_m, stream_k)


@pytest.mark.parametrize("args,expect", [
    ((-1, 8, 8), ST_INV), ((8, -1, 8), ST_INV), ((8, 8, -1), ST_INV), ((1 << 31, 8, 8), ST_INV),
    ((8, 12, 8), ST_MIS), ((8, 8, 12), ST_MIS), ((0, 12, 8), ST_OK), ((8, 0, 8), ST_OK), ((8, 8, 0), ST_OK),
    ((3, 8, 8), ST_OK)])
def test_plan_size_validation(args, expect):
    assert plan(*args)[0] == expect


def test_plan_dtype_and_layout_validation():
    assert plan(64, 64, 64, layout=2)[0] == ST_INV
    assert plan(64, 64, 64, fin=5)[0] == ST_INV
    assert plan(64, 64, 64, fin=H.HGEMM_BF16, acc=H.HGEMM_F16)[0] == ST_UNS
    assert plan(64, 64, 64, fin=H.HGEMM_F32)[0] == ST_UNS
    assert plan(64, 64, 64, out=H.HGEMM_F32)[0] == ST_UNS
    assert plan(64, 64, 64, acc=H.HGEMM_BF16)[0] == ST_UNS
    assert plan(64, 64, 64, fin=H.HGEMM_F16, acc=H.HGEMM_F16, out=H.HGEMM_F16)[0] == ST_OK
    assert plan(64, 64, 64, sms=0)[0] == ST_INV
    assert plan(64, 64, 64, variant=9)[0] == ST_INV
    assert plan(64, 64, 64, variant=6)[0] == ST_INV


def test_plan_variant_choice():
    st, p = plan(4096, 4096, 4096)
    assert st == ST_OK and p.variant == H.HGEMM_VARIANT_2SM_256x256 and p.cta_group == 2
    assert (p.tile_m, p.tile_n, p.tiles_m, p.tiles_n, p.num_tiles, p.k_blocks) == (256, 256, 16, 16, 256, 64)
    assert p.grid == 152 and p.tmem_cols == 512 and p.smem_bytes <= 232448
    # 256 tiles over 76 pairs: three whole waves data-parallel, the remaining
    # 28 tiles each cut into 2 K pieces
    assert p.stream_k == 1 and p.dp_tiles == 228 and p.sk_units == (256 - 228) * 64 and p.sk_pieces == 2
    st, p = plan(4096, 4096, 4096, stream_k=0, variant=3)
    assert st == ST_OK and p.stream_k == 0 and p.dp_tiles == 256 and p.sk_units == 0 and p.workspace_bytes == 0
    # a tile count that is a whole number of waves stays data-parallel
    st, p = plan(256 * 76, 256, 4096)
    assert st == ST_OK and p.variant == H.HGEMM_VARIANT_2SM_256x256 and p.stream_k == 0
    st, p = plan(16, 16384, 8192)
    assert st == ST_OK and p.variant == H.HGEMM_VARIANT_SPLITK and p.tile_n == 16 and p.num_tiles == 128
    # whole tiles: one 128-row tile per CTA on 128 of the 152 SMs, no partials
    assert p.grid == 128 and p.block_k == 128 and p.k_blocks == 64 and p.splitk_align == 64 and p.workspace_bytes == 0
    st, p = plan(16, 16384, 8192, stream_k=2)
    assert st == ST_OK and p.grid == 152 and p.splitk_align == 1 and p.workspace_bytes > 0
    st, p = plan(16, 16384, 8192, layout=H.HGEMM_LAYOUT_NN)
    assert st == ST_OK and p.variant != H.HGEMM_VARIANT_SPLITK  # split-K is TN only
    st, p = plan(16, 16384, 8192, fin=0, acc=0, out=0)
    assert st == ST_OK and p.variant != H.HGEMM_VARIANT_SPLITK  # and fp32 accumulate only
    assert plan(16, 64, 64, layout=1, variant=H.HGEMM_VARIANT_SPLITK)[0] == ST_UNS
    assert plan(65, 64, 64, variant=H.HGEMM_VARIANT_SPLITK)[0] == ST_UNS
    for v in (1, 2, 3, 5):
        st, p = plan(1000, 3000, 4104, variant=v)
        assert st == ST_OK and p.variant == v
    # the ragged shape: 256 x 192 tiles give 64 tiles (one wave, no stream-K fix-ups)
    st, p = plan(1000, 3000, 4104)
    assert st == ST_OK and p.variant == H.HGEMM_VARIANT_2SM_256x192 and p.num_tiles == 64 and p.stream_k == 0
    assert plan(1000, 3000, 4104, layout=H.HGEMM_LAYOUT_NN, variant=5)[0] == ST_UNS
    st, p = plan(1000, 3000, 4104, layout=H.HGEMM_LAYOUT_NN)
    assert st == ST_OK and p.variant != H.HGEMM_VARIANT_2SM_256x192
    st, p = plan(1000, 3000, 4104, variant=1)
    assert (p.tiles_m, p.tiles_n, p.k_blocks) == (8, 24, 65)


def test_automatic_group_height():
    # All of A within 32 MiB: one group spans every tile row (A read from HBM once).
    assert plan(4096, 4096, 4096)[1].group_m == 16
    assert plan(6144, 4096, 2048)[1].group_m == 24
    assert plan(4096, 4096, 4096, fin=0, acc=0, out=0)[1].group_m == 16
    # Larger A, or no more than 8 tile rows: 8.
    assert plan(8192, 8192, 8192)[1].group_m == 8
    assert plan(4096, 4096, 4104)[1].group_m == 8  # A just over 32 MiB
    assert plan(2048, 2048, 2048)[1].group_m == 8
    assert plan(1000, 3000, 4104)[1].group_m == 8
    # An explicit height is kept.
    assert plan(4096, 4096, 4096, group_m=4)[1].group_m == 4


@pytest.mark.parametrize("M,N,K,variant", [(4096, 4096, 4096, 3), (1000, 3000, 4104, 1), (1000, 3000, 4104, 2),
                                           (8192, 8192, 64, 3), (129, 8, 8, 3), (5000, 136, 64, 1)])
@pytest.mark.parametrize("group_m", [1, 3, 8, 100])
def test_tile_map_is_a_bijection(M, N, K, variant, group_m):
    st, p = plan(M, N, K, variant=variant, group_m=group_m)
    assert st == ST_OK
    seen = set()
    for t in range(p.num_tiles):
        s, m, n = H.hgemm_plan_tile(p, t)
        assert s == ST_OK and 0 <= m < p.tiles_m and 0 <= n < p.tiles_n
        seen.add((m, n))
    assert len(seen) == p.num_tiles
    assert H.hgemm_plan_tile(p, p.num_tiles)[0] == ST_INV
    assert H.hgemm_plan_tile(p, -1)[0] == ST_INV


def test_tile_map_groups_rows():
    # Within a full group, consecutive tiles walk down group_m tile rows before
    # moving one tile column on ("block swizzle" band order).
    st, p = plan(4096, 4096, 4096, variant=3, group_m=4)
    coords = [H.hgemm_plan_tile(p, t)[1:] for t in range(12)]
    assert coords[:5] == [(0, 0), (1, 0), (2, 0), (3, 0), (0, 1)]
    assert coords[8] == (0, 2)
    # odd groups walk the tile columns right to left (serpentine), so a group
    # starts on the columns its predecessor read last
    second = [H.hgemm_plan_tile(p, t)[1:] for t in range(4 * 16, 4 * 16 + 6)]
    assert second == [(4, 15), (5, 15), (6, 15), (7, 15), (4, 14), (5, 14)]
    third = H.hgemm_plan_tile(p, 8 * 16)[1:]
    assert third == (8, 0)
    # the last group is shorter when tiles_m is not a multiple of group_m
    st, p = plan(5 * 256, 512, 64, variant=3, group_m=4)
    tail = [H.hgemm_plan_tile(p, t)[1:] for t in range(8, 10)]
    assert tail == [(4, 1), (4, 0)]


@pytest.mark.parametrize("M,N,K,sms", [(16, 16384, 8192, 152), (1, 8, 64, 152), (64, 1000, 72, 152),
                                       (16, 4096, 4096, 7), (33, 100000, 640, 152), (16, 128, 8192, 152)])
def test_splitk_partition(M, N, K, sms):
    st, p = plan(M, N, K, sms=sms)
    assert st == ST_OK and p.variant == H.HGEMM_VARIANT_SPLITK
    units = p.num_tiles * p.k_blocks
    prev_end, sizes = 0, []
    for c in range(p.grid):
        s, b, e = H.hgemm_plan_splitk_range(p, c)
        assert s == ST_OK and b == prev_end and e > b
        if p.splitk_align > 1:  # whole tiles: ranges start and end on tile boundaries
            assert p.splitk_align == p.k_blocks and b % p.k_blocks == 0 and e % p.k_blocks == 0
        sizes.append(e - b)
        prev_end = e
    assert prev_end == units
    assert max(sizes) - min(sizes) <= max(1, p.splitk_align)
    assert H.hgemm_plan_splitk_range(p, p.grid)[0] == ST_INV


@pytest.mark.parametrize("M,N,K,sms,whole,grid", [
    (16, 16384, 8192, 152, True, 128),    # 128 tiles: one per CTA, 24 SMs idle, HBM still saturated
    (16, 32768, 4096, 152, True, 128),    # 256 tiles: two per CTA
    (16, 12288, 8192, 152, True, 96),     # 96 CTAs reach ~5.9 of 6.25 TB/s: still ahead of split + fix-up
    (16, 8192, 8192, 152, False, 152),    # 64 CTAs would reach ~4 TB/s: split over every SM
    (16, 20480, 8192, 152, False, 152),   # 160 tiles -> 80 CTAs of two tiles: too few
    (16, 4096, 4096, 152, False, 152),
    (16, 16384, 8192, 148, True, 128),
    (64, 16384, 8192, 152, True, 128),    # the split's fix-up grows with M
    (32, 14336, 4096, 152, True, 112),
    (1, 16384, 16384, 152, True, 128),    # long K: whole tiles stream as fast as all SMs, with no fix-up
    (4, 32768, 8192, 152, True, 128),     # 256 tiles: two per CTA
    (1, 8192, 16384, 152, False, 152)])   # 64 tiles: 64 CTAs would stream at ~4 TB/s
def test_splitk_whole_tile_choice(M, N, K, sms, whole, grid):
    """The planner's layout for skinny products: whole tiles per CTA (no
    tile's K range split, no fix-up) when 128-row tiles at the CTA count that
    takes them saturate HBM about as well as all SMs, else the balanced split;
    HGEMM_OPT_STREAM_K 0 / 2 force one or the other."""
    st, p = plan(M, N, K, sms=sms)
    assert st == ST_OK and p.variant == H.HGEMM_VARIANT_SPLITK
    assert (p.splitk_align == p.k_blocks) == whole and p.grid == grid
    assert (p.workspace_bytes == 0) == whole
    st, p0 = plan(M, N, K, sms=sms, stream_k=0)
    per = -(-p0.num_tiles // sms)
    assert p0.splitk_align == p0.k_blocks and p0.grid == -(-p0.num_tiles // per) and p0.workspace_bytes == 0
    st, p2 = plan(M, N, K, sms=sms, stream_k=2)
    assert p2.splitk_align == 1 and p2.grid == min(sms, p2.num_tiles * p2.k_blocks)
    st, pd = H.hgemm_plan(M, N, K, num_sms=sms, schedule=H.HGEMM_SCHEDULE_DYNAMIC)
    assert pd.splitk_align == 1  # the dynamic schedule always splits


@pytest.mark.parametrize("schedule", [H.HGEMM_SCHEDULE_STATIC, H.HGEMM_SCHEDULE_DYNAMIC])
@pytest.mark.parametrize("M,N,K,sms", [(16, 16384, 8192, 152), (1, 8, 64, 152), (64, 1000, 72, 148),
                                       (16, 4096, 4096, 7), (33, 100000, 640, 152), (16, 128, 8192, 152)])
def test_splitk_segment_order(M, N, K, sms, schedule):
    """The segments a chunk is processed in: one per N tile its range touches
    (found here by walking the chunk unit by unit), all of them once, the
    longest last (the later one on a tie), the rest in ascending order, and
    'first' on the one that starts the range."""
    st, p = H.hgemm_plan(M, N, K, num_sms=sms, schedule=schedule)
    assert st == ST_OK and p.variant == H.HGEMM_VARIANT_SPLITK
    kb = p.k_blocks
    for g in range(p.splitk_chunks):
        s, b, e = H.hgemm_plan_splitk_range(p, g)
        assert s == ST_OK
        pieces = {}
        for u in range(b, e):
            t, k = divmod(u, kb)
            lo, hi = pieces.get(t, (k, k))
            pieces[t] = (min(lo, k), max(hi, k + 1))
        expect = [(t,) + pieces[t] for t in sorted(pieces)]
        got = []
        for i in range(len(expect)):
            s, t, k0, k1, first = H.hgemm_plan_splitk_segment(p, g, i)
            assert s == ST_OK
            assert first == (t * kb + k0 == b)
            got.append((t, k0, k1))
        assert H.hgemm_plan_splitk_segment(p, g, len(expect))[0] == ST_INV
        assert sorted(got) == expect
        lengths = [x[2] - x[1] for x in expect]
        longest = max(i for i, n in enumerate(lengths) if n == max(lengths))
        assert got == expect[:longest] + expect[longest + 1:] + [expect[longest]]
    assert H.hgemm_plan_splitk_segment(p, p.splitk_chunks, 0)[0] == ST_INV
    assert H.hgemm_plan_splitk_segment(p, 0, -1)[0] == ST_INV


@pytest.mark.parametrize("M,N,K,sms", [(16, 16384, 8192, 152), (1, 8, 64, 152), (64, 1000, 72, 148),
                                       (33, 4096, 1024, 152), (16, 16384, 8192, 7), (8, 256, 16384, 152)])
def test_splitk_dynamic_chunks(M, N, K, sms):
    """Dynamic split-K chunks: the first `grid` chunks (one per SM) hold about
    three quarters of the units, the small chunks (about a quarter of an SM's
    share each) the rest; all of them together cover every unit once, in
    order, and no chunk is empty."""
    st, p = H.hgemm_plan(M, N, K, num_sms=sms, schedule=H.HGEMM_SCHEDULE_DYNAMIC)
    assert st == ST_OK and p.variant == H.HGEMM_VARIANT_SPLITK and p.schedule == H.HGEMM_SCHEDULE_DYNAMIC
    units = p.num_tiles * p.k_blocks
    sizes, prev_end = [], 0
    for g in range(p.splitk_chunks):
        s, b, e = H.hgemm_plan_splitk_range(p, g)
        assert s == ST_OK and b == prev_end and e > b
        sizes.append(e - b)
        prev_end = e
    assert prev_end == units
    assert H.hgemm_plan_splitk_range(p, p.splitk_chunks)[0] == ST_INV
    big, small = sizes[:p.grid], sizes[p.grid:]
    assert max(big) - min(big) <= 1
    if units >= 4 * p.grid:
        assert small and max(small) - min(small) <= 1 and max(small) < min(big)
        assert sum(big) == p.splitk_head_units and abs(sum(small) - units // 4) <= 1
        assert max(small) <= max(1, units // (p.grid * 4)) + 1
    else:
        assert not small and p.splitk_head_units == units  # too little work to split further
    # the static plan of the same problem split over every SM: one range per CTA
    st, q = H.hgemm_plan(M, N, K, num_sms=sms, stream_k=2, schedule=H.HGEMM_SCHEDULE_STATIC)
    assert q.splitk_chunks == q.grid == p.grid and q.splitk_head_units == units and q.splitk_align == 1


# ------------------------------------------------------------ descriptors ----
# Expected words are written out by hand from the field tables:
#   idesc: D fmt bits 4-5 (f32 = 1), A fmt 7-9 / B fmt 10-12 (bf16 = 1),
#          A major bit 15, B major bit 16, N>>3 at 17-22, M>>4 at 24-28.
#   smem desc: addr>>4 at 0-13, LBO>>4 at 16-29, SBO>>4 at 32-45, bit 46 = 1,
#          swizzle at 61-63 (128-byte swizzle = 2).
@pytest.mark.parametrize("args,word", [
    ((128, 256, H.HGEMM_BF16, H.HGEMM_F32, 0, 0), 0x08400490),  # 0x10|0x80|0x400|(32<<17)|(8<<24)
    ((256, 256, H.HGEMM_BF16, H.HGEMM_F32, 0, 0), 0x10400490),  # M=256: 16<<24
    ((128, 128, H.HGEMM_F16, H.HGEMM_F32, 0, 0), 0x08200010),   # fp16 in: format 0; N=128: 16<<17
    ((128, 128, H.HGEMM_F16, H.HGEMM_F16, 0, 0), 0x08200000),   # fp16 accumulate: D format 0
    ((128, 16, H.HGEMM_BF16, H.HGEMM_F32, 0, 0), 0x08040490),   # N=16: 2<<17
    ((256, 256, H.HGEMM_F16, H.HGEMM_F32, 0, 1), 0x10410010),   # NN: B MN-major bit 16
    ((128, 64, H.HGEMM_F16, H.HGEMM_F32, 1, 0), 0x08108010),    # A MN-major bit 15; N=64: 8<<17
])
def test_instruction_descriptor_bits(args, word):
    assert H.hgemm_encode_idesc(*args) == word


@pytest.mark.parametrize("args,word", [
    ((0x400, 16, 1024, 2), 0x4000404000010040),
    ((0x1C400 + 32, 16, 1024, 2), 0x4000404000011C42),   # +32 B K step inside the swizzle atom
    ((0x2000, 8192, 1024, 2), 0x4000404002000200),       # MN-major: LBO 8 KiB
    ((0x0, 128, 1024, 0), 0x0000404000080000),           # no swizzle
    ((0x3FFF0, 0, 0, 2), 0x4000400000003FFF),            # top of the 18-bit shared window
])
def test_shared_memory_descriptor_bits(args, word):
    assert H.hgemm_encode_smem_desc(*args) == word


STREAMK_CASES = [(4096, 4096, 4096, 3), (2048, 2048, 2048, 3), (1000, 3000, 4104, 1), (1000, 3000, 4104, 3),
                 (4096, 4096, 4096, 5), (3000, 6000, 2048, 5),
                 (8192, 8192, 8192, 3), (256, 256, 4096, 3), (640, 1024, 2048, 2), (256, 512, 128, 3)]


@pytest.mark.parametrize("M,N,K,variant", STREAMK_CASES)
def test_work_lists_cover_every_unit_once(M, N, K, variant):
    st, p = plan(M, N, K, variant=variant)
    assert st == ST_OK
    clusters = p.grid // p.cta_group
    covered = {}
    per_cluster = []
    slots = {}
    for c in range(clusters):
        i, work = 0, 0
        while True:
            s, t, a, b, slot = H.hgemm_plan_work_item(p, c, i)
            if s != ST_OK:
                break
            assert 0 <= t < p.num_tiles and 0 <= a < b <= p.k_blocks
            if slot < 0:
                assert (a, b) == (0, p.k_blocks)
            else:
                assert t >= p.dp_tiles and (a, b) != (0, p.k_blocks)
                assert (c, slot) not in slots  # at most one partial per slot
                slots[(c, slot)] = t
            for kb in range(a, b):
                assert (t, kb) not in covered
                covered[(t, kb)] = c
            work += b - a
            i += 1
        per_cluster.append(work)
    assert len(covered) == p.num_tiles * p.k_blocks
    if p.stream_k and p.sk_pieces == 0:
        # equal ranges: every cluster does the same number of k-blocks, up to one
        assert max(per_cluster) - min(per_cluster) <= 1
        # a split tile's pieces come from consecutive clusters, in K order
        for t in range(p.dp_tiles, p.num_tiles):
            owners = [covered[(t, kb)] for kb in range(p.k_blocks)]
            assert owners == sorted(owners)
            assert set(owners) == set(range(owners[0], owners[-1] + 1))
    if p.stream_k and p.sk_pieces:
        # K pieces: each split tile is cut into sk_pieces pieces of equal
        # length (up to one k-block) that start at the same K offsets in
        # every split tile, one piece per cluster
        piece = -(-p.k_blocks // p.sk_pieces)
        starts = None
        for t in range(p.dp_tiles, p.num_tiles):
            owners = [covered[(t, kb)] for kb in range(p.k_blocks)]
            cuts = [0] + [kb for kb in range(1, p.k_blocks) if owners[kb] != owners[kb - 1]]
            assert len(cuts) == p.sk_pieces and len(set(owners)) == p.sk_pieces
            starts = starts or cuts
            assert cuts == starts
            lens = [b - a for a, b in zip(cuts, cuts[1:] + [p.k_blocks])]
            assert max(lens) - min(lens) <= 1
        assert max(per_cluster) - min(per_cluster) <= piece


@pytest.mark.parametrize("M,N,K,variant", STREAMK_CASES)
def test_work_ids_partition_the_work(M, N, K, variant):
    """The dynamic schedule runs whole work ids in any order: the ids must cut
    the work into disjoint pieces that cover it, the static walk of cluster c
    must be exactly ids c, c + P, ... in order, and the stream-K ranges must
    come first."""
    st, p = plan(M, N, K, variant=variant)
    assert st == ST_OK
    clusters = p.grid // p.cta_group
    assert p.work_ids == p.sk_ranges + p.dp_tiles
    if not p.stream_k:
        assert p.sk_ranges == 0
    elif p.sk_pieces == 0:
        assert p.sk_ranges == clusters
    else:
        assert p.sk_ranges == (p.num_tiles - p.dp_tiles) * p.sk_pieces <= clusters
    items = {}
    covered = set()
    for i in range(p.work_ids):
        lst, j = [], 0
        while True:
            s, t, a, b, slot = H.hgemm_plan_id_item(p, i, j)
            if s != ST_OK:
                break
            lst.append((t, a, b, slot))
            for kb in range(a, b):
                assert (t, kb) not in covered
                covered.add((t, kb))
            j += 1
        assert lst, "every id has work"
        if i >= p.sk_ranges:
            assert lst == [(i - p.sk_ranges, 0, p.k_blocks, -1)]
        else:
            assert all(t >= p.dp_tiles for t, _, _, _ in lst)
            # slot 0 only on the first piece, slot 1 only on the last
            for k, (t, a, b, slot) in enumerate(lst):
                if slot == 0:
                    assert k == 0
                if slot == 1:
                    assert k == len(lst) - 1 and k > 0
        items[i] = lst
    assert len(covered) == p.num_tiles * p.k_blocks
    for c in range(clusters):
        walk, j = [], 0
        while True:
            s, t, a, b, slot = H.hgemm_plan_work_item(p, c, j)
            if s != ST_OK:
                break
            walk.append((t, a, b, slot))
            j += 1
        expect = [it for i in range(c, p.work_ids, clusters) for it in items[i]]
        assert walk == expect


def test_work_id_arguments():
    st, p = plan(4096, 4096, 4096)
    assert H.hgemm_plan_id_item(p, -1, 0)[0] == ST_INV
    assert H.hgemm_plan_id_item(p, p.work_ids, 0)[0] == ST_INV
    assert H.hgemm_plan_id_item(p, 0, -1)[0] == ST_INV
    st, sp = plan(16, 16384, 8192)
    assert H.hgemm_plan_id_item(sp, 0, 0)[0] == ST_INV


def test_schedule_option_values():
    # no device here: only the option's validation path is reachable without a handle
    assert H.SCHEDULES == {"static": 0, "dynamic": 1}


def test_tma_bench_validates_before_touching_the_device():
    fake = 1 << 20  # never dereferenced: every case below is rejected or finds no device
    assert H.hgemm_tma_bench(None, 1024, 1024, 0, 128, 64, 2, 8)[0] == ST_INV
    assert H.hgemm_tma_bench(fake, 1024, 1024, 5, 128, 64, 2, 8)[0] == ST_INV
    assert H.hgemm_tma_bench(fake, 1000, 1024, 0, 128, 64, 2, 8)[0] == ST_INV  # height % tile_rows
    assert H.hgemm_tma_bench(fake, 1024, 1024, 2, 128, 32, 2, 8)[0] == ST_INV  # 128-byte box needs 64 columns
    assert H.hgemm_tma_bench(fake + 64, 1024, 1024, 0, 128, 64, 2, 8)[0] == H.HGEMM_ERR_MISALIGNED
    assert H.hgemm_tma_bench(fake, 1024, 1024, 0, 128, 64, 2, 8)[0] == H.HGEMM_ERR_NO_DEVICE


def test_tma_bench_reference_sums():
    from tensor_core_half_gb300 import tma_bench
    import numpy as np
    words = tma_bench.source(64, 256, device="cpu").view(torch.int16).numpy().view(np.uint16).astype(np.uint64)
    # tile 3 of a 32 x 64 grid is rows 0..31, columns 192..255
    t = words[0:32, 192:256]
    assert tma_bench.expected_sums(64, 256, H.HGEMM_TMA_2D_128B, 32, 64, [3, -1]) == (int(t.sum()), int((t * t).sum()))
    # bulk tile 1: the second 2048 words in memory order
    f = words.reshape(-1)[2048:4096]
    assert tma_bench.expected_sums(64, 256, H.HGEMM_TMA_BULK, 32, 64, [1]) == (int(f.sum()), int((f * f).sum()))


def test_stream_k_split_by_remainder():
    # 2-SM 256 x 256 tiles, 76 pairs.  Equal ranges (stream_k = 2), 86 tiles: a
    # remainder of 10 (< 76 / 4) would be cut among ~8 pairs each, so the whole
    # first round joins the split.
    st, p = plan(512, 256 * 43, 4096, variant=3, stream_k=2)
    assert st == ST_OK and p.num_tiles == 86 and p.stream_k == 1 and p.dp_tiles == 0 and p.sk_units == 86 * 64
    assert p.sk_pieces == 0 and p.sk_ranges == 76
    # 106 tiles: a remainder of 30 (>= 19) is split alone; 76 tiles stay whole.
    st, p = plan(512, 256 * 53, 4096, variant=3, stream_k=2)
    assert st == ST_OK and p.num_tiles == 106 and p.stream_k == 1 and p.dp_tiles == 76 and p.sk_units == 30 * 64
    # The estimate's choice: K pieces.  A remainder of 10 tiles is cut into 4
    # pieces each (76 / 10 = 7, capped at 4), 30 tiles into 2 pieces each;
    # the first round stays whole.
    st, p = plan(512, 256 * 43, 4096, variant=3)
    assert st == ST_OK and p.stream_k == 1 and p.dp_tiles == 76 and p.sk_units == 10 * 64
    assert p.sk_pieces == 4 and p.sk_ranges == 40 and p.grid == 152
    st, p = plan(512, 256 * 53, 4096, variant=3)
    assert st == ST_OK and p.dp_tiles == 76 and p.sk_pieces == 2 and p.sk_ranges == 60


def test_stream_k_option_values():
    # ragged 1000 x 3000 x 4104 on 2-SM 256 x 256 tiles: 48 tiles for 76 pairs.
    # The estimate keeps whole tiles; stream_k = 2 splits them anyway; 0 never.
    st, p = plan(1000, 3000, 4104, variant=3, stream_k=1)
    assert st == ST_OK and p.stream_k == 0 and p.dp_tiles == 48
    st, p = plan(1000, 3000, 4104, variant=3, stream_k=2)
    assert st == ST_OK and p.stream_k == 1 and p.dp_tiles == 0 and p.sk_units == 48 * 65
    st, p = plan(4096, 4096, 4096, variant=3, stream_k=2)
    assert st == ST_OK and p.stream_k == 1 and p.dp_tiles == 228 and p.sk_pieces == 0 and p.sk_ranges == 76
    # 3: K pieces (the estimate's choice here): 28 leftover tiles, 2 pieces each
    st, p = plan(4096, 4096, 4096, variant=3, stream_k=3)
    assert st == ST_OK and p.stream_k == 1 and p.dp_tiles == 228 and p.sk_pieces == 2 and p.sk_ranges == 56
    st, q = plan(4096, 4096, 4096, variant=3, stream_k=1)
    assert (q.dp_tiles, q.sk_units, q.sk_ranges, q.sk_pieces) == (228, 28 * 64, 56, 2)
    # 48 tiles for 76 pairs: one piece per tile fits, so 3 forces two
    st, p = plan(1000, 3000, 4104, variant=3, stream_k=3)
    assert st == ST_OK and p.dp_tiles == 0 and p.sk_pieces == 2 and p.sk_ranges == 96 and p.grid == 152
    st, p = plan(4096, 4096, 4096, variant=3, stream_k=4)
    assert st == ST_INV


def test_work_list_arguments():
    st, p = plan(4096, 4096, 4096)
    assert H.hgemm_plan_work_item(p, -1, 0)[0] == ST_INV
    assert H.hgemm_plan_work_item(p, p.grid // 2, 0)[0] == ST_INV
    assert H.hgemm_plan_work_item(p, 0, -1)[0] == ST_INV
    st, sp = plan(16, 16384, 8192)
    assert H.hgemm_plan_work_item(sp, 0, 0)[0] == ST_INV  # split-K plans have no dense work list


def test_trace_read_requires_tracing():
    st, n, rows = H.hgemm_trace_read(None, 4)
    assert st == ST_INV and rows == []


def test_trace_summary_and_chrome_format():
    from tensor_core_half_gb300 import trace
    rows = [(1000, 0, 0, 1, -1, 0), (1100, 0, 1, 3, 5, 0), (1900, 0, 1, 4, 5, 64), (1200, 0, 2, 3, 5, 0),
            (2000, 0, 2, 4, 5, 64), (2100, 0, 3, 3, 5, -1), (2600, 0, 3, 4, 5, -1), (2700, 0, 0, 2, -1, 0),
            (1000, 1, 0, 1, -1, 1), (2900, 1, 0, 2, -1, 1)]
    s = trace.summary(rows)
    assert s["span_ns"] == 1900 and s["items"] == 3 and s["cta_end_ns"] == [1700, 1900]
    assert s["busy_ns_per_cta"]["tma"] == 400.0
    doc = trace.chrome_trace(rows)
    names = sorted(e["name"] for e in doc["traceEvents"])
    assert names.count("tile 5") == 3 and "kernel_end" in names


def test_operand_shape_accepts_one_product_and_names_each_mismatch():
    f16, bf16 = torch.float16, torch.bfloat16
    A = torch.zeros((6, 16), dtype=f16)
    B_tn = torch.zeros((8, 16), dtype=f16)
    B_nn = torch.zeros((16, 8), dtype=f16)
    C = torch.zeros((6, 8), dtype=f16)
    assert H.operand_shape(A, B_tn, C, "TN", cuda=False) == (6, 8, 16)
    assert H.operand_shape(A, B_nn, C, "NN", cuda=False) == (6, 8, 16)
    assert H.operand_shape(A[:, :0].contiguous(), B_tn[:, :0].contiguous(), C, "TN", cuda=False) == (6, 8, 0)
    bad = [
        ((A, B_tn, C, "TT"), "layout"),
        ((A, B_nn.t(), C, "TN"), "contiguous"),           # a transposed view is not packed
        ((A, B_tn, C.t().contiguous().t(), "TN"), "contiguous"),
        ((A, B_tn.to(bf16), C, "TN"), "element type"),
        ((A, B_nn, C, "TN"), "K"),                         # NN storage passed as TN
        ((A, B_tn, C[:, :4], "TN"), "C must be"),
        ((A.unsqueeze(0), B_tn, C, "TN"), "2-D"),
    ]
    for args, word in bad:
        with pytest.raises(ValueError, match=word):
            H.operand_shape(*args, cuda=False)
    with pytest.raises(ValueError, match="CUDA"):
        H.operand_shape(A, B_tn, C, "TN", cuda=True)      # host tensors handed to the device call


@pytest.mark.parametrize("M,N,K", [(4096, 4096, 4096), (2048, 2048, 2048), (1000, 3000, 4104), (16, 16384, 8192),
                                   (16, 8192, 8192), (1, 16384, 16384), (64, 16384, 8192), (256, 256, 256)])
@pytest.mark.parametrize("stream_k", [0, 1, 2])
def test_workspace_only_where_a_tile_is_split(M, N, K, stream_k):
    # A launch needs the workspace (fp32 partials and fix-up counters) exactly
    # when some tile's K range is split: dense stream-K, or a split-K plan
    # that is not whole tiles.  Whole-tile plans allocate nothing, which is
    # what lets them be captured into a graph on a fresh handle.
    st, p = H.hgemm_plan(M, N, K, num_sms=152, stream_k=stream_k)
    assert st == ST_OK
    if p.variant == H.HGEMM_VARIANT_SPLITK:
        split = p.splitk_align == 1
    else:
        split = p.stream_k == 1
    assert (p.workspace_bytes > 0) == split, (p.variant, p.stream_k, p.splitk_align, p.workspace_bytes)


def test_tile_count_beyond_32_bits_is_rejected():
    # Each dimension is allowed up to 2^31 - 1, but the 128 x 128 tile count
    # must stay 32-bit: the largest square product that fits is accepted, the
    # next size up is refused before any plan is made.
    big = 2 ** 31 - 8
    st, _ = H.hgemm_plan(big, big, 64, num_sms=152)
    assert st == H.HGEMM_ERR_INVALID_ARG
    st, _ = H.hgemm_plan(128 * 46340, 128 * 46340, 64, num_sms=152)   # 46340^2 < 2^31 tiles
    assert st == ST_OK
    st, _ = H.hgemm_plan(128 * 46341, 128 * 46341, 64, num_sms=152)   # 46341^2 > 2^31 - 1
    assert st == H.HGEMM_ERR_INVALID_ARG


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device path")
def test_noalloc_size_limit_at_its_boundary():
    """The allocation-free entry point keeps one arrival counter per 128-column
    tile in a 2 MiB area: N up to 67,108,864 passes the size check (and then
    finds no device here); one more tile's worth is refused before any device
    call.  The pointers are never dereferenced."""
    R = H.hgemm_run_splitk_noalloc
    bf = H.HGEMM_BF16
    A, B, C = 1 << 40, 2 << 40, 3 << 40
    n_max = (2 << 20) // 4 * 128
    assert n_max == 67108864
    assert R(A, B, C, 16, n_max + 8, 64, bf, bf, 0) == ST_UNS
    assert R(A, B, C, 16, n_max, 64, bf, bf, 0) == H.HGEMM_ERR_NO_DEVICE
    assert R(A, B, C, 64, 64, 64, bf, bf, 0) == H.HGEMM_ERR_NO_DEVICE
    assert R(A, B, C, 65, 64, 64, bf, bf, 0) == ST_UNS
