"""Randomised properties of the planner and the schedulers (no GPU needed).

For many seeded (M, N, K, SM count, variant, stream-K, schedule) draws:
  - dense plans: the work ids partition the (tile, k-block) units, stream-K
    ranges first; every cluster's static walk visits whole ids and all
    clusters together do equal work up to one k-block in the split part;
  - split-K plans: the chunks partition the units in order, none is empty.
"""
import numpy as np
import pytest

from tensor_core_half_gb300 import hgemm as H

ST_OK = H.HGEMM_OK


def _dense_cases(n, seed):
    r = np.random.default_rng(seed)
    for _ in range(n):
        M = int(r.choice([1, 7, 64, 129, 256, 1000, 2048, 4096, 8192, 12000]))
        N = int(r.choice([8, 64, 136, 1000, 3000, 4096, 8192, 16384]))
        K = int(8 * r.integers(1, 1200))
        sms = int(r.choice([8, 16, 40, 76, 132, 148, 152]))
        variant = int(r.choice([1, 2, 3, 5]))
        stream_k = int(r.choice([0, 1, 2, 3]))
        yield M, N, K, sms, variant, stream_k


@pytest.mark.parametrize("seed", range(4))
def test_dense_work_ids_partition_units(seed):
    for M, N, K, sms, variant, stream_k in _dense_cases(40, seed):
        st, p = H.hgemm_plan(M, N, K, H.HGEMM_LAYOUT_TN, H.HGEMM_BF16, H.HGEMM_F32, H.HGEMM_BF16, sms, variant, 0,
                             stream_k)
        assert st == ST_OK, (M, N, K, sms, variant, stream_k)
        if p.variant == H.HGEMM_VARIANT_SPLITK:
            continue
        clusters = p.grid // p.cta_group
        assert 1 <= clusters <= max(1, sms // p.cta_group)
        assert p.work_ids == p.sk_ranges + p.dp_tiles
        assert p.dp_tiles + (p.sk_units // p.k_blocks if p.k_blocks else 0) == p.num_tiles
        seen = np.zeros((p.num_tiles, p.k_blocks), np.int8)
        id_kb = []
        for i in range(p.work_ids):
            j, kb = 0, 0
            while True:
                s, t, a, b, slot = H.hgemm_plan_id_item(p, i, j)
                if s != ST_OK:
                    break
                assert 0 <= t < p.num_tiles and 0 <= a < b <= p.k_blocks
                assert (slot < 0) == (a == 0 and b == p.k_blocks)
                seen[t, a:b] += 1
                kb += b - a
                j += 1
            assert j > 0
            id_kb.append(kb)
        assert (seen == 1).all(), (M, N, K, sms, variant, stream_k)
        if p.sk_ranges:
            sk = id_kb[:p.sk_ranges]
            assert max(sk) - min(sk) <= 1  # equal stream-K ranges
            # the kernel keeps two fp32 partial slots [cta_group][tile_n][128]
            # per range id: the workspace the plan asks for must hold them all
            slots = 2 * p.sk_ranges * p.cta_group * p.tile_n * 128 * 4
            assert p.workspace_bytes >= slots + p.num_tiles * p.cta_group * 8
        if p.sk_pieces:
            assert 2 <= p.sk_pieces <= 4 and p.sk_ranges == (p.num_tiles - p.dp_tiles) * p.sk_pieces
        # the static walk of every cluster: ids c, c + P, ... and nothing else
        per_cluster = []
        for c in range(clusters):
            j, kb = 0, 0
            while True:
                s, t, a, b, slot = H.hgemm_plan_work_item(p, c, j)
                if s != ST_OK:
                    break
                kb += b - a
                j += 1
            assert kb == sum(id_kb[c::clusters])
            per_cluster.append(kb)
        if p.sk_ranges:  # stream-K evens the work out
            assert max(per_cluster) - min(per_cluster) <= p.k_blocks + 1


@pytest.mark.parametrize("seed", range(4))
def test_splitk_chunks_partition_units(seed):
    r = np.random.default_rng(100 + seed)
    for _ in range(60):
        M = int(r.integers(1, 65))
        N = int(8 * r.integers(1, 40000))
        K = int(8 * r.integers(1, 4000))
        sms = int(r.choice([4, 16, 76, 148, 152]))
        schedule = int(r.choice([0, 1]))
        st, p = H.hgemm_plan(M, N, K, num_sms=sms, schedule=schedule)
        assert st == ST_OK and p.variant == H.HGEMM_VARIANT_SPLITK
        units = p.num_tiles * p.k_blocks
        prev = 0
        for g in range(p.splitk_chunks):
            s, b, e = H.hgemm_plan_splitk_range(p, g)
            assert s == ST_OK and b == prev and e > b
            prev = e
        assert prev == units
        assert p.grid <= sms and p.splitk_chunks >= p.grid
