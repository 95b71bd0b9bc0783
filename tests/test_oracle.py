"""Pins for the CPU oracle: it is checked against things other than itself.

- exact decode of every fp16 / bf16 bit pattern against numpy / torch widening;
- RNE encode against numpy's double->half conversion and against a brute-force
  nearest-value search over all bf16 values;
- hand-derived golden products (tests/golden/small_products.txt);
- closed forms: identity and permutation matrices, all-ones (C = K), a ones
  row (C = column sums of B);
- small-integer inputs against an independent int64 matrix product (exact);
- the tiled loop nest against the naive one (same k order, bitwise equal);
- float64 torch.matmul as a third opinion on small shapes;
- TN and NN storage of the same B give the same C;
- selected entries agree with the full product.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "small_products.txt")


def _rng(seed):
    return np.random.default_rng(seed)


def _all_bits():
    return np.arange(65536, dtype=np.uint32).astype(np.uint16)


# ---------------------------------------------------------------- decode ----

def test_decode_f16_all_patterns_matches_numpy():
    bits = _all_bits()
    got = oracle.decode(bits, "f16")
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # signed zeros keep their sign
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_decode_bf16_all_patterns_matches_torch():
    bits = _all_bits()
    got = oracle.decode(bits, "bf16")
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


# ---------------------------------------------------------------- encode ----

def _interesting_doubles(fmt, n, seed):
    r = _rng(seed)
    if fmt == "f16":
        lo, hi = -30, 17
        maxf, tiny = 65504.0, 2.0 ** -24
    else:
        lo, hi = -140, 129
        maxf, tiny = float(torch.finfo(torch.bfloat16).max), 2.0 ** -133
    mags = 2.0 ** r.uniform(lo, hi, n)
    signs = r.choice([-1.0, 1.0], n)
    vals = list(mags * signs)
    # exact ties and near-ties around representable values
    dec = oracle.decode(_all_bits(), fmt)
    finite = np.sort(np.unique(dec[np.isfinite(dec) & (dec >= 0)]))
    idx = r.integers(0, len(finite) - 1, n // 4)
    mids = (finite[idx] + finite[idx + 1]) / 2.0
    vals += list(mids) + list(-mids) + list(np.nextafter(mids, 0)) + list(np.nextafter(mids, np.inf))
    vals += [0.0, -0.0, tiny, tiny / 2, tiny * 1.5, maxf, -maxf, math.inf, -math.inf]
    # around the overflow threshold: max + half a step
    half_step = (maxf - finite[-2]) / 2.0
    vals += [maxf + half_step, np.nextafter(maxf + half_step, 0), -(maxf + half_step)]
    return np.array(vals, dtype=np.float64)


def test_encode_f16_matches_numpy_rne():
    x = _interesting_doubles("f16", 200000, 1)
    got = oracle.encode(x, "f16")
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, ref)


def _brute_force_rne(x, fmt):
    """Nearest representable value by exhaustive search; ties to even bits."""
    bits = _all_bits()
    dec = oracle.decode(bits, fmt)
    ok = np.isfinite(dec)
    vals, vbits = dec[ok], bits[ok]
    order = np.argsort(vals, kind="stable")
    vals, vbits = vals[order], vbits[order]
    maxf = vals[-1]
    step_top = maxf - vals[-2]
    out = np.empty(x.shape, np.uint16)
    for i, v in enumerate(x):
        if math.isnan(v):
            out[i] = 0
            continue
        if abs(v) >= maxf + step_top / 2:
            out[i] = (0xFC00 if fmt == "f16" else 0xFF80) if v < 0 else (0x7C00 if fmt == "f16" else 0x7F80)
            continue
        j = np.searchsorted(vals, v)
        cands = [k for k in (j - 1, j) if 0 <= k < len(vals)]
        dists = [abs(vals[k] - v) for k in cands]
        best = min(dists)
        tied = [cands[t] for t in range(len(cands)) if dists[t] == best]
        if len(tied) == 1:
            pick = tied[0]
        else:  # tie: the one with an even significand (last bit 0)
            pick = [k for k in tied if int(vbits[k]) & 1 == 0][0]
        b = int(vbits[pick])
        if vals[pick] == 0.0:
            b = 0x8000 if math.copysign(1.0, v) < 0 else 0
        out[i] = b
    return out


def test_encode_bf16_matches_brute_force():
    x = _interesting_doubles("bf16", 6000, 2)
    x = x[np.isfinite(x) | np.isinf(x)]
    got = oracle.encode(x, "bf16")
    ref = _brute_force_rne(x, "bf16")
    assert np.array_equal(got, ref)


def test_encode_f16_matches_brute_force_sample():
    x = _interesting_doubles("f16", 4000, 3)
    got = oracle.encode(x, "f16")
    ref = _brute_force_rne(x, "f16")
    assert np.array_equal(got, ref)


def test_encode_decode_roundtrip_all_patterns():
    for fmt in ("f16", "bf16"):
        bits = _all_bits()
        dec = oracle.decode(bits, fmt)
        ok = ~np.isnan(dec)
        assert np.array_equal(oracle.encode(dec[ok], fmt), bits[ok])


def test_encode_nan_is_nan():
    for fmt in ("f16", "bf16"):
        b = oracle.encode(np.array([math.nan]), fmt)
        assert math.isnan(oracle.decode(b, fmt)[0])


# ---------------------------------------------------------------- golden ----

def _parse_golden():
    cases, cur = [], None
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            tok = line.split()
            if tok[0] == "case":
                cur = dict(name=tok[1], M=int(tok[2]), N=int(tok[3]), K=int(tok[4]), layout=tok[5],
                           fin=tok[6], fout=tok[7])
                cases.append(cur)
            else:
                cur[tok[0]] = [float.fromhex(t) if t.startswith(("0x", "-0x")) else float(t) for t in tok[1:]]
    return cases


GOLDEN_CASES = _parse_golden()


@pytest.mark.parametrize("case", GOLDEN_CASES, ids=[c["name"] for c in GOLDEN_CASES])
def test_golden_products(case):
    M, N, K = case["M"], case["N"], case["K"]
    a = oracle.encode(np.array(case["A"]), case["fin"])
    b = oracle.encode(np.array(case["B"]), case["fin"])
    # inputs must be exact in the input format
    assert np.array_equal(oracle.decode(a, case["fin"]), np.array(case["A"]))
    assert np.array_equal(oracle.decode(b, case["fin"]), np.array(case["B"]))
    C, _, _ = oracle.gemm(a, b, M, N, K, case["layout"], case["fin"], case["fout"])
    got = oracle.decode(C.ravel(), case["fout"])
    exp = np.array(case["C"])
    assert np.array_equal(got, exp), (got, exp)
    assert not np.any(np.signbit(got[exp == 0]))


# ---------------------------------------------------------- closed forms ----

def _enc(x, fmt):
    return oracle.encode(np.asarray(x, dtype=np.float64), fmt)


@pytest.mark.parametrize("fmt", ["f16", "bf16"])
@pytest.mark.parametrize("layout", ["TN", "NN"])
def test_identity_and_permutation(fmt, layout):
    r = _rng(10)
    K = N = 37
    M = K
    bvals = r.uniform(-3, 3, (K, N))
    Bkn = oracle.decode(_enc(bvals, fmt), fmt).reshape(K, N)  # exact B[k][n]
    B_store = _enc(Bkn.T if layout == "TN" else Bkn, fmt)
    I = _enc(np.eye(M, K), fmt)
    C, ex, _ = oracle.gemm(I, B_store, M, N, K, layout, fmt, fmt, want_exact=True)
    assert np.array_equal(ex, Bkn)
    perm = r.permutation(M)
    P = np.zeros((M, K))
    P[np.arange(M), perm] = 1.0
    C, ex, _ = oracle.gemm(_enc(P, fmt), B_store, M, N, K, layout, fmt, fmt, want_exact=True)
    assert np.array_equal(ex, Bkn[perm])
    assert np.array_equal(C, _enc(Bkn[perm], fmt))


@pytest.mark.parametrize("fmt,K", [("f16", 1), ("f16", 100), ("f16", 2048), ("f16", 3001),
                                   ("bf16", 255), ("bf16", 513), ("bf16", 4104)])
def test_all_ones_gives_K(fmt, K):
    M, N = 3, 5
    A = _enc(np.ones((M, K)), fmt)
    B = _enc(np.ones((N, K)), fmt)
    C, ex, ab = oracle.gemm(A, B, M, N, K, "TN", fmt, fmt, want_exact=True, want_abs=True)
    assert np.all(ex == K) and np.all(ab == K)
    assert np.all(C == _enc(float(K), fmt))
    # K rounded to the format: e.g. 3001 -> 3000 in fp16 (spacing 2), 513 -> 512 in bf16
    assert oracle.decode(C[:1, :1].ravel(), fmt)[0] == {("f16", 3001): 3000.0, ("bf16", 513): 512.0,
                                                        ("bf16", 4104): 4096.0}.get((fmt, K), float(K))


@pytest.mark.parametrize("layout", ["TN", "NN"])
def test_ones_row_gives_column_sums(layout):
    r = _rng(11)
    K, N = 300, 40
    Bkn = oracle.decode(_enc(r.integers(-50, 50, (K, N)) / 8.0, "bf16"), "bf16").reshape(K, N)
    B_store = _enc(Bkn.T if layout == "TN" else Bkn, "bf16")
    A = _enc(np.ones((1, K)), "bf16")
    _, ex, _ = oracle.gemm(A, B_store, 1, N, K, layout, "bf16", "bf16", want_exact=True)
    assert np.array_equal(ex[0], Bkn.sum(axis=0))
    # and a ones column on the right gives row sums of A
    Avals = oracle.decode(_enc(r.integers(-50, 50, (6, K)) / 4.0, "bf16"), "bf16").reshape(6, K)
    ones = _enc(np.ones((1, K)) if layout == "TN" else np.ones((K, 1)), "bf16")
    _, ex, _ = oracle.gemm(_enc(Avals, "bf16"), ones, 6, 1, K, layout, "bf16", "bf16", want_exact=True)
    assert np.array_equal(ex[:, 0], Avals.sum(axis=1))


@pytest.mark.parametrize("fmt", ["f16", "bf16"])
@pytest.mark.parametrize("layout", ["TN", "NN"])
@pytest.mark.parametrize("shape", [(1, 1, 1), (7, 9, 17), (31, 8, 64), (64, 33, 200)])
def test_small_integers_exact_vs_int64(fmt, layout, shape):
    M, N, K = shape
    r = _rng(M * 1000 + N * 10 + K)
    a = r.integers(-4, 5, (M, K))
    bkn = r.integers(-4, 5, (K, N))
    ref = a.astype(np.int64) @ bkn.astype(np.int64)
    A = _enc(a, fmt)
    B = _enc(bkn.T if layout == "TN" else bkn, fmt)
    C, ex, ab = oracle.gemm(A, B, M, N, K, layout, fmt, fmt, want_exact=True, want_abs=True)
    assert np.array_equal(ex, ref.astype(np.float64))
    assert np.array_equal(ab, (np.abs(a) @ np.abs(bkn)).astype(np.float64))
    assert np.array_equal(C, _enc(ref, fmt))


@pytest.mark.parametrize("layout", ["TN", "NN"])
@pytest.mark.parametrize("shape", [(1, 1, 1), (2, 3, 7), (8, 9, 17), (31, 17, 64), (64, 64, 9), (3, 2, 72)])
def test_tiled_matches_naive(layout, shape):
    M, N, K = shape
    r = _rng(sum(shape))
    A = _enc(r.normal(0, 1, (M, K)), "f16")
    B = _enc(r.normal(0, 1, (N, K) if layout == "TN" else (K, N)), "f16")
    _, ex, _ = oracle.gemm(A, B, M, N, K, layout, "f16", "f16", want_exact=True)
    for bm, bn, bk in [(1, 1, 1), (2, 4, 8), (8, 8, 16), (128, 128, 64)]:
        tiled = oracle.gemm_tiled(A, B, M, N, K, layout, "f16", bm, bn, bk)
        assert np.array_equal(tiled, ex)


@pytest.mark.parametrize("fmt", ["f16", "bf16"])
@pytest.mark.parametrize("layout", ["TN", "NN"])
def test_float64_torch_matmul_third_opinion(fmt, layout):
    M, N, K = 40, 24, 333
    r = _rng(5)
    A = _enc(r.uniform(-1, 1, (M, K)), fmt)
    B = _enc(r.uniform(-1, 1, (N, K) if layout == "TN" else (K, N)), fmt)
    a = torch.from_numpy(oracle.decode(A, fmt).reshape(M, K))
    b = torch.from_numpy(oracle.decode(B, fmt).reshape((N, K) if layout == "TN" else (K, N)))
    ref = (a @ (b.T if layout == "TN" else b)).numpy()
    _, ex, ab = oracle.gemm(A, B, M, N, K, layout, fmt, fmt, want_exact=True, want_abs=True)
    assert np.all(np.abs(ex - ref) <= 1e-12 * ab + 1e-300)


def test_tn_and_nn_storage_agree():
    M, N, K = 19, 23, 129
    r = _rng(6)
    A = _enc(r.normal(0, 1, (M, K)), "bf16")
    Bkn = _enc(r.normal(0, 1, (K, N)), "bf16").reshape(K, N)
    C1, e1, _ = oracle.gemm(A, np.ascontiguousarray(Bkn.T), M, N, K, "TN", "bf16", "f16", want_exact=True)
    C2, e2, _ = oracle.gemm(A, Bkn, M, N, K, "NN", "bf16", "f16", want_exact=True)
    assert np.array_equal(e1, e2) and np.array_equal(C1, C2)


@pytest.mark.parametrize("layout", ["TN", "NN"])
def test_entries_agree_with_full(layout):
    M, N, K = 33, 65, 100
    r = _rng(7)
    A = _enc(r.normal(0, 1, (M, K)), "f16")
    B = _enc(r.normal(0, 1, (N, K) if layout == "TN" else (K, N)), "f16")
    _, ex, ab = oracle.gemm(A, B, M, N, K, layout, "f16", "f16", want_exact=True, want_abs=True, nthreads=3)
    rows = r.integers(0, M, 500)
    cols = r.integers(0, N, 500)
    e, a = oracle.gemm_entries(A, B, M, N, K, layout, "f16", rows, cols, nthreads=4)
    assert np.array_equal(e, ex[rows, cols]) and np.array_equal(a, ab[rows, cols])


def test_thread_count_does_not_change_results():
    M, N, K = 50, 20, 300
    r = _rng(8)
    A = _enc(r.normal(0, 1, (M, K)), "bf16")
    B = _enc(r.normal(0, 1, (N, K)), "bf16")
    outs = [oracle.gemm(A, B, M, N, K, "TN", "bf16", "bf16", nthreads=t, want_exact=True)[1] for t in (1, 3, 64)]
    assert all(np.array_equal(outs[0], o) for o in outs[1:])


def test_empty_dimensions():
    A = np.zeros((0,), np.uint16)
    C, ex, _ = oracle.gemm(A, np.zeros((0,), np.uint16), 0, 0, 5, "TN", "f16", "f16", want_exact=True)
    assert C.shape == (0, 0)
    # K = 0: the empty sum is +0
    C, ex, ab = oracle.gemm(np.zeros((0,), np.uint16), np.zeros((0,), np.uint16), 3, 4, 0, "TN", "f16", "bf16",
                            want_exact=True, want_abs=True)
    assert np.all(ex == 0) and np.all(C == 0) and np.all(ab == 0)


def test_bad_entry_index_is_rejected():
    A = _enc(np.ones((2, 2)), "f16")
    with pytest.raises(RuntimeError):
        oracle.gemm_entries(A, A, 2, 2, 2, "TN", "f16", [0, 2], [0, 0])


@pytest.mark.parametrize("layout", [-1, 2, 7])
def test_bad_layout_is_rejected_by_the_c_entry_points(layout):
    """The C functions themselves refuse a layout that is neither TN nor NN
    (the Python wrapper checks too, but a caller of the library must not get
    B silently read as NN), and leave the outputs untouched."""
    import ctypes
    lib = oracle._load()
    A = _enc(np.ones((2, 3)), "f16")
    u16p = ctypes.POINTER(ctypes.c_uint16)
    f64p = ctypes.POINTER(ctypes.c_double)
    i64p = ctypes.POINTER(ctypes.c_int64)
    rows = np.array([0, 1], np.int64)
    cols = np.array([1, 0], np.int64)
    ex = np.full(2, 7.0)
    ab = np.full(2, 7.0)
    st = lib.oracle_gemm_entries(A.ctypes.data_as(u16p), A.ctypes.data_as(u16p), 2, 2, 3, layout, 0,
                                 rows.ctypes.data_as(i64p), cols.ctypes.data_as(i64p), 2, ex.ctypes.data_as(f64p),
                                 ab.ctypes.data_as(f64p), 1)
    assert st == -1 and np.all(ex == 7.0) and np.all(ab == 7.0)
    C = np.zeros(4, np.uint16)
    full = np.full(4, 7.0)
    st = lib.oracle_gemm(A.ctypes.data_as(u16p), A.ctypes.data_as(u16p), 2, 2, 3, layout, 0, 0,
                         C.ctypes.data_as(u16p), full.ctypes.data_as(f64p), None, 1)
    assert st == -1 and np.all(full == 7.0)
    st = lib.oracle_gemm_tiled(A.ctypes.data_as(u16p), A.ctypes.data_as(u16p), 2, 2, 3, layout, 0, 1, 1, 1,
                               full.ctypes.data_as(f64p))
    assert st == -1 and np.all(full == 7.0)
    # the same call with a valid layout succeeds
    st = lib.oracle_gemm_entries(A.ctypes.data_as(u16p), A.ctypes.data_as(u16p), 2, 2, 3, 0, 0,
                                 rows.ctypes.data_as(i64p), cols.ctypes.data_as(i64p), 2, ex.ctypes.data_as(f64p),
                                 ab.ctypes.data_as(f64p), 1)
    assert st == 0 and np.all(ex == 3.0) and np.all(ab == 3.0)
