"""Parity helpers shared by the GPU tests, the smoke check and the benchmark.

Tolerances (what the tests assert, per output entry, with ref the oracle's
exact double result and S = sum_k |a_mk * b_kn|):
  fp32 accumulation:  |gpu - ref| <= ulp_out(ref) + 2^-20 * S
  fp16 accumulation:  |gpu - ref| <= 2^-9 * S            (fp16 output)
                      |gpu - ref| <= 2^-9 * S + ulp_out(ref)   (bf16 output)
  small-integer inputs: bit-exact against the oracle's rounded result.
ulp_out(r) is the spacing of the output format at |r|,
2^(floor(log2|r|) - p + 1), never below the subnormal spacing (p = 11, spacing
2^-24 for fp16; p = 8, spacing 2^-133 for bf16).
"""
from __future__ import annotations

import numpy as np

import oracle
from tensor_core_half_gb300 import workloads

_FMT = {"f16": (11, -24), "bf16": (8, -133)}


def ulp_out(ref: np.ndarray, fmt: str) -> np.ndarray:
    p, sub = _FMT[fmt]
    a = np.abs(np.asarray(ref, dtype=np.float64))
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    spacing = np.exp2(e - p + 1)
    spacing = np.where(a > 0, spacing, 0.0)
    return np.maximum(spacing, 2.0 ** sub)


def bound(ref, absdot, acc: str, out: str) -> np.ndarray:
    if acc == "f32":
        return ulp_out(ref, out) + 2.0 ** -20 * absdot
    b = 2.0 ** -9 * absdot
    if out == "bf16":
        b = b + ulp_out(ref, out)
    return b


def boundary_indices(extent: int, tiles=(128, 256)) -> np.ndarray:
    """Rows (or columns) at tile boundaries: 0, T-1, T, 2T-1, 2T, the middle,
    the start of the last full tile and the row before it, and the last."""
    idx = set()
    for T in tiles:
        last_full = (extent // T) * T
        for v in (0, T - 1, T, 2 * T - 1, 2 * T, extent // 2 - 1, extent // 2, last_full - 1, last_full,
                  extent - 1):
            if 0 <= v < extent:
                idx.add(v)
    return np.array(sorted(idx), dtype=np.int64)


def sample_entries(M: int, N: int, n_random: int, seed: int):
    """n_random seeded entries plus every entry of the boundary rows and columns."""
    r = np.random.default_rng(seed)
    rows = [r.integers(0, M, n_random)]
    cols = [r.integers(0, N, n_random)]
    for i in boundary_indices(M):
        rows.append(np.full(N, i, np.int64))
        cols.append(np.arange(N, dtype=np.int64))
    for j in boundary_indices(N):
        rows.append(np.arange(M, dtype=np.int64))
        cols.append(np.full(M, j, np.int64))
    return np.concatenate(rows), np.concatenate(cols)


def sample_entries_sparse(M: int, N: int, n_random: int, seed: int, per_line: int = 2048):
    """For outputs too large to check whole rows: n_random seeded entries plus
    per_line seeded entries of every boundary row and column (including the
    last row and column)."""
    r = np.random.default_rng(seed)
    rows = [r.integers(0, M, n_random)]
    cols = [r.integers(0, N, n_random)]
    for i in boundary_indices(M):
        rows.append(np.full(per_line, i, np.int64))
        cols.append(np.concatenate([[0, N - 1], r.integers(0, N, per_line - 2)]))
    for j in boundary_indices(N):
        rows.append(np.concatenate([[0, M - 1], r.integers(0, M, per_line - 2)]))
        cols.append(np.full(per_line, j, np.int64))
    return np.concatenate(rows), np.concatenate(cols)


def check_gathered(C, A, B, M, N, K, layout, in_dtype, acc, out, n_random=8192, seed=0):
    """Sampled parity for operands and results that stay on the device.

    C, A, B are device tensors (A [M, K]; B [N, K] for TN, [K, N] for NN).
    The sampled entries of C, and the rows of A and B they need, are gathered
    to the host; the oracle computes those dot products from the exact input
    bits (on the gathered sub-matrices, with the indices mapped)."""
    import torch

    rows, cols = sample_entries_sparse(M, N, n_random, seed)
    ur, ri = np.unique(rows, return_inverse=True)
    uc, ci = np.unique(cols, return_inverse=True)
    dev = C.device
    tr = torch.from_numpy(ur).to(dev)
    tc = torch.from_numpy(uc).to(dev)
    a_sub = A.view(torch.int16).index_select(0, tr).cpu().numpy().view(np.uint16)
    if layout == "TN":
        b_sub = B.view(torch.int16).index_select(0, tc).cpu().numpy().view(np.uint16)
    else:
        b_sub = B.view(torch.int16).index_select(1, tc).cpu().numpy().view(np.uint16)
    g_bits = C.view(torch.int16)[torch.from_numpy(rows).to(dev), torch.from_numpy(cols).to(dev)]
    g = oracle.decode(g_bits.cpu().numpy().view(np.uint16), out)
    ref, absdot = oracle.gemm_entries(a_sub, b_sub, ur.size, uc.size, K, layout, in_dtype, ri, ci)
    b = bound(ref, absdot, acc, out)
    err = np.abs(g - ref)
    bad = ~(err <= b)
    if bad.any():
        k = np.nonzero(bad)[0][:8]
        detail = ", ".join("[%d,%d] gpu=%r ref=%r bound=%.3g" % (rows[i], cols[i], g[i], ref[i], b[i]) for i in k)
        raise AssertionError("%d of %d sampled entries out of tolerance: %s" % (int(bad.sum()), ref.size, detail))
    return dict(entries=int(ref.size), max_err=float(err.max()))


def check(got_bits: np.ndarray, A_bits, B_bits, M, N, K, layout, in_dtype, acc, out, sampled=False, n_random=8192,
          seed=0, nthreads=0):
    """Compares a device result with the oracle.  Returns a dict of statistics
    and raises AssertionError with details on the first violation."""
    got_bits = np.asarray(got_bits).reshape(M, N)
    if sampled:
        rows, cols = sample_entries(M, N, n_random, seed)
        ref, absdot = oracle.gemm_entries(A_bits, B_bits, M, N, K, layout, in_dtype, rows, cols, nthreads=nthreads)
        g = oracle.decode(got_bits[rows, cols], out)
    else:
        _, ref, absdot = oracle.gemm(A_bits, B_bits, M, N, K, layout, in_dtype, out, nthreads=nthreads,
                                     want_exact=True, want_abs=True)
        ref = ref.ravel()
        absdot = absdot.ravel()
        g = oracle.decode(got_bits.ravel(), out)
        rows = np.repeat(np.arange(M), N)
        cols = np.tile(np.arange(N), M)
    b = bound(ref, absdot, acc, out)
    err = np.abs(g - ref)
    bad = ~(err <= b)  # also catches NaN
    stats = dict(entries=int(ref.size), max_err=float(np.nanmax(err)) if err.size else 0.0,
                 max_ratio=float(np.nanmax(err / np.maximum(b, 1e-300))) if err.size else 0.0)
    if bad.any():
        k = np.nonzero(bad)[0][:8]
        detail = ", ".join("[%d,%d] gpu=%r ref=%r bound=%.3g" % (rows[i], cols[i], g[i], ref[i], b[i]) for i in k)
        raise AssertionError("%d of %d entries out of tolerance (%s acc, %s out): %s" %
                             (int(bad.sum()), ref.size, acc, out, detail))
    return stats


def inputs(M, N, K, layout, in_dtype, dist, seed, scale_inv_sqrt_k=False):
    """CPU tensors from the shared seeded generator and their raw bits."""
    a, b = workloads.generate(M, N, K, layout, in_dtype, dist, seed, scale_inv_sqrt_k)
    return a, b, workloads.bits(a), workloads.bits(b)
