"""TMA-engine micro-benchmark (hgemm_tma_bench) with a checked sweep.

"tcgen05 for dummies: a B200 GEMM from scratch" (translated) sees its GEMM
run 2.7x faster once its TMA boxes are 128 bytes wide instead of 16, and finds
one 3-D copy per tile no faster than several 2-D copies; it guesses that the
TMA engine prefers wide inner boxes and asks for a micro-benchmark.  This
module runs that benchmark on the GPU: for each copy form and tile shape,
every SM streams tiles from a source that fits in L2 or from one far larger
than L2, and the table reports bytes per SM clock and aggregate GB/s.  Each
run also checks what landed in shared memory against sums computed here from
the same tiles.

    python -m tensor_core_half_gb300.tma_bench            # markdown table
"""
from __future__ import annotations

import argparse
import itertools
import json

import numpy as np
import torch

from . import hgemm


def _words(y, x):
    """Source word at (row y, column x): depends on both (uint16 bits)."""
    y = np.asarray(y, dtype=np.int64)
    x = np.asarray(x, dtype=np.int64)
    return ((y * 131 + x * 7 + (y * x) % 17) & 0xFFFF).astype(np.uint64)


def expected_sums(height, width, mode, tile_rows, tile_cols, tiles):
    """Sum and sum of squares of the 16-bit words of the listed tiles."""
    tiles_x = width // tile_cols
    s1 = s2 = 0
    for t in tiles:
        if t < 0:
            continue
        if mode == hgemm.HGEMM_TMA_BULK:
            i = np.arange(t * tile_rows * tile_cols, (t + 1) * tile_rows * tile_cols, dtype=np.int64)
            v = _words(i // width, i % width)
        else:
            ty, tx = divmod(t, tiles_x)
            y = np.arange(ty * tile_rows, (ty + 1) * tile_rows)[:, None]
            x = np.arange(tx * tile_cols, (tx + 1) * tile_cols)[None, :]
            v = _words(y, x)
        s1 += int(v.sum())
        s2 += int((v * v).sum())
    return s1 & (2**64 - 1), s2 & (2**64 - 1)


def source(height, width, device="cuda"):
    """The words as a bf16 device tensor (bits copied unchanged), built on the GPU."""
    out = torch.empty((height, width), dtype=torch.int16, device=device)
    x = torch.arange(width, dtype=torch.int32, device=device)[None, :]
    rows = max(1, (1 << 26) // width)
    for y0 in range(0, height, rows):
        y = torch.arange(y0, min(height, y0 + rows), dtype=torch.int32, device=device)[:, None]
        v = (y * 131 + x * 7 + torch.remainder(y * x, 17)) & 0xFFFF
        out[y0:y0 + y.shape[0]] = (v - ((v >> 15) << 16)).to(torch.int16)  # same 16 bits, signed
    return out.view(torch.bfloat16)


def run_checked(src, mode, tile_rows, tile_cols, depth, iters, issuers=1, ctas=0, check_ctas=8,
                walk=hgemm.HGEMM_TMA_WALK_SCATTERED):
    height, width = src.shape
    st, res, sums, last = hgemm.hgemm_tma_bench(src.data_ptr(), height, width, mode, tile_rows, tile_cols, depth, iters,
                                                issuers, ctas, torch.cuda.current_stream().cuda_stream, walk=walk)
    if st != hgemm.HGEMM_OK:
        raise hgemm.HgemmError(st, "hgemm_tma_bench")
    step = max(1, len(sums) // check_ctas)
    for i in range(0, len(sums), step):
        if tuple(sums[i]) != expected_sums(height, width, mode, tile_rows, tile_cols, last[i]):
            raise AssertionError("TMA bench: CTA %d holds the wrong bytes (mode %d)" % (i, mode))
    return res


def sweep(per_cta_mb=32):
    names = {v: k for k, v in hgemm.TMA_MODES.items()}
    rows = []
    windows = [("L2 (32 MiB)", 4096, 4096), ("HBM (2 GiB)", 32768, 32768)]
    configs = []
    for mode in (hgemm.HGEMM_TMA_2D_16B, hgemm.HGEMM_TMA_3D_16B, hgemm.HGEMM_TMA_2D_128B, hgemm.HGEMM_TMA_3D_128B,
                 hgemm.HGEMM_TMA_BULK):
        configs.append((mode, 128, 64, 1))  # the GEMM's A stage: 128 rows x 64 columns (16 KiB)
        configs.append((mode, 128, 128, 1))
    for r in (32, 64, 256):
        configs.append((hgemm.HGEMM_TMA_2D_128B, r, 64, 1))  # box height
    configs.append((hgemm.HGEMM_TMA_2D_128B, 128, 128, 2))  # two issuing warps
    configs.append((hgemm.HGEMM_TMA_2D_128B, 256, 128, 2))
    configs.append((hgemm.HGEMM_TMA_BULK, 256, 128, 1))  # 64 KiB per copy
    configs.append((hgemm.HGEMM_TMA_BULK, 128, 32, 1))   # 8 KiB per copy
    for wname, h, w in windows:
        src = source(h, w)
        for (mode, r, c, iss), (walk_name, walk) in itertools.product(configs, hgemm.TMA_WALKS.items()):
            tile_bytes = r * c * 2
            depth = max(1, min(8, (160 * 1024) // tile_bytes))
            iters = max(depth, (per_cta_mb << 20) // tile_bytes)
            run_checked(src, mode, r, c, depth, max(depth, iters // 8), iss, walk=walk)  # warm-up
            res = run_checked(src, mode, r, c, depth, iters, iss, walk=walk)
            rows.append({"source": wname, "walk": walk_name, "mode": names[mode], "tile": "%dx%d" % (r, c),
                         "copies_per_tile": res.copies_per_tile, "copy_bytes": tile_bytes // res.copies_per_tile,
                         "issuers": iss, "depth": depth, "bytes_per_clk_sm": round(res.bytes_per_clk_sm, 1),
                         "gbs": round(res.gbs, 0), "sm_mhz": round(res.sm_mhz, 0), "checked": True})
        del src
        torch.cuda.empty_cache()
    return rows


def markdown(rows):
    head = ["source", "walk", "mode", "tile", "copies_per_tile", "copy_bytes", "issuers", "depth", "bytes_per_clk_sm", "gbs",
            "sm_mhz"]
    out = ["| " + " | ".join(head) + " |", "|" + "---|" * len(head)]
    for r in rows:
        out.append("| " + " | ".join(str(r[k]) for k in head) + " |")
    return "\n".join(out)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--per-cta-mb", type=int, default=32)
    ap.add_argument("--json", action="store_true")
    args = ap.parse_args()
    rows = sweep(args.per_cta_mb)
    print(json.dumps(rows) if args.json else markdown(rows))


if __name__ == "__main__":
    main()
