// sched.cuh -- persistent tile scheduling (host + device, pure functions).
//
// Persistent kernel, static schedule: "tcgen05 for dummies: a B200 GEMM from
// scratch" (translated), section "Persistent kernel: static scheduling" -- one
// CTA (or CTA pair) per SM walks tiles t = id, id + count, ...
// Grouped rasterisation ("block swizzle" in "HGEMM: WMMA and MMA PTX study
// notes" and "HGEMM CuTe version study notes", section on block swizzle): the
// linear tile index walks a band of group_m tile rows column by column, so the
// tiles in flight at one time share a few rows of A and columns of B in L2.
// The CTA-pair mapping of the 2-SM section (the two CTAs of a pair take
// adjacent 128-row halves of one M tile) is built into the tile height.
#pragma once

#include <stdint.h>

#include "desc.cuh"  // HG_HD

namespace hg {

struct TileCoord {
  int32_t m;  // tile row index
  int32_t n;  // tile column index
};

// Linear tile index -> (tile row, tile column), grouped by group_m rows.
HG_HD TileCoord tile_coord(int32_t t, int32_t tiles_m, int32_t tiles_n, int32_t group_m) {
  const int32_t per_group = group_m * tiles_n;
  const int32_t g = t / per_group;
  const int32_t first_m = g * group_m;
  const int32_t rows_left = tiles_m - first_m;
  const int32_t gsz = rows_left < group_m ? rows_left : group_m;
  const int32_t r = t - g * per_group;
  TileCoord c;
  c.m = first_m + r % gsz;
  c.n = r / gsz;
  return c;
}

// Split-K (skinny M): the work is the tile-major list of (tile, k-block) units,
// U = num_tiles * k_blocks; CTA c of G owns the contiguous range
// [floor(c U / G), floor((c+1) U / G)).  Every CTA gets the same number of
// k-blocks up to one, whatever the tile count.
HG_HD int64_t splitk_begin(int64_t c, int64_t units, int64_t ctas) { return (c * units) / ctas; }

// The CTA that owns unit u: the largest c with floor(c U / G) <= u.
HG_HD int64_t splitk_owner(int64_t u, int64_t units, int64_t ctas) { return ((u + 1) * ctas - 1) / units; }

}  // namespace hg
