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

// One item of a cluster's work list: k-blocks [kb0, kb1) of tile `tile`.
// slot < 0: the item covers the whole K range, its result goes straight to C.
// slot 0 / 1: a stream-K partial; it is the first (0) or last (1) item of the
// cluster's stream-K range, which fixes where its fp32 partial is kept.
struct WorkItem {
  int32_t tile, kb0, kb1, slot;
};

// The persistent dense kernel's schedule ("Persistent kernel: static
// scheduling", extended with stream-K).  Tiles [0, dp_tiles) are dealt
// round-robin to the clusters and computed over the whole K range.  The
// remaining tiles form sk_units = (num_tiles - dp_tiles) * k_blocks units of
// one k-block each, cut into one contiguous range per cluster, so that every
// cluster does the same number of k-blocks.  A tile cut between clusters is
// finished by whichever contributor arrives last.  Each cluster walks its
// stream-K range FIRST: the fix-ups of split tiles then overlap the mainloops
// of the data-parallel tiles instead of ending the kernel.
struct WorkIter {
  int32_t t, step, dp_tiles, k_blocks;
  int64_t u, u_begin, u_end;

  HG_HD WorkIter(int32_t cluster, int32_t nclusters, int32_t dp_tiles_, int64_t sk_units, int32_t k_blocks_)
      : t(cluster), step(nclusters), dp_tiles(dp_tiles_), k_blocks(k_blocks_) {
    u_begin = splitk_begin(cluster, sk_units, nclusters);
    u_end = splitk_begin((int64_t)cluster + 1, sk_units, nclusters);
    u = u_begin;
  }

  HG_HD bool next(WorkItem& w) {
    if (u < u_end) {
      const int64_t rel = u / k_blocks;
      const int32_t kb0 = (int32_t)(u - rel * k_blocks);
      const int64_t left = u_end - u;
      const int32_t room = k_blocks - kb0;
      const int32_t kb1 = kb0 + (int32_t)(left < room ? left : room);
      w.tile = dp_tiles + (int32_t)rel;
      w.kb0 = kb0;
      w.kb1 = kb1;
      w.slot = (kb0 == 0 && kb1 == k_blocks) ? -1 : (u == u_begin ? 0 : 1);
      u += kb1 - kb0;
      return true;
    }
    if (t < dp_tiles) {
      w.tile = t;
      w.kb0 = 0;
      w.kb1 = k_blocks;
      w.slot = -1;
      t += step;
      return true;
    }
    return false;
  }
};

// Contributors of stream-K tile `tile`: clusters [*first, *last], in K order.
HG_HD void sk_contributors(int32_t tile, int32_t dp_tiles, int64_t sk_units, int32_t k_blocks, int32_t nclusters,
                           int64_t* first, int64_t* last) {
  const int64_t u0 = (int64_t)(tile - dp_tiles) * k_blocks;
  *first = splitk_owner(u0, sk_units, nclusters);
  *last = splitk_owner(u0 + k_blocks - 1, sk_units, nclusters);
}

// Where contributor `c` keeps its partial of stream-K tile `tile`: slot 0 if
// the tile is the first of c's range, else slot 1 (it is then c's last).
HG_HD int32_t sk_slot_of(int64_t c, int32_t tile, int32_t dp_tiles, int64_t sk_units, int32_t k_blocks,
                         int32_t nclusters) {
  const int64_t first_tile = splitk_begin(c, sk_units, nclusters) / k_blocks;
  return (first_tile == (int64_t)(tile - dp_tiles)) ? 0 : 1;
}

}  // namespace hg
