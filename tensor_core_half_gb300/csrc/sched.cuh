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

// Linear tile index -> (tile row, tile column), grouped by group_m rows: down
// the rows of a group column by column, even groups left to right and odd
// groups right to left, so that each group starts on the tile columns of B
// the group before it read last, which are still in L2 (8192^3 on GB300:
// 1.05 GB of DRAM traffic per launch instead of 1.11).
HG_HD TileCoord tile_coord(int32_t t, int32_t tiles_m, int32_t tiles_n, int32_t group_m) {
  const int32_t per_group = group_m * tiles_n;
  const int32_t g = t / per_group;
  const int32_t first_m = g * group_m;
  const int32_t rows_left = tiles_m - first_m;
  const int32_t gsz = rows_left < group_m ? rows_left : group_m;
  const int32_t r = t - g * per_group;
  TileCoord c;
  c.m = first_m + r % gsz;
  c.n = (g & 1) ? tiles_n - 1 - r / gsz : r / gsz;
  return c;
}

// Split-K (skinny M): the work is the tile-major list of (tile, k-block) units,
// U = num_tiles * k_blocks; CTA c of G owns the contiguous range
// [floor(c U / G), floor((c+1) U / G)).  Every CTA gets the same number of
// k-blocks up to one, whatever the tile count.
HG_HD int64_t splitk_begin(int64_t c, int64_t units, int64_t ctas) { return (c * units) / ctas; }

// The CTA that owns unit u: the largest c with floor(c U / G) <= u.
HG_HD int64_t splitk_owner(int64_t u, int64_t units, int64_t ctas) { return ((u + 1) * ctas - 1) / units; }

// Split-K work ids ("chunks"): contiguous ranges of the tile-major unit list.
// The first `big` chunks cut the first `head` units evenly; the remaining
// units are cut evenly into `n_small` chunks.  Static schedule: head = units,
// n_small = 0, one chunk per CTA (the balanced split above).  Dynamic
// schedule: about three quarters of the units in one big chunk per SM, the
// rest in small chunks that the SMs which finish first take over, so that
// work still spreads when some SMs are busy with other kernels.
// align > 1 (whole-tile split, align = k_blocks): the big chunks cut the
// head in steps of `align` units, so that every chunk is whole tiles.
struct SplitChunks {
  int64_t units, head;
  int32_t big, n_small;
  int32_t align = 1;

  HG_HD int64_t count() const { return (int64_t)big + n_small; }
  HG_HD int64_t begin(int64_t g) const {
    if (g <= big) return align * splitk_begin(g, head / align, big);
    return head + splitk_begin(g - big, units - head, n_small);
  }
  // The chunk that holds unit u.
  HG_HD int64_t owner(int64_t u) const {
    if (u < head) return splitk_owner(u / align, head / align, big);
    return big + splitk_owner(u - head, units - head, n_small);
  }
};

// The chunk layout the planner picks: static, or (dynamic, when there are at
// least four units per SM) a quarter of the units in chunks of about a
// quarter of an SM's share.  Smaller chunks balance finer but cost more than
// they save on GB300: a CTA that takes a short k-slice of a tile and moves on
// loses the DRAM row locality of one long run (measured: 1/8-share chunks
// 22 % slower than the static split on an idle GPU, 1/4-share 8 %).
HG_HD SplitChunks splitk_chunks(int64_t units, int32_t ctas, bool dynamic) {
  SplitChunks c;
  c.units = units;
  c.big = ctas;
  c.head = units;
  c.n_small = 0;
  if (dynamic && units >= 4 * (int64_t)ctas) {
    const int64_t tail = units / 4;
    int64_t size = units / ((int64_t)ctas * 4);
    if (size < 1) size = 1;
    c.head = units - tail;
    c.n_small = (int32_t)((tail + size - 1) / size);
  }
  return c;
}

// The segments of a split-K chunk [begin, end): one per N tile it touches,
// k-blocks [kb0, kb1) of that tile.  They are processed in ascending order,
// except that the longest (the later one on a tie) goes last.  A segment's
// fix-up runs in the epilogue after its MMAs, one segment after another, so a
// short segment at the end of a chunk would wait behind the fix-up of the
// long one before it and both would end the kernel; with the long segment
// last, the other fix-ups finish under its mainloop.  Where a segment sits in
// K (first of its chunk or not) still decides where its partial is kept.
struct ChunkSegments {
  int64_t begin, end, tile_lo;
  int32_t k_blocks, count, longest;

  HG_HD void init(int64_t b, int64_t e, int32_t kb) {
    begin = b;
    end = e;
    k_blocks = kb;
    tile_lo = b / kb;
    count = (e > b) ? (int32_t)((e - 1) / kb - tile_lo + 1) : 0;
    longest = 0;
    if (count >= 2) {
      int64_t best = (tile_lo + 1) * kb - b;  // segment 0
      if (count >= 3 && kb >= best) {         // the last whole tile in between
        longest = count - 2;
        best = kb;
      }
      if (e - (tile_lo + count - 1) * kb >= best) longest = count - 1;
    }
  }
  // Segment index processed at position i (0 <= i < count).
  HG_HD int32_t at(int32_t i) const {
    if (i < longest) return i;
    return (i + 1 < count) ? i + 1 : longest;
  }
  HG_HD void get(int32_t idx, int32_t* tile, int32_t* kb0, int32_t* kb1) const {
    const int64_t t = tile_lo + idx;
    const int64_t lo = (idx == 0) ? begin : t * k_blocks;
    const int64_t hi = (t + 1) * k_blocks < end ? (t + 1) * k_blocks : end;
    *tile = (int32_t)t;
    *kb0 = (int32_t)(lo - t * k_blocks);
    *kb1 = (int32_t)(hi - t * k_blocks);
  }
};

// Whole tiles, none split along K: CTA c of `ctas` takes tiles
// [floor(c T / ctas), floor((c+1) T / ctas)).
HG_HD SplitChunks splitk_whole_tiles(int64_t tiles, int32_t k_blocks, int32_t ctas) {
  SplitChunks c;
  c.units = tiles * k_blocks;
  c.head = c.units;
  c.big = ctas;
  c.n_small = 0;
  c.align = k_blocks;
  return c;
}

// One item of a cluster's work list: k-blocks [kb0, kb1) of tile `tile`.
// slot < 0: the item covers the whole K range, its result goes straight to C.
// slot 0 / 1: a stream-K partial; it is the first (0) or last (1) item of
// stream-K range `owner`, which fixes where its fp32 partial is kept.
struct WorkItem {
  int32_t tile, kb0, kb1, slot, owner;
};

// The dense kernel's work, cut into work ids ("Persistent kernel: static
// scheduling", extended with stream-K).  Ids [0, sk_ranges) are stream-K
// ranges: the last tiles (num_tiles - dp_tiles of them) form sk_units =
// (num_tiles - dp_tiles) * k_blocks units of one k-block each, cut into
// sk_ranges contiguous ranges of equal size (up to one).  Ids [sk_ranges,
// sk_ranges + dp_tiles) are whole tiles.  A tile cut between ranges is
// finished by whichever contributor arrives last.
//
// Static schedule: cluster c of P walks ids c, c + P, c + 2P, ... with
// sk_ranges = P, so that every cluster does the same number of k-blocks and
// takes its stream-K range FIRST: the fix-ups of split tiles then overlap the
// mainloops of the whole tiles instead of ending the kernel.  Dynamic
// schedule: one cluster is launched per id; a running cluster that finishes
// an id takes the id of a cluster that has not started yet (cluster launch
// control), so the same ids are spread over the clusters that are running.
struct WorkIter {
  int32_t sk_ranges, dp_tiles, k_blocks;
  int64_t sk_units;
  int64_t id, step, n_ids;  // current id; the static walk's stride; id count
  int64_t u, u_begin, u_end;
  int32_t dp_tile;  // whole tile still to hand out, or -1

  HG_HD WorkIter(int32_t sk_ranges_, int32_t dp_tiles_, int64_t sk_units_, int32_t k_blocks_)
      : sk_ranges(sk_units_ > 0 ? sk_ranges_ : 0), dp_tiles(dp_tiles_), k_blocks(k_blocks_), sk_units(sk_units_),
        id(-1), step(0), u(0), u_begin(0), u_end(0), dp_tile(-1) {
    n_ids = (int64_t)sk_ranges + dp_tiles;
  }

  // Make `id_` the current id (0 <= id_ < n_ids).
  HG_HD void start(int64_t id_) {
    id = id_;
    if (id_ < sk_ranges) {
      u_begin = splitk_begin(id_, sk_units, sk_ranges);
      u_end = splitk_begin(id_ + 1, sk_units, sk_ranges);
      u = u_begin;
      dp_tile = -1;
    } else {
      u = u_begin = u_end = 0;
      dp_tile = (int32_t)(id_ - sk_ranges);
    }
  }

  // The next item of the current id; false once the id is used up.
  HG_HD bool next_in_id(WorkItem& w) {
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
      w.owner = (int32_t)id;
      u += kb1 - kb0;
      return true;
    }
    if (dp_tile >= 0) {
      w.tile = dp_tile;
      w.kb0 = 0;
      w.kb1 = k_blocks;
      w.slot = -1;
      w.owner = -1;
      dp_tile = -1;
      return true;
    }
    return false;
  }

  // k-blocks of the current id after the item next_in_id returned last.
  HG_HD int64_t left_after_item() const { return u_end - u; }
  // k-blocks of the current id in all.
  HG_HD int64_t id_length() const { return id < sk_ranges ? u_end - u_begin : (int64_t)k_blocks; }

  // Static schedule of cluster `cluster` of `nclusters`.
  HG_HD void start_static(int32_t cluster, int32_t nclusters) {
    step = nclusters;
    if (cluster < n_ids) start(cluster);
  }

  HG_HD bool next_static(WorkItem& w) {
    if (id < 0) return false;
    for (;;) {
      if (next_in_id(w)) return true;
      if (id + step >= n_ids) return false;
      start(id + step);
    }
  }
};

// Contributors of stream-K tile `tile`: ranges [*first, *last], in K order.
HG_HD void sk_contributors(int32_t tile, int32_t dp_tiles, int64_t sk_units, int32_t k_blocks, int32_t sk_ranges,
                           int64_t* first, int64_t* last) {
  const int64_t u0 = (int64_t)(tile - dp_tiles) * k_blocks;
  *first = splitk_owner(u0, sk_units, sk_ranges);
  *last = splitk_owner(u0 + k_blocks - 1, sk_units, sk_ranges);
}

// Where range `c` keeps its partial of stream-K tile `tile`: slot 0 if the
// tile is the first of c's range, else slot 1 (it is then c's last).
HG_HD int32_t sk_slot_of(int64_t c, int32_t tile, int32_t dp_tiles, int64_t sk_units, int32_t k_blocks,
                         int32_t sk_ranges) {
  const int64_t first_tile = splitk_begin(c, sk_units, sk_ranges) / k_blocks;
  return (first_tile == (int64_t)(tile - dp_tiles)) ? 0 : 1;
}

}  // namespace hg
