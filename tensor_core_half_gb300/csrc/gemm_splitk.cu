// gemm_splitk.cu -- bandwidth-oriented split-K GEMM for skinny M (TN layout).
//
// With M <= 64 the product C[M,N] = A[M,K] . B[K,N] is bound by streaming B
// (N x K values) from HBM once.  The pages contain no skinny kernel; this one
// reuses the tcgen05 machinery of "tcgen05 for dummies: a B200 GEMM from
// scratch" (translated) -- TMA + mbarrier ring, warp specialisation, tensor-
// memory accumulators, persistent CTAs -- with these changes:
//   - swap A and B: the MMA computes C^T[N,M] = B[N,K] . A[M,K]^T, so that the
//     large N fills the MMA's 128 rows and M (padded to 16..64) is the MMA's N;
//   - the work is the tile-major list of (128-row N tile, 128-wide K block)
//     units, cut into contiguous chunks (splitk_shape): whole tiles per CTA
//     where that streams as fast, else one equal range per SM so that every
//     SM streams the same number of bytes of B;
//   - deterministic reduction of a tile whose K range is split: one fp32
//     partial per contributor in a workspace; the last contributor (an
//     atomic ticket, or all the others seen published while it computed)
//     adds the partials in K order and writes C.  No float atomics, so
//     repeated runs give identical bits.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "clc.cuh"
#include "desc.cuh"
#include "kernels.h"
#include "ptx.cuh"
#include "sched.cuh"

namespace hg {

namespace {
constexpr int kRowsPerTile = 128;  // N rows per tile = MMA M
// K per stage: two 64-wide boxes (the 128-byte swizzle's row) side by side.
// Measured on GB300 with this kernel's access pattern (each CTA a run of
// k-blocks of 128-row tiles): 128-wide stages stream 4-6 % faster from HBM
// than 64-wide ones with the same bytes in flight.
constexpr int kBoxK = 64;
constexpr int kBK = 2 * kBoxK;
constexpr int kWHalf = kRowsPerTile * kBoxK * 2;  // one box of B: 16 KiB
constexpr int kWBytes = kRowsPerTile * kBK * 2;   // B per stage: 32 KiB
constexpr int kThreads = 192;
constexpr int kClcSlots = 16;  // responses in flight: the epilogue may trail the producer by several chunks
constexpr int kMaxAcc = 8;  // tensor-memory accumulators (one per segment in flight)
}  // namespace

// Layout: ring (stages x stage_bytes, 1 KiB aligned) | barriers | misc (16 B) |
// cluster-launch-control responses (16 B each) | C staging ([mma_n][128]
// 16-bit) | prefetched partials (pf_slots x [128 rows][mma_n] fp32, in
// whatever shared memory the rest leaves over).
static_assert(kBK == kSplitKBlockK, "the planner's k-block is the kernel's stage depth in K");
__host__ __device__ __forceinline__ int sk_stage_bytes(int mma_n) { return kWBytes + mma_n * kBK * 2; }
__host__ __device__ __forceinline__ int sk_bar_off(int mma_n, int stages) { return stages * sk_stage_bytes(mma_n); }
// full[S], empty[S], tmem_full[A], tmem_empty[A], drain, clc_full[C], clc_empty[C]
__host__ __device__ __forceinline__ int sk_num_bars(int stages) { return 2 * stages + 2 * kMaxAcc + 1 + 2 * kClcSlots; }
__host__ __device__ __forceinline__ int sk_clc_off(int mma_n, int stages) {
  return (sk_bar_off(mma_n, stages) + sk_num_bars(stages) * 8 + 16 + 15) / 16 * 16;
}
// Accumulators: as many as fit in 256 columns, at most kMaxAcc.  The epilogue
// can then fall several segments behind (a fix-up that waits for other
// contributors) before the MMA issuer has to wait for a free accumulator.
__host__ __device__ __forceinline__ int sk_num_acc(int mma_n) {
  const int n = 256 / mma_n;
  return n < kMaxAcc ? n : kMaxAcc;
}
__host__ __device__ __forceinline__ int sk_tmem_cols(int mma_n) {
  int cols = 32;
  while (cols < sk_num_acc(mma_n) * mma_n) cols *= 2;
  return cols;
}

__host__ __device__ __forceinline__ int sk_cstage_off(int mma_n, int stages) {
  return sk_clc_off(mma_n, stages) + 16 * kClcSlots;
}
__host__ __device__ __forceinline__ int sk_pf_off(int mma_n, int stages) {
  return sk_cstage_off(mma_n, stages) + mma_n * kRowsPerTile * 2;
}
__host__ __device__ __forceinline__ int sk_partial_bytes(int mma_n) { return kRowsPerTile * mma_n * 4; }

int splitk_stage_bytes(int mma_n) { return sk_stage_bytes(mma_n); }
int splitk_pf_slots(int mma_n, int stages, int smem_optin) {
  const int left = smem_optin - (sk_pf_off(mma_n, stages) + 1024);
  const int slots = left > 0 ? left / sk_partial_bytes(mma_n) : 0;
  return slots < kSplitKMaxPrefetch ? slots : kSplitKMaxPrefetch;
}
int splitk_smem_bytes(int mma_n, int stages, int pf_slots) {
  return sk_pf_off(mma_n, stages) + pf_slots * sk_partial_bytes(mma_n) + 1024;
}

// The deepest ring up to `most` stages that fits.  With every SM streaming,
// 144-180 KB of B and A in flight per SM are several times what HBM latency
// needs (on GB300, 16 x 16384 x 8192 with 64-wide stages: 7-10 stages
// within 0.5 % of each other, 12 stages 3 % slower).  Fewer CTAs, each
// streaming faster, want more in flight: with 128 CTAs, 144 KB reach 6.0
// TB/s and 180-200 KB 6.2 TB/s.
int splitk_stages_for(int mma_n, int smem_optin, int most) {
  int s = most;
  while (s > 2 && splitk_smem_bytes(mma_n, s, 0) > smem_optin) --s;
  return s;
}

namespace {
// GB300 streaming rates behind the layout choice (a CTA streaming B tiles
// along K through an 11-stage ring, measured with 32-152 CTAs): one CTA
// reaches 62-68 GB/s, and the GPU as a whole about 6250 GB/s, which about 100
// CTAs already reach.  Whole tiles, their K walks started at eight offsets
// (SegmentOrder), keep all of that in the kernel (128 CTAs: 6.3-6.5 TB/s of
// streaming; 0.94 of it while every tile walked K from its start).  A split
// of some tile's K range between CTAs costs the fix-up at the end of the
// kernel: ~4 us at M <= 16 (16 x 16384 x 8192, the same launches with the
// fix-ups left out), growing with the fp32 partials, ~1.5 us per further 16
// columns of M.  Measured choices this reproduces (the faster layout, timed
// both ways on one box): whole tiles at 16 x 16384 x 8192, 16 x 12288 x 8192,
// 32 x 14336 x 4096, 64 x 16384 x 8192, 16 x 32768 x 4096, 4 x 32768 x 8192
// and {1, 8, 16} x 16384 x 16384; the split at 16 x 20480 x 8192,
// 16 x 8192 x 8192 and 1 x 8192 x 16384.
constexpr double kSplitKCtaGBs = 62.0;
constexpr double kSplitKGpuGBs = 6250.0;
constexpr double kSplitKWholeEff = 1.0;
constexpr double kSplitKFixupNs = 4000.0;
constexpr double kSplitKFixupPer16Ns = 1500.0;
constexpr int kSplitKSplitStages = 5;  // 180 KB in flight at M <= 16
constexpr int kSplitKWholeStages = 6;  // 216 KB: fewer CTAs, each streaming faster

double splitk_rate(int64_t ctas) {
  const double r = kSplitKCtaGBs * (double)ctas;
  return r < kSplitKGpuGBs ? r : kSplitKGpuGBs;
}
}  // namespace

// Whole tiles (each CTA the full K range of ceil(T / CTAs) or one fewer
// tiles, no partials, no fix-up) when that is estimated no slower than the
// balanced split over every CTA plus its fix-up; the split otherwise, and
// always under the dynamic schedule.  With 128 tiles on 152 SMs (16 x 16384 x
// 8192) the whole-tile layout leaves 24 SMs idle and loses nothing: 128 CTAs
// stream as fast as 152.
SplitKShape splitk_shape(int64_t tiles, int32_t k_blocks, int64_t K, int mma_n, int num_sms, int max_ctas,
                         int smem_optin, int split_k, bool dynamic) {
  int64_t sms = num_sms;
  if (max_ctas > 0 && max_ctas < sms) sms = max_ctas;
  if (sms < 1) sms = 1;
  const int64_t units = tiles * k_blocks;
  bool whole = false;
  if (!dynamic && split_k != 2) {
    if (split_k == 0) {
      whole = true;
    } else {
      const double tile_bytes = (double)kRowsPerTile * (double)K * 2.0;
      const int64_t per = (tiles + sms - 1) / sms;
      const int64_t p_whole = (tiles + per - 1) / per;
      const double t_whole = (double)per * tile_bytes / (kSplitKWholeEff * splitk_rate(p_whole) / (double)p_whole);
      const int64_t p_split = units < sms ? units : sms;
      const double fixup = kSplitKFixupNs + kSplitKFixupPer16Ns * (double)(mma_n / 16 - 1);
      const double t_split = (double)tiles * tile_bytes / splitk_rate(p_split) + fixup;
      whole = t_whole <= t_split;
    }
  }
  SplitKShape sh;
  if (whole) {
    const int64_t per = (tiles + sms - 1) / sms;
    sh.ctas = (int32_t)((tiles + per - 1) / per);
    sh.chunks = splitk_whole_tiles(tiles, k_blocks, sh.ctas);
    sh.stages = splitk_stages_for(mma_n, smem_optin, kSplitKWholeStages);
    sh.pf_slots = 0;
  } else {
    sh.ctas = (int32_t)(units < sms ? units : sms);
    sh.chunks = splitk_chunks(units, sh.ctas, dynamic);
    sh.stages = splitk_stages_for(mma_n, smem_optin, kSplitKSplitStages);
    sh.pf_slots = splitk_pf_slots(mma_n, sh.stages, smem_optin);
  }
  sh.smem_bytes = splitk_smem_bytes(mma_n, sh.stages, sh.pf_slots);
  return sh;
}

int splitk_tmem_cols(int mma_n) { return sk_tmem_cols(mma_n); }

size_t splitk_workspace_bytes(int64_t chunks, int mma_n, int n_tiles) {
  size_t partial = (size_t)chunks * 2 * kRowsPerTile * (size_t)mma_n * sizeof(float);
  partial = (partial + 255) & ~(size_t)255;
  return partial + (size_t)n_tiles * kSplitKTicketStride * sizeof(int32_t);  // one arrival counter per tile
}

__device__ __forceinline__ void sk_report(int32_t* status, int32_t role, volatile uint32_t* abort_flag) {
  *abort_flag = 1u;
  atomicCAS(status, 0, kStatusTimeout | (role << 8) | ((int32_t)(blockIdx.x & 0xFFFF) << 16));
}

// One segment: the k-blocks [kb0, kb1) of N tile `tile`, part of chunk `chunk`
// (ChunkSegments gives the order).
struct Segment {
  int32_t tile, kb0, kb1;
  bool first;     // it starts at its chunk's first unit (it is first in K, not necessarily in time)
  int64_t chunk;
};

// The order in which a segment's k-blocks are loaded and multiplied.  A
// segment that covers its tile's whole K range (whole-tile layout) starts at
// ((tile mod 8) / 8) of the range and wraps around; any other segment walks
// K in order.  With every CTA streaming its own rows of B at the same K
// offset, the concurrent reads share their low address bits; spreading the
// tiles over eight starting offsets measured 0-12 % faster on GB300 over
// eight skinny shapes (16 x 16384 x 8192: 0.8 %, 64 x 16384 x 8192: 2.6 %,
// 16 x 16384 x 16384: 12 %), where 4 or 16 offsets each lost up to 9 % on
// some shape.  Only the fp32 summation order of such a tile changes, the
// same on every run.
constexpr int kKPhases = 8;
struct SegmentOrder {
  int32_t kb0, len, rot;
  __device__ SegmentOrder(const Segment& sg, int32_t k_blocks)
      : kb0(sg.kb0), len(sg.kb1 - sg.kb0),
        rot((sg.kb0 == 0 && sg.kb1 == k_blocks) ? (int32_t)(((int64_t)(sg.tile % kKPhases) * len) / kKPhases) : 0) {}
  // The k-block the segment's j-th step handles (0 <= j < len).
  __device__ int32_t kb(int32_t j) const { return kb0 + (j + rot < len ? j + rot : j + rot - len); }
};

// The segments one role walks through: its CTA's own chunk, then (dynamic
// schedule) the chunks it takes over from CTAs that have not started.
struct ChunkFeed {
  ClcIds<1, kClcSlots> clc;
  SplitChunks ch;
  int32_t k_blocks;
  bool dynamic;
  bool checks;
  int32_t* status;
  bool started = false, finished = false;
  bool want = false;  // issuer: the current chunk's request is still to be made
  int64_t chunk = -1;
  ChunkSegments segs;
  int32_t pos = 0;    // segments of the current chunk handed out
  int64_t rest = 0;   // units of the current chunk not handed out yet

  __device__ ChunkFeed(const SplitKArgs& a, uint32_t resp0, uint32_t full0, uint32_t empty0, bool issuer,
                       bool warp_wide, bool arrive)
      : clc(resp0, full0, empty0, issuer, warp_wide, arrive),
        k_blocks(a.k_blocks),
        dynamic(a.dynamic != 0),
        checks(a.checks != 0),
        status(a.status) {
    ch.units = a.units;
    ch.head = a.head;
    ch.big = a.big;
    ch.n_small = a.n_small;
    ch.align = a.align;
  }

  __device__ void set(int64_t g) {
    chunk = g;
    segs.init(ch.begin(g), ch.begin(g + 1), k_blocks);
    pos = 0;
    rest = segs.end - segs.begin;
  }

  // 1: a segment in sg; 0: no work left; -1: a wait gave up.
  __device__ int next(Segment& sg, const WaitCtl& ctl) {
    for (;;) {
      if (!started) {
        if (finished) return 0;
        started = true;
        set(blockIdx.x);
        want = dynamic && clc.issuer;
      }
      if (pos < segs.count) {
        const int32_t idx = segs.at(pos++);
        segs.get(idx, &sg.tile, &sg.kb0, &sg.kb1);
        sg.first = (idx == 0);
        sg.chunk = chunk;
        rest -= sg.kb1 - sg.kb0;
        return 1;
      }
      if (!dynamic) {
        finished = true;
        return 0;
      }
      if (want) {  // a chunk shorter than the lead: ask now
        want = false;
        if (!clc.request(ctl)) return -1;
      }
      int64_t g = 0;
      const int got = clc.fetch(&g, ctl);
      if (got < 0) return -1;
      if (got > 0 && checks && (g < 0 || g >= ch.count())) {
        report_check(status, kCheckWorkId, nullptr);
        return -1;
      }
      if (got == 0) {
        finished = true;
        return 0;
      }
      set(g);
      want = clc.issuer;
    }
  }

  // Issuer, after loading a k-block: `left` k-blocks of the current segment
  // remain; ask for the next chunk when clc_time_to_ask says so.
  __device__ bool poll(int64_t left, const WaitCtl& ctl) {
    if (!want || !clc_time_to_ask(left + rest, segs.end - segs.begin)) return true;
    want = false;
    return clc.request(ctl);
  }
};

// The fix-up sum of a split tile: s = the contributors' partials in
// contributor (= K) order, the caller's own values (chunk `own`) taken from
// its registers and the others read from the workspace.  Columns go in slabs
// of 16 (four float4 per row); within a slab the partials of three
// contributors are loaded before any is added, so a tile with many
// contributors costs a third as many dependent L2 round trips.  p0: this
// thread's row of chunk 0, slot 0; a partial is [128 rows][mma_n] fp32.
__device__ __forceinline__ const float4* partial_row(const float4* p0, int64_t c, int64_t c_first, int slot_first,
                                                     int mma_n) {
  const int64_t per_slot = (int64_t)kRowsPerTile * mma_n / 4;  // float4s in one partial
  return p0 + (c * 2 + ((c == c_first) ? slot_first : 0)) * per_slot;
}

__device__ __forceinline__ void sum_contributors(float (&s)[kSplitKMaxM], const float (&v)[kSplitKMaxM],
                                                 const float4* p0, int64_t c_first, int64_t c_last, int64_t own,
                                                 int slot_first, int mma_n) {
  constexpr int B = 3;
#pragma unroll
  for (int j0 = 0; j0 < kSplitKMaxM / 4; j0 += 4) {
    if (4 * j0 >= mma_n) break;  // mma_n is a multiple of 16: whole slabs
    for (int64_t c0 = c_first; c0 <= c_last; c0 += B) {
      float4 g[B][4];
#pragma unroll
      for (int b = 0; b < B; ++b) {
        const int64_t cc = c0 + b;
        if (cc <= c_last && cc != own) {
          const float4* src = partial_row(p0, cc, c_first, slot_first, mma_n) + j0;
#pragma unroll
          for (int j = 0; j < 4; ++j) g[b][j] = __ldcg(src + j);
        }
      }
#pragma unroll
      for (int b = 0; b < B; ++b) {
        const int64_t cc = c0 + b;
        if (cc > c_last) break;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int k = 4 * (j0 + j);
          if (cc == own) {
            s[k] += v[k];
            s[k + 1] += v[k + 1];
            s[k + 2] += v[k + 2];
            s[k + 3] += v[k + 3];
          } else {
            s[k] += g[b][j].x;
            s[k + 1] += g[b][j].y;
            s[k + 2] += g[b][j].z;
            s[k + 3] += g[b][j].w;
          }
        }
      }
    }
  }
}

// The same sum when the other contributors' rows were copied to shared memory
// beforehand (pf: this thread's row of the first copied partial; the copies
// follow in contributor order, `own` skipped, each [128 rows][mma_n] fp32).
__device__ __forceinline__ void sum_prefetched(float (&s)[kSplitKMaxM], const float (&v)[kSplitKMaxM],
                                               const float4* pf, int64_t c_first, int64_t c_last, int64_t own,
                                               int mma_n) {
  const int per_slot = kRowsPerTile * mma_n / 4;
  int k = 0;
  for (int64_t cc = c_first; cc <= c_last; ++cc) {
    const float4* src = pf + (int64_t)k * per_slot;
#pragma unroll
    for (int j = 0; j < kSplitKMaxM / 4; ++j) {
      if (4 * j >= mma_n) break;
      const float4 g = (cc == own) ? make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]) : src[j];
      s[4 * j] += g.x;
      s[4 * j + 1] += g.y;
      s[4 * j + 2] += g.z;
      s[4 * j + 3] += g.w;
    }
    if (cc != own) ++k;
  }
}

// Watches a split tile's arrival counter while this CTA's accumulator for the
// tile is still being computed (one thread).  1: every other contributor has
// already published (acquired: their partials may be read), so this CTA is
// the tile's last contributor; 0: the accumulator became ready first; -1: a
// time limit or the CTA's abort flag; -2: a count past the contributors
// (checked mode).  The counter is polled with relaxed loads, each overlapped
// with a wait of up to 1 us on the accumulator's barrier, and upgraded with a
// fence once it shows every other contributor.
__device__ __noinline__ int watch_arrivals(const int32_t* arrivals, int32_t others, uint32_t tfull, uint32_t parity,
                                           WaitCtl ctl, bool checks) {
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    const int32_t seen = ld_relaxed_gpu(arrivals);
    const bool ready = mbar_try_wait_hint(tfull, parity, 1000u);
    if (seen == others) {
      fence_acq_rel_gpu();
      return 1;
    }
    if (checks && (seen < 0 || seen > others)) return -2;
    if (ready) return 0;
    if ((i & 15u) == 0) {
      if (ctl.abort_flag != nullptr && *ctl.abort_flag != 0u) return -1;
      if (globaltimer_ns() - t0 > ctl.timeout_ns) return -1;
    }
  }
}

// Writes one tile's slice of C, [M rows][128 columns of N] of 16-bit values
// (all 128 epilogue threads; x: this thread's column).  Each thread rounds
// its column into the staging area, then the threads copy the slice out in
// 16-byte pieces along N: at M = 16, two stores per thread instead of
// sixteen 2-byte ones, which is what the kernel's last segment waits on.
// N % 8 == 0 and C is 16-byte aligned, so a piece is wholly inside or
// outside C.
__device__ __forceinline__ void store_tile(uint8_t* cstage, const float (&x)[kSplitKMaxM], int row, int M, int N,
                                           int32_t tile, void* C, bool out_bf16) {
  uint16_t* const st = reinterpret_cast<uint16_t*>(cstage);
#pragma unroll
  for (int m = 0; m < kSplitKMaxM; ++m) {
    if (m < M) {
      const float f = x[m];
      st[m * kRowsPerTile + row] = out_bf16 ? __bfloat16_as_ushort(__float2bfloat16_rn(f))
                                            : __half_as_ushort(__float2half_rn(f));
    }
  }
  named_bar_sync(3, 128);
  const int64_t n0 = (int64_t)tile * kRowsPerTile;
  for (int c = row; c < M * (kRowsPerTile / 8); c += 128) {
    const int m = c / (kRowsPerTile / 8);
    const int col = (c % (kRowsPerTile / 8)) * 8;
    if (n0 + col < N)
      *reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(C) + (int64_t)m * N + n0 + col) =
          *reinterpret_cast<const uint4*>(st + m * kRowsPerTile + col);
  }
  named_bar_sync(3, 128);  // the staging area is free for the next tile
}

__global__ void __launch_bounds__(192, 1)
    splitk_gemm_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                       const SplitKArgs args) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const int stages = args.stages;
  const int mma_n = args.mma_n;
  const uint32_t stage_bytes = (uint32_t)sk_stage_bytes(mma_n);
  const uint32_t bars = base + (uint32_t)sk_bar_off(mma_n, stages);
  const uint32_t misc_off = (uint32_t)(sk_bar_off(mma_n, stages) + sk_num_bars(stages) * 8);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + misc_off);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(gbase + misc_off + 4);
  volatile int32_t* ticket_slot = reinterpret_cast<volatile int32_t*>(gbase + misc_off + 8);
  volatile int32_t* watch_slot = reinterpret_cast<volatile int32_t*>(gbase + misc_off + 12);

  auto full_bar = [&](int s) -> uint32_t { return bars + 8u * s; };
  auto empty_bar = [&](int s) -> uint32_t { return bars + 8u * (stages + s); };
  auto tfull_bar = [&](int b) -> uint32_t { return bars + 8u * (2 * stages + b); };
  auto tempty_bar = [&](int b) -> uint32_t { return bars + 8u * (2 * stages + kMaxAcc + b); };
  const uint32_t drain_bar = bars + 8u * (2 * stages + 2 * kMaxAcc);
  const uint32_t clc_full0 = drain_bar + 8u;
  const uint32_t clc_empty0 = clc_full0 + 8u * kClcSlots;
  const uint32_t clc_resp0 = base + (uint32_t)sk_clc_off(mma_n, stages);

  const int warp = threadIdx.x / 32;
  const uint32_t lane = threadIdx.x % 32;
  SplitChunks chunks;
  chunks.units = args.units;
  chunks.head = args.head;
  chunks.big = args.big;
  chunks.n_small = args.n_small;
  chunks.align = args.align;
  const int tmem_cols = sk_tmem_cols(mma_n);
  const int nacc = sk_num_acc(mma_n);
  const WaitCtl ctl{args.timeout_ns, abort_flag};
  const WaitCtl drain_ctl{kDrainTimeoutNs, nullptr};

  if (warp == 0) {
    if (lane == 0) {
      for (int s = 0; s < stages; ++s) {
        mbar_init(full_bar(s), 1);
        mbar_init(empty_bar(s), 1);
      }
      for (int b = 0; b < nacc; ++b) {
        mbar_init(tfull_bar(b), 1);
        mbar_init(tempty_bar(b), 4);
      }
      mbar_init(drain_bar, 1);
      ClcIds<1, kClcSlots>::init(clc_full0, clc_empty0, 6);  // producer, MMA issuer, 4 epilogue warps
      *abort_flag = 0u;
      fence_mbar_init();
      prefetch_tmap(&tmW);
      prefetch_tmap(&tmX);
    }
    __syncwarp();
  } else if (warp == 1) {
    tmem_alloc<1>(smem_addr(tmem_slot), (uint32_t)tmem_cols);
    tmem_relinquish<1>();
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(tmem_slot);
  // The prologue above touched no global memory; from here on the previous
  // kernel in the stream (launched with programmatic serialisation) must be done.
  pdl_launch_dependents();
  pdl_wait_prior_grid();
  TraceBuf* const tb = args.trace;
  TraceBuf* const tbi = args.trace_items ? tb : nullptr;  // work-item events (else only begin/end)
  // This CTA's kernel begin and end records (with the SM cycle counter): both
  // slots are reserved here by an epilogue thread, idle until the first
  // accumulator is ready, so that neither the producer's first copy nor the
  // CTA's exit waits for the trace's atomic.
  unsigned long long stamp_slot = 0;
  if (tb != nullptr && threadIdx.x == kStampThread) {
    const uint64_t t = globaltimer_ns();
    const int32_t clk = (int32_t)(clock64() & 0x7fffffff);
    stamp_slot = trace_reserve(tb, 2ull);
    trace_put(tb, stamp_slot, t, 0, kTraceKernelBegin, -1, clk);
  }

  if (warp == 0) {
    // ---------------------------------------------------- TMA producer ----
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int64_t issued = 0;
      bool ok = true;
      ChunkFeed feed(args, clc_resp0, clc_full0, clc_empty0, true, false, true);
      Segment sg;
      while (ok) {
        const int more = feed.next(sg, ctl);
        if (more < 0) ok = false;
        if (more <= 0) break;
        trace_event(tbi, kRoleProducer, kTraceItemBegin, sg.tile, sg.kb0);
        if (args.checks && (sg.tile < 0 || sg.tile >= args.n_tiles || sg.kb0 < 0 || sg.kb0 >= sg.kb1 ||
                            sg.kb1 > args.k_blocks || sg.chunk < 0 || sg.chunk >= chunks.count())) {
          report_check(args.status, kCheckItem, abort_flag);
          ok = false;
          break;
        }
        const SegmentOrder order(sg, args.k_blocks);
        for (int j = 0; j < order.len; ++j) {
          const int kb = order.kb(j);
          if (!mbar_wait(empty_bar(stage), phase ^ 1u, ctl)) {
            ok = false;
            break;
          }
          const bool drop = (args.inject == 1) && (blockIdx.x == 0) && (issued == 0);
          if (!drop) {
            const uint32_t w_dst = base + (uint32_t)stage * stage_bytes;
            const uint32_t x_dst = w_dst + kWBytes;
            const uint32_t x_half = (uint32_t)(mma_n * kBoxK * 2);
            const uint32_t fb = full_bar(stage);
            mbar_arrive_expect_tx(fb, stage_bytes);
            // A box that starts at or past K is zero-filled (and counted in full).
#pragma unroll
            for (int h = 0; h < kBK / kBoxK; ++h) {
              tma_load_2d(w_dst + (uint32_t)(h * kWHalf), &tmW, fb, kb * kBK + h * kBoxK, sg.tile * kRowsPerTile);
              tma_load_2d(x_dst + (uint32_t)h * x_half, &tmX, fb, kb * kBK + h * kBoxK, 0);
            }
          }
          ++issued;
          if (++stage == stages) {
            stage = 0;
            phase ^= 1u;
          }
          if (!feed.poll(order.len - j - 1, ctl)) {
            ok = false;
            break;
          }
        }
      }
      trace_event(tbi, kRoleProducer, kTraceItemEnd, -1, (int32_t)issued);
      if (!ok) sk_report(args.status, kRoleProducer, abort_flag);
      if (!feed.clc.drain(drain_ctl)) sk_report(args.status, kRoleTeardown, abort_flag);
      for (int s = 0; s < stages; ++s) {
        if (issued <= s) break;
        const int64_t last = s + (int64_t)stages * ((issued - 1 - s) / stages);
        if ((args.inject == 1) && (blockIdx.x == 0) && (last == 0)) continue;
        if (!mbar_wait(full_bar(s), (uint32_t)((last / stages) & 1), drain_ctl))
          sk_report(args.status, kRoleTeardown, abort_flag);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------ MMA issuer ----
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      ChunkFeed feed(args, clc_resp0, clc_full0, clc_empty0, false, false, true);
      Segment sg;
      while (ok) {
        const int more = feed.next(sg, ctl);
        if (more < 0) ok = false;
        if (more <= 0) break;
        if (!mbar_wait(tempty_bar(acc), acc_phase ^ 1u, ctl)) {
          ok = false;
          break;
        }
        tc_fence_after();
        trace_event(tbi, kRoleMma, kTraceItemBegin, sg.tile, sg.kb0);
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * mma_n);
        const int32_t steps = sg.kb1 - sg.kb0;  // in SegmentOrder's order; the first step starts the sum
        for (int j = 0; j < steps; ++j) {
          if (!mbar_wait(full_bar(stage), phase, ctl)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t w_addr = base + (uint32_t)stage * stage_bytes;
          const uint32_t x_addr = w_addr + kWBytes;
#pragma unroll
          for (int h = 0; h < kBK / kBoxK; ++h) {  // the two 64-wide halves of the stage
            const uint64_t w_desc = make_smem_desc(w_addr + (uint32_t)(h * kWHalf), 16u, kKMajorSBO, kSwizzle128B);
            const uint64_t x_desc =
                make_smem_desc(x_addr + (uint32_t)(h * mma_n * kBoxK * 2), 16u, kKMajorSBO, kSwizzle128B);
#pragma unroll
            for (int kk = 0; kk < kBoxK / 16; ++kk) {
              const uint64_t step = (uint64_t)(kk * (kKMajorStepBytes >> 4));
              mma_f16<1>(d_tmem, w_desc + step, x_desc + step, args.idesc,
                         (uint32_t)((j != 0) || (h != 0) || (kk != 0)));
            }
          }
          tc_commit(empty_bar(stage));
          if (++stage == stages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(tfull_bar(acc));
        trace_event(tbi, kRoleMma, kTraceItemEnd, sg.tile, sg.kb1);
        if (++acc == nacc) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      if (!ok) sk_report(args.status, kRoleMma, abort_flag);
      tc_commit(drain_bar);
      if (!mbar_wait(drain_bar, 0u, WaitCtl{args.timeout_ns, nullptr})) sk_report(args.status, kRoleTeardown, abort_flag);
    }
    __syncwarp();
  } else {
    // -------------------------------------------------------- epilogue ----
    const int q = warp & 3;
    const int row = q * 32 + (int)lane;  // N row within the tile = TMEM lane
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    const bool out_bf16 = args.out_bf16 != 0;
    float* partials = args.partials;
    ChunkFeed feed(args, clc_resp0, clc_full0, clc_empty0, false, true, lane == 0);
    const float4* const row_partials = reinterpret_cast<const float4*>(partials + (int64_t)row * mma_n);
    uint8_t* const cstage = gbase + sk_cstage_off(mma_n, stages);
    const uint32_t pf_base = base + (uint32_t)sk_pf_off(mma_n, stages);
    const float4* const pf_rows = reinterpret_cast<const float4*>(gbase + sk_pf_off(mma_n, stages)) + row * mma_n / 4;
    Segment sg;
    for (;;) {
      const int more = feed.next(sg, ctl);
      // The four epilogue warps read the same chunks; they stop together.
      if (named_bar_or(2, 128, more < 0)) {
        ok = false;
        break;
      }
      if (more == 0) break;
      const bool whole = (sg.kb0 == 0 && sg.kb1 == args.k_blocks);
      const int64_t u_first = (int64_t)sg.tile * args.k_blocks;
      const int64_t c_first = whole ? sg.chunk : chunks.owner(u_first);
      const int64_t c_last = whole ? sg.chunk : chunks.owner(u_first + args.k_blocks - 1);
      const int32_t others = (int32_t)(c_last - c_first);
      int32_t* const arrivals = args.tickets + (int64_t)sg.tile * args.ticket_stride;
      // Contributors after the first start inside this tile, so their
      // partial of it is their first (slot 0); the first contributor's range
      // may start in an earlier tile (slot 1).
      const int slot_first = (chunks.begin(c_first) >= u_first) ? 0 : 1;
      // A split tile: while the MMA still works on this segment, watch the
      // tile's counter.  When the other contributors have all published
      // before this one is done (the usual case for a CTA's last segment,
      // whose tile the next CTA began with), this CTA completes the tile
      // without publishing its partial or drawing a ticket.
      int early = 0;
      bool prefetched = false;
      if (!whole) {
        if (threadIdx.x == 64) {
          const int w = watch_arrivals(arrivals, others, tfull_bar(acc), acc_phase, ctl, args.checks);
          // The check's status goes in before any warp leaves and reports a stop.
          if (w == -2) report_check(args.status, kCheckTicket, abort_flag);
          *watch_slot = w;
        }
        named_bar_sync(1, 128);
        early = *watch_slot;
        if (early < 0) {
          ok = false;
          break;
        }
        if (early == 1 && others <= args.pf_slots) {
          // The others' partials are acquired: copy this thread's rows of
          // them into shared memory while the MMA finishes, so that the sum
          // after it waits on no global load (the C stores that follow it
          // have to reach memory before the kernel can end).
          int k = 0;
          for (int64_t cc = c_first; cc <= c_last; ++cc) {
            if (cc == sg.chunk) continue;
            const float4* src = partial_row(row_partials, cc, c_first, slot_first, mma_n);
            const uint32_t dst = pf_base + (uint32_t)((k * kRowsPerTile + row) * mma_n * 4);
            for (int j = 0; j < mma_n / 4; ++j) cp_async_16(dst + 16u * (uint32_t)j, src + j);
            ++k;
          }
          cp_async_commit();
          prefetched = true;
        }
      }
      const bool got = mbar_wait(tfull_bar(acc), acc_phase, ctl);
      // The four epilogue warps meet at named barriers below, so they give up together.
      if (named_bar_or(2, 128, !got)) {
        ok = false;
        break;
      }
      tc_fence_after();
      if (threadIdx.x == 64) trace_event(tbi, kRoleEpilogue, kTraceItemBegin, sg.tile, sg.kb0);
      float v[kSplitKMaxM];
      const uint32_t t_row = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * mma_n);
#pragma unroll
      for (int j = 0; j < kSplitKMaxM / 16; ++j) {
        if (j * 16 < mma_n) {
          uint32_t r[16];
          tmem_ld_x16(t_row + (uint32_t)(j * 16), r);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) v[j * 16 + i] = __uint_as_float(r[i]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty_bar(acc));
      if (++acc == nacc) {
        acc = 0;
        acc_phase ^= 1u;
      }

      if (args.checks && threadIdx.x == 64 && !whole) {
        if (sg.chunk < c_first || sg.chunk > c_last) report_check(args.status, kCheckContributor, abort_flag);
        if (c_first < 0 || c_last >= chunks.count()) report_check(args.status, kCheckPartial, abort_flag);
      }
      if (whole) {
        // The whole K range of this tile is ours: write C directly.
        store_tile(cstage, v, row, args.M, args.N, sg.tile, args.C, out_bf16);
      } else {
        // Publish, then count: a contributor stores its fp32 partial and,
        // once all rows are written, one thread takes a ticket with an
        // acquire-release add; the contributor that draws the last ticket has
        // thereby acquired every other contributor's partial.  A contributor
        // that saw all the others published while it computed (early == 1)
        // is the last one already: it neither publishes nor draws a ticket.
        // The last contributor sums the partials, its own from registers, in
        // contributor (= K) order and writes C, so the result does not depend
        // on who finishes last.
        bool last = (early == 1);
        if (!last) {
          const int slot = sg.first ? 0 : 1;
          float* mine = partials + ((sg.chunk * 2 + slot) * kRowsPerTile + row) * mma_n;
#pragma unroll
          for (int j = 0; j < kSplitKMaxM / 4; ++j)
            if (j * 4 < mma_n)
              reinterpret_cast<float4*>(mine)[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
          named_bar_sync(1, 128);  // every row of the partial is written ...
          if (threadIdx.x == 64) *ticket_slot = atom_add_acq_rel_gpu(arrivals, 1);  // ... before the ticket
          named_bar_sync(1, 128);  // ... and the acquire orders the partial reads below
          const int32_t ticket = *ticket_slot;
          if (threadIdx.x == 64) trace_event(tbi, kRoleEpilogue, kTracePartialStored, sg.tile, ticket);
          if (args.checks && threadIdx.x == 64 && (ticket < 0 || ticket > others))
            report_check(args.status, kCheckTicket, abort_flag);
          last = (ticket == others);
        }
        if (last) {
          float s[kSplitKMaxM];
#pragma unroll
          for (int m = 0; m < kSplitKMaxM; ++m) s[m] = 0.0f;
          if (prefetched) {
            cp_async_wait_all();  // this thread's own copies: no barrier needed
            sum_prefetched(s, v, pf_rows, c_first, c_last, sg.chunk, mma_n);
          } else {
            sum_contributors(s, v, row_partials, c_first, c_last, sg.chunk, slot_first, mma_n);
          }
          store_tile(cstage, s, row, args.M, args.N, sg.tile, args.C, out_bf16);
          if (threadIdx.x == 64) {
            *arrivals = 0;  // ready for the next launch
            trace_event(tbi, kRoleEpilogue, kTraceReduced, sg.tile, others + 1);
          }
        }
        named_bar_sync(1, 128);  // ticket_slot and watch_slot are reused by the next segment
      }
      if (threadIdx.x == 64) trace_event(tbi, kRoleEpilogue, kTraceItemEnd, sg.tile, sg.kb1);
    }
    cp_async_wait_all();  // copies a segment that gave up had in flight
    if (!ok && lane == 0) sk_report(args.status, kRoleEpilogue, abort_flag);
  }

  __syncthreads();
  // every role of the CTA is done: the end of the CTA's work
  if (tb != nullptr && threadIdx.x == kStampThread)
    trace_put(tb, stamp_slot + 1, globaltimer_ns(), 0, kTraceKernelEnd, -1, (int32_t)(clock64() & 0x7fffffff));
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc<1>(tmem_base, (uint32_t)tmem_cols);
  }
}

cudaError_t splitk_prepare(int smem_bytes) {
  return cudaFuncSetAttribute(reinterpret_cast<const void*>(&splitk_gemm_kernel),
                              cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
}

cudaError_t splitk_launch(const CUtensorMap& tmW, const CUtensorMap& tmX, const SplitKArgs& args, int grid,
                          int smem_bytes, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3((unsigned)grid, 1, 1);
  cfg.blockDim = dim3((unsigned)kThreads, 1, 1);
  cfg.dynamicSmemBytes = (size_t)smem_bytes;
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // overlap launch with the previous kernel
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, splitk_gemm_kernel, tmW, tmX, args);
}

// ------------------------------------------------------------ zero fill ----
// K == 0: C is the empty sum, +0 everywhere.  16-byte stores, grid-stride.
__global__ void fill_zero_kernel(uint4* p, size_t n16) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n16; i += (size_t)gridDim.x * blockDim.x)
    p[i] = make_uint4(0u, 0u, 0u, 0u);
}

cudaError_t fill_zero_launch(void* p, size_t bytes, cudaStream_t stream) {
  const size_t n16 = bytes / 16;
  if (n16 == 0) return cudaSuccess;
  size_t blocks = (n16 + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  fill_zero_kernel<<<(unsigned)blocks, 256, 0, stream>>>(reinterpret_cast<uint4*>(p), n16);
  return cudaGetLastError();
}

}  // namespace hg
