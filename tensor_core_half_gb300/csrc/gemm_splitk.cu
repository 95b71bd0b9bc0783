// gemm_splitk.cu -- bandwidth-oriented split-K GEMM for skinny M (TN layout).
//
// With M <= 64 the product C[M,N] = A[M,K] . B[K,N] is bound by streaming B
// (N x K values) from HBM once.  The pages contain no skinny kernel; this one
// reuses the tcgen05 machinery of "tcgen05 for dummies: a B200 GEMM from
// scratch" (translated) -- TMA + mbarrier ring, warp specialisation, tensor-
// memory accumulators, persistent CTAs -- with three changes:
//   - swap A and B: the MMA computes C^T[N,M] = B[N,K] . A[M,K]^T, so that the
//     large N fills the MMA's 128 rows and M (padded to 16..64) is the MMA's N;
//   - balanced split-K: the tile-major list of (128-row N tile, 64-wide K
//     block) units is cut into one contiguous range per CTA, so every SM
//     streams the same number of bytes of B;
//   - deterministic reduction: a tile covered by several CTAs gets one fp32
//     partial per CTA in a workspace; the last CTA to finish the tile (an
//     atomic ticket) adds the partials in K order and writes C.  No float
//     atomics, so repeated runs give identical bits.
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
constexpr int kBK = 64;            // K per stage
constexpr int kWBytes = kRowsPerTile * kBK * 2;  // B tile per stage: 16 KiB
constexpr int kThreads = 192;
constexpr int kClcSlots = 16;  // responses in flight: the epilogue may trail the producer by several chunks
constexpr int kMaxAcc = 8;  // tensor-memory accumulators (one per segment in flight)
}  // namespace

// Layout: ring (stages x stage_bytes, 1 KiB aligned) | barriers | misc (16 B) |
// cluster-launch-control responses (16 B each).
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

int splitk_stage_bytes(int mma_n) { return sk_stage_bytes(mma_n); }
int splitk_smem_bytes(int mma_n, int stages) { return sk_clc_off(mma_n, stages) + 16 * kClcSlots + 1024; }

// 8 stages: 144 KB of B and A in flight per SM at M <= 16, several times what
// HBM latency needs.  Measured on GB300 (16 x 16384 x 8192): 7-10 stages
// within 0.5 % of each other, 12 stages 3 % slower (more requests queued
// than the memory system serves well).
int splitk_stages_for(int mma_n, int smem_optin) {
  int s = 8;
  while (s > 2 && splitk_smem_bytes(mma_n, s) > smem_optin) --s;
  return s;
}

int splitk_tmem_cols(int mma_n) { return sk_tmem_cols(mma_n); }

size_t splitk_workspace_bytes(int64_t chunks, int mma_n, int n_tiles) {
  size_t partial = (size_t)chunks * 2 * kRowsPerTile * (size_t)mma_n * sizeof(float);
  partial = (partial + 255) & ~(size_t)255;
  return partial + (size_t)n_tiles * 2 * sizeof(int32_t);  // arrival counters (one per tile used)
}

__device__ __forceinline__ void sk_report(int32_t* status, int32_t role, volatile uint32_t* abort_flag) {
  *abort_flag = 1u;
  atomicCAS(status, 0, kStatusTimeout | (role << 8) | ((int32_t)(blockIdx.x & 0xFFFF) << 16));
}

// One segment: the k-blocks [kb0, kb1) of N tile `tile`, part of chunk `chunk`.
struct Segment {
  int32_t tile, kb0, kb1;
  bool first;     // the first segment of its chunk
  int64_t chunk;
};

__device__ __forceinline__ Segment segment_at(int64_t u, int64_t end, int32_t k_blocks, int64_t begin) {
  Segment s;
  s.tile = (int32_t)(u / k_blocks);
  s.kb0 = (int32_t)(u - (int64_t)s.tile * k_blocks);
  const int64_t left = end - u;
  const int64_t room = k_blocks - s.kb0;
  s.kb1 = s.kb0 + (int32_t)(left < room ? left : room);
  s.first = (u == begin);
  s.chunk = -1;
  return s;
}

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
  int64_t chunk = -1, begin = 0, u = 0, end = 0;

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
  }

  __device__ void set(int64_t g) {
    chunk = g;
    begin = ch.begin(g);
    end = ch.begin(g + 1);
    u = begin;
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
      if (u < end) {
        sg = segment_at(u, end, k_blocks, begin);
        sg.chunk = chunk;
        u += sg.kb1 - sg.kb0;
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
    if (!want || !clc_time_to_ask(left + (end - u), end - begin)) return true;
    want = false;
    return clc.request(ctl);
  }
};

// The fix-up sum of a split tile: s = the contributors' partials in
// contributor (= K) order, read from the workspace (the caller has stored its
// own values there too).  Columns go in slabs of 16 (four float4 per row);
// within a slab the partials of four contributors are loaded before any is
// added, so a tile with many contributors costs a quarter as many dependent
// L2 round trips.  p0: this thread's row of chunk 0, slot 0; a partial is
// [128 rows][mma_n] fp32.
__device__ __forceinline__ void sum_contributors(float (&s)[kSplitKMaxM], const float4* p0, int64_t c_first,
                                                 int64_t c_last, int slot_first, int mma_n) {
  constexpr int B = 4;
  const int64_t per_slot = (int64_t)kRowsPerTile * mma_n / 4;  // float4s in one partial
#pragma unroll
  for (int j0 = 0; j0 < kSplitKMaxM / 4; j0 += 4) {
    if (4 * j0 >= mma_n) break;  // mma_n is a multiple of 16: whole slabs
    for (int64_t c0 = c_first; c0 <= c_last; c0 += B) {
      float4 g[B][4];
#pragma unroll
      for (int b = 0; b < B; ++b) {
        const int64_t cc = c0 + b;
        if (cc <= c_last) {
          const int slot = (cc == c_first) ? slot_first : 0;
          const float4* src = p0 + (cc * 2 + slot) * per_slot + j0;
#pragma unroll
          for (int j = 0; j < 4; ++j) g[b][j] = __ldcg(src + j);
        }
      }
#pragma unroll
      for (int b = 0; b < B; ++b) {
        if (c0 + b > c_last) break;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          s[4 * (j0 + j)] += g[b][j].x;
          s[4 * (j0 + j) + 1] += g[b][j].y;
          s[4 * (j0 + j) + 2] += g[b][j].z;
          s[4 * (j0 + j) + 3] += g[b][j].w;
        }
      }
    }
  }
}

__device__ __forceinline__ void store_out(void* C, int64_t idx, float v, bool out_bf16) {
  if (out_bf16)
    reinterpret_cast<__nv_bfloat16*>(C)[idx] = __float2bfloat16_rn(v);
  else
    reinterpret_cast<__half*>(C)[idx] = __float2half_rn(v);
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
  if (threadIdx.x == 0) trace_event(tb, 0, kTraceKernelBegin, -1, (int32_t)(clock64() & 0x7fffffff));

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
        trace_event(tb, kRoleProducer, kTraceItemBegin, sg.tile, sg.kb0);
        if (args.checks && (sg.tile < 0 || sg.tile >= args.n_tiles || sg.kb0 < 0 || sg.kb0 >= sg.kb1 ||
                            sg.kb1 > args.k_blocks || sg.chunk < 0 || sg.chunk >= chunks.count())) {
          report_check(args.status, kCheckItem, abort_flag);
          ok = false;
          break;
        }
        for (int kb = sg.kb0; kb < sg.kb1; ++kb) {
          if (!mbar_wait(empty_bar(stage), phase ^ 1u, ctl)) {
            ok = false;
            break;
          }
          const bool drop = (args.inject == 1) && (blockIdx.x == 0) && (issued == 0);
          if (!drop) {
            const uint32_t w_dst = base + (uint32_t)stage * stage_bytes;
            const uint32_t x_dst = w_dst + kWBytes;
            const uint32_t fb = full_bar(stage);
            mbar_arrive_expect_tx(fb, stage_bytes);
            tma_load_2d(w_dst, &tmW, fb, kb * kBK, sg.tile * kRowsPerTile);
            tma_load_2d(x_dst, &tmX, fb, kb * kBK, 0);
          }
          ++issued;
          if (++stage == stages) {
            stage = 0;
            phase ^= 1u;
          }
          if (!feed.poll(sg.kb1 - kb - 1, ctl)) {
            ok = false;
            break;
          }
        }
      }
      trace_event(tb, kRoleProducer, kTraceItemEnd, -1, (int32_t)issued);
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
        trace_event(tb, kRoleMma, kTraceItemBegin, sg.tile, sg.kb0);
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * mma_n);
        for (int kb = sg.kb0; kb < sg.kb1; ++kb) {
          if (!mbar_wait(full_bar(stage), phase, ctl)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t w_addr = base + (uint32_t)stage * stage_bytes;
          const uint32_t x_addr = w_addr + kWBytes;
          const uint64_t w_desc = make_smem_desc(w_addr, 16u, kKMajorSBO, kSwizzle128B);
          const uint64_t x_desc = make_smem_desc(x_addr, 16u, kKMajorSBO, kSwizzle128B);
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            const uint64_t step = (uint64_t)(kk * (kKMajorStepBytes >> 4));
            mma_f16<1>(d_tmem, w_desc + step, x_desc + step, args.idesc, (uint32_t)((kb != sg.kb0) || (kk != 0)));
          }
          tc_commit(empty_bar(stage));
          if (++stage == stages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(tfull_bar(acc));
        trace_event(tb, kRoleMma, kTraceItemEnd, sg.tile, sg.kb1);
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
    Segment sg;
    for (;;) {
      const int more = feed.next(sg, ctl);
      // The four epilogue warps read the same chunks; they stop together.
      if (named_bar_or(2, 128, more < 0)) {
        ok = false;
        break;
      }
      if (more == 0) break;
      const bool got = mbar_wait(tfull_bar(acc), acc_phase, ctl);
      // The four epilogue warps meet at named barriers below, so they give up together.
      if (named_bar_or(2, 128, !got)) {
        ok = false;
        break;
      }
      tc_fence_after();
      if (threadIdx.x == 64) trace_event(tb, kRoleEpilogue, kTraceItemBegin, sg.tile, sg.kb0);
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

      const int64_t n = (int64_t)sg.tile * kRowsPerTile + row;
      if (sg.kb0 == 0 && sg.kb1 == args.k_blocks) {
        // The whole K range of this tile is ours: write C directly.
        if (n < args.N) {
#pragma unroll
          for (int m = 0; m < kSplitKMaxM; ++m)
            if (m < args.M) store_out(args.C, (int64_t)m * args.N + n, v[m], out_bf16);
        }
      } else {
        // Publish, then count: every contributor stores its fp32 partial, and
        // once all rows are written one thread takes a ticket with an
        // acquire-release add.  The contributor that draws the last ticket
        // has thereby acquired every other contributor's partial; it sums all
        // of them (its own read back) in contributor (= K) order and writes C,
        // so the result does not depend on who finishes last.
        const int64_t u_first = (int64_t)sg.tile * args.k_blocks;
        const int64_t u_last = u_first + args.k_blocks - 1;
        const int64_t c_first = chunks.owner(u_first);
        const int64_t c_last = chunks.owner(u_last);
        const int32_t others = (int32_t)(c_last - c_first);
        int32_t* const arrivals = args.tickets + sg.tile;
        {
          const int slot = sg.first ? 0 : 1;
          float* mine = partials + ((sg.chunk * 2 + slot) * kRowsPerTile + row) * mma_n;
#pragma unroll
          for (int j = 0; j < kSplitKMaxM / 4; ++j)
            if (j * 4 < mma_n)
              reinterpret_cast<float4*>(mine)[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
        }
        named_bar_sync(1, 128);  // every row of the partial is written ...
        if (threadIdx.x == 64) *ticket_slot = atom_add_acq_rel_gpu(arrivals, 1);  // ... before the ticket
        named_bar_sync(1, 128);  // ... and the acquire orders the partial reads below
        const int32_t ticket = *ticket_slot;
        if (args.checks && threadIdx.x == 64) {
          if (ticket < 0 || ticket > others) report_check(args.status, kCheckTicket, abort_flag);
          if (sg.chunk < c_first || sg.chunk > c_last) report_check(args.status, kCheckContributor, abort_flag);
          if (c_first < 0 || c_last >= chunks.count()) report_check(args.status, kCheckPartial, abort_flag);
        }
        if (ticket == others) {
          float s[kSplitKMaxM];
#pragma unroll
          for (int m = 0; m < kSplitKMaxM; ++m) s[m] = 0.0f;
          // Contributors after the first start inside this tile, so their
          // partial of it is their first (slot 0); the first contributor's
          // range may start in an earlier tile (slot 1).
          const int slot_first = (chunks.begin(c_first) >= u_first) ? 0 : 1;
          const float4* const tile_partials = reinterpret_cast<const float4*>(partials + (int64_t)row * mma_n);
          sum_contributors(s, tile_partials, c_first, c_last, slot_first, mma_n);
          if (n < args.N) {
#pragma unroll
            for (int m = 0; m < kSplitKMaxM; ++m)
              if (m < args.M) store_out(args.C, (int64_t)m * args.N + n, s[m], out_bf16);
          }
          if (threadIdx.x == 64) *arrivals = 0;  // ready for the next launch
        }
        named_bar_sync(1, 128);  // ticket_slot is reused by the next segment
      }
      if (threadIdx.x == 64) trace_event(tb, kRoleEpilogue, kTraceItemEnd, sg.tile, sg.kb1);
    }
    if (!ok && lane == 0) sk_report(args.status, kRoleEpilogue, abort_flag);
  }

  __syncthreads();
  // every role of the CTA is done: the end of the CTA's work
  if (threadIdx.x == 0) trace_event(tb, 0, kTraceKernelEnd, -1, (int32_t)(clock64() & 0x7fffffff));
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
