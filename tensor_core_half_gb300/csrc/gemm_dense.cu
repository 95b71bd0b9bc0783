// gemm_dense.cu -- persistent, warp-specialised tcgen05 GEMM for sm_103a.
//
// C[M,N] = A[M,K] . B[K,N], fp16/bf16 inputs, fp32 or fp16 accumulators in
// tensor memory, fp16/bf16 output.  The kernel structure follows the steps of
// "tcgen05 for dummies: a B200 GEMM from scratch" (translated):
//   - "TMA and mbarrier": tiles move global -> shared with cp.async.bulk.tensor,
//     completion tracked by transaction-count mbarriers;
//   - "128-byte global loads and swizzle": 64-element (128 B) boxes with the
//     128-byte swizzle, matched by the MMA's shared-memory descriptor;
//   - "Pipelining" and "Warp specialization": a STAGES-deep ring with full /
//     empty barrier pairs, one TMA warp, one MMA warp;
//   - "2-SM MMA": cta_group::2, a CTA pair computes a 256-row tile, each CTA
//     loads its own 128 rows of A and half of the B tile;
//   - "Persistent kernel: static scheduling": one CTA (pair) per SM walks its
//     tiles; tensor-memory accumulators are double-buffered so the epilogue of
//     one tile overlaps the mainloop of the next.
// Differences from the page: the epilogue goes tcgen05.ld -> cast -> swizzled
// shared staging -> TMA store (the page stored from registers); tiles are
// visited in grouped (L2-friendly) order; every wait is bounded and a wait
// that gives up reports HGEMM_ERR_TIMEOUT instead of hanging; ragged M, N and
// K are handled by TMA zero fill on loads and clipping on stores; NN layout
// (B row-major, MN-major operand) and fp16 accumulation are supported.
//
// Warp roles (192 threads):
//   warp 0      TMA producer (one thread)
//   warp 1      TMEM allocator; MMA issuer (one thread; in a CTA pair only CTA 0)
//   warps 2..5  epilogue; warp w reads TMEM lanes 32*(w%4) .. 32*(w%4)+31
#include <cuda_fp16.h>

#include "clc.cuh"
#include "desc.cuh"
#include "kernels.h"
#include "ptx.cuh"
#include "sched.cuh"

namespace hg {

template <int CG, int BN, int STAGES>
struct DenseShape {
  static constexpr int BM = 128;                  // C rows per CTA
  static constexpr int BK = 64;                   // K elements per stage: one 128 B swizzle row
  static constexpr int A_BYTES = BM * BK * 2;     // 16 KiB
  static constexpr int B_ROWS = BN / CG;          // N extent of the B slice this CTA loads
  static constexpr int B_BYTES = B_ROWS * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int EPI_BOX_COLS = 64;         // output columns per TMA store box (128 B)
  static constexpr int EPI_BOX_BYTES = 32 * 128;  // 32 rows x 128 B
  static constexpr int EPI_BYTES = 4 * 2 * EPI_BOX_BYTES;  // 4 warps x double buffer
  static constexpr int RING_BYTES = STAGES * STAGE_BYTES;
  static constexpr int BAR_OFF = RING_BYTES + EPI_BYTES;
  static constexpr int CLC_SLOTS = 4;             // cluster-launch-control responses in flight
  // full[S], empty[S], tmem_full[2], tmem_empty[2], drain, clc_full[C], clc_empty[C]
  static constexpr int NUM_BARS = 2 * STAGES + 5 + 2 * CLC_SLOTS;
  static constexpr int MISC_OFF = BAR_OFF + NUM_BARS * 8;
  static constexpr int CLC_OFF = (MISC_OFF + 16 + 15) / 16 * 16;  // 16-byte responses
  static constexpr int SMEM_BYTES = CLC_OFF + 16 * CLC_SLOTS + 1024;  // + alignment slack for the 1 KiB base
  static constexpr int TMEM_COLS = 2 * BN <= 256 ? 256 : 512;  // two accumulators, power of two
  static constexpr int THREADS = 192;
  static_assert(BN % 64 == 0 && BN <= 256, "BN");
  static_assert((BN / CG) % 8 == 0, "B slice rows");
  // An MN-major (NN) B slice is loaded as 64-column boxes.
  static constexpr bool kMNMajorOK = (BN / CG) % 64 == 0;
  static_assert(TMEM_COLS == 256 || TMEM_COLS == 512, "TMEM allocation must be a power of two");
  static_assert(SMEM_BYTES <= 232448, "shared memory");
};

__device__ __forceinline__ void report_timeout(int32_t* status, int32_t role, volatile uint32_t* abort_flag) {
  *abort_flag = 1u;
  atomicCAS(status, 0, kStatusTimeout | (role << 8) | ((int32_t)(blockIdx.x & 0xFFFF) << 16));
}

// fp16x2 (packed) -> the output's packed pair.
__device__ __forceinline__ uint32_t f16x2_to_out(uint32_t h2, bool out_bf16) {
  if (!out_bf16) return h2;
  __half2 h = *reinterpret_cast<__half2*>(&h2);
  float2 f = __half22float2(h);
  return pack_f32x2_to_bf16x2(f.x, f.y);
}

// The work ids one role walks through.  Static schedule: the cluster's fixed
// walk.  Dynamic schedule: the cluster's own id, then ids taken over from
// clusters that have not started (ClcIds, cluster launch control).
template <int CG, int SLOTS>
struct IdFeed {
  WorkIter it;
  ClcIds<CG, SLOTS> clc;
  int32_t cluster, nclusters;
  bool dynamic;
  bool checks;
  int32_t* status;
  bool started = false, finished = false;
  bool want = false;  // issuer: the current id's request is still to be made

  __device__ IdFeed(const DenseArgs& a, int32_t cluster_, int32_t nclusters_, uint32_t resp0, uint32_t full0,
                    uint32_t empty0, bool issuer, bool warp_wide, bool arrive)
      : it(a.sk_ranges, a.dp_tiles, a.sk_units, a.k_blocks),
        clc(resp0, full0, empty0, issuer, warp_wide, arrive),
        cluster(cluster_),
        nclusters(nclusters_),
        dynamic(a.dynamic != 0),
        checks(a.checks != 0),
        status(a.status) {}

  // 1: an item in w; 0: no work left; -1: a wait gave up.
  __device__ int next(WorkItem& w, const WaitCtl& ctl) {
    for (;;) {
      if (!started) {
        if (finished) return 0;
        started = true;
        if (!dynamic) {
          it.start_static(cluster, nclusters);
        } else {
          it.start(cluster);
          want = clc.issuer;
        }
      }
      if (!dynamic) return it.next_static(w) ? 1 : 0;
      if (it.next_in_id(w)) return 1;
      if (want) {  // an id shorter than the lead: ask now
        want = false;
        if (!clc.request(ctl)) return -1;
      }
      int64_t id = 0;
      const int got = clc.fetch(&id, ctl);
      if (got < 0) return -1;
      if (got > 0 && checks && (id < 0 || id >= it.n_ids)) {
        report_check(status, kCheckWorkId, nullptr);
        return -1;
      }
      if (got == 0) {
        finished = true;
        started = false;
        return 0;
      }
      it.start(id);
      want = clc.issuer;
    }
  }

  // Issuer, after loading a k-block of the current item: `left` k-blocks of
  // the item remain; ask for the next id when clc_time_to_ask says so.
  __device__ bool poll(int64_t left, const WaitCtl& ctl) {
    if (!want || !clc_time_to_ask(left + it.left_after_item(), it.id_length())) return true;
    want = false;
    return clc.request(ctl);
  }

  __device__ bool drain(const WaitCtl& ctl) { return clc.drain(ctl); }
};

template <int CG, int BN, int STAGES>
__global__ void __launch_bounds__(192, 1)
    dense_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                      const __grid_constant__ CUtensorMap tmC, const DenseArgs args) {
  using S = DenseShape<CG, BN, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;  // 128 B swizzle atoms need 1 KiB alignment
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t ring = base;
  const uint32_t epi = base + S::RING_BYTES;
  const uint32_t bars = base + S::BAR_OFF;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + S::MISC_OFF);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(gbase + S::MISC_OFF + 4);
  volatile int32_t* ticket_slot = reinterpret_cast<volatile int32_t*>(gbase + S::MISC_OFF + 8);

  auto full_bar = [&](int s) -> uint32_t { return bars + 8u * s; };
  auto empty_bar = [&](int s) -> uint32_t { return bars + 8u * (STAGES + s); };
  auto tfull_bar = [&](int b) -> uint32_t { return bars + 8u * (2 * STAGES + b); };
  auto tempty_bar = [&](int b) -> uint32_t { return bars + 8u * (2 * STAGES + 2 + b); };
  const uint32_t drain_bar = bars + 8u * (2 * STAGES + 4);
  const uint32_t clc_full0 = bars + 8u * (2 * STAGES + 5);
  const uint32_t clc_empty0 = clc_full0 + 8u * S::CLC_SLOTS;
  const uint32_t clc_resp0 = base + S::CLC_OFF;
  using Feed = IdFeed<CG, S::CLC_SLOTS>;

  const int warp = threadIdx.x / 32;
  const uint32_t lane = threadIdx.x % 32;
  const uint32_t rank = (CG == 2) ? cluster_ctarank() : 0u;
  const int cluster = (CG == 2) ? (int)cluster_id_x() : (int)blockIdx.x;
  const int nclusters = (CG == 2) ? (int)num_clusters_x() : (int)gridDim.x;
  constexpr bool kCS = (CG == 2);  // cluster-scope waits on barriers that see peer signals
  const WaitCtl ctl{args.timeout_ns, abort_flag};
  const WaitCtl drain_ctl{kDrainTimeoutNs, nullptr};

  // ------------------------------------------------------------ setup ----
  if (warp == 0) {
    if (lane == 0) {
      for (int s = 0; s < STAGES; ++s) {
        mbar_init(full_bar(s), 1);
        mbar_init(empty_bar(s), 1);
      }
      for (int b = 0; b < 2; ++b) {
        mbar_init(tfull_bar(b), 1);
        mbar_init(tempty_bar(b), 4 * CG);  // every epilogue warp of the pair arrives
      }
      mbar_init(drain_bar, 1);
      // readers of every response: producer, MMA issuer and 4 epilogue warps
      // of CTA 0, producer and 4 epilogue warps of CTA 1
      ClcIds<CG, S::CLC_SLOTS>::init(clc_full0, clc_empty0, CG == 2 ? 11 : 6);
      *abort_flag = 0u;
      fence_mbar_init();
      prefetch_tmap(&tmA);
      prefetch_tmap(&tmB);
      prefetch_tmap(&tmC);
    }
    __syncwarp();
  } else if (warp == 1) {
    tmem_alloc<CG>(smem_addr(tmem_slot), S::TMEM_COLS);
    tmem_relinquish<CG>();
    tc_fence_before();
  }
  if constexpr (CG == 2)
    cluster_sync();
  else
    __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(tmem_slot);
  bool aborted = false;
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
    // ------------------------------------------------- TMA producer ----
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int64_t issued = 0;
      bool ok = true;
      const uint32_t full_rank0 = (CG == 2) ? mapa_shared(full_bar(0), 0) : full_bar(0);
      Feed feed(args, cluster, nclusters, clc_resp0, clc_full0, clc_empty0, rank == 0, false, true);
      WorkItem w;
      for (;;) {
        const int got = feed.next(w, ctl);
        if (got < 0) ok = false;
        if (got <= 0) break;
        trace_event(tbi, kRoleProducer, kTraceItemBegin, w.tile, w.kb0);
        uint32_t stall = 0;
        const TileCoord tc = tile_coord(w.tile, args.tiles_m, args.tiles_n, args.group_m);
        if (args.checks) {
          const bool bad = w.tile < 0 || w.tile >= args.num_tiles || w.kb0 < 0 || w.kb0 >= w.kb1 ||
                           w.kb1 > args.k_blocks || tc.m < 0 || tc.m >= args.tiles_m || tc.n < 0 ||
                           tc.n >= args.tiles_n ||
                           (w.slot >= 0 && (w.tile < args.dp_tiles || w.owner < 0 || w.owner >= args.sk_ranges));
          if (bad) {
            report_check(args.status, kCheckItem, abort_flag);
            ok = false;
            break;
          }
        }
        const int m_row = tc.m * (S::BM * CG) + (int)rank * S::BM;
        const int n_row = tc.n * BN + (int)rank * S::B_ROWS;
        for (int kb = w.kb0; kb < w.kb1; ++kb) {
          if (!mbar_wait_stall<kCS>(empty_bar(stage), phase ^ 1u, ctl, &stall)) {
            ok = false;
            break;
          }
          // Test hook: the first cluster drops its first stage in every CTA of
          // the pair (no expect_tx, no copy), so the MMA issuer's wait for it
          // runs out and no copy is left in flight when the CTAs exit.
          const bool drop = (args.inject == 1) && (blockIdx.x / CG == 0) && (issued == 0);
          if (!drop) {
            const uint32_t a_dst = ring + (uint32_t)stage * S::STAGE_BYTES;
            const uint32_t b_dst = a_dst + S::A_BYTES;
            const int k0 = kb * S::BK;
            if constexpr (CG == 1) {
              const uint32_t fb = full_bar(stage);
              mbar_arrive_expect_tx(fb, S::STAGE_BYTES);
              tma_load_2d(a_dst, &tmA, fb, k0, m_row);
              if (!args.b_mn_major) {
                tma_load_2d(b_dst, &tmB, fb, k0, n_row);
              } else if constexpr (S::kMNMajorOK) {
#pragma unroll
                for (int j = 0; j < S::B_ROWS / 64; ++j) tma_load_2d(b_dst + j * 8192, &tmB, fb, n_row + 64 * j, k0);
              }
            } else {
              // Both CTAs report their bytes to CTA 0's barrier, which expects the pair's total.
              const uint32_t fb = full_rank0 + 8u * (uint32_t)stage;
              if (rank == 0) mbar_arrive_expect_tx(full_bar(stage), 2 * S::STAGE_BYTES);
              tma_load_2d_pair(a_dst, &tmA, fb, k0, m_row);
              if (!args.b_mn_major) {
                tma_load_2d_pair(b_dst, &tmB, fb, k0, n_row);
              } else if constexpr (S::kMNMajorOK) {
#pragma unroll
                for (int j = 0; j < S::B_ROWS / 64; ++j)
                  tma_load_2d_pair(b_dst + j * 8192, &tmB, fb, n_row + 64 * j, k0);
              }
            }
          }
          ++issued;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
          if (!feed.poll(w.kb1 - kb - 1, ctl)) {
            ok = false;
            break;
          }
        }
        trace_event(tbi, kRoleProducer, kTraceStall, w.tile, (int32_t)stall);
        trace_event(tbi, kRoleProducer, kTraceItemEnd, w.tile, w.kb1);
        if (!ok) break;
      }
      if (!ok) {
        report_timeout(args.status, kRoleProducer, abort_flag);
        aborted = true;
      }
      if (!feed.drain(drain_ctl)) {
        report_timeout(args.status, kRoleTeardown, abort_flag);
        aborted = true;
      }
      // Every load this CTA issued and signalled on its own barrier must land
      // before the CTA can exit.  In the normal path these waits return at once.
      if (CG == 1 || rank == 0) {
        for (int s = 0; s < STAGES; ++s) {
          if (issued <= s) break;
          const int64_t last = s + (int64_t)STAGES * ((issued - 1 - s) / STAGES);
          const bool dropped = (args.inject == 1) && (blockIdx.x / CG == 0) && (last == 0);
          if (dropped) continue;
          if (!mbar_wait<kCS>(full_bar(s), (uint32_t)((last / STAGES) & 1), drain_ctl)) {
            report_timeout(args.status, kRoleTeardown, abort_flag);
            aborted = true;
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // --------------------------------------------------- MMA issuer ----
    if ((CG == 1 || rank == 0) && lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      const uint32_t b_step = args.b_mn_major ? (kMNMajorStepBytes >> 4) : (kKMajorStepBytes >> 4);
      const uint32_t b_lbo = args.b_mn_major ? kMNMajorLBO : 16u;
      const uint32_t b_sbo = args.b_mn_major ? kMNMajorSBO : kKMajorSBO;
      Feed feed(args, cluster, nclusters, clc_resp0, clc_full0, clc_empty0, false, false, true);
      WorkItem w;
      for (;;) {
        const int got = feed.next(w, ctl);
        if (got < 0) ok = false;
        if (got <= 0) break;
        // Wait until the epilogue has drained this accumulator buffer.
        if (!mbar_wait<kCS>(tempty_bar(acc), acc_phase ^ 1u, ctl)) {
          ok = false;
          break;
        }
        tc_fence_after();
        trace_event(tbi, kRoleMma, kTraceItemBegin, w.tile, w.kb0);
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
        uint32_t stall = 0;
        for (int kb = w.kb0; kb < w.kb1; ++kb) {
          if (!mbar_wait_stall<kCS>(full_bar(stage), phase, ctl, &stall)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = ring + (uint32_t)stage * S::STAGE_BYTES;
          const uint32_t b_addr = a_addr + S::A_BYTES;
          const uint64_t a_desc = make_smem_desc(a_addr, 16u, kKMajorSBO, kSwizzle128B);
          const uint64_t b_desc = make_smem_desc(b_addr, b_lbo, b_sbo, kSwizzle128B);
#pragma unroll
          for (int kk = 0; kk < S::BK / 16; ++kk) {
            mma_f16<CG>(d_tmem, a_desc + (uint64_t)(kk * (kKMajorStepBytes >> 4)), b_desc + (uint64_t)(kk * b_step),
                        args.idesc, (uint32_t)((kb != w.kb0) || (kk != 0)));
          }
          tc_commit_cg<CG>(empty_bar(stage), (uint16_t)0x3);  // frees the stage once these MMAs finish
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit_cg<CG>(tfull_bar(acc), (uint16_t)0x3);  // accumulator ready for the epilogue
        trace_event(tbi, kRoleMma, kTraceStall, w.tile, (int32_t)stall);
        trace_event(tbi, kRoleMma, kTraceItemEnd, w.tile, w.kb1);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      if (!ok) {
        report_timeout(args.status, kRoleMma, abort_flag);
        aborted = true;
      }
      // Drain: every MMA issued above completes before tensor memory is released.
      tc_commit_cg<CG>(drain_bar, (uint16_t)0x1);
      if (!mbar_wait<false>(drain_bar, 0u, WaitCtl{args.timeout_ns, nullptr})) {
        report_timeout(args.status, kRoleTeardown, abort_flag);
        aborted = true;
      }
    }
    __syncwarp();
  } else {
    // ----------------------------------------------------- epilogue ----
    const int q = warp & 3;   // TMEM lane quarter this warp may access
    const int ew = warp - 2;  // staging slot
    const int row = q * 32 + (int)lane;  // row of this thread within the CTA's 128 rows
    int acc = 0;
    uint32_t acc_phase = 0;
    uint32_t nstores = 0;
    bool ok = true;
    const bool out_bf16 = args.out_bf16 != 0;
    const bool acc_f16 = args.acc_f16 != 0;
    const bool epi_direct = args.epi_direct != 0;

    // 64 accumulator columns of this thread's row, as fp32.
    auto load_chunk = [&](uint32_t t_row, int c, float (&f)[64]) {
      uint32_t v[64];
      tmem_ld_x32(t_row + (uint32_t)(c * 64), v);
      tmem_ld_x32(t_row + (uint32_t)(c * 64 + 32), v + 32);
      tmem_ld_wait();
      if (!acc_f16) {
#pragma unroll
        for (int i = 0; i < 64; ++i) f[i] = __uint_as_float(v[i]);
      } else {
        // fp16 accumulators occupy one 32-bit TMEM column each, in the low half.
#pragma unroll
        for (int i = 0; i < 64; ++i) f[i] = __half2float(__ushort_as_half((unsigned short)(v[i] & 0xFFFFu)));
      }
    };

    // Round 64 columns to the output type and store them (warp: 32 rows x 64 columns).
    auto emit_chunk = [&](const float (&f)[64], int m0, int nc) {
      if (!(m0 < args.M && nc < args.N)) return;  // warp-uniform; TMA clips partial boxes
      uint32_t p[32];
      if (out_bf16) {
#pragma unroll
        for (int i = 0; i < 32; ++i) p[i] = pack_f32x2_to_bf16x2(f[2 * i], f[2 * i + 1]);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) p[i] = pack_f32x2_to_f16x2(f[2 * i], f[2 * i + 1]);
      }
      if (epi_direct) {
        // Straight from registers: this thread's row, eight 16-byte pieces
        // (N is a multiple of 8, so a piece is wholly inside C or outside).
        const int r = m0 + (int)lane;
        if (r < args.M) {
          uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(args.C) + (size_t)r * (size_t)args.N + nc);
#pragma unroll
          for (int j = 0; j < 8; ++j)
            if (nc + 8 * j < args.N) dst[j] = make_uint4(p[4 * j], p[4 * j + 1], p[4 * j + 2], p[4 * j + 3]);
        }
        return;
      }
      const uint32_t buf = epi + (uint32_t)(ew * 2 + (int)(nstores & 1u)) * S::EPI_BOX_BYTES;
      if (lane == 0) bulk_wait_read<1>();  // the store that last used this buffer has read it
      __syncwarp();
      const uint32_t srow = buf + lane * 128u;
#pragma unroll
      for (int j = 0; j < 8; ++j)
        st_shared_v4(srow + ((uint32_t)(j ^ (int)(lane & 7u)) << 4), p[4 * j], p[4 * j + 1], p[4 * j + 2],
                     p[4 * j + 3]);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_store_2d(&tmC, buf, nc, m0);
        bulk_commit();
      }
      ++nstores;
    };

    auto release_tmem = [&](int b) {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if constexpr (CG == 1)
          mbar_arrive(tempty_bar(b));
        else
          mbar_arrive_cluster(mapa_shared(tempty_bar(b), 0));
      }
    };

    // Stream-K partial of cluster c, slot s, this CTA: BN/4 groups of 4 columns,
    // each [128 rows] of float4, so a warp's accesses are 512 contiguous bytes.
    auto partial_of = [&](int64_t c, int s) -> float4* {  // c: stream-K range
      return reinterpret_cast<float4*>(args.partials + (((c * 2 + s) * CG + rank) * (int64_t)BN * 128));
    };

    Feed feed(args, cluster, nclusters, clc_resp0, clc_full0, clc_empty0, false, true, lane == 0);
    WorkItem w;
    int deferred = -1;  // accumulator buffer of a whole tile whose release waits for the next item
    for (;;) {
      const int more = feed.next(w, ctl);
      // The four epilogue warps read the same ids; they stop together.
      if (named_bar_or(2, 128, more < 0)) {
        ok = false;
        break;
      }
      if (more == 0) break;
      // A whole tile's buffer is handed back to the MMA issuer only once
      // another item follows: after the last item nobody waits for it, and
      // its fence and (in a pair) cluster-scope arrive, ~0.6 us measured on
      // GB300, would otherwise sit between the last store and the CTA's exit.
      if (deferred >= 0) {
        release_tmem(deferred);
        deferred = -1;
      }
      const bool got = mbar_wait<kCS>(tfull_bar(acc), acc_phase, ctl);
      // The four epilogue warps meet at named barriers, so they give up together.
      if (named_bar_or(2, 128, !got)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const bool tracer = threadIdx.x == 64;
      if (tracer) trace_event(tbi, kRoleEpilogue, kTraceItemBegin, w.tile, w.slot);
      const TileCoord tc = tile_coord(w.tile, args.tiles_m, args.tiles_n, args.group_m);
      const int m0 = tc.m * (S::BM * CG) + (int)rank * S::BM + q * 32;  // first C row of this warp
      const int n0 = tc.n * BN;
      const uint32_t t_row = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN);
      if (w.slot < 0) {
#pragma unroll 1
        for (int c = 0; c < BN / 64; ++c) {
          float f[64];
          load_chunk(t_row, c, f);
          emit_chunk(f, m0, n0 + c * 64);
        }
        // All reads of this accumulator are done; it is released at the next
        // item (above), after this tile's stores are issued.  The MMA issuer
        // needs the buffer only after the tile that follows.
        deferred = acc;
      } else {
        // A piece of a stream-K tile.  The ticket comes first: the contributor
        // that arrives last keeps its accumulator in TMEM and adds the other
        // contributors' fp32 partials to it; every other contributor publishes
        // its partial and bumps the tile's publication count.  The sum always
        // runs over the contributors in K order, whoever arrives last, so the
        // result does not depend on timing.
        const int32_t tix = w.tile * CG + (int32_t)rank;
        int32_t* const arrivals = args.tickets + tix;
        int32_t* const pubs = args.tickets + (int64_t)args.num_tiles * CG + tix;
        int64_t c_first, c_last;
        sk_contributors(w.tile, args.dp_tiles, args.sk_units, args.k_blocks, args.sk_ranges, &c_first, &c_last);
        const int32_t others = (int32_t)(c_last - c_first);
        if (threadIdx.x == 64) *ticket_slot = atomicAdd(arrivals, 1);
        named_bar_sync(1, 128);
        const int32_t ticket = *ticket_slot;
        named_bar_sync(1, 128);
        if (args.checks && threadIdx.x == 64) {
          // A ticket past the count would leave the tile unreduced; the owner
          // and its partial slots must lie inside the contributor range and
          // the workspace.
          if (ticket < 0 || ticket > others) report_check(args.status, kCheckTicket, abort_flag);
          if (w.owner < c_first || w.owner > c_last) report_check(args.status, kCheckContributor, abort_flag);
          if (c_first < 0 || c_last >= args.sk_ranges) report_check(args.status, kCheckPartial, abort_flag);
        }
        if (ticket != others) {
          float4* mine = partial_of(w.owner, w.slot) + row;
#pragma unroll 1
          for (int c = 0; c < BN / 64; ++c) {
            float f[64];
            load_chunk(t_row, c, f);
            if (c == BN / 64 - 1) release_tmem(acc);
#pragma unroll
            for (int j = 0; j < 16; ++j)
              mine[(c * 16 + j) * 128] = make_float4(f[4 * j], f[4 * j + 1], f[4 * j + 2], f[4 * j + 3]);
          }
          named_bar_sync(1, 128);  // every row of the partial is written ...
          if (threadIdx.x == 64) red_add_release_gpu(pubs, 1);  // ... before it is published
          if (tracer) trace_event(tbi, kRoleEpilogue, kTracePartialStored, w.tile, ticket);
        } else {
          if (threadIdx.x == 64) {
            const bool all_in = wait_counter_geq(pubs, others, ctl);
            if (!all_in) report_timeout(args.status, kRoleEpilogue, abort_flag);
            *ticket_slot = all_in ? 1 : 0;
          }
          named_bar_sync(1, 128);  // the acquire above orders the partial reads below
          const bool have_all = *ticket_slot != 0;
#pragma unroll 1
          for (int c = 0; c < BN / 64; ++c) {
            float f[64];
#pragma unroll
            for (int j = 0; j < 64; ++j) f[j] = 0.0f;
            for (int64_t cc = c_first; cc <= c_last; ++cc) {
              if (cc == w.owner) {
                float own[64];
                load_chunk(t_row, c, own);
                if (c == BN / 64 - 1) release_tmem(acc);
#pragma unroll
                for (int j = 0; j < 64; ++j) f[j] += own[j];
              } else if (have_all) {
                const float4* src =
                    partial_of(cc, sk_slot_of(cc, w.tile, args.dp_tiles, args.sk_units, args.k_blocks, args.sk_ranges)) +
                    row;
                float4 g[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) g[j] = __ldcg(src + (c * 16 + j) * 128);
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                  f[4 * j] += g[j].x;
                  f[4 * j + 1] += g[j].y;
                  f[4 * j + 2] += g[j].z;
                  f[4 * j + 3] += g[j].w;
                }
              }
            }
            emit_chunk(f, m0, n0 + c * 64);
          }
          if (tracer) trace_event(tbi, kRoleEpilogue, kTraceReduced, w.tile, others + 1);
          if (threadIdx.x == 64) {  // ready for the next launch
            *arrivals = 0;
            *pubs = 0;
          }
        }
        named_bar_sync(1, 128);  // ticket_slot is reused by the next item
      }
      if (tracer) trace_event(tbi, kRoleEpilogue, kTraceItemEnd, w.tile, w.slot);
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    if (!ok) {
      if (lane == 0) report_timeout(args.status, kRoleEpilogue, abort_flag);
      aborted = true;
    }
    tc_fence_before();  // this warp's tensor-memory reads precede the teardown's dealloc
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }

  // --------------------------------------------------------- teardown ----
  if constexpr (CG == 2) {
    // In a pair, the peer's loads signal CTA 0 and CTA 0's MMAs read the peer's
    // shared memory; after a give-up, leave time for copies still in flight.
    if (__syncthreads_or(aborted ? 1 : 0)) {
      const uint64_t t0 = globaltimer_ns();
      while (globaltimer_ns() - t0 < 50000ull) {
      }
    }
    cluster_sync();
  } else {
    __syncthreads();
  }
  // every role of the CTA (pair) is done: the end of the CTA's work
  if (tb != nullptr && threadIdx.x == kStampThread)
    trace_put(tb, stamp_slot + 1, globaltimer_ns(), 0, kTraceKernelEnd, -1, (int32_t)(clock64() & 0x7fffffff));
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc<CG>(tmem_base, S::TMEM_COLS);
  }
}

// --------------------------------------------------------------- host ----
#define HG_DENSE_KINDS(X) \
  X(kDense1Sm128, 1, 128, 6) \
  X(kDense1Sm256, 1, 256, 4) \
  X(kDense2Sm256, 2, 256, 6) \
  X(kDense2Sm192, 2, 192, 6)

DenseKindInfo dense_kind_info(DenseKind kind) {
  switch (kind) {
#define X(KIND, CG, BN, ST)                                                                                 \
  case KIND:                                                                                                \
    return DenseKindInfo{CG, BN, ST, DenseShape<CG, BN, ST>::SMEM_BYTES, DenseShape<CG, BN, ST>::TMEM_COLS, \
                         DenseShape<CG, BN, ST>::THREADS};
    HG_DENSE_KINDS(X)
#undef X
  }
  return DenseKindInfo{0, 0, 0, 0, 0, 0};
}

static const void* dense_fn(DenseKind kind) {
  switch (kind) {
#define X(KIND, CG, BN, ST) \
  case KIND:                \
    return reinterpret_cast<const void*>(&dense_gemm_kernel<CG, BN, ST>);
    HG_DENSE_KINDS(X)
#undef X
  }
  return nullptr;
}

cudaError_t dense_prepare(DenseKind kind) {
  const DenseKindInfo info = dense_kind_info(kind);
  const void* fn = dense_fn(kind);
  if (!fn) return cudaErrorInvalidValue;
  return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, info.smem_bytes);
}

// Launch configuration: cluster shape for the CTA-pair kernel, and programmatic
// stream serialisation so that back-to-back GEMMs overlap launch and prologue.
static void fill_config(cudaLaunchConfig_t& cfg, cudaLaunchAttribute* attr, const DenseKindInfo& info, int grid,
                        cudaStream_t stream, bool pdl) {
  cfg = cudaLaunchConfig_t{};
  cfg.gridDim = dim3((unsigned)grid, 1, 1);
  cfg.blockDim = dim3((unsigned)info.threads, 1, 1);
  cfg.dynamicSmemBytes = (size_t)info.smem_bytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 0;
  if (info.cta_group > 1) {
    attr[cfg.numAttrs].id = cudaLaunchAttributeClusterDimension;
    attr[cfg.numAttrs].val.clusterDim.x = (unsigned)info.cta_group;
    attr[cfg.numAttrs].val.clusterDim.y = 1;
    attr[cfg.numAttrs].val.clusterDim.z = 1;
    ++cfg.numAttrs;
  }
  if (pdl) {
    attr[cfg.numAttrs].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[cfg.numAttrs].val.programmaticStreamSerializationAllowed = 1;
    ++cfg.numAttrs;
  }
}

cudaError_t dense_max_active_clusters(DenseKind kind, int* clusters) {
  const DenseKindInfo info = dense_kind_info(kind);
  if (info.cta_group == 1) {
    int dev = 0, sms = 0, per_sm = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, dense_fn(kind), info.threads, (size_t)info.smem_bytes);
    *clusters = per_sm * sms;
    return e;
  }
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[2];
  fill_config(cfg, attr, info, info.cta_group * 64, nullptr, false);
  return cudaOccupancyMaxActiveClusters(clusters, dense_fn(kind), &cfg);
}

cudaError_t dense_launch(DenseKind kind, const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmC,
                         const DenseArgs& args, int grid_ctas, cudaStream_t stream) {
  const DenseKindInfo info = dense_kind_info(kind);
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[2];
  fill_config(cfg, attr, info, grid_ctas, stream, true);
  switch (kind) {
#define X(KIND, CG, BN, ST) \
  case KIND:                \
    return cudaLaunchKernelEx(&cfg, dense_gemm_kernel<CG, BN, ST>, tmA, tmB, tmC, args);
    HG_DENSE_KINDS(X)
#undef X
  }
  return cudaErrorInvalidValue;
}

}  // namespace hg
