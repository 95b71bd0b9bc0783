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
}  // namespace

// Layout: ring (stages x stage_bytes, 1 KiB aligned) | barriers | misc.
__host__ __device__ __forceinline__ int sk_stage_bytes(int mma_n) { return kWBytes + mma_n * kBK * 2; }
__host__ __device__ __forceinline__ int sk_bar_off(int mma_n, int stages) { return stages * sk_stage_bytes(mma_n); }
__host__ __device__ __forceinline__ int sk_num_bars(int stages) { return 2 * stages + 5; }
__host__ __device__ __forceinline__ int sk_tmem_cols(int mma_n) {
  int cols = 32;
  while (cols < 2 * mma_n) cols *= 2;
  return cols;
}

int splitk_stage_bytes(int mma_n) { return sk_stage_bytes(mma_n); }
int splitk_smem_bytes(int mma_n, int stages) { return sk_bar_off(mma_n, stages) + sk_num_bars(stages) * 8 + 16 + 1024; }

int splitk_stages_for(int mma_n, int smem_optin) {
  int s = 12;
  while (s > 2 && splitk_smem_bytes(mma_n, s) > smem_optin) --s;
  return s;
}

int splitk_tmem_cols(int mma_n) { return sk_tmem_cols(mma_n); }

size_t splitk_workspace_bytes(int grid, int mma_n, int n_tiles) {
  size_t partial = (size_t)grid * 2 * kRowsPerTile * (size_t)mma_n * sizeof(float);
  partial = (partial + 255) & ~(size_t)255;
  return partial + (size_t)n_tiles * 2 * sizeof(int32_t);  // arrivals and publications
}

__device__ __forceinline__ void sk_report(int32_t* status, int32_t role, volatile uint32_t* abort_flag) {
  *abort_flag = 1u;
  atomicCAS(status, 0, kStatusTimeout | (role << 8) | ((int32_t)(blockIdx.x & 0xFFFF) << 16));
}

// One segment: the k-blocks [kb0, kb1) of N tile `tile`.
struct Segment {
  int32_t tile, kb0, kb1;
  bool first;  // the first segment of this CTA's range
};

__device__ __forceinline__ Segment segment_at(int64_t u, int64_t end, int32_t k_blocks, int64_t begin) {
  Segment s;
  s.tile = (int32_t)(u / k_blocks);
  s.kb0 = (int32_t)(u - (int64_t)s.tile * k_blocks);
  const int64_t left = end - u;
  const int64_t room = k_blocks - s.kb0;
  s.kb1 = s.kb0 + (int32_t)(left < room ? left : room);
  s.first = (u == begin);
  return s;
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
  auto tempty_bar = [&](int b) -> uint32_t { return bars + 8u * (2 * stages + 2 + b); };
  const uint32_t drain_bar = bars + 8u * (2 * stages + 4);

  const int warp = threadIdx.x / 32;
  const uint32_t lane = threadIdx.x % 32;
  const int64_t G = gridDim.x;
  const int64_t c = blockIdx.x;
  const int64_t begin = splitk_begin(c, args.units, G);
  const int64_t end = splitk_begin(c + 1, args.units, G);
  const int tmem_cols = sk_tmem_cols(mma_n);
  const WaitCtl ctl{args.timeout_ns, abort_flag};
  const WaitCtl drain_ctl{kDrainTimeoutNs, nullptr};

  if (warp == 0) {
    if (lane == 0) {
      for (int s = 0; s < stages; ++s) {
        mbar_init(full_bar(s), 1);
        mbar_init(empty_bar(s), 1);
      }
      for (int b = 0; b < 2; ++b) {
        mbar_init(tfull_bar(b), 1);
        mbar_init(tempty_bar(b), 4);
      }
      mbar_init(drain_bar, 1);
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
      for (int64_t u = begin; ok && u < end;) {
        const Segment sg = segment_at(u, end, args.k_blocks, begin);
        trace_event(tb, kRoleProducer, kTraceItemBegin, sg.tile, sg.kb0);
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
        }
        u += sg.kb1 - sg.kb0;
      }
      trace_event(tb, kRoleProducer, kTraceItemEnd, -1, (int32_t)issued);
      if (!ok) sk_report(args.status, kRoleProducer, abort_flag);
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
      for (int64_t u = begin; ok && u < end;) {
        const Segment sg = segment_at(u, end, args.k_blocks, begin);
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
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
        u += sg.kb1 - sg.kb0;
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
    for (int64_t u = begin; u < end;) {
      const Segment sg = segment_at(u, end, args.k_blocks, begin);
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
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;

      const int64_t n = (int64_t)sg.tile * kRowsPerTile + row;
      if (sg.kb0 == 0 && sg.kb1 == args.k_blocks) {
        // The whole K range of this tile is ours: write C directly.
        if (n < args.N) {
#pragma unroll
          for (int m = 0; m < kSplitKMaxM; ++m)
            if (m < args.M) store_out(args.C, (int64_t)m * args.N + n, v[m], out_bf16);
        }
      } else {
        // Take a ticket first.  The last contributor keeps its own values in
        // registers and adds the others' published partials to them; every other
        // contributor publishes its partial and bumps the publication count.  The
        // sum runs over the contributors in K order whoever arrives last.
        const int64_t u_first = (int64_t)sg.tile * args.k_blocks;
        const int64_t u_last = u_first + args.k_blocks - 1;
        const int64_t c_first = splitk_owner(u_first, args.units, G);
        const int64_t c_last = splitk_owner(u_last, args.units, G);
        const int32_t others = (int32_t)(c_last - c_first);
        int32_t* const arrivals = args.tickets + sg.tile;
        int32_t* const pubs = args.tickets + args.n_tiles + sg.tile;
        if (threadIdx.x == 64) *ticket_slot = atomicAdd(arrivals, 1);
        named_bar_sync(1, 128);
        const int32_t ticket = *ticket_slot;
        named_bar_sync(1, 128);
        if (ticket != others) {
          const int slot = sg.first ? 0 : 1;
          float* mine = partials + (((int64_t)c * 2 + slot) * kRowsPerTile + row) * mma_n;
#pragma unroll
          for (int j = 0; j < kSplitKMaxM / 4; ++j)
            if (j * 4 < mma_n)
              reinterpret_cast<float4*>(mine)[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
          named_bar_sync(1, 128);  // every row of the partial is written ...
          if (threadIdx.x == 64) red_add_release_gpu(pubs, 1);  // ... before it is published
        } else {
          if (threadIdx.x == 64) {
            const bool all_in = wait_counter_geq(pubs, others, ctl);
            if (!all_in) sk_report(args.status, kRoleEpilogue, abort_flag);
            *ticket_slot = all_in ? 1 : 0;
          }
          named_bar_sync(1, 128);  // the acquire above orders the partial reads below
          const bool have_all = *ticket_slot != 0;
          float s[kSplitKMaxM];
#pragma unroll
          for (int m = 0; m < kSplitKMaxM; ++m) s[m] = 0.0f;
          for (int64_t cc = c_first; cc <= c_last; ++cc) {
            if (cc == c) {
#pragma unroll
              for (int m = 0; m < kSplitKMaxM; ++m) s[m] += v[m];
            } else if (have_all) {
              const int64_t cc_first_tile = splitk_begin(cc, args.units, G) / args.k_blocks;
              const int cslot = (cc_first_tile == sg.tile) ? 0 : 1;
              const float4* src =
                  reinterpret_cast<const float4*>(partials + ((cc * 2 + cslot) * kRowsPerTile + row) * mma_n);
#pragma unroll
              for (int j = 0; j < kSplitKMaxM / 4; ++j) {
                if (j * 4 < mma_n) {
                  const float4 f = __ldcg(src + j);
                  s[4 * j] += f.x;
                  s[4 * j + 1] += f.y;
                  s[4 * j + 2] += f.z;
                  s[4 * j + 3] += f.w;
                }
              }
            }
          }
          if (n < args.N) {
#pragma unroll
            for (int m = 0; m < kSplitKMaxM; ++m)
              if (m < args.M) store_out(args.C, (int64_t)m * args.N + n, s[m], out_bf16);
          }
          if (threadIdx.x == 64) {  // ready for the next launch
            *arrivals = 0;
            *pubs = 0;
          }
        }
        named_bar_sync(1, 128);  // ticket_slot is reused by the next segment
      }
      if (threadIdx.x == 64) trace_event(tb, kRoleEpilogue, kTraceItemEnd, sg.tile, sg.kb1);
      u += sg.kb1 - sg.kb0;
    }
    if (!ok && lane == 0) sk_report(args.status, kRoleEpilogue, abort_flag);
  }

  if (threadIdx.x == 0) trace_event(tb, 0, kTraceKernelEnd, -1, (int32_t)(clock64() & 0x7fffffff));
  __syncthreads();
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
