// tma_bench.cu -- micro-benchmark of the TMA engine: global -> shared copies.
//
// "tcgen05 for dummies: a B200 GEMM from scratch" (translated) measures its
// first kernels with 16-byte-wide TMA boxes, then with 128-byte-wide boxes and
// the 128-byte swizzle (2.7x faster), each in a 2-D form (several copies per
// tile) and a 3-D form (one copy per tile), and guesses that the TMA engine
// moves wide inner boxes faster; its section on the 128-byte swizzle asks for
// a TMA micro-benchmark to settle it.  This kernel is that benchmark: every
// CTA (one per SM) streams tiles of a bf16 matrix into a ring of shared-memory
// slots, one mbarrier per slot, and the host reports bytes per SM clock and
// aggregate bandwidth.  The copies are checked: after the last round every
// CTA sums the 16-bit words of what its slots hold (a sum does not depend on
// the swizzle or the box order in shared memory) and the caller compares the
// sums with its own over the same tiles.
//
// One tile is tile_rows x tile_cols elements, moved as
//   2D_16B  : tile_cols / 8 copies of a {8, tile_rows} box (16-byte rows)
//   3D_16B  : one copy of a {8, tile_rows, tile_cols / 8} box
//   2D_128B : tile_cols / 64 copies of a {64, tile_rows} box, 128-byte swizzle
//   3D_128B : one copy of a {64, tile_rows, tile_cols / 64} box, 128-byte swizzle
//   BULK    : one 1-D bulk copy of the tile's bytes (tiles stored contiguously)
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <mutex>
#include <vector>

#include "../../include/hgemm.h"
#include "kernels.h"
#include "ptx.cuh"

namespace hg {
namespace {

constexpr int kBenchThreads = 128;
constexpr int kMaxDepth = 16;

struct BenchArgs {
  int32_t mode, tile_rows, tile_cols, depth, issuers, iters, walk;
  int32_t tiles_y, tiles_x;  // tile grid over the source
  int32_t tile_bytes, copies;
  uint64_t timeout_ns;
  const uint8_t* src;  // BULK: tile t is bytes [t * tile_bytes, (t + 1) * tile_bytes)
  int32_t* status;
  long long* cycles;               // [ctas]
  unsigned long long* ns;          // [ctas]
  unsigned long long* sums;        // [ctas][2]: sum of words, sum of squared words
  int32_t* last_tiles;             // [ctas][depth]
};

// Tile that CTA `cta` loads in round j.  SCATTERED: neighbouring CTAs and
// rounds hit unrelated tiles.  ALONG_K: CTA c keeps one band of tile_rows rows
// (band c mod tiles_y) and walks it column tile by column tile, as a GEMM's
// producer walks K over the same rows of A.
__host__ __device__ inline int32_t bench_tile(int walk, int cta, int j, int tiles_y, int tiles_x) {
  if (walk == HGEMM_TMA_WALK_ALONG_K)
    return (int32_t)((cta % tiles_y) * tiles_x + ((cta / tiles_y) * 7 + j) % tiles_x);
  return (int32_t)(((int64_t)cta * 7919 + (int64_t)j * 13) % ((int64_t)tiles_y * tiles_x));
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* m, uint32_t bar, int32_t x, int32_t y,
                                            int32_t z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

__global__ void __launch_bounds__(kBenchThreads, 1)
    tma_bench_kernel(const __grid_constant__ CUtensorMap tm, const BenchArgs a) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bars[kMaxDepth];
  __shared__ uint32_t abort_flag;
  __shared__ unsigned long long red[2];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;  // 128-byte swizzle needs 1 KiB alignment
  const uint8_t* gbase = smem_raw + (base - raw);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    for (int i = 0; i < a.depth; ++i) mbar_init(smem_addr(&bars[i]), (uint32_t)a.issuers);
    abort_flag = 0u;
    red[0] = red[1] = 0ull;
    fence_mbar_init();
    prefetch_tmap(&tm);
  }
  __syncthreads();
  const WaitCtl ctl{a.timeout_ns, &abort_flag};
  const long long c0 = clock64();
  const uint64_t t0 = globaltimer_ns();
  bool ok = true;

  if (warp < a.issuers && lane == 0) {
    // This warp issues copies [cb, ce) of every tile.  The loop keeps only
    // counters (slot, phase, tile coordinates stepped in place): a division
    // or a 64-bit modulo per round costs the issuing thread hundreds of
    // cycles, which would be measured instead of the copy engine.
    const int cb = warp * a.copies / a.issuers, ce = (warp + 1) * a.copies / a.issuers;
    const uint32_t copy_bytes = (uint32_t)(a.tile_bytes / a.copies);
    const uint32_t mine = copy_bytes * (uint32_t)(ce - cb);
    const int32_t t0 = bench_tile(a.walk, blockIdx.x, 0, a.tiles_y, a.tiles_x);
    int32_t ty = t0 / a.tiles_x, tx = t0 % a.tiles_x;
    // SCATTERED: tile t + 13 (mod n_tiles) = 13 / tiles_x rows and 13 % tiles_x columns on.
    const int32_t step_y = (a.walk == HGEMM_TMA_WALK_ALONG_K) ? 0 : 13 / a.tiles_x;
    const int32_t step_x = (a.walk == HGEMM_TMA_WALK_ALONG_K) ? 1 : 13 % a.tiles_x;
    int slot = 0;
    uint32_t phase = 0;
    for (int j = 0; j < a.iters; ++j) {
      const uint32_t bar = smem_addr(&bars[slot]);
      if (j >= a.depth && !mbar_wait<false>(bar, phase ^ 1u, ctl)) {
        ok = false;
        break;
      }
      mbar_arrive_expect_tx(bar, mine);
      const uint32_t dst = base + (uint32_t)slot * (uint32_t)a.tile_bytes;
      const int32_t x0 = tx * a.tile_cols, y0 = ty * a.tile_rows;
      for (int c = cb; c < ce; ++c) {
        switch (a.mode) {
          case HGEMM_TMA_2D_16B:
            tma_load_2d(dst + (uint32_t)c * copy_bytes, &tm, bar, x0 + 8 * c, y0);
            break;
          case HGEMM_TMA_3D_16B:
            tma_load_3d(dst, &tm, bar, 0, y0, x0 / 8);
            break;
          case HGEMM_TMA_2D_128B:
            tma_load_2d(dst + (uint32_t)c * copy_bytes, &tm, bar, x0 + 64 * c, y0);
            break;
          case HGEMM_TMA_3D_128B:
            tma_load_3d(dst, &tm, bar, 0, y0, x0 / 64);
            break;
          default:  // HGEMM_TMA_BULK
            bulk_load(dst + (uint32_t)c * copy_bytes,
                      a.src + ((size_t)ty * a.tiles_x + tx) * a.tile_bytes + (size_t)c * copy_bytes, copy_bytes, bar);
            break;
        }
      }
      // next tile, in the order bench_tile gives
      tx += step_x;
      int32_t carry = 0;
      if (tx >= a.tiles_x) {
        tx -= a.tiles_x;
        carry = (a.walk == HGEMM_TMA_WALK_ALONG_K) ? 0 : 1;
      }
      ty += step_y + carry;
      while (ty >= a.tiles_y) ty -= a.tiles_y;  // at most 14 times: step_y + carry <= 14
      if (++slot == a.depth) {
        slot = 0;
        phase ^= 1u;
      }
    }
    if (!ok) {
      abort_flag = 1u;
      atomicCAS(a.status, 0, kStatusTimeout | (1 << 8) | ((int32_t)(blockIdx.x & 0xFFFF) << 16));
    }
  }
  // The other threads idle at this barrier rather than polling the slots'
  // barriers: lanes of the issuing warp that spin in try_wait take issue
  // slots from the issuing lane and slow every copy down.
  __syncthreads();
  // Every thread waits for the last round of every slot (bounded), then the
  // block sums what the slots hold.
  const int used = a.iters < a.depth ? a.iters : a.depth;
  for (int s = 0; s < used; ++s) {
    const int j_last = s + a.depth * ((a.iters - 1 - s) / a.depth);
    const WaitCtl end_ctl{a.timeout_ns, nullptr};
    if (!mbar_wait<false>(smem_addr(&bars[s]), (uint32_t)((j_last / a.depth) & 1), end_ctl)) ok = false;
  }
  const long long c1 = clock64();
  const uint64_t t1 = globaltimer_ns();
  if (__syncthreads_or(ok ? 0 : 1)) {
    if (threadIdx.x == 0) atomicCAS(a.status, 0, kStatusTimeout | (4 << 8) | ((int32_t)(blockIdx.x & 0xFFFF) << 16));
    return;
  }
  unsigned long long s1 = 0, s2 = 0;
  const int words = a.tile_bytes / 2;
  for (int s = 0; s < used; ++s) {
    const uint16_t* w = reinterpret_cast<const uint16_t*>(gbase + (size_t)s * a.tile_bytes);
    for (int i = threadIdx.x; i < words; i += kBenchThreads) {
      const unsigned long long v = w[i];
      s1 += v;
      s2 += v * v;
    }
  }
  atomicAdd(&red[0], s1);
  atomicAdd(&red[1], s2);
  __syncthreads();
  if (threadIdx.x == 0) {
    a.cycles[blockIdx.x] = c1 - c0;
    a.ns[blockIdx.x] = t1 - t0;
    a.sums[2 * blockIdx.x] = red[0];
    a.sums[2 * blockIdx.x + 1] = red[1];
    for (int s = 0; s < a.depth; ++s)
      a.last_tiles[blockIdx.x * a.depth + s] =
          s < used ? bench_tile(a.walk, blockIdx.x, s + a.depth * ((a.iters - 1 - s) / a.depth), a.tiles_y, a.tiles_x)
                   : -1;
  }
}

PFN_cuTensorMapEncodeTiled_v12000 g_bench_encode = nullptr;
std::once_flag g_bench_encode_once;

void load_bench_encode() {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    g_bench_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
}

hgemm_status_t status_of(cudaError_t e) {
  if (e == cudaSuccess) return HGEMM_OK;
  if (e == cudaErrorMemoryAllocation) return HGEMM_ERR_OOM;
  if (e == cudaErrorNoDevice || e == cudaErrorInsufficientDriver) return HGEMM_ERR_NO_DEVICE;
  return HGEMM_ERR_CUDA;
}

}  // namespace
}  // namespace hg

using namespace hg;

extern "C" hgemm_status_t hgemm_tma_bench(const void* src, int64_t height, int64_t width,
                                          const hgemm_tma_bench_config_t* cfg, hgemm_tma_bench_result_t* res,
                                          uint64_t* sums, int32_t* last_tiles, void* stream) {
  if (!cfg || !res || !src) return HGEMM_ERR_INVALID_ARG;
  const hgemm_tma_bench_config_t c = *cfg;
  const int R = c.tile_rows, C = c.tile_cols;
  if (c.mode < HGEMM_TMA_2D_16B || c.mode > HGEMM_TMA_BULK) return HGEMM_ERR_INVALID_ARG;
  if (R < 8 || R > 256 || R % 8 != 0 || C < 8 || C % 8 != 0) return HGEMM_ERR_INVALID_ARG;
  const bool wide = c.mode == HGEMM_TMA_2D_128B || c.mode == HGEMM_TMA_3D_128B;
  if (wide && C % 64 != 0) return HGEMM_ERR_INVALID_ARG;
  if (c.mode == HGEMM_TMA_3D_16B && C / 8 > 256) return HGEMM_ERR_INVALID_ARG;
  if (c.depth < 1 || c.depth > kMaxDepth || c.iters < 1 || c.issuers < 1 || c.issuers > 2 || c.ctas < 0 ||
      (c.walk != HGEMM_TMA_WALK_SCATTERED && c.walk != HGEMM_TMA_WALK_ALONG_K))
    return HGEMM_ERR_INVALID_ARG;
  if (height < R || width < C || height % R != 0 || width % C != 0 || width > ((int64_t)1 << 31) ||
      height > ((int64_t)1 << 31))
    return HGEMM_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(src) & 127u) != 0) return HGEMM_ERR_MISALIGNED;
  const int copies = c.mode == HGEMM_TMA_2D_16B ? C / 8 : (c.mode == HGEMM_TMA_2D_128B ? C / 64 : 1);
  if (c.issuers > copies) return HGEMM_ERR_INVALID_ARG;
  const int tile_bytes = R * C * 2;
  if (c.mode == HGEMM_TMA_BULK && tile_bytes % 16 != 0) return HGEMM_ERR_INVALID_ARG;

  int dev = 0, sms = 0, optin = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return HGEMM_ERR_NO_DEVICE;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return HGEMM_ERR_NO_DEVICE;
  if (major != 10 || minor != 3) return HGEMM_ERR_UNSUPPORTED;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
    return HGEMM_ERR_CUDA;
  const size_t smem = (size_t)c.depth * (size_t)tile_bytes + 1024;
  if (smem + 1024 > (size_t)optin) return HGEMM_ERR_UNSUPPORTED;  // static shared memory + slack
  const int ctas = c.ctas > 0 ? c.ctas : sms;
  std::call_once(g_bench_encode_once, load_bench_encode);
  if (!g_bench_encode) return HGEMM_ERR_NO_DEVICE;

  // The tensor map (unused by BULK, which still needs a valid one to pass).
  CUtensorMap tm;
  const CUtensorMapDataType bf16 = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult cr;
  if (c.mode == HGEMM_TMA_3D_16B || c.mode == HGEMM_TMA_3D_128B) {
    const cuuint64_t inner = wide ? 64 : 8;
    const cuuint64_t dims[3] = {inner, (cuuint64_t)height, (cuuint64_t)width / inner};
    const cuuint64_t strides[2] = {(cuuint64_t)width * 2, inner * 2};
    const cuuint32_t box[3] = {(cuuint32_t)inner, (cuuint32_t)R, (cuuint32_t)(C / inner)};
    cr = g_bench_encode(&tm, bf16, 3, const_cast<void*>(src), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        wide ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  } else {
    const cuuint32_t inner = (c.mode == HGEMM_TMA_2D_16B) ? 8 : 64;
    const cuuint64_t dims[2] = {(cuuint64_t)width, (cuuint64_t)height};
    const cuuint64_t strides[1] = {(cuuint64_t)width * 2};
    const cuuint32_t box[2] = {inner, (cuuint32_t)R};
    cr = g_bench_encode(&tm, bf16, 2, const_cast<void*>(src), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        c.mode == HGEMM_TMA_2D_128B ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  }
  if (cr != CUDA_SUCCESS) return HGEMM_ERR_CUDA;

  // Per-CTA outputs: cycles, ns, two sums, depth tile indices, and a status word.
  const size_t per = sizeof(long long) + sizeof(unsigned long long) + 2 * sizeof(unsigned long long) +
                     (size_t)c.depth * sizeof(int32_t);
  uint8_t* d = nullptr;
  cudaError_t e = cudaMalloc(&d, (size_t)ctas * per + 16);
  if (e != cudaSuccess) return status_of(e);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  BenchArgs a;
  a.mode = c.mode;
  a.tile_rows = R;
  a.tile_cols = C;
  a.depth = c.depth;
  a.issuers = c.issuers;
  a.iters = c.iters;
  a.walk = c.walk;
  a.tiles_y = (int32_t)(height / R);
  a.tiles_x = (int32_t)(width / C);
  a.tile_bytes = tile_bytes;
  a.copies = copies;
  a.timeout_ns = kDefaultTimeoutNs;
  a.src = static_cast<const uint8_t*>(src);
  a.cycles = reinterpret_cast<long long*>(d);
  a.ns = reinterpret_cast<unsigned long long*>(d + (size_t)ctas * 8);
  a.sums = reinterpret_cast<unsigned long long*>(d + (size_t)ctas * 16);
  a.last_tiles = reinterpret_cast<int32_t*>(d + (size_t)ctas * 32);
  a.status = reinterpret_cast<int32_t*>(d + (size_t)ctas * per);
  float ms = 0.0f;
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  e = cudaMemsetAsync(a.status, 0, 16, s);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(tma_bench_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e == cudaSuccess) e = cudaEventCreate(&e0);
  if (e == cudaSuccess) e = cudaEventCreate(&e1);
  if (e == cudaSuccess) e = cudaEventRecord(e0, s);
  if (e == cudaSuccess) {
    tma_bench_kernel<<<ctas, kBenchThreads, smem, s>>>(tm, a);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) e = cudaEventRecord(e1, s);
  if (e == cudaSuccess) e = cudaEventSynchronize(e1);
  if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, e0, e1);
  std::vector<long long> cyc(ctas);
  std::vector<unsigned long long> ns(ctas), sm(2 * (size_t)ctas);
  std::vector<int32_t> lt((size_t)ctas * c.depth);
  int32_t status = 0;
  if (e == cudaSuccess) e = cudaMemcpy(cyc.data(), a.cycles, (size_t)ctas * 8, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemcpy(ns.data(), a.ns, (size_t)ctas * 8, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemcpy(sm.data(), a.sums, (size_t)ctas * 16, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemcpy(lt.data(), a.last_tiles, lt.size() * 4, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemcpy(&status, a.status, 4, cudaMemcpyDeviceToHost);
  if (e0) cudaEventDestroy(e0);
  if (e1) cudaEventDestroy(e1);
  cudaFree(d);
  if (e != cudaSuccess) return status_of(e);
  if (status != 0) return (hgemm_status_t)(status & 0xFF);

  // Per-SM rate: each CTA's bytes over its own cycle count (median CTA).
  std::vector<double> rate(ctas), mhz(ctas);
  const double cta_bytes = (double)c.iters * tile_bytes;
  for (int i = 0; i < ctas; ++i) {
    rate[i] = cyc[i] > 0 ? cta_bytes / (double)cyc[i] : 0.0;
    mhz[i] = ns[i] > 0 ? (double)cyc[i] / (double)ns[i] * 1e3 : 0.0;
  }
  std::sort(rate.begin(), rate.end());
  std::sort(mhz.begin(), mhz.end());
  res->ms = ms;
  res->bytes = cta_bytes * ctas;
  res->gbs = ms > 0 ? res->bytes / ((double)ms * 1e-3) / 1e9 : 0.0;
  res->bytes_per_clk_sm = rate[ctas / 2];
  res->sm_mhz = mhz[ctas / 2];
  res->copies_per_tile = copies;
  res->ctas = ctas;
  res->tile_bytes = tile_bytes;
  res->reserved = 0;
  if (sums)
    for (size_t i = 0; i < sm.size(); ++i) sums[i] = sm[i];
  if (last_tiles)
    for (size_t i = 0; i < lt.size(); ++i) last_tiles[i] = lt[i];
  return HGEMM_OK;
}
