// noalloc.cu -- a skinny-M (split-K) entry point that allocates no device memory.
//
// Who needs it: callers that must not call cudaMalloc while they multiply.
// Examples are code running inside a caching allocator or an out-of-memory
// handler, a process whose device memory is all reserved by its own pool, and
// latency-critical loops that cannot absorb cudaMalloc's implicit device-wide
// synchronisation.  Such callers cannot create a handle (hgemm_create
// allocates a status word) and cannot let hgemm_run allocate or grow its
// split-K workspace.  hgemm_run_splitk_noalloc runs the same split-K kernel,
// but its scratch (partial sums, per-tile tickets, a status word) lives in a
// fixed array compiled into the library's device image.  Every GPU that loads
// the library holds that array until the process exits.
//
// The pages have no counterpart for this entry point; it is a deployment
// convenience around the split-K kernel.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/hgemm.h"
#include "desc.cuh"
#include "kernels.h"

namespace {

// Scratch layout: [status word | per-tile tickets | fp32 partial sums].
constexpr size_t kNoAllocScratchBytes = (size_t)16 << 20;  // 16 MiB
constexpr size_t kStatusBytes = 256;
// One arrival counter per N tile (the split-K kernel keeps no other per-tile
// state): 2 MiB holds 524,288 counters, so N <= 67,108,864.  Counters sit one
// per 128-byte line while that fits (up to 16,384 tiles), else packed.
constexpr size_t kTicketBytes = (size_t)2 << 20;
constexpr int64_t kMaxN = (int64_t)(kTicketBytes / sizeof(int32_t)) * 128;
constexpr size_t kPartialOffset = kStatusBytes + kTicketBytes;
constexpr size_t kPartialBytes = kNoAllocScratchBytes - kPartialOffset;
constexpr int kMaxDevices = 64;

}  // namespace

// The scratch itself.  In host code this name is only a stand-in for the
// device symbol; the device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {

struct DeviceSetup {
  std::mutex mu;
  bool done = false;  // set only by a set-up that succeeded; a failed one is retried by the next call
  hgemm_status_t status = HGEMM_ERR_NO_DEVICE;
  unsigned char* scratch = nullptr;  // device address of g_noalloc_scratch
  int sm_count = 0;
  int smem_optin = 0;
};

DeviceSetup g_devices[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_noalloc_encode = nullptr;
std::mutex g_noalloc_encode_mu;

void load_encode_fn() {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    g_noalloc_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
}

// Once per device, with that device current: find the scratch's device
// address, read the SM count, and set the split-K kernel's shared-memory limit.
void setup_device(DeviceSetup* d, int dev) {
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
    d->status = HGEMM_ERR_NO_DEVICE;
    return;
  }
  if (major != 10 || minor != 3) {
    d->status = HGEMM_ERR_UNSUPPORTED;
    return;
  }
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
    d->status = HGEMM_ERR_CUDA;
    return;
  }
  if (cudaDeviceGetAttribute(&d->sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&d->smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
      hg::splitk_prepare(d->smem_optin) != cudaSuccess) {
    d->status = HGEMM_ERR_CUDA;
    return;
  }
  d->scratch = static_cast<unsigned char*>(p);
  d->status = HGEMM_OK;
}

bool encode(CUtensorMap* m, int dtype, const void* ptr, uint64_t inner, uint64_t outer, uint32_t box_inner,
            uint32_t box_outer) {
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {inner * 2};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  const CUtensorMapDataType t =
      dtype == HGEMM_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  return g_noalloc_encode(m, t, 2, const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B,
                          (inner * 2) % 128 == 0 ? CU_TENSOR_MAP_L2_PROMOTION_L2_256B : CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool ranges_overlap(uintptr_t a, size_t an, uintptr_t b, size_t bn) {
  return an > 0 && bn > 0 && a < b + bn && b < a + an;
}

}  // namespace

extern "C" hgemm_status_t hgemm_run_splitk_noalloc(const void* A, const void* B, void* C, int64_t M, int64_t N,
                                                   int64_t K, hgemm_dtype_t in_dtype, hgemm_dtype_t out_dtype,
                                                   void* stream) {
  // Arguments first: nothing below touches the device until they are valid.
  if (M < 0 || N < 0 || K < 0 || M > 2147483647 || N > 2147483647 || K > 2147483647) return HGEMM_ERR_INVALID_ARG;
  if ((in_dtype != HGEMM_F16 && in_dtype != HGEMM_BF16 && in_dtype != HGEMM_F32) ||
      (out_dtype != HGEMM_F16 && out_dtype != HGEMM_BF16 && out_dtype != HGEMM_F32))
    return HGEMM_ERR_INVALID_ARG;
  if (in_dtype == HGEMM_F32 || out_dtype == HGEMM_F32) return HGEMM_ERR_UNSUPPORTED;
  if (M == 0 || N == 0) return HGEMM_OK;
  if (M > hg::kSplitKMaxM) return HGEMM_ERR_UNSUPPORTED;  // beyond the scratch layout's maximum
  if (N > kMaxN) return HGEMM_ERR_UNSUPPORTED;  // one ticket per 128-column tile must fit the ticket area
  const int64_t n_tiles = (N + 127) / 128;
  if (N % 8 != 0 || (K > 0 && K % 8 != 0)) return HGEMM_ERR_MISALIGNED;
  if (!C || (K > 0 && (!A || !B))) return HGEMM_ERR_INVALID_ARG;
  const uintptr_t a = reinterpret_cast<uintptr_t>(A), b = reinterpret_cast<uintptr_t>(B),
                  c = reinterpret_cast<uintptr_t>(C);
  if ((c & 15u) != 0 || (K > 0 && ((a & 15u) != 0 || (b & 15u) != 0))) return HGEMM_ERR_MISALIGNED;
  const size_t c_bytes = (size_t)M * (size_t)N * 2;
  if (ranges_overlap(c, c_bytes, a, (size_t)M * (size_t)K * 2) || ranges_overlap(c, c_bytes, b, (size_t)N * (size_t)K * 2))
    return HGEMM_ERR_ALIAS;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return HGEMM_ERR_NO_DEVICE;
  if (dev < 0 || dev >= kMaxDevices) return HGEMM_ERR_UNSUPPORTED;
  DeviceSetup* d = &g_devices[dev];
  {
    // Once per device, with that device current.  A set-up that failed (a
    // sticky error left by earlier work, say) is not remembered: the next call
    // tries again.
    std::lock_guard<std::mutex> lock(d->mu);
    if (!d->done) {
      setup_device(d, dev);
      d->done = d->status == HGEMM_OK;
    }
    if (!d->done) return d->status;
  }
  {
    std::lock_guard<std::mutex> lock(g_noalloc_encode_mu);
    if (!g_noalloc_encode) load_encode_fn();  // retried while it fails
    if (!g_noalloc_encode) return HGEMM_ERR_NO_DEVICE;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (K == 0) return hg::fill_zero_launch(C, c_bytes, s) == cudaSuccess ? HGEMM_OK : HGEMM_ERR_CUDA;

  // Plan: the same layout as hgemm_run's split-K variant (whole tiles or the
  // balanced split), with the CTA count capped so the partial sums fit the
  // scratch.
  const int mma_n = (int)((M + 15) / 16) * 16;
  const int64_t k_blocks = (K + hg::kSplitKBlockK - 1) / hg::kSplitKBlockK;
  const size_t per_cta = (size_t)2 * 128 * (size_t)mma_n * sizeof(float);
  const hg::SplitKShape sh = hg::splitk_shape(n_tiles, (int32_t)k_blocks, K, mma_n, d->sm_count,
                                              (int)(kPartialBytes / per_cta), d->smem_optin, 1, false);
  const int64_t units = n_tiles * k_blocks;
  const int64_t grid = sh.ctas;
  const int stages = sh.stages;
  const int pf_slots = sh.pf_slots;
  const int smem = sh.smem_bytes;

  CUtensorMap tmW, tmX;
  if (!encode(&tmW, in_dtype, B, (uint64_t)K, (uint64_t)N, 64, 128) ||
      !encode(&tmX, in_dtype, A, (uint64_t)K, (uint64_t)M, 64, (uint32_t)mma_n))
    return HGEMM_ERR_CUDA;

  // The array keeps whatever the previous call left: clear the status word and
  // the tickets this call uses (they must start at zero), on the same stream.
  // One counter per 128-byte line where they fit, else packed.
  const int32_t stride = ((size_t)n_tiles * hg::kSplitKTicketStride * sizeof(int32_t) <= kTicketBytes)
                             ? hg::kSplitKTicketStride
                             : 1;
  const size_t clear = (kStatusBytes + (size_t)n_tiles * stride * sizeof(int32_t) + 15) & ~(size_t)15;
  if (hg::fill_zero_launch(d->scratch, clear, s) != cudaSuccess) return HGEMM_ERR_CUDA;

  hg::SplitKArgs args;
  args.M = (int32_t)M;
  args.N = (int32_t)N;
  args.K = (int32_t)K;
  args.mma_n = mma_n;
  args.n_tiles = (int32_t)n_tiles;
  args.k_blocks = (int32_t)k_blocks;
  args.units = units;
  args.head = sh.chunks.head;  // static: one range per CTA
  args.big = (int32_t)grid;
  args.n_small = 0;
  args.align = sh.chunks.align;
  args.dynamic = 0;
  args.checks = 0;
  args.stages = stages;
  args.pf_slots = pf_slots;
  args.idesc = hg::make_idesc(128, mma_n, in_dtype == HGEMM_BF16, true, false, false);
  args.out_bf16 = out_dtype == HGEMM_BF16;
  args.inject = 0;
  args.timeout_ns = hg::kDefaultTimeoutNs;
  args.status = reinterpret_cast<int32_t*>(d->scratch);
  args.tickets = reinterpret_cast<int32_t*>(d->scratch + kStatusBytes);
  args.ticket_stride = stride;
  args.partials = reinterpret_cast<float*>(d->scratch + kPartialOffset);
  args.C = C;
  args.trace = nullptr;
  args.trace_items = 0;
  return hg::splitk_launch(tmW, tmX, args, (int)grid, smem, s) == cudaSuccess ? HGEMM_OK : HGEMM_ERR_CUDA;
}
