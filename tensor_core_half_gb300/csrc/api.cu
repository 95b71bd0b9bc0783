// api.cu -- the C ABI declared in include/hgemm.h: argument validation, launch
// planning, TMA tensor-map encoding and kernel dispatch (host code).
//
// Tensor maps follow "tcgen05 for dummies: a B200 GEMM from scratch"
// (translated), section "TMA and mbarrier" (cuTensorMapEncodeTiled, dims and
// strides innermost first, strides in bytes) and section "128-byte global
// loads and swizzle" (64-element inner box with CU_TENSOR_MAP_SWIZZLE_128B).
// The driver entry point is fetched through the runtime, so the library has no
// link-time dependency on the driver and loads on machines without a GPU.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <mutex>
#include <new>

#include "../../include/hgemm.h"
#include "desc.cuh"
#include "kernels.h"
#include "sched.cuh"

using namespace hg;

namespace {

constexpr int32_t kVersion = 100;
constexpr int kDefaultGroupM = 8;
constexpr int64_t kWholeABytes = 32ll << 20;  // A up to this size is read from HBM once (one group)
constexpr int kDefaultSmemOptin = 232448;  // 227 KiB, sm_100-class parts
constexpr int64_t kMaxDim = 2147483647;

struct Ctx {
  int device = 0;
  int sm_count = 0;
  int smem_optin = 0;
  int32_t* status = nullptr;  // device status word
  float* partials = nullptr;  // split-K fp32 partial sums
  size_t partials_bytes = 0;
  int32_t* tickets = nullptr;  // split-K per-tile tickets, all zero between launches
  size_t ticket_count = 0;
  bool tickets_dirty = false;  // a launch gave up and may have left tickets behind
  int force_variant = HGEMM_VARIANT_AUTO;
  uint64_t timeout_ns = kDefaultTimeoutNs;
  int inject = 0;
  int group_m = 0;  // 0: auto_group_m
  int max_ctas = 0;
  int stream_k = 1;  // 0 never, 1 when the estimate says so, 2 whenever the tile count leaves a partial wave
  int schedule = HGEMM_SCHEDULE_STATIC;
  int epilogue = HGEMM_EPILOGUE_TMA_STORE;
  bool checks = false;
  TraceBuf* trace = nullptr;  // device trace buffer (HGEMM_OPT_TRACE)
  int64_t trace_capacity = 0;
  bool trace_items = true;  // HGEMM_OPT_TRACE_ITEMS: false keeps only the kernel begin/end records
  // hgemm_run_host: two staging sets (double buffering across calls), three
  // internal streams and the events that chain them.
  struct HostStage {
    void* A = nullptr;
    void* B = nullptr;
    void* C = nullptr;
    size_t a_cap = 0, b_cap = 0, c_cap = 0;
    cudaEvent_t ev_free = nullptr;  // recorded when the last copy out of this set is done
    cudaEvent_t ev_a[8] = {};       // chunk i of A (and all of B) is on the device
    cudaEvent_t ev_c[8] = {};       // chunk i of C is computed
    bool used = false;
  } stage[2];
  int stage_next = 0;
  cudaStream_t s_h2d = nullptr, s_compute = nullptr, s_d2h = nullptr;
  cudaEvent_t ev_entry = nullptr, ev_done = nullptr;
  int capacity[kNumDenseKinds] = {};  // resident clusters per dense kind
  int splitk_prepared_smem = 0;
};

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

void load_encode() {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
}

bool valid_dtype(int d) { return d == HGEMM_F16 || d == HGEMM_BF16 || d == HGEMM_F32; }

// Test-only pin of the variant for every new handle: HGEMM_FORCE_VARIANT =
// auto | 1sm128 | 1sm256 | 2sm256 | splitk | 2sm192, or the hgemm_variant_t
// number.  Unset or unrecognised: automatic choice (HGEMM_VARIANT_AUTO).
int env_force_variant() {
  const char* v = getenv("HGEMM_FORCE_VARIANT");
  if (v == nullptr || *v == 0) return HGEMM_VARIANT_AUTO;
  static const struct { const char* name; int id; } names[] = {
      {"auto", HGEMM_VARIANT_AUTO},        {"1sm128", HGEMM_VARIANT_1SM_128x128}, {"1sm256", HGEMM_VARIANT_1SM_128x256},
      {"2sm256", HGEMM_VARIANT_2SM_256x256}, {"splitk", HGEMM_VARIANT_SPLITK},    {"2sm192", HGEMM_VARIANT_2SM_256x192}};
  for (const auto& n : names)
    if (strcmp(v, n.name) == 0) return n.id;
  if (v[0] >= '0' && v[0] <= '5' && v[1] == 0) return v[0] - '0';
  return HGEMM_VARIANT_AUTO;
}

// Checks that do not involve pointers.  Order: sizes, enums, combinations, pitches.
hgemm_status_t check_problem(int64_t M, int64_t N, int64_t K, int layout, int in, int acc, int out) {
  if (M < 0 || N < 0 || K < 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim) return HGEMM_ERR_INVALID_ARG;
  // Tile counts are 32-bit in the plans and on the device: the smallest tile
  // (128 x 128) must leave them in range (each factor is below 2^24 here, so
  // the product cannot overflow 64 bits).
  if (((M + 127) / 128) * ((N + 127) / 128) > (int64_t)INT32_MAX) return HGEMM_ERR_INVALID_ARG;
  if (layout != HGEMM_LAYOUT_TN && layout != HGEMM_LAYOUT_NN) return HGEMM_ERR_INVALID_ARG;
  if (!valid_dtype(in) || !valid_dtype(acc) || !valid_dtype(out)) return HGEMM_ERR_INVALID_ARG;
  if (in == HGEMM_F32 || out == HGEMM_F32) return HGEMM_ERR_UNSUPPORTED;
  if (acc == HGEMM_BF16) return HGEMM_ERR_UNSUPPORTED;
  if (acc == HGEMM_F16 && in != HGEMM_F16) return HGEMM_ERR_UNSUPPORTED;
  if (M == 0 || N == 0) return HGEMM_OK;
  if (N % 8 != 0) return HGEMM_ERR_MISALIGNED;           // C (and NN B) row pitch
  if (K > 0 && K % 8 != 0) return HGEMM_ERR_MISALIGNED;  // A (and TN B) row pitch
  return HGEMM_OK;
}

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

DenseKind kind_of(int variant) {
  switch (variant) {
    case HGEMM_VARIANT_1SM_128x128: return kDense1Sm128;
    case HGEMM_VARIANT_1SM_128x256: return kDense1Sm256;
    case HGEMM_VARIANT_2SM_256x192: return kDense2Sm192;
    default: return kDense2Sm256;
  }
}

int variant_of(DenseKind k) {
  switch (k) {
    case kDense1Sm128: return HGEMM_VARIANT_1SM_128x128;
    case kDense1Sm256: return HGEMM_VARIANT_1SM_128x256;
    case kDense2Sm192: return HGEMM_VARIANT_2SM_256x192;
    default: return HGEMM_VARIANT_2SM_256x256;
  }
}

// A dense schedule: data-parallel tiles, then an optional stream-K range.
struct DenseChoice {
  double cost;        // estimated time in units of one full tile on one CTA pair
  int clusters;       // persistent clusters launched
  int dp_tiles;       // tiles computed whole
  int64_t sk_units;   // k-block units of the stream-K range
  int sk_ranges;      // stream-K work ids (0 without stream-K)
  int sk_pieces;      // 0: one equal range per cluster; p: each split tile cut into p equal K pieces
};

// Data-parallel: ceil(T / P) rounds of whole tiles.  Stream-K: the remainder
// (T mod P tiles) is cut into equal k-block ranges over the P clusters, so the
// time is T / P tiles plus the fix-up of the split tiles, which costs about 30
// k-blocks of mainloop time per cluster (measured on GB300 with the kernel's
// event trace: publishing or reducing a 256 x 256 fp32 partial).  When the
// remainder is under P / 4 tiles, each of them would be cut among more than
// four clusters; the last full round then joins the split, so that each split
// tile has one or two contributors.  (Measured: splitting the remainder alone
// equals the wider split at 4096^3 and beats it by 1-2 % at 8192^3 and
// 8192 x 8192 x 16384, with single launches 1.5-4 % faster: fewer tiles are
// split, so less partial traffic and fewer work items per cluster.)
DenseChoice dense_choice(DenseKind kind, int64_t M, int64_t N, int64_t K, int capacity, int max_ctas,
                         int allow_sk) {
  const DenseKindInfo info = dense_kind_info(kind);
  const int64_t tiles = cdiv(M, 128 * info.cta_group) * cdiv(N, info.block_n);
  const int64_t kb = cdiv(K, 64);
  int64_t P = capacity > 0 ? capacity : 1;
  if (max_ctas > 0) P = std::max<int64_t>(1, std::min<int64_t>(P, max_ctas / info.cta_group));
  DenseChoice dp{(double)cdiv(tiles, P), (int)std::min<int64_t>(tiles, P), (int)tiles, 0, 0, 0};
  DenseChoice best = dp;
  if (allow_sk && kb >= 2 && tiles % P != 0) {
    const int64_t waves = tiles / P;
    const int64_t rem = tiles - waves * P;
    DenseChoice sk;
    sk.dp_tiles = (int)(waves >= 1 ? (rem * 4 >= P ? waves : waves - 1) * P : 0);
    sk.sk_units = (tiles - sk.dp_tiles) * kb;
    sk.clusters = (int)std::min<int64_t>(P, sk.sk_units);
    sk.sk_ranges = sk.clusters;
    sk.sk_pieces = 0;
    sk.cost = (double)tiles / (double)sk.clusters + 30.0 / (double)kb;
    // K pieces: each of the rem leftover tiles is cut into p = P / rem equal
    // K pieces, one per cluster.  All pieces start together, the first
    // pieces of every split tile at k = 0, the second ones at k = kb / p, ...,
    // so the clusters walk K side by side and share each A and B line fetch
    // the way a wave of whole tiles does; equal ranges per cluster start at
    // scattered K offsets and fetch nearly every line alone.  The price: the
    // makespan is ceil(kb / p) instead of rem * kb / P k-blocks.
    // At most kMaxPieces contributors per split tile: every further one adds
    // a published fp32 partial to the tile's fix-up.
    DenseChoice pc{};
    constexpr int64_t kMaxPieces = 4;
    const int64_t pieces = rem > 0 ? std::min<int64_t>(std::min<int64_t>(P / rem, kb), kMaxPieces) : 0;
    if (pieces >= 2 || (allow_sk == 3 && kb >= 2)) {
      pc.sk_pieces = (int)std::max<int64_t>(2, pieces);
      pc.dp_tiles = (int)(waves * P);
      pc.sk_units = rem * kb;
      pc.sk_ranges = (int)(rem * pc.sk_pieces);
      pc.clusters = (int)std::min<int64_t>(P, std::max<int64_t>(pc.dp_tiles, pc.sk_ranges));
      // The fix-ups of split tiles run under the whole tiles' mainloops when
      // there are whole tiles; they still cost their partial traffic.
      pc.cost = (double)waves + (double)cdiv(kb, pc.sk_pieces) / (double)kb + (waves >= 1 ? 8.0 : 30.0) / (double)kb;
    }
    if (allow_sk == 2) {
      best = sk;
    } else if (allow_sk == 3) {
      best = pc.sk_pieces ? pc : sk;
    } else {
      if (sk.cost < best.cost) best = sk;
      if (pc.sk_pieces && pc.cost < best.cost) best = pc;
    }
  }
  // relative mainloop efficiency per tile area (2-SM 256-wide tiles are the reference)
  const double eff = (kind == kDense2Sm256) ? 1.0 : (kind == kDense2Sm192 ? 0.78 : (kind == kDense1Sm256 ? 0.85 : 0.70));
  best.cost *= (double)(128 * info.cta_group) * (double)info.block_n / (double)info.cta_group / eff;
  return best;
}

// Rasterisation group height when the caller sets none.  Tiles are visited
// in groups of group_m tile rows, down the rows of a group column by column,
// so a wave of clusters reads the A rows of one group and a few tile columns
// of B.  When all of A fits in 32 MiB, one group spans every tile row: A then
// stays in L2 and is read from HBM once, and the waves stream B once (4096^3
// bf16 on GB300: 96 MB of DRAM traffic per launch instead of 131 MB, and 0.6-
// 1.4 % faster, the lower DRAM power leaving the SMs a higher clock).  Larger
// A keeps 8 tile rows: from K = 8192 to 16384 (8192^3, 12288^3, 16384^3,
// 8192 x 8192 x 16384) heights of 4-5 measured 1-2 % slower and 16-32 up to
// 10 % slower, their extra DRAM traffic lowering the clock under the power
// limit.
int auto_group_m(int64_t M, int64_t K, int32_t tiles_m) {
  if (M * K * 2 <= kWholeABytes && tiles_m > kDefaultGroupM) return tiles_m;
  return kDefaultGroupM;
}

void fill_dense_plan(DenseKind kind, const DenseChoice& ch, int64_t M, int64_t N, int64_t K, int group_m,
                     hgemm_plan_t* p) {
  const DenseKindInfo info = dense_kind_info(kind);
  p->variant = variant_of(kind);
  p->cta_group = info.cta_group;
  p->tile_m = 128 * info.cta_group;
  p->tile_n = info.block_n;
  p->block_k = 64;
  p->stages = info.stages;
  p->tiles_m = (int32_t)cdiv(M, p->tile_m);
  p->tiles_n = (int32_t)cdiv(N, p->tile_n);
  p->num_tiles = p->tiles_m * p->tiles_n;
  p->k_blocks = (int32_t)cdiv(K, 64);
  p->grid = ch.clusters * info.cta_group;
  p->group_m = group_m > 0 ? group_m : auto_group_m(M, K, p->tiles_m);
  p->smem_bytes = info.smem_bytes;
  p->tmem_cols = info.tmem_cols;
  p->dp_tiles = ch.dp_tiles;
  p->sk_units = ch.sk_units;
  p->stream_k = ch.sk_units > 0 ? 1 : 0;
  p->sk_ranges = p->stream_k ? ch.sk_ranges : 0;
  p->sk_pieces = p->stream_k ? ch.sk_pieces : 0;
  p->work_ids = p->sk_ranges + ch.dp_tiles;
  // partial slots: two per stream-K range (ranges may outnumber the clusters when pieces are forced)
  p->workspace_bytes =
      p->stream_k ? (int64_t)std::max(ch.clusters, ch.sk_ranges) * 2 * info.cta_group * info.block_n * 128 * 4 +
                        (int64_t)p->num_tiles * info.cta_group * 8
                  : 0;
}

hgemm_status_t make_plan(int64_t M, int64_t N, int64_t K, int layout, int in, int acc, int out, int num_sms,
                         int smem_optin, const int capacity_in[kNumDenseKinds], int variant, int group_m, int max_ctas,
                         int allow_sk, int schedule, hgemm_plan_t* p) {
  memset(p, 0, sizeof(*p));
  if (schedule != HGEMM_SCHEDULE_STATIC && schedule != HGEMM_SCHEDULE_DYNAMIC) return HGEMM_ERR_INVALID_ARG;
  p->schedule = schedule;
  hgemm_status_t st = check_problem(M, N, K, layout, in, acc, out);
  if (st != HGEMM_OK) return st;
  if (num_sms <= 0) return HGEMM_ERR_INVALID_ARG;
  if (variant < HGEMM_VARIANT_AUTO || variant > HGEMM_VARIANT_2SM_256x192) return HGEMM_ERR_INVALID_ARG;
  int capacity[kNumDenseKinds];
  for (int i = 0; i < kNumDenseKinds; ++i) {
    const DenseKindInfo info = dense_kind_info((DenseKind)i);
    capacity[i] = (capacity_in && capacity_in[i] > 0) ? capacity_in[i] : num_sms / info.cta_group;
  }
  const bool splitk_ok = (M >= 1 && M <= kSplitKMaxM && layout == HGEMM_LAYOUT_TN && acc == HGEMM_F32);
  if (variant == HGEMM_VARIANT_SPLITK && !splitk_ok) return HGEMM_ERR_UNSUPPORTED;
  if (M == 0 || N == 0 || K == 0) {
    p->variant = variant == HGEMM_VARIANT_AUTO ? HGEMM_VARIANT_1SM_128x128 : variant;
    p->group_m = group_m > 0 ? group_m : kDefaultGroupM;
    return HGEMM_OK;  // nothing or a zero fill to launch
  }
  if (variant == HGEMM_VARIANT_SPLITK || (variant == HGEMM_VARIANT_AUTO && splitk_ok)) {
    const int mma_n = (int)cdiv(M, 16) * 16;
    p->variant = HGEMM_VARIANT_SPLITK;
    p->cta_group = 1;
    p->tile_m = 128;
    p->tile_n = mma_n;
    p->block_k = kSplitKBlockK;
    const int optin = smem_optin > 0 ? smem_optin : kDefaultSmemOptin;
    p->tiles_m = (int32_t)cdiv(N, 128);
    p->tiles_n = 1;
    p->num_tiles = p->tiles_m;
    p->k_blocks = (int32_t)cdiv(K, kSplitKBlockK);
    const SplitKShape sh = splitk_shape(p->num_tiles, p->k_blocks, K, mma_n, num_sms, max_ctas, optin,
                                        allow_sk == 3 ? 2 : allow_sk,
                                        schedule == HGEMM_SCHEDULE_DYNAMIC);
    p->stages = sh.stages;
    p->grid = sh.ctas;
    p->group_m = 1;
    p->smem_bytes = sh.smem_bytes;
    p->tmem_cols = splitk_tmem_cols(mma_n);
    const SplitChunks ch = sh.chunks;
    p->splitk_chunks = (int32_t)ch.count();
    p->splitk_head_units = ch.head;
    p->splitk_align = ch.align;
    p->workspace_bytes = ch.align > 1 ? 0 : (int64_t)splitk_workspace_bytes(ch.count(), mma_n, p->num_tiles);
    return HGEMM_OK;
  }
  DenseKind kind = kDense2Sm256;
  DenseChoice choice{};
  if (variant != HGEMM_VARIANT_AUTO) {
    kind = kind_of(variant);
    if (layout == HGEMM_LAYOUT_NN && !dense_kind_allows_nn(kind)) return HGEMM_ERR_UNSUPPORTED;
    choice = dense_choice(kind, M, N, K, capacity[kind], max_ctas, allow_sk);
  } else {
    bool first = true;
    for (DenseKind k : {kDense2Sm256, kDense2Sm192, kDense1Sm256, kDense1Sm128}) {
      if (layout == HGEMM_LAYOUT_NN && !dense_kind_allows_nn(k)) continue;
      const DenseChoice c = dense_choice(k, M, N, K, capacity[k], max_ctas, allow_sk);
      if (first || c.cost < choice.cost) {
        choice = c;
        kind = k;
        first = false;
      }
    }
  }
  fill_dense_plan(kind, choice, M, N, K, group_m, p);
  return HGEMM_OK;
}

// L2 fetch size of a TMA miss.  With a row pitch that is a multiple of 128 B,
// each 128-byte box row is one L2 line and 256-byte promotion brings the next
// k-block's line along.  With any other pitch a box row straddles two lines,
// and promoting both to 256 B fetches bytes no box asks for: measured on
// GB300 at 1000 x 3000 x 4104 (pitch 8208 B), 27.4-27.5 us per launch with
// 128-byte, 64-byte or no promotion against 28.5 us with 256-byte; with
// aligned pitches (2048^3, 4096^3, 8192^3, 16 x 16384 x 8192) 256 B was as
// fast or faster.
CUtensorMapL2promotion l2_promotion(uint64_t row_pitch_bytes) {
  return (row_pitch_bytes % 128 == 0) ? CU_TENSOR_MAP_L2_PROMOTION_L2_256B : CU_TENSOR_MAP_L2_PROMOTION_L2_128B;
}

bool encode_2d(CUtensorMap* m, int dtype, const void* ptr, uint64_t inner, uint64_t outer, uint32_t box_inner,
               uint32_t box_outer) {
  if (!g_encode) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {inner * 2};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  const CUtensorMapDataType t =
      dtype == HGEMM_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  return g_encode(m, t, 2, const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, l2_promotion(inner * 2), CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

bool overlaps(uintptr_t a, size_t an, uintptr_t b, size_t bn) { return an > 0 && bn > 0 && a < b + bn && b < a + an; }

hgemm_status_t cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return HGEMM_OK;
  if (e == cudaErrorMemoryAllocation) return HGEMM_ERR_OOM;
  if (e == cudaErrorNoDevice || e == cudaErrorInsufficientDriver) return HGEMM_ERR_NO_DEVICE;
  return HGEMM_ERR_CUDA;
}

bool stream_capturing(cudaStream_t s) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  return cudaStreamIsCapturing(s, &cs) == cudaSuccess && cs != cudaStreamCaptureStatusNone;
}

// Partial sums and tickets shared by split-K and stream-K launches of a handle.
// While `s` is being captured into a CUDA graph nothing may be allocated or
// freed: a workspace that would have to grow is refused (UNSUPPORTED).
hgemm_status_t ensure_workspace(Ctx* c, size_t partial_bytes, size_t n_tiles, cudaStream_t s) {
  if ((c->partials_bytes < partial_bytes || c->ticket_count < n_tiles) && stream_capturing(s))
    return HGEMM_ERR_UNSUPPORTED;
  if (c->partials_bytes < partial_bytes) {
    if (c->partials) cudaFree(c->partials);
    c->partials = nullptr;
    c->partials_bytes = 0;
    if (cudaMalloc(reinterpret_cast<void**>(&c->partials), partial_bytes) != cudaSuccess) return HGEMM_ERR_OOM;
    c->partials_bytes = partial_bytes;
  }
  if (c->ticket_count < n_tiles) {
    if (c->tickets) cudaFree(c->tickets);
    c->tickets = nullptr;
    c->ticket_count = 0;
    const size_t count = (n_tiles + 3) & ~(size_t)3;  // whole 16-byte groups for the zero fill
    if (cudaMalloc(reinterpret_cast<void**>(&c->tickets), count * sizeof(int32_t)) != cudaSuccess)
      return HGEMM_ERR_OOM;
    c->ticket_count = count;
    c->tickets_dirty = true;
  }
  if (c->tickets_dirty) {
    cudaError_t e = fill_zero_launch(c->tickets, c->ticket_count * sizeof(int32_t), s);
    if (e != cudaSuccess) return cuda_status(e);
    c->tickets_dirty = false;
  }
  return HGEMM_OK;
}

// HGEMM_OPT_INJECT_FAULT = 2 (tests): fill the fix-up ticket counters with
// 0x01 bytes, so every ticket is far past its tile's contributor count.  The
// kernels only compare tickets, so nothing is accessed out of range and no
// wait depends on them; HGEMM_OPT_CHECKS reports HGEMM_ERR_CHECK.  The next
// launch zeroes the counters again.
hgemm_status_t inject_ticket_fault(Ctx* c, cudaStream_t s) {
  if (c->inject != 2) return HGEMM_OK;
  c->tickets_dirty = true;
  return cuda_status(cudaMemsetAsync(c->tickets, 0x01, c->ticket_count * sizeof(int32_t), s));
}

}  // namespace

struct hgemm_ctx : Ctx {};

extern "C" {

const char* hgemm_status_string(hgemm_status_t s) {
  switch (s) {
    case HGEMM_OK: return "HGEMM_OK";
    case HGEMM_ERR_INVALID_ARG: return "HGEMM_ERR_INVALID_ARG: invalid argument";
    case HGEMM_ERR_UNSUPPORTED: return "HGEMM_ERR_UNSUPPORTED: unsupported combination or device";
    case HGEMM_ERR_MISALIGNED: return "HGEMM_ERR_MISALIGNED: pointer or row pitch not 16-byte aligned";
    case HGEMM_ERR_ALIAS: return "HGEMM_ERR_ALIAS: C overlaps A or B";
    case HGEMM_ERR_NO_DEVICE: return "HGEMM_ERR_NO_DEVICE: no usable CUDA device";
    case HGEMM_ERR_CUDA: return "HGEMM_ERR_CUDA: a CUDA call failed";
    case HGEMM_ERR_TIMEOUT: return "HGEMM_ERR_TIMEOUT: a device-side wait gave up";
    case HGEMM_ERR_OOM: return "HGEMM_ERR_OOM: device allocation failed";
    case HGEMM_ERR_CHECK: return "HGEMM_ERR_CHECK: a device-side invariant check failed";
  }
  return "unknown hgemm status";
}

int32_t hgemm_version(void) { return kVersion; }

uint32_t hgemm_encode_idesc(int32_t mma_m, int32_t mma_n, hgemm_dtype_t in_dtype, hgemm_dtype_t acc_dtype,
                            int32_t a_mn_major, int32_t b_mn_major) {
  return make_idesc(mma_m, mma_n, in_dtype == HGEMM_BF16, acc_dtype == HGEMM_F32, a_mn_major != 0, b_mn_major != 0);
}

uint64_t hgemm_encode_smem_desc(uint32_t smem_addr, uint32_t lbo_bytes, uint32_t sbo_bytes, int32_t swizzle_mode) {
  return make_smem_desc(smem_addr, lbo_bytes, sbo_bytes, swizzle_mode);
}

hgemm_status_t hgemm_plan_ex(int64_t M, int64_t N, int64_t K, hgemm_layout_t layout, hgemm_dtype_t in_dtype,
                             hgemm_dtype_t acc_dtype, hgemm_dtype_t out_dtype, int32_t num_sms, int32_t variant,
                             int32_t group_m, int32_t stream_k, int32_t schedule, hgemm_plan_t* plan) {
  if (!plan || group_m < 0 || stream_k < 0 || stream_k > 3) return HGEMM_ERR_INVALID_ARG;
  return make_plan(M, N, K, layout, in_dtype, acc_dtype, out_dtype, num_sms, kDefaultSmemOptin, nullptr, variant,
                   group_m, 0, stream_k, schedule, plan);
}

hgemm_status_t hgemm_plan(int64_t M, int64_t N, int64_t K, hgemm_layout_t layout, hgemm_dtype_t in_dtype,
                          hgemm_dtype_t acc_dtype, hgemm_dtype_t out_dtype, int32_t num_sms, int32_t variant,
                          int32_t group_m, int32_t stream_k, hgemm_plan_t* plan) {
  return hgemm_plan_ex(M, N, K, layout, in_dtype, acc_dtype, out_dtype, num_sms, variant, group_m, stream_k,
                       HGEMM_SCHEDULE_STATIC, plan);
}

hgemm_status_t hgemm_plan_work_item(const hgemm_plan_t* plan, int32_t cluster, int32_t index, int32_t* tile,
                                    int32_t* kb0, int32_t* kb1, int32_t* slot) {
  if (!plan || !tile || !kb0 || !kb1 || !slot || plan->variant == HGEMM_VARIANT_SPLITK || plan->cta_group < 1 ||
      index < 0)
    return HGEMM_ERR_INVALID_ARG;
  const int32_t nclusters = plan->grid / plan->cta_group;
  if (cluster < 0 || cluster >= nclusters) return HGEMM_ERR_INVALID_ARG;
  WorkIter it(plan->sk_ranges, plan->dp_tiles, plan->sk_units, plan->k_blocks);
  it.start_static(cluster, nclusters);
  WorkItem w;
  for (int32_t i = 0; i <= index; ++i)
    if (!it.next_static(w)) return HGEMM_ERR_INVALID_ARG;
  *tile = w.tile;
  *kb0 = w.kb0;
  *kb1 = w.kb1;
  *slot = w.slot;
  return HGEMM_OK;
}

hgemm_status_t hgemm_plan_id_item(const hgemm_plan_t* plan, int32_t id, int32_t index, int32_t* tile, int32_t* kb0,
                                  int32_t* kb1, int32_t* slot) {
  if (!plan || !tile || !kb0 || !kb1 || !slot || plan->variant == HGEMM_VARIANT_SPLITK || plan->cta_group < 1 ||
      index < 0 || id < 0 || id >= plan->work_ids)
    return HGEMM_ERR_INVALID_ARG;
  WorkIter it(plan->sk_ranges, plan->dp_tiles, plan->sk_units, plan->k_blocks);
  it.start(id);
  WorkItem w;
  for (int32_t i = 0; i <= index; ++i)
    if (!it.next_in_id(w)) return HGEMM_ERR_INVALID_ARG;
  *tile = w.tile;
  *kb0 = w.kb0;
  *kb1 = w.kb1;
  *slot = w.slot;
  return HGEMM_OK;
}

hgemm_status_t hgemm_plan_tile(const hgemm_plan_t* plan, int32_t t, int32_t* tile_m_idx, int32_t* tile_n_idx) {
  if (!plan || !tile_m_idx || !tile_n_idx || t < 0 || t >= plan->num_tiles || plan->group_m <= 0)
    return HGEMM_ERR_INVALID_ARG;
  const TileCoord c = tile_coord(t, plan->tiles_m, plan->tiles_n, plan->group_m);
  *tile_m_idx = c.m;
  *tile_n_idx = c.n;
  return HGEMM_OK;
}

hgemm_status_t hgemm_plan_splitk_range(const hgemm_plan_t* plan, int32_t chunk, int64_t* begin, int64_t* end) {
  if (!plan || !begin || !end || plan->variant != HGEMM_VARIANT_SPLITK || chunk < 0 || chunk >= plan->splitk_chunks)
    return HGEMM_ERR_INVALID_ARG;
  SplitChunks ch;
  ch.units = (int64_t)plan->num_tiles * plan->k_blocks;
  ch.head = plan->splitk_head_units;
  ch.big = plan->grid;
  ch.n_small = plan->splitk_chunks - plan->grid;
  ch.align = plan->splitk_align > 1 ? plan->splitk_align : 1;
  *begin = ch.begin(chunk);
  *end = ch.begin((int64_t)chunk + 1);
  return HGEMM_OK;
}

hgemm_status_t hgemm_plan_splitk_segment(const hgemm_plan_t* plan, int32_t chunk, int32_t index, int32_t* tile,
                                         int32_t* kb0, int32_t* kb1, int32_t* first) {
  int64_t b = 0, e = 0;
  if (!tile || !kb0 || !kb1 || !first || plan == nullptr || plan->k_blocks <= 0) return HGEMM_ERR_INVALID_ARG;
  const hgemm_status_t st = hgemm_plan_splitk_range(plan, chunk, &b, &e);
  if (st != HGEMM_OK) return st;
  ChunkSegments segs;
  segs.init(b, e, plan->k_blocks);
  if (index < 0 || index >= segs.count) return HGEMM_ERR_INVALID_ARG;
  const int32_t idx = segs.at(index);
  segs.get(idx, tile, kb0, kb1);
  *first = idx == 0 ? 1 : 0;
  return HGEMM_OK;
}

hgemm_status_t hgemm_create(hgemm_handle_t* out) {
  if (!out) return HGEMM_ERR_INVALID_ARG;
  *out = nullptr;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return HGEMM_ERR_NO_DEVICE;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return HGEMM_ERR_NO_DEVICE;
  if (major != 10 || minor != 3) return HGEMM_ERR_UNSUPPORTED;
  std::call_once(g_encode_once, load_encode);
  if (!g_encode) return HGEMM_ERR_NO_DEVICE;
  hgemm_ctx* c = new (std::nothrow) hgemm_ctx();
  if (!c) return HGEMM_ERR_OOM;
  c->device = dev;
  if (cudaDeviceGetAttribute(&c->sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&c->smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) {
    delete c;
    return HGEMM_ERR_CUDA;
  }
  e = cudaMalloc(&c->status, 16);
  if (e == cudaSuccess) e = cudaMemset(c->status, 0, 16);
  for (int k = 0; e == cudaSuccess && k < kNumDenseKinds; ++k) {
    e = dense_prepare((DenseKind)k);
    if (e == cudaSuccess) e = dense_max_active_clusters((DenseKind)k, &c->capacity[k]);
  }
  if (e == cudaSuccess) {
    e = splitk_prepare(c->smem_optin);
    c->splitk_prepared_smem = c->smem_optin;
  }
  if (e != cudaSuccess) {
    if (c->status) cudaFree(c->status);
    delete c;
    return cuda_status(e);
  }
  c->force_variant = env_force_variant();
  *out = c;
  return HGEMM_OK;
}

hgemm_status_t hgemm_destroy(hgemm_handle_t h) {
  if (!h) return HGEMM_OK;
  int prev = 0;
  cudaGetDevice(&prev);
  cudaSetDevice(h->device);
  cudaError_t e = cudaDeviceSynchronize();
  if (h->partials) cudaFree(h->partials);
  if (h->tickets) cudaFree(h->tickets);
  if (h->trace) cudaFree(h->trace);
  for (auto& st : h->stage) {
    if (st.A) cudaFree(st.A);
    if (st.B) cudaFree(st.B);
    if (st.C) cudaFree(st.C);
    if (st.ev_free) cudaEventDestroy(st.ev_free);
    for (int i = 0; i < 8; ++i) {
      if (st.ev_a[i]) cudaEventDestroy(st.ev_a[i]);
      if (st.ev_c[i]) cudaEventDestroy(st.ev_c[i]);
    }
  }
  if (h->s_h2d) cudaStreamDestroy(h->s_h2d);
  if (h->s_compute) cudaStreamDestroy(h->s_compute);
  if (h->s_d2h) cudaStreamDestroy(h->s_d2h);
  if (h->ev_entry) cudaEventDestroy(h->ev_entry);
  if (h->ev_done) cudaEventDestroy(h->ev_done);
  if (h->status) cudaFree(h->status);
  cudaSetDevice(prev);
  delete h;
  return e == cudaSuccess ? HGEMM_OK : HGEMM_ERR_CUDA;
}

hgemm_status_t hgemm_set_option(hgemm_handle_t h, int32_t option, int64_t value) {
  if (!h) return HGEMM_ERR_INVALID_ARG;
  switch (option) {
    case HGEMM_OPT_FORCE_VARIANT:
      if (value < HGEMM_VARIANT_AUTO || value > HGEMM_VARIANT_2SM_256x192) return HGEMM_ERR_INVALID_ARG;
      h->force_variant = (int)value;
      return HGEMM_OK;
    case HGEMM_OPT_TIMEOUT_NS:
      if (value <= 0) return HGEMM_ERR_INVALID_ARG;
      h->timeout_ns = (uint64_t)value;
      return HGEMM_OK;
    case HGEMM_OPT_INJECT_FAULT:
      if (value < 0 || value > 2) return HGEMM_ERR_INVALID_ARG;
      h->inject = (int)value;
      return HGEMM_OK;
    case HGEMM_OPT_GROUP_M:
      if (value < 0 || value > 65536) return HGEMM_ERR_INVALID_ARG;
      h->group_m = (int)value;
      return HGEMM_OK;
    case HGEMM_OPT_MAX_CTAS:
      if (value < 0 || value > 65536) return HGEMM_ERR_INVALID_ARG;
      h->max_ctas = (int)value;
      return HGEMM_OK;
    case HGEMM_OPT_STREAM_K:
      if (value < 0 || value > 3) return HGEMM_ERR_INVALID_ARG;
      h->stream_k = (int)value;
      return HGEMM_OK;
    case HGEMM_OPT_SCHEDULE:
      if (value != HGEMM_SCHEDULE_STATIC && value != HGEMM_SCHEDULE_DYNAMIC) return HGEMM_ERR_INVALID_ARG;
      h->schedule = (int)value;
      return HGEMM_OK;
    case HGEMM_OPT_CHECKS:
      if (value < 0 || value > 1) return HGEMM_ERR_INVALID_ARG;
      h->checks = value != 0;
      return HGEMM_OK;
    case HGEMM_OPT_TRACE_ITEMS:
      if (value < 0 || value > 1) return HGEMM_ERR_INVALID_ARG;
      h->trace_items = value != 0;
      return HGEMM_OK;
    case HGEMM_OPT_EPILOGUE:
      if (value != HGEMM_EPILOGUE_TMA_STORE && value != HGEMM_EPILOGUE_DIRECT) return HGEMM_ERR_INVALID_ARG;
      h->epilogue = (int)value;
      return HGEMM_OK;
    case HGEMM_OPT_TRACE: {
      if (value < 0 || value > (int64_t)1 << 26) return HGEMM_ERR_INVALID_ARG;
      if (h->trace) {
        cudaDeviceSynchronize();
        cudaFree(h->trace);
        h->trace = nullptr;
        h->trace_capacity = 0;
      }
      if (value == 0) return HGEMM_OK;
      const size_t bytes = sizeof(TraceBuf) + (size_t)value * sizeof(TraceRecord);
      if (cudaMalloc(reinterpret_cast<void**>(&h->trace), bytes) != cudaSuccess) {
        h->trace = nullptr;
        return HGEMM_ERR_OOM;
      }
      const unsigned long long head[2] = {0ull, (unsigned long long)value};
      if (cudaMemcpy(h->trace, head, sizeof(head), cudaMemcpyHostToDevice) != cudaSuccess) return HGEMM_ERR_CUDA;
      h->trace_capacity = value;
      return HGEMM_OK;
    }
  }
  return HGEMM_ERR_INVALID_ARG;
}

hgemm_status_t hgemm_run(hgemm_handle_t h, const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K,
                         hgemm_layout_t layout, hgemm_dtype_t in_dtype, hgemm_dtype_t acc_dtype,
                         hgemm_dtype_t out_dtype, void* stream) {
  if (!h) return HGEMM_ERR_INVALID_ARG;
  hgemm_status_t st = check_problem(M, N, K, layout, in_dtype, acc_dtype, out_dtype);
  if (st != HGEMM_OK) return st;
  if (M == 0 || N == 0) return HGEMM_OK;
  if (!C || (K > 0 && (!A || !B))) return HGEMM_ERR_INVALID_ARG;
  const uintptr_t a = reinterpret_cast<uintptr_t>(A), b = reinterpret_cast<uintptr_t>(B),
                  c = reinterpret_cast<uintptr_t>(C);
  if ((c & 15u) != 0 || (K > 0 && ((a & 15u) != 0 || (b & 15u) != 0))) return HGEMM_ERR_MISALIGNED;
  const size_t a_bytes = (size_t)M * (size_t)K * 2, b_bytes = (size_t)K * (size_t)N * 2,
               c_bytes = (size_t)M * (size_t)N * 2;
  if (overlaps(c, c_bytes, a, a_bytes) || overlaps(c, c_bytes, b, b_bytes)) return HGEMM_ERR_ALIAS;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (K == 0) return cuda_status(fill_zero_launch(C, c_bytes, s));

  hgemm_plan_t p;
  st = make_plan(M, N, K, layout, in_dtype, acc_dtype, out_dtype, h->sm_count, h->smem_optin, h->capacity,
                 h->force_variant, h->group_m, h->max_ctas, h->stream_k, h->schedule, &p);
  if (st != HGEMM_OK) return st;

  if (p.variant == HGEMM_VARIANT_SPLITK) {
    const int mma_n = p.tile_n;
    CUtensorMap tmW, tmX;
    if (!encode_2d(&tmW, in_dtype, B, (uint64_t)K, (uint64_t)N, 64, 128) ||
        !encode_2d(&tmX, in_dtype, A, (uint64_t)K, (uint64_t)M, 64, (uint32_t)mma_n))
      return HGEMM_ERR_CUDA;
    // Whole tiles need neither partials nor counters: no tile has a second contributor.
    const bool whole = p.splitk_align > 1;
    const size_t partial_bytes = whole ? 0 : (size_t)p.splitk_chunks * 2 * 128 * (size_t)mma_n * sizeof(float);
    st = ensure_workspace(h, partial_bytes, whole ? 0 : (size_t)p.num_tiles * kSplitKTicketStride, s);
    if (st != HGEMM_OK) return st;
    if ((st = inject_ticket_fault(h, s)) != HGEMM_OK) return st;
    if (p.smem_bytes > h->splitk_prepared_smem) return HGEMM_ERR_UNSUPPORTED;
    SplitKArgs args;
    args.M = (int32_t)M;
    args.N = (int32_t)N;
    args.K = (int32_t)K;
    args.mma_n = mma_n;
    args.n_tiles = p.num_tiles;
    args.k_blocks = p.k_blocks;
    args.units = (int64_t)p.num_tiles * p.k_blocks;
    args.head = p.splitk_head_units;
    args.big = p.grid;
    args.n_small = p.splitk_chunks - p.grid;
    args.align = p.splitk_align > 1 ? p.splitk_align : 1;
    args.dynamic = h->schedule == HGEMM_SCHEDULE_DYNAMIC ? 1 : 0;
    args.checks = h->checks ? 1 : 0;
    args.stages = p.stages;
    // the plan's shared memory beyond the ring holds this many prefetched partials
    args.pf_slots = (p.smem_bytes - splitk_smem_bytes(mma_n, p.stages, 0)) / (128 * mma_n * (int)sizeof(float));
    args.idesc = make_idesc(128, mma_n, in_dtype == HGEMM_BF16, true, false, false);
    args.out_bf16 = out_dtype == HGEMM_BF16;
    args.inject = h->inject;
    args.timeout_ns = h->timeout_ns;
    args.status = h->status;
    args.partials = h->partials;
    args.tickets = h->tickets;
    args.ticket_stride = kSplitKTicketStride;
    args.C = C;
    args.trace = h->trace;
    args.trace_items = h->trace_items ? 1 : 0;
    // Dynamic schedule: one CTA per chunk; the CTAs that run take over the rest.
    return cuda_status(splitk_launch(tmW, tmX, args, args.dynamic ? p.splitk_chunks : p.grid, p.smem_bytes, s));
  }

  const DenseKind kind = kind_of(p.variant);
  const DenseKindInfo info = dense_kind_info(kind);
  const bool nn = layout == HGEMM_LAYOUT_NN;
  CUtensorMap tmA, tmB, tmC;
  bool ok = encode_2d(&tmA, in_dtype, A, (uint64_t)K, (uint64_t)M, 64, 128);
  if (!nn)
    ok = ok && encode_2d(&tmB, in_dtype, B, (uint64_t)K, (uint64_t)N, 64, (uint32_t)(info.block_n / info.cta_group));
  else
    ok = ok && encode_2d(&tmB, in_dtype, B, (uint64_t)N, (uint64_t)K, 64, 64);
  ok = ok && encode_2d(&tmC, out_dtype, C, (uint64_t)N, (uint64_t)M, 64, 32);
  if (!ok) return HGEMM_ERR_CUDA;
  DenseArgs args;
  args.M = (int32_t)M;
  args.N = (int32_t)N;
  args.K = (int32_t)K;
  args.tiles_m = p.tiles_m;
  args.tiles_n = p.tiles_n;
  args.num_tiles = p.num_tiles;
  args.k_blocks = p.k_blocks;
  args.group_m = p.group_m;
  args.idesc = make_idesc(128 * info.cta_group, info.block_n, in_dtype == HGEMM_BF16, acc_dtype == HGEMM_F32, false, nn);
  args.b_mn_major = nn ? 1 : 0;
  args.acc_f16 = acc_dtype == HGEMM_F16;
  args.out_bf16 = out_dtype == HGEMM_BF16;
  args.inject = h->inject;
  args.timeout_ns = h->timeout_ns;
  args.status = h->status;
  args.trace = h->trace;
  args.trace_items = h->trace_items ? 1 : 0;
  args.dp_tiles = p.dp_tiles;
  args.sk_ranges = p.sk_ranges;
  args.sk_units = p.sk_units;
  args.dynamic = h->schedule == HGEMM_SCHEDULE_DYNAMIC ? 1 : 0;
  args.epi_direct = h->epilogue == HGEMM_EPILOGUE_DIRECT ? 1 : 0;
  args.checks = h->checks ? 1 : 0;
  args.C = C;
  args.partials = nullptr;
  args.tickets = nullptr;
  if (p.stream_k) {
    // two partial slots per stream-K range (the kernel indexes them by range id)
    const size_t ranges = (size_t)std::max(p.grid / info.cta_group, p.sk_ranges);
    const size_t partial_bytes = ranges * 2 * (size_t)info.cta_group * (size_t)info.block_n * 128 * sizeof(float);
    // two counters per tile and CTA of the pair: arrivals, then publications
    st = ensure_workspace(h, partial_bytes, (size_t)p.num_tiles * (size_t)info.cta_group * 2, s);
    if (st != HGEMM_OK) return st;
    if ((st = inject_ticket_fault(h, s)) != HGEMM_OK) return st;
    args.partials = h->partials;
    args.tickets = h->tickets;
  }
  // Dynamic schedule: one cluster per work id; the clusters that run first
  // take over the ids of those that have not started.
  const int grid = args.dynamic ? p.work_ids * info.cta_group : p.grid;
  return cuda_status(dense_launch(kind, tmA, tmB, tmC, args, grid, s));
}

namespace {

cudaError_t grow(void** p, size_t* cap, size_t need) {
  if (*cap >= need) return cudaSuccess;
  if (*p) {
    cudaError_t e = cudaFree(*p);
    *p = nullptr;
    *cap = 0;
    if (e != cudaSuccess) return e;
  }
  cudaError_t e = cudaMalloc(p, need);
  if (e == cudaSuccess) *cap = need;
  return e;
}

cudaError_t ensure_host_path(Ctx* c, Ctx::HostStage& st) {
  cudaError_t e = cudaSuccess;
  if (!c->s_h2d) e = cudaStreamCreateWithFlags(&c->s_h2d, cudaStreamNonBlocking);
  if (e == cudaSuccess && !c->s_compute) e = cudaStreamCreateWithFlags(&c->s_compute, cudaStreamNonBlocking);
  if (e == cudaSuccess && !c->s_d2h) e = cudaStreamCreateWithFlags(&c->s_d2h, cudaStreamNonBlocking);
  if (e == cudaSuccess && !c->ev_entry) e = cudaEventCreateWithFlags(&c->ev_entry, cudaEventDisableTiming);
  if (e == cudaSuccess && !c->ev_done) e = cudaEventCreateWithFlags(&c->ev_done, cudaEventDisableTiming);
  if (e == cudaSuccess && !st.ev_free) e = cudaEventCreateWithFlags(&st.ev_free, cudaEventDisableTiming);
  for (int i = 0; e == cudaSuccess && i < 8; ++i) {
    if (!st.ev_a[i]) e = cudaEventCreateWithFlags(&st.ev_a[i], cudaEventDisableTiming);
    if (e == cudaSuccess && !st.ev_c[i]) e = cudaEventCreateWithFlags(&st.ev_c[i], cudaEventDisableTiming);
  }
  return e;
}

}  // namespace

hgemm_status_t hgemm_run_host(hgemm_handle_t h, const void* A, const void* B, void* C, int64_t M, int64_t N,
                              int64_t K, hgemm_layout_t layout, hgemm_dtype_t in_dtype, hgemm_dtype_t acc_dtype,
                              hgemm_dtype_t out_dtype, void* stream) {
  if (!h) return HGEMM_ERR_INVALID_ARG;
  hgemm_status_t st = check_problem(M, N, K, layout, in_dtype, acc_dtype, out_dtype);
  if (st != HGEMM_OK) return st;
  if (M == 0 || N == 0) return HGEMM_OK;
  if (!C || (K > 0 && (!A || !B))) return HGEMM_ERR_INVALID_ARG;
  const size_t a_bytes = (size_t)M * (size_t)K * 2, b_bytes = (size_t)K * (size_t)N * 2,
               c_bytes = (size_t)M * (size_t)N * 2;
  const uintptr_t a = reinterpret_cast<uintptr_t>(A), b = reinterpret_cast<uintptr_t>(B),
                  c = reinterpret_cast<uintptr_t>(C);
  if (overlaps(c, c_bytes, a, K > 0 ? a_bytes : 0) || overlaps(c, c_bytes, b, K > 0 ? b_bytes : 0))
    return HGEMM_ERR_ALIAS;

  Ctx::HostStage& sg = h->stage[h->stage_next];
  cudaError_t e = ensure_host_path(h, sg);
  if (e != cudaSuccess) return cuda_status(e);
  // A set is reused two calls later: its previous copies out must be done
  // before its buffers are reallocated or overwritten.
  if (sg.used && (sg.a_cap < a_bytes || sg.b_cap < b_bytes || sg.c_cap < c_bytes)) {
    e = cudaEventSynchronize(sg.ev_free);
    if (e != cudaSuccess) return cuda_status(e);
  }
  if ((e = grow(&sg.A, &sg.a_cap, a_bytes > 0 ? a_bytes : 16)) != cudaSuccess ||
      (e = grow(&sg.B, &sg.b_cap, b_bytes > 0 ? b_bytes : 16)) != cudaSuccess ||
      (e = grow(&sg.C, &sg.c_cap, c_bytes)) != cudaSuccess)
    return e == cudaErrorMemoryAllocation ? HGEMM_ERR_OOM : cuda_status(e);

  // Row chunks of A and C: at least 1024 rows (whole 256-row tiles), at most
  // 4.  A chunk's GEMM must run at least as fast as the link delivers the
  // next chunk of A (about 840 TFLOPS at 4096 x 4096 and 205 GB/s); 512-row
  // chunks do not (measured 297 TFLOPS end to end at 4096^3 vs 306 with 4).
  int64_t rows = ((M + 3) / 4 + 255) / 256 * 256;
  if (rows < 1024) rows = 1024;
  const int nch = (int)((M + rows - 1) / rows);

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  char* Ad = static_cast<char*>(sg.A);
  char* Cd = static_cast<char*>(sg.C);
  const char* Ah = static_cast<const char*>(A);
  char* Ch = static_cast<char*>(C);
  // inputs go in after earlier work on the caller's stream and after the set is free
  if ((e = cudaEventRecord(h->ev_entry, s)) != cudaSuccess ||
      (e = cudaStreamWaitEvent(h->s_h2d, h->ev_entry, 0)) != cudaSuccess ||
      (sg.used && (e = cudaStreamWaitEvent(h->s_h2d, sg.ev_free, 0)) != cudaSuccess))
    return cuda_status(e);
  if (K > 0 && (e = cudaMemcpyAsync(sg.B, B, b_bytes, cudaMemcpyHostToDevice, h->s_h2d)) != cudaSuccess)
    return cuda_status(e);
  for (int i = 0; i < nch; ++i) {
    const int64_t r0 = i * rows, r1 = (r0 + rows < M) ? r0 + rows : M;
    if (K > 0 && (e = cudaMemcpyAsync(Ad + r0 * K * 2, Ah + r0 * K * 2, (size_t)(r1 - r0) * K * 2,
                                      cudaMemcpyHostToDevice, h->s_h2d)) != cudaSuccess)
      return cuda_status(e);
    if ((e = cudaEventRecord(sg.ev_a[i], h->s_h2d)) != cudaSuccess) return cuda_status(e);
  }
  for (int i = 0; i < nch; ++i) {
    const int64_t r0 = i * rows, r1 = (r0 + rows < M) ? r0 + rows : M;
    if ((e = cudaStreamWaitEvent(h->s_compute, sg.ev_a[i], 0)) != cudaSuccess) return cuda_status(e);
    st = hgemm_run(h, K > 0 ? Ad + r0 * K * 2 : nullptr, K > 0 ? sg.B : nullptr, Cd + r0 * N * 2, r1 - r0, N, K,
                   layout, in_dtype, acc_dtype, out_dtype, h->s_compute);
    if (st != HGEMM_OK) return st;
    if ((e = cudaEventRecord(sg.ev_c[i], h->s_compute)) != cudaSuccess) return cuda_status(e);
  }
  for (int i = 0; i < nch; ++i) {
    const int64_t r0 = i * rows, r1 = (r0 + rows < M) ? r0 + rows : M;
    if ((e = cudaStreamWaitEvent(h->s_d2h, sg.ev_c[i], 0)) != cudaSuccess ||
        (e = cudaMemcpyAsync(Ch + r0 * N * 2, Cd + r0 * N * 2, (size_t)(r1 - r0) * N * 2, cudaMemcpyDeviceToHost,
                             h->s_d2h)) != cudaSuccess)
      return cuda_status(e);
  }
  if ((e = cudaEventRecord(sg.ev_free, h->s_d2h)) != cudaSuccess ||
      (e = cudaEventRecord(h->ev_done, h->s_d2h)) != cudaSuccess ||
      (e = cudaStreamWaitEvent(s, h->ev_done, 0)) != cudaSuccess)
    return cuda_status(e);
  sg.used = true;
  h->stage_next ^= 1;
  return HGEMM_OK;
}

hgemm_status_t hgemm_trace_read(hgemm_handle_t h, hgemm_trace_record_t* out, int64_t capacity, int64_t* n_events) {
  static_assert(sizeof(hgemm_trace_record_t) == sizeof(TraceRecord), "trace record layout");
  if (!h || !h->trace || capacity < 0 || (capacity > 0 && !out) || !n_events) return HGEMM_ERR_INVALID_ARG;
  cudaError_t e = cudaDeviceSynchronize();
  unsigned long long count = 0;
  if (e == cudaSuccess) e = cudaMemcpy(&count, h->trace, sizeof(count), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_status(e);
  *n_events = (int64_t)count;
  int64_t n = (int64_t)count;
  if (n > h->trace_capacity) n = h->trace_capacity;
  if (n > capacity) n = capacity;
  if (n > 0) e = cudaMemcpy(out, h->trace->rec, (size_t)n * sizeof(TraceRecord), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemset(h->trace, 0, sizeof(unsigned long long));
  return cuda_status(e);
}

hgemm_status_t hgemm_sync_status(hgemm_handle_t h, void* stream, int32_t* detail) {
  if (!h) return HGEMM_ERR_INVALID_ARG;
  if (detail) *detail = 0;
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_status(e);
  int32_t word = 0;
  e = cudaMemcpy(&word, h->status, sizeof(word), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_status(e);
  if (detail) *detail = word;
  if (word == 0) return HGEMM_OK;
  e = cudaMemset(h->status, 0, sizeof(int32_t));
  if (e != cudaSuccess) return cuda_status(e);
  h->tickets_dirty = true;  // a split-K launch that gave up may leave tickets behind
  return (hgemm_status_t)(word & 0xFF);
}

}  // extern "C"
