// kernels.h -- internal interface between the C-ABI layer and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "sched.cuh"

namespace hg {

// Device status word layout (shared with hgemm_sync_status).
constexpr int32_t kStatusTimeout = 7;  // == HGEMM_ERR_TIMEOUT
constexpr int32_t kStatusCheck = 9;    // == HGEMM_ERR_CHECK
// Invariant checks (== hgemm_check_t)
enum CheckId : int32_t { kCheckWorkId = 1, kCheckItem = 2, kCheckTicket = 3, kCheckContributor = 4, kCheckPartial = 5 };
enum Role : int32_t { kRoleProducer = 1, kRoleMma = 2, kRoleEpilogue = 3, kRoleTeardown = 4 };

// Intra-kernel event trace (HGEMM_OPT_TRACE): a device buffer of fixed-size
// records appended with an atomic counter.  Kinds are listed in hgemm.h.
struct TraceRecord {
  uint64_t t_ns;     // %globaltimer
  uint32_t cta;      // blockIdx.x
  uint16_t role;     // Role
  uint16_t kind;     // event kind
  int32_t item;      // tile index (or -1)
  int32_t value;     // kind-specific (k-block range start, ticket, ...)
};
enum TraceKind : uint16_t {
  kTraceKernelBegin = 1,    // after setup (value: SM clock counter, low 31 bits)
  kTraceKernelEnd = 2,      // before teardown (value: SM clock counter, low 31 bits)
  kTraceItemBegin = 3,      // a role starts a work item (value: first k-block, or slot for the epilogue)
  kTraceItemEnd = 4,        // a role finishes it
  kTracePartialStored = 5,  // stream-K / split-K partial published (value: ticket drawn)
  kTraceReduced = 6,        // a split tile reduced and stored (value: contributors)
  kTraceStall = 7,          // SM cycles the role spent blocked on barriers during the item
};
struct TraceBuf {
  unsigned long long count;  // records requested (may exceed capacity)
  unsigned long long capacity;
  TraceRecord rec[1];
};

// Thread that records each CTA's kernel begin/end trace events: lane 0 of the
// first epilogue warp (both kernels run a producer warp, an MMA warp, then
// the epilogue warps).
constexpr int kStampThread = 64;

// Default limit of every bounded device-side wait.
constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;
// Limit used when draining in-flight copies after another role gave up.
constexpr uint64_t kDrainTimeoutNs = 2000000ull;

// ---------------------------------------------------------------- dense ----
struct DenseArgs {
  int32_t M, N, K;
  int32_t tiles_m, tiles_n, num_tiles, k_blocks, group_m;
  int32_t dp_tiles;   // tiles computed over the whole K range
  int32_t sk_ranges;  // stream-K ranges (work ids before the whole tiles); 0 without stream-K
  int64_t sk_units;   // (num_tiles - dp_tiles) * k_blocks, split evenly over the ranges
  int32_t dynamic;    // 1: one cluster per work id, ids taken over by cluster launch control
  int32_t epi_direct; // 1: the epilogue stores C from registers (16-byte stores), no TMA store
  int32_t checks;     // 1: check invariants, report violations as kStatusCheck
  void* C;            // [M][N] row-major output (used by the direct epilogue)
  float* partials;    // stream-K partials [sk_ranges][2][cta_group][BN/4][128] float4 (null if sk_units == 0)
  int32_t* tickets;  // [2][num_tiles * cta_group] arrivals, publications; all zero between launches
  uint32_t idesc;
  int32_t b_mn_major;      // NN layout: B tile is MN-major in shared memory
  int32_t acc_f16;         // fp16 accumulators in tensor memory (one per 32-bit column, low half)
  int32_t out_bf16;        // output dtype: 1 bf16, 0 fp16
  int32_t inject;          // test-only fault injection (HGEMM_OPT_INJECT_FAULT)
  uint64_t timeout_ns;
  int32_t* status;
  TraceBuf* trace;         // null unless tracing
  int32_t trace_items;     // 1: trace every event kind; 0: only each CTA's kernel begin/end
};

enum DenseKind : int { kDense1Sm128 = 0, kDense1Sm256 = 1, kDense2Sm256 = 2, kDense2Sm192 = 3 };
constexpr int kNumDenseKinds = 4;
// Kinds whose B slice per CTA is a whole number of 64-column boxes (NN layout).
inline bool dense_kind_allows_nn(DenseKind k) { return k != kDense2Sm192; }

struct DenseKindInfo {
  int cta_group, block_n, stages, smem_bytes, tmem_cols, threads;
};
DenseKindInfo dense_kind_info(DenseKind kind);

// Sets the kernel attributes (dynamic shared memory) on the current device.
cudaError_t dense_prepare(DenseKind kind);
// Number of CTA clusters of this kernel that fit on the device at once.
cudaError_t dense_max_active_clusters(DenseKind kind, int* clusters);
cudaError_t dense_launch(DenseKind kind, const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmC,
                         const DenseArgs& args, int grid_ctas, cudaStream_t stream);

// ---------------------------------------------------------------- split-K ----
struct SplitKArgs {
  int32_t M, N, K;
  int32_t mma_n;     // M rounded up to a multiple of 16 (the MMA's N)
  int32_t n_tiles;   // ceil(N / 128)
  int32_t k_blocks;  // ceil(K / kSplitKBlockK)
  int64_t units;     // n_tiles * k_blocks
  int64_t head;      // units covered by the first `big` chunks (all units under the static schedule)
  int32_t big;       // big chunks (= CTAs of the static schedule)
  int32_t n_small;   // small chunks after them (dynamic schedule), else 0
  int32_t align;     // big chunks cut in steps of this many units: k_blocks (whole tiles) or 1
  int32_t dynamic;   // 1: one CTA per chunk, chunks taken over by cluster launch control
  int32_t checks;    // 1: check invariants, report violations as kStatusCheck
  int32_t stages;
  int32_t pf_slots;  // partials that fit in the shared-memory prefetch area (splitk_pf_slots)
  uint32_t idesc;
  int32_t out_bf16;
  int32_t inject;
  uint64_t timeout_ns;
  int32_t* status;
  float* partials;   // [big + n_small chunks][2][128][mma_n] fp32
  int32_t* tickets;  // arrival counters, tile t's at tickets[t * ticket_stride]; all zero between launches
  int32_t ticket_stride;  // int32 words between counters: kSplitKTicketStride (one 128-byte line each), or 1
  void* C;           // [M][N] row-major
  TraceBuf* trace;   // null unless tracing
  int32_t trace_items;  // 1: trace every event kind; 0: only each CTA's kernel begin/end
};

constexpr int kSplitKMaxM = 64;
constexpr int kSplitKBlockK = 128;  // K per pipeline stage (and per work unit)
// Split-K arrival counters, one per 128-byte line: a counter is polled by its
// tile's last contributor while the others draw tickets on it, and counters
// packed 32 to a line made every such access queue behind those of 31 other
// tiles.
constexpr int kSplitKTicketStride = 32;
// The last contributor of a split tile copies up to this many other partials
// into shared memory ahead of its sum.
constexpr int kSplitKMaxPrefetch = 4;
int splitk_stage_bytes(int mma_n);
int splitk_pf_slots(int mma_n, int stages, int smem_optin);
int splitk_smem_bytes(int mma_n, int stages, int pf_slots);
int splitk_stages_for(int mma_n, int smem_optin, int most);

// How a skinny product is laid out over the CTAs (splitk_shape).
struct SplitKShape {
  SplitChunks chunks;  // the work ids; chunks.align > 1: whole tiles, no fix-up
  int32_t ctas;        // CTAs launched (static schedule) / running at most (dynamic)
  int32_t stages, pf_slots, smem_bytes;
};
// split_k: 0 never splits a tile's K range between CTAs, 2 always does, 1
// decides by the estimate in gemm_splitk.cu.  max_ctas > 0 caps the CTAs.
SplitKShape splitk_shape(int64_t tiles, int32_t k_blocks, int64_t K, int mma_n, int num_sms, int max_ctas,
                         int smem_optin, int split_k, bool dynamic);
int splitk_tmem_cols(int mma_n);
size_t splitk_workspace_bytes(int64_t chunks, int mma_n, int n_tiles);
cudaError_t splitk_prepare(int smem_bytes);
cudaError_t splitk_launch(const CUtensorMap& tmW, const CUtensorMap& tmX, const SplitKArgs& args, int grid,
                          int smem_bytes, cudaStream_t stream);

// ---------------------------------------------------------------- misc ----
cudaError_t fill_zero_launch(void* p, size_t bytes, cudaStream_t stream);

}  // namespace hg
