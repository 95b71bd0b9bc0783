/*
 * hgemm.h -- C ABI of a GB300 (sm_103a) dense half-precision matrix multiply
 *
 *     C[M,N] = A[M,K] . B[K,N]
 *
 * with fp16 or bf16 inputs, fp32 (or, for fp16 inputs, fp16) accumulation and
 * fp16 or bf16 output, computed by hand-written tcgen05 / TMA kernels.
 *
 * The operation is the plain matrix product of "tcgen05 for dummies: a B200
 * GEMM from scratch" (translated), section "Recap: how to write a fast matmul
 * kernel": every C[m][n] is the dot product of row m of A and column n of B.
 * Layout names follow "HGEMM: WMMA and MMA PTX study notes" (kernel header
 * comment): TN = A row-major, B column-major (stored as [N,K]), C row-major;
 * NN = A, B and C all row-major.
 *
 * Conventions shared by every entry point:
 *   - All pointers passed to hgemm_run are DEVICE pointers of the device that
 *     was current when the handle was created.  The caller owns them.
 *   - Matrices are dense and packed (no leading-dimension arguments).
 *   - A stream argument is a cudaStream_t passed as void* (0 = legacy default
 *     stream).  Work is enqueued on it; nothing blocks the host except
 *     hgemm_sync_status.
 *   - Every entry point returns an hgemm_status_t; argument errors are
 *     detected on the host before anything is launched and leave the device
 *     untouched.  There is no CPU fallback and no vendor GEMM library call.
 *   - A handle is not thread-safe: use one handle per host thread.
 */
#ifndef HGEMM_H_
#define HGEMM_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct hgemm_ctx* hgemm_handle_t;

typedef enum {
  HGEMM_OK = 0,
  HGEMM_ERR_INVALID_ARG = 1, /* null handle/pointer, negative size, bad enum, size too large */
  HGEMM_ERR_UNSUPPORTED = 2, /* valid combination this library does not implement, or not sm_103 */
  HGEMM_ERR_MISALIGNED = 3,  /* a base pointer is not 16-byte aligned, or a row pitch is not a
                                multiple of 16 bytes (K % 8 != 0 or N % 8 != 0) */
  HGEMM_ERR_ALIAS = 4,       /* C overlaps A or B */
  HGEMM_ERR_NO_DEVICE = 5,   /* no CUDA device / driver */
  HGEMM_ERR_CUDA = 6,        /* a CUDA runtime or driver call failed */
  HGEMM_ERR_TIMEOUT = 7,     /* a bounded device-side wait gave up (reported by hgemm_sync_status) */
  HGEMM_ERR_OOM = 8,         /* workspace allocation failed */
  HGEMM_ERR_CHECK = 9        /* a device-side invariant check failed (HGEMM_OPT_CHECKS; reported by
                                hgemm_sync_status, which gives the check's number in detail bits 8-15) */
} hgemm_status_t;

typedef enum { HGEMM_LAYOUT_TN = 0, HGEMM_LAYOUT_NN = 1 } hgemm_layout_t;

typedef enum { HGEMM_F16 = 0, HGEMM_BF16 = 1, HGEMM_F32 = 2 } hgemm_dtype_t;

/* Kernel variants (hgemm_plan / HGEMM_OPT_FORCE_VARIANT). */
typedef enum {
  HGEMM_VARIANT_AUTO = 0,
  HGEMM_VARIANT_1SM_128x128 = 1, /* persistent tcgen05, one CTA per 128x128 C tile          */
  HGEMM_VARIANT_1SM_128x256 = 2, /* persistent tcgen05, one CTA per 128x256 C tile          */
  HGEMM_VARIANT_2SM_256x256 = 3, /* persistent tcgen05 cta_group::2, a CTA pair per 256x256 */
  HGEMM_VARIANT_SPLITK = 4,      /* skinny M (TN, fp32 accumulate, M <= 64): swap-AB split-K */
  HGEMM_VARIANT_2SM_256x192 = 5  /* as 2SM_256x256 with 192-column tiles (TN only)            */
} hgemm_variant_t;

/* Handle options (hgemm_set_option). */
typedef enum {
  HGEMM_OPT_FORCE_VARIANT = 1, /* value: an hgemm_variant_t; AUTO restores automatic choice   */
  HGEMM_OPT_TIMEOUT_NS = 2,    /* value: limit of every device-side wait, ns (default 2e9)    */
  HGEMM_OPT_INJECT_FAULT = 3,  /* value: 0 off; 1 = the producers of the first CTA (both CTAs
                                  of a pair) drop their first stage, issuing no copy for it,
                                  so the consumer's bounded wait must give up; 2 = the
                                  host fills the fix-up ticket counters with 0x01 bytes before
                                  a stream-K or split-K launch, which HGEMM_OPT_CHECKS must
                                  report (tests)                                              */
  HGEMM_OPT_GROUP_M = 4,       /* value: rasterisation group height in tiles; 0 (default) =
                                  automatic: every tile row when all of A fits in 32 MiB
                                  (A then stays in L2), else 8                             */
  HGEMM_OPT_MAX_CTAS = 5,      /* value: cap on persistent CTAs (0 = one per SM)              */
  HGEMM_OPT_STREAM_K = 6,      /* value: 1 (default) lets the planner split the last wave of
                                  dense tiles along K (stream-K) when its estimate favours it;
                                  0 keeps every tile whole; 2 splits whenever the tile count
                                  leaves a partial wave, into one equal range per cluster; 3
                                  splits each leftover tile into equal K pieces (as many as
                                  fit the clusters, at least 2; else as 2).  Split-K (skinny
                                  M) plans likewise (3 acts as 2):
                                  1 chooses between whole tiles per CTA and the balanced
                                  K split over every SM by estimate, 0 always takes whole
                                  tiles, 2 always splits                                     */
  HGEMM_OPT_TRACE = 7,         /* value: capacity in events of a device trace buffer that the
                                  kernels append to (0 = off, the default); hgemm_trace_read */
  HGEMM_OPT_SCHEDULE = 8,      /* value: an hgemm_schedule_t for the dense kernels           */
  HGEMM_OPT_EPILOGUE = 9,      /* value: an hgemm_epilogue_t for the dense kernels           */
  HGEMM_OPT_CHECKS = 10,       /* value: 1 = the kernels check their invariants (work ids from
                                  launch control in range, work items and tiles in range,
                                  fix-up tickets not past the contributor count, partial
                                  slots in range) and report a violation as HGEMM_ERR_CHECK
                                  instead of trapping; 0 (default) = no checks              */
  HGEMM_OPT_TRACE_ITEMS = 11   /* value: 1 (default) = the trace (HGEMM_OPT_TRACE) records every
                                  event kind; 0 = only each CTA's kernel begin and end records,
                                  two per CTA per launch, whose SM cycle counter and global
                                  timer give the SM clock of every launch (both records are
                                  reserved by one atomic of a thread that is idle then, so no
                                  role of the kernel waits on the trace)                     */
} hgemm_option_t;

/* Check numbers reported with HGEMM_ERR_CHECK (detail bits 8-15). */
typedef enum {
  HGEMM_CHECK_WORK_ID = 1,     /* a work id or chunk from launch control out of range */
  HGEMM_CHECK_ITEM = 2,        /* a work item's tile or k-block range out of range    */
  HGEMM_CHECK_TICKET = 3,      /* a fix-up ticket past the tile's contributor count   */
  HGEMM_CHECK_CONTRIBUTOR = 4, /* the item's owner outside the tile's contributors    */
  HGEMM_CHECK_PARTIAL = 5      /* a partial-sum slot outside the workspace            */
} hgemm_check_t;

/*
 * How the dense kernels' epilogue writes C (HGEMM_OPT_EPILOGUE); both give
 * the same bits.
 *   TMA_STORE (default): tcgen05.ld -> round -> 128-byte-swizzled shared
 *     staging (per warp, double-buffered) -> TMA tensor store of 32 x 64 boxes.
 *   DIRECT: tcgen05.ld -> round -> 16-byte global stores from registers, each
 *     thread writing its own row, as the first kernel of "tcgen05 for
 *     dummies: a B200 GEMM from scratch" (translated) writes its tile back;
 *     that page reports plain stores beating its TMA store.
 */
typedef enum { HGEMM_EPILOGUE_TMA_STORE = 0, HGEMM_EPILOGUE_DIRECT = 1 } hgemm_epilogue_t;

/*
 * Work schedules (HGEMM_OPT_SCHEDULE).  Dense kernels: both cut the same
 * work into the same work ids (hgemm_plan_t: sk_ranges stream-K ranges, then
 * dp_tiles whole tiles) and give bitwise identical results.  Split-K: the
 * static schedule gives each CTA one equal range of units; the dynamic one
 * keeps about 3/4 of the units in one range per SM and cuts the rest into
 * small chunks that the SMs that finish first take over (results are
 * deterministic for each schedule; the two differ in fp32 summation order).
 *   STATIC (default): plan->grid / cta_group persistent clusters; cluster c
 *     takes ids c, c + P, c + 2P, ... (P clusters).
 *   DYNAMIC: plan->work_ids clusters are launched, one per id; a cluster that
 *     finishes an id cancels the launch of a cluster that has not started
 *     (Blackwell cluster launch control) and takes over its id, so the ids
 *     spread over the clusters that actually run (other work on the GPU,
 *     uneven SM speed).  The "Persistent kernel" section of "tcgen05 for
 *     dummies: a B200 GEMM from scratch" names this as the step after static
 *     scheduling.
 */
typedef enum { HGEMM_SCHEDULE_STATIC = 0, HGEMM_SCHEDULE_DYNAMIC = 1 } hgemm_schedule_t;

/* One intra-kernel trace event (HGEMM_OPT_TRACE).  t_ns is the GPU's global
 * nanosecond timer.  role: 0 CTA, 1 TMA producer, 2 MMA issuer, 3 epilogue.
 * kind: 1 kernel begin, 2 kernel end (after setup / before teardown; value =
 * the SM cycle counter's low 31 bits, so cycles / ns gives the clock), 3 item
 * begin, 4 item end, 5 stream-K or split-K partial stored and its ticket
 * drawn (value = ticket), 6 split tile reduced (value = contributors),
 * 7 cycles the role spent blocked on its barriers during the item (value).  item = tile index (-1 if none); value
 * for item begin/end = first / last k-block (epilogue: the stream-K slot). */
typedef struct {
  uint64_t t_ns;
  uint32_t cta;
  uint16_t role;
  uint16_t kind;
  int32_t item;
  int32_t value;
} hgemm_trace_record_t;

/*
 * hgemm_create -- bind a new handle to the CURRENT CUDA device.
 *   out: receives the handle (owned by the caller, release with hgemm_destroy).
 * The device must be compute capability 10.3 (sm_103).  Allocates a 16-byte
 * device status word.  Returns NO_DEVICE when no device/driver is usable,
 * UNSUPPORTED for another architecture, CUDA on any other CUDA failure.
 * For tests, the environment variable HGEMM_FORCE_VARIANT (auto, 1sm128,
 * 1sm256, 2sm256, splitk, 2sm192, or the hgemm_variant_t number) sets the new
 * handle's HGEMM_OPT_FORCE_VARIANT; unset or unrecognised means automatic.
 */
hgemm_status_t hgemm_create(hgemm_handle_t* out);

/*
 * hgemm_destroy -- synchronise the handle's device and free everything the
 * handle owns (status word, split-K workspace).  Null is accepted (no-op).
 */
hgemm_status_t hgemm_destroy(hgemm_handle_t h);

/*
 * hgemm_run -- enqueue C = A . B on `stream`.
 *   A: device pointer, M x K, row-major (element [m][k] at A + m*K + k).
 *   B: device pointer; TN: stored N x K row-major (element B[k][n] at B + n*K + k);
 *      NN: stored K x N row-major (element B[k][n] at B + k*N + n).
 *   C: device pointer, M x N, row-major, written (never read).  Must not overlap A or B.
 *   M, N, K >= 0, each <= 2^31 - 1, and ceil(M/128) * ceil(N/128) <= 2^31 - 1
 *      (the tile count is 32-bit); INVALID_ARG otherwise.
 *      M == 0 or N == 0: nothing to do, HGEMM_OK.
 *      K == 0: C is filled with +0 (the empty sum).
 *   in_dtype:  HGEMM_F16 or HGEMM_BF16 (A and B share it).
 *   acc_dtype: HGEMM_F32, or HGEMM_F16 with in_dtype == HGEMM_F16.
 *   out_dtype: HGEMM_F16 or HGEMM_BF16; the result is rounded to nearest even.
 * Alignment: A, B, C 16-byte aligned; K % 8 == 0 and N % 8 == 0 (every row
 * pitch is a multiple of 16 bytes, a TMA requirement).  K == 0 skips the K
 * check and A, B may then be null.
 * Asynchronous: returns once the kernel is enqueued.  A device-side timeout
 * is reported later by hgemm_sync_status.  Stream-K launches and split-K
 * launches that split a tile's K range use a workspace that the handle
 * allocates on first use (cudaMalloc; HGEMM_ERR_OOM on failure); plans without
 * stream-K and split-K plans of whole tiles need none.  Consecutive launches
 * on different streams must not overlap when they share a handle.
 * CUDA graphs: hgemm_run may be captured into a graph.  A capture cannot
 * contain the workspace allocation, so warm the handle up outside the
 * capture with the largest problem the graph will hold; during a capture a
 * call whose workspace would have to grow returns HGEMM_ERR_UNSUPPORTED and
 * enqueues nothing.  Replays use the handle's workspace, so replays of graphs
 * holding launches of one handle must not overlap each other or other
 * launches of that handle.
 */
hgemm_status_t hgemm_run(hgemm_handle_t h, const void* A, const void* B, void* C, int64_t M, int64_t N,
                         int64_t K, hgemm_layout_t layout, hgemm_dtype_t in_dtype, hgemm_dtype_t acc_dtype,
                         hgemm_dtype_t out_dtype, void* stream);

/*
 * hgemm_run_host -- C = A . B with A, B and C in HOST memory (end to end).
 *   Same arguments, layouts and rules as hgemm_run, except that A, B and C are
 *   host pointers (page-locked memory lets the copies run asynchronously and
 *   overlap; pageable memory works but its copies block the host).
 * B is copied to the device once; A and C move in row chunks (1024 rows or
 * more, whole 256-row tiles, at most 4 chunks) on two internal copy streams,
 * so that the upload of chunk i+1, the GEMM of chunk i and the download of
 * chunk i-1 overlap.  The handle owns two sets of device staging buffers
 * (allocated on first use, grown on demand) and alternates between them, so
 * consecutive calls on DIFFERENT streams overlap too: one call's uploads run
 * beside the previous call's GEMM and download.  Calls on one stream run one
 * after another.  The work starts after earlier work on `stream`, and
 * `stream` waits for its end: C is complete once `stream` is synchronised.
 * A, B and C must stay valid and unmodified until then.  C must not overlap
 * A or B.
 */
hgemm_status_t hgemm_run_host(hgemm_handle_t h, const void* A, const void* B, void* C, int64_t M, int64_t N,
                              int64_t K, hgemm_layout_t layout, hgemm_dtype_t in_dtype, hgemm_dtype_t acc_dtype,
                              hgemm_dtype_t out_dtype, void* stream);

/*
 * hgemm_sync_status -- synchronise `stream`, then return and clear the device
 * status word: HGEMM_OK, or HGEMM_ERR_TIMEOUT when a bounded wait in any
 * kernel launched through this handle gave up since the last call (the
 * launch's output is then undefined), or HGEMM_ERR_CUDA when the stream
 * reports an error.  *detail (nullable) receives the raw status word: bits
 * 0-7 the status, bits 8-15 the role that gave up (1 producer, 2 MMA issuer,
 * 3 epilogue, 4 teardown), bits 16-31 the CTA index.
 */
hgemm_status_t hgemm_sync_status(hgemm_handle_t h, void* stream, int32_t* detail);

/* Set a handle option (hgemm_option_t).  INVALID_ARG for an unknown option or
 * value; OOM when the trace buffer cannot be allocated. */
hgemm_status_t hgemm_set_option(hgemm_handle_t h, int32_t option, int64_t value);

/*
 * hgemm_trace_read -- synchronise the device, copy up to `capacity` recorded
 * events (oldest first in append order, which is not time order) to `out`
 * (host memory, capacity records), store in *n_events how many were recorded
 * since the last read (may exceed both capacities: the excess was dropped),
 * and empty the buffer.  INVALID_ARG when tracing is off.
 */
hgemm_status_t hgemm_trace_read(hgemm_handle_t h, hgemm_trace_record_t* out, int64_t capacity, int64_t* n_events);

/* Static, human-readable name of a status code. */
const char* hgemm_status_string(hgemm_status_t s);

/* ------------------------------------------------------------------------- */
/* Planning and introspection (host only; no device needed).                  */

typedef struct {
  int32_t variant;       /* hgemm_variant_t chosen                                        */
  int32_t cta_group;     /* 1, or 2 for the CTA-pair MMA                                 */
  int32_t tile_m;        /* C rows per tile (per CTA pair for cta_group 2); split-K: N rows */
  int32_t tile_n;        /* C columns per tile; split-K: padded M (the MMA N)            */
  int32_t block_k;       /* K elements per pipeline stage                                */
  int32_t stages;        /* shared-memory ring depth                                     */
  int32_t tiles_m;       /* tile grid                                                    */
  int32_t tiles_n;
  int32_t num_tiles;
  int32_t k_blocks;      /* ceil(K / block_k)                                            */
  int32_t grid;          /* CTAs launched                                                */
  int32_t group_m;       /* rasterisation group height (tiles)                           */
  int32_t smem_bytes;    /* dynamic shared memory per CTA                                */
  int32_t tmem_cols;     /* tensor-memory columns allocated per CTA                      */
  int64_t workspace_bytes; /* split-K / stream-K partial sums + tickets                  */
  int32_t dp_tiles;      /* dense: tiles computed whole, dealt round-robin (all if no stream-K) */
  int32_t stream_k;      /* dense: 1 when the remaining tiles are split along K            */
  int64_t sk_units;      /* dense: (num_tiles - dp_tiles) * k_blocks, cut evenly into sk_ranges ranges */
  int32_t sk_ranges;     /* dense: stream-K ranges, work ids [0, sk_ranges); 0 without stream-K */
  int32_t work_ids;      /* dense: sk_ranges + dp_tiles; ids >= sk_ranges are whole tiles  */
  int32_t schedule;      /* hgemm_schedule_t the plan was made for                         */
  int32_t splitk_chunks; /* split-K: work ids (chunks of units); = grid under STATIC         */
  int64_t splitk_head_units; /* split-K: units in chunks [0, grid) (all of them under STATIC;
                                under DYNAMIC about 3/4, the rest in splitk_chunks - grid
                                small chunks)                                             */
  int32_t splitk_align;  /* split-K: k_blocks when every chunk is whole tiles (no tile's K
                            range is split, no partials or fix-up), else 1                */
  int32_t sk_pieces;     /* dense stream-K: 0 when the split k-blocks are cut into one equal
                            range per cluster (sk_ranges = clusters); p >= 2 when each split
                            tile is cut into p equal K pieces (sk_ranges = split tiles * p
                            <= clusters), so that all pieces walk K side by side          */
} hgemm_plan_t;

/*
 * hgemm_plan -- the launch plan hgemm_run would use for these arguments on a
 * GPU with `num_sms` SMs (cluster capacity assumed num_sms / 2 pairs).
 * `variant` = HGEMM_VARIANT_AUTO or a forced variant; group_m = 0 for the
 * automatic height (as HGEMM_OPT_GROUP_M); stream_k = 1 to allow stream-K, 0 to forbid it, 2 to force equal
 * ranges, 3 to force equal K pieces (as HGEMM_OPT_STREAM_K).  Validates the
 * sizes, dtypes and layout like hgemm_run (pointers are not involved).
 */
hgemm_status_t hgemm_plan(int64_t M, int64_t N, int64_t K, hgemm_layout_t layout, hgemm_dtype_t in_dtype,
                          hgemm_dtype_t acc_dtype, hgemm_dtype_t out_dtype, int32_t num_sms, int32_t variant,
                          int32_t group_m, int32_t stream_k, hgemm_plan_t* plan);

/* hgemm_plan for a given hgemm_schedule_t (hgemm_plan plans for STATIC). */
hgemm_status_t hgemm_plan_ex(int64_t M, int64_t N, int64_t K, hgemm_layout_t layout, hgemm_dtype_t in_dtype,
                             hgemm_dtype_t acc_dtype, hgemm_dtype_t out_dtype, int32_t num_sms, int32_t variant,
                             int32_t group_m, int32_t stream_k, int32_t schedule, hgemm_plan_t* plan);

/*
 * hgemm_plan_work_item -- the index-th item of cluster `cluster`'s work list
 * in a dense plan: k-blocks [*kb0, *kb1) of linear tile *tile; *slot = -1 for
 * a whole tile, 0 or 1 for a stream-K partial (first or last item of the
 * cluster's stream-K range).  INVALID_ARG past the end of the list.  The same
 * iterator runs on the device in the producer, MMA and epilogue roles.
 */
hgemm_status_t hgemm_plan_work_item(const hgemm_plan_t* plan, int32_t cluster, int32_t index, int32_t* tile,
                                    int32_t* kb0, int32_t* kb1, int32_t* slot);

/*
 * hgemm_plan_id_item -- the index-th item of work id `id` (0 <= id <
 * plan->work_ids) of a dense plan, in the same form as hgemm_plan_work_item.
 * Under HGEMM_SCHEDULE_DYNAMIC a cluster runs whole ids in whatever order
 * cluster launch control hands them out.  INVALID_ARG past the id's end.
 */
hgemm_status_t hgemm_plan_id_item(const hgemm_plan_t* plan, int32_t id, int32_t index, int32_t* tile, int32_t* kb0,
                                  int32_t* kb1, int32_t* slot);

/*
 * hgemm_plan_tile -- the persistent scheduler's map from a linear tile index
 * (0 <= t < plan->num_tiles) to tile coordinates: grouped rasterisation,
 * group_m tile rows swept together along N, even groups left to right and
 * odd groups right to left (serpentine).  The same function runs on the
 * device.  For split-K plans, tile t is the t-th block of 128 rows of N.
 */
hgemm_status_t hgemm_plan_tile(const hgemm_plan_t* plan, int32_t t, int32_t* tile_m_idx, int32_t* tile_n_idx);

/*
 * hgemm_plan_splitk_range -- for a split-K plan, the contiguous range of
 * (tile, k-block) work units in chunk `chunk` (0 <= chunk <
 * plan->splitk_chunks): units [*begin, *end) of the tile-major linear order
 * (unit u = tile * k_blocks + kb).  Under STATIC chunk c is CTA c's range;
 * under DYNAMIC the first plan->grid chunks start on the CTAs that run first
 * and the small chunks after them go to whichever CTA finishes first.
 */
hgemm_status_t hgemm_plan_splitk_range(const hgemm_plan_t* plan, int32_t chunk, int64_t* begin, int64_t* end);

/*
 * hgemm_plan_splitk_segment -- for a split-K plan, the index-th segment
 * (0 <= index) that the kernel processes of chunk `chunk`: k-blocks
 * [*kb0, *kb1) of N tile *tile.  A chunk has one segment per tile its range
 * touches; they come in ascending order except that the longest (the later
 * one on a tie) comes last, so the fix-ups of the others finish under its
 * mainloop.  *first is 1 for the segment that starts the chunk's range (it
 * decides where the segment's fp32 partial is kept).  INVALID_ARG past the
 * chunk's last segment or for a bad chunk.
 */
hgemm_status_t hgemm_plan_splitk_segment(const hgemm_plan_t* plan, int32_t chunk, int32_t index, int32_t* tile,
                                         int32_t* kb0, int32_t* kb1, int32_t* first);

/*
 * hgemm_encode_idesc -- the 32-bit tcgen05.mma instruction descriptor the
 * kernels use (kind::f16: D format bit 4-5, A/B format bits 7-9/10-12,
 * A/B major bits 15/16, N>>3 at bit 17, M>>4 at bit 24).
 */
uint32_t hgemm_encode_idesc(int32_t mma_m, int32_t mma_n, hgemm_dtype_t in_dtype, hgemm_dtype_t acc_dtype,
                            int32_t a_mn_major, int32_t b_mn_major);

/*
 * hgemm_encode_smem_desc -- the 64-bit shared-memory matrix descriptor
 * (start address >> 4 at bits 0-13, leading byte offset >> 4 at 16-29, stride
 * byte offset >> 4 at 32-45, version 1 at bit 46, swizzle mode at 61-63 with
 * 2 = 128-byte swizzle).
 */
uint64_t hgemm_encode_smem_desc(uint32_t smem_addr, uint32_t lbo_bytes, uint32_t sbo_bytes, int32_t swizzle_mode);

/*
 * hgemm_run_splitk_noalloc -- C = A . B for skinny M without allocating any
 * device memory and without a handle.
 *
 * The pages have no counterpart for this entry point.  It exists for callers
 * that cannot call cudaMalloc while they multiply (code inside a caching
 * allocator or an out-of-memory handler, a process whose device memory is
 * all held by its own pool, latency-critical loops that cannot take
 * cudaMalloc's implicit synchronisation): such callers can neither create a
 * handle nor let hgemm_run grow its split-K workspace.
 *
 * It runs the split-K kernel of hgemm_run (TN layout, fp32 accumulation) with
 * its scratch -- partial sums, per-tile tickets and a status word -- in a
 * fixed 16 MiB array inside the library's device image, which every GPU that
 * loads the library holds until the process exits.  No cudaMalloc, cudaFree
 * or allocating library routine is called.
 *   A: device pointer, M x K row-major; B: device pointer, N x K row-major
 *   (TN); C: device pointer, M x N row-major, written.  The caller owns all three.
 *   Limits: 1 <= M <= 64 and N <= 67,108,864 (one arrival counter for each
 *   of the ceil(N/128) tiles, in a 2 MiB part of the array); larger sizes
 *   return HGEMM_ERR_UNSUPPORTED.  M == 0 or N == 0 is a no-op; K == 0 writes +0.  Alignment and aliasing rules are those of
 *   hgemm_run (HGEMM_ERR_MISALIGNED, HGEMM_ERR_ALIAS, HGEMM_ERR_INVALID_ARG).
 *   in_dtype, out_dtype: HGEMM_F16 or HGEMM_BF16.
 * The first call on each device does a one-time set-up with that device
 * current (the array's device address, the SM count, the kernel's shared-
 * memory limit); make that first call before any stream capture.  A set-up
 * that fails returns its error and is tried again by the next call.  Every call
 * clears the status word and the tickets it uses, on `stream`, before the
 * kernel.  All calls on a device share the one array, so calls whose kernels
 * overlap on the GPU (different streams without ordering) race and give
 * wrong results.  A device-side wait that gives up is not reported: there is
 * no handle to read a status from.
 */
hgemm_status_t hgemm_run_splitk_noalloc(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K,
                                        hgemm_dtype_t in_dtype, hgemm_dtype_t out_dtype, void* stream);

/* ------------------------------------------------------------------------- */
/* TMA-engine micro-benchmark.                                                */

/*
 * How one tile of tile_rows x tile_cols bf16 elements is copied global ->
 * shared.  "tcgen05 for dummies: a B200 GEMM from scratch" (translated)
 * compares 16-byte and 128-byte inner boxes, each as several 2-D copies or
 * one 3-D copy per tile (its v1a/v1b and v2a/v2b kernels), and in its section
 * on the 128-byte swizzle asks for a micro-benchmark of the TMA engine.
 */
typedef enum {
  HGEMM_TMA_2D_16B = 0,  /* tile_cols / 8 copies of a {8, tile_rows} box, no swizzle          */
  HGEMM_TMA_3D_16B = 1,  /* one copy of a {8, tile_rows, tile_cols / 8} box, no swizzle       */
  HGEMM_TMA_2D_128B = 2, /* tile_cols / 64 copies of a {64, tile_rows} box, 128-byte swizzle  */
  HGEMM_TMA_3D_128B = 3, /* one copy of a {64, tile_rows, tile_cols / 64} box, 128-byte swizzle */
  HGEMM_TMA_BULK = 4     /* one 1-D bulk copy of the tile's bytes (tiles stored back to back) */
} hgemm_tma_mode_t;

typedef struct {
  int32_t mode;       /* hgemm_tma_mode_t                                                    */
  int32_t tile_rows;  /* 8..256, a multiple of 8                                              */
  int32_t tile_cols;  /* a multiple of 8 (of 64 for the 128-byte modes; <= 2048 for 3D_16B)   */
  int32_t depth;      /* tiles in flight per CTA (shared-memory slots), 1..16                 */
  int32_t issuers;    /* warps issuing a tile's copies, 1 or 2 (<= copies per tile)           */
  int32_t ctas;       /* CTAs, one per SM; 0 = every SM                                       */
  int32_t iters;      /* tiles each CTA copies                                                */
  int32_t walk;       /* hgemm_tma_walk_t: the order in which a CTA visits tiles              */
} hgemm_tma_bench_config_t;

typedef enum {
  HGEMM_TMA_WALK_SCATTERED = 0, /* CTA c, round j: tile (c * 7919 + j * 13) mod n_tiles          */
  HGEMM_TMA_WALK_ALONG_K = 1    /* CTA c stays on row band c mod tiles_y and takes its column
                                   tiles in order from ((c / tiles_y) * 7) mod tiles_x, the way a
                                   GEMM's producer walks K over the same rows of A            */
} hgemm_tma_walk_t;

typedef struct {
  double ms;               /* event-timed kernel duration                                     */
  double bytes;            /* bytes copied by all CTAs                                        */
  double gbs;              /* bytes / ms, GB/s                                                */
  double bytes_per_clk_sm; /* median over CTAs of the CTA's bytes / its SM cycles             */
  double sm_mhz;           /* median SM clock seen by the CTAs                                */
  int32_t copies_per_tile;
  int32_t ctas;
  int32_t tile_bytes;
  int32_t reserved;
} hgemm_tma_bench_result_t;

/*
 * hgemm_tma_bench -- every CTA copies cfg->iters tiles of `src` (device
 * pointer, height x width bf16 row-major, 128-byte aligned; height a
 * multiple of tile_rows, width of tile_cols; for BULK the same bytes are read
 * as height*width/(tile_rows*tile_cols) tiles stored one after another) into
 * a ring of cfg->depth shared-memory slots, visiting tiles in the order
 * cfg->walk gives (tiles numbered row-major over the height/tile_rows x
 * width/tile_cols grid).  Synchronous: returns after
 * the kernel, with *res filled.  Checks: sums (host, 2 per CTA, nullable)
 * receives the sum of the 16-bit words in the CTA's slots after the last
 * round and the sum of their squares; last_tiles (host, depth per CTA,
 * nullable) the tile index each slot held (-1 if unused), so the caller can
 * recompute both sums.  Allocates a small result buffer with cudaMalloc.
 * INVALID_ARG / MISALIGNED / UNSUPPORTED (slots do not fit in shared memory)
 * before any launch; TIMEOUT if a bounded wait gave up.
 */
hgemm_status_t hgemm_tma_bench(const void* src, int64_t height, int64_t width, const hgemm_tma_bench_config_t* cfg,
                               hgemm_tma_bench_result_t* res, uint64_t* sums, int32_t* last_tiles, void* stream);

/* Library version, e.g. 100 for 0.1.0. */
int32_t hgemm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* HGEMM_H_ */
