/*
 * topk_paged.h — C ABI of the GB300 (sm_103a) indexer top-k + paged slot library.
 *
 * Operation ("Serving GLM5.2 NVFP4 Agentic Workload with SGLang", section
 * "Kernel Optimization > TopK-V2", Figs. 2-4 and the paragraphs after them):
 * for every query row of fp32 indexer scores over the historical KV positions,
 * select the top k (runtime k <= 2048) exactly in fp32 and translate each selected
 * logical position into a physical indexer KV-cache slot through a paged block
 * table, in one kernel. A planning kernel bins rows by length and builds a work
 * list once per batch; the plan is reused by every select call (every indexer
 * layer) of that batch (the reuse contract is stated at topk_plan).
 *
 * Readings of what the pages leave open (they define the exact result):
 *   - order: position p ranks before q iff s(p) > s(q), or s(p) == s(q) and p < q;
 *     IEEE equality, so -0.0 == +0.0; every NaN ranks below -inf;
 *   - a row of valid length L yields min(k, L) entries; the remaining
 *     k - min(k, L) entries of its output row are -1;
 *   - slot(p) = block_table[t][p / page_size] * page_size + p % page_size with
 *     t = row_to_table[r] (t = r when row_to_table is NULL), computed in 64 bits;
 *   - the entries of a row are a set: their order inside the row is unspecified.
 *
 * Conventions for every call:
 *   - "device" pointers point to memory of the current CUDA device; the caller owns
 *     all memory. The library never allocates, frees or synchronizes, except
 *     topk_read_status, which synchronizes `stream` to read the status word.
 *   - work is enqueued on `stream` (a cudaStream_t; NULL = legacy default stream);
 *   - a negative return value is a host-side argument error: nothing was enqueued.
 *   - errors found on the device (bad lengths, bad table entries, a bounded wait
 *     that expired) set bits in a sticky status word inside the workspace; read it
 *     with topk_read_status. After a nonzero status, call topk_plan again before
 *     the next select: the plan's counters may be left mid-call.
 *   - one workspace serves one stream at a time: two calls that use the same
 *     workspace must not run concurrently.
 */
#ifndef TOPK_PAGED_H
#define TOPK_PAGED_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* topk_stream_t; /* identical to cudaStream_t */

/* Host-side return codes. */
enum {
  TOPK_OK = 0,
  TOPK_ERR_NULL = -1,        /* a required pointer is NULL */
  TOPK_ERR_ROWS = -2,        /* rows < 0 */
  TOPK_ERR_K = -3,           /* k outside [1, TOPK_MAX_K] */
  TOPK_ERR_PAGE_SIZE = -4,   /* page_size < 1 */
  TOPK_ERR_LD = -5,          /* ld < max_len, or table_ld < 1 */
  TOPK_ERR_WORKSPACE = -6,   /* workspace too small or not 256-byte aligned */
  TOPK_ERR_MAX_LEN = -7,     /* max_len < 0 or above topk_max_row_len() */
  TOPK_ERR_ALIGN = -8,       /* scores not 4-byte aligned / outputs not 4-byte aligned */
  TOPK_ERR_CUDA = -9,        /* a CUDA runtime call failed (launch, attribute query) */
  TOPK_ERR_DEVICE = -10,     /* current device cannot run the kernels (not sm_103) */
  TOPK_ERR_CHUNK = -11,      /* forced chunk size outside [16, topk_chunk_capacity()] */
  TOPK_ERR_STATIC_ROWS = -12 /* rows above TOPK_STATIC_MAX_ROWS (topk_select_paged_noalloc) */
};

/* Device status bits (sticky, OR-ed together; 0 = no error). */
enum {
  TOPK_STATUS_LEN = 1,            /* lens[r] outside [0, max_len]: row written as -1 */
  TOPK_STATUS_TABLE_WIDTH = 2,    /* ceil(lens[r] / page_size) > table_ld: row written as -1 */
  TOPK_STATUS_TABLE_ENTRY = 4,    /* a selected position's table entry is negative: that entry -1 */
  TOPK_STATUS_SLOT_OVERFLOW = 8,  /* a slot exceeds INT32_MAX: that entry -1 */
  TOPK_STATUS_TIMEOUT = 16,       /* a bounded cross-CTA wait expired: row contents undefined */
  TOPK_STATUS_PLAN_MISMATCH = 32, /* lens/rows/max_len differ from the plan, or no plan: rows -1 */
  TOPK_STATUS_ORDER = 64          /* a row barrier found a CTA already past it: row contents undefined */
};

#define TOPK_MAX_K 2048

/* Bytes of workspace needed for a batch of `rows` rows whose lengths are at most
 * `max_len`. Host only, pure (no CUDA call). Returns 0 for invalid arguments. */
size_t topk_workspace_bytes(int rows, int max_len);

/* Largest max_len supported on the current device (rows longer than this cannot be
 * spread over the co-resident CTAs). Host only; queries the device. <= 0 on error. */
int64_t topk_max_row_len(void);

/* Elements one CTA keeps resident in shared memory (the largest chunk of a row one
 * CTA processes). Host only, pure. */
int topk_chunk_capacity(void);

/* Planning kernel (one launch). Reads the device-resident lengths lens[rows] (int32,
 * device) and writes the plan into `workspace` (device, 256-byte aligned, at least
 * topk_workspace_bytes(rows, max_len) bytes). The batch's max_len picks the path:
 *   - max_len <= 256: one warp per row, the row in registers;
 *   - max_len <= 16384: one CTA per row, several CTAs per SM, the row in shared memory;
 *   - max_len <= 131072 with rows * C <= topk_grid_size(), where C = 2, 4 or 8 CTAs
 *     per row for max_len up to 32768, 65536 or 131072: one thread-block cluster of C
 *     CTAs per row, each CTA holding a range of the row's positions in shared memory;
 *     the CTAs merge their histograms through distributed shared memory;
 *   - otherwise every row is binned by length into a single-CTA path (the row
 *     resident in one CTA's shared memory) or a multi-CTA path (the row split into
 *     chunks processed by co-resident CTAs that combine their histograms through
 *     global memory), and the plan holds that work list.
 * For the first three paths the plan is its header alone. A forced chunk (see
 * topk_plan_ex) builds the work list; the register and medium paths do not read it,
 * and a batch of the cluster path then runs on the work list instead. Rows with
 * len <= k are copied whole on every path. Also resets the workspace counters and the
 * status word.
 *
 * Reuse: one plan serves every select call on the same rows, max_len and lens, for
 * any k, scores, block table, row map, page size and outputs; plan again when the
 * lengths change, and after a call that left a nonzero status. A select whose lens
 * differ from a work-list plan's reports TOPK_STATUS_PLAN_MISMATCH; header-only plans
 * record no lengths, and those paths serve any lens up to max_len. */
int topk_plan(const int32_t* lens, int rows, int max_len, void* workspace,
              size_t ws_bytes, topk_stream_t stream);

/* topk_plan with a forced chunk size (elements per CTA, 16 <= chunk <=
 * topk_chunk_capacity()): rows longer than `chunk` are split into ceil(len / chunk)
 * CTAs. The result must not depend on the chunking; tests use this to drive the
 * same rows through every path. chunk == 0 means the automatic choice. */
int topk_plan_ex(const int32_t* lens, int rows, int max_len, int chunk, void* workspace,
                 size_t ws_bytes, topk_stream_t stream);

/* Select + page translation (one launch: the path the plan's batch falls in).
 *   scores      device fp32 [rows, ld], row-major, 4-byte aligned; entries past
 *               lens[r] never affect the result. The cluster path copies a row's
 *               whole aligned 16-byte vectors below max_len before it reads lens[r]
 *               (memory inside the row's stride, as ld >= max_len); the other paths
 *               read the first lens[r] entries (in whole aligned 16-byte vectors)
 *   ld          row stride in elements, ld >= max_len
 *   lens        device int32 [rows]: must equal the lens given to topk_plan
 *   k           1 <= k <= TOPK_MAX_K
 *   block_table device int32 [n_tables, table_ld]: physical page ids
 *   row_to_table device int32 [rows] (table row of each query row) or NULL (identity)
 *   page_size   tokens per page, >= 1
 *   out_slots   device int32 [rows, k]: selected slots, then -1 padding
 *   out_pos     device int32 [rows, k] or NULL: the selected logical positions, in
 *               the same order as out_slots, then -1 padding
 *   workspace   the workspace holding a plan built for these lens/rows/max_len */
int topk_select_paged(const float* scores, int64_t ld, const int32_t* lens, int rows,
                      int max_len, int k, const int32_t* block_table, int64_t table_ld,
                      const int32_t* row_to_table, int page_size, int32_t* out_slots,
                      int32_t* out_pos, void* workspace, topk_stream_t stream);

/* Synchronizes `stream`, then copies the device status word into *status. */
int topk_read_status(const void* workspace, topk_stream_t stream, int* status);

/* Enqueues a reset of the device status word to 0 on `stream`. */
int topk_clear_status(void* workspace, topk_stream_t stream);

/* Text for a host return code (negative) or a device status bit set (positive). */
const char* topk_status_str(int code);

/* Number of CTAs of the persistent select grid on the current device. */
int topk_grid_size(void);

/* Test entry: topk_select_paged with every bounded wait limited to `wait_ns`
 * nanoseconds (0 = the default 200 ms) and CTA `skip_cta` (>= 0; -1 = none) never
 * arriving at the first row barrier of its multi-CTA units: the other CTAs of that row
 * then give up after `wait_ns`, the call ends, TOPK_STATUS_TIMEOUT is set and the first
 * expired wait is recorded in the workspace header (bytes 128..159: kind (1 = row
 * barrier, 2 = piece copy), row, rank, barrier sequence, stuck rank, target, CTA).
 * Rows served by other CTAs are unaffected. Used to test that expired waits end the
 * call cleanly; after it, call topk_plan again. */
int topk_select_paged_test(const float* scores, int64_t ld, const int32_t* lens, int rows,
                           int max_len, int k, const int32_t* block_table, int64_t table_ld,
                           const int32_t* row_to_table, int page_size, int32_t* out_slots,
                           int32_t* out_pos, void* workspace, topk_stream_t stream,
                           uint64_t wait_ns, int skip_cta);

/* Limits of topk_select_paged_noalloc: its scratch is a fixed 10 MiB array in the
 * library's device image, enough for the plan and group states of 64 rows. */
#define TOPK_STATIC_MAX_ROWS 64
#define TOPK_STATIC_SCRATCH_BYTES (10u * 1024u * 1024u)

/* Plan + select + page translation in one call that allocates nothing and takes no
 * workspace. The pages have no counterpart of this entry point: it serves callers
 * that cannot provide device memory (a plain C host without a device allocator, a
 * plug-in in an engine whose free device memory is all reserved for the KV cache,
 * code that must not call cudaMalloc/cudaFree because they synchronize the device).
 * It enqueues topk_plan and then topk_select_paged on `stream`, both on a scratch
 * array of TOPK_STATIC_SCRATCH_BYTES bytes that is a file-scope __device__ object of
 * the library (allocated when the module loads). The planning kernel clears what
 * must start at zero (group-state flags, histograms, counters, the status word) on
 * every call, so every call starts clean.
 *   arguments   as for topk_select_paged (scores, ld, lens, rows, max_len, k,
 *               block_table, table_ld, row_to_table, page_size, out_slots, out_pos)
 *   status      device int32 [1] or NULL: receives this call's device status bits
 *               (TOPK_STATUS_*) once the stream reaches the end of the call
 * Returns TOPK_ERR_STATIC_ROWS for rows > TOPK_STATIC_MAX_ROWS, otherwise the codes
 * of topk_plan / topk_select_paged. Argument errors are found before anything is
 * enqueued; TOPK_ERR_CUDA (a launch or copy that failed) may leave the planning
 * kernel enqueued on the scratch array, with no select after it.
 * The first call on each device looks up the scratch array's address with
 * cudaGetSymbolAddress (with that device current) and queries the device; make that
 * first call before any stream capture begins. There is one scratch array per
 * device: calls that overlap in time on one device (two streams, two host threads)
 * race on it and give undefined results; serialize them on one stream. */
int topk_select_paged_noalloc(const float* scores, int64_t ld, const int32_t* lens, int rows,
                              int max_len, int k, const int32_t* block_table, int64_t table_ld,
                              const int32_t* row_to_table, int page_size, int32_t* out_slots,
                              int32_t* out_pos, int32_t* status, topk_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* TOPK_PAGED_H */
