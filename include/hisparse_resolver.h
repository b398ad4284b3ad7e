/* Fused top-K resolver over a paged KV cache whose older pages may live only in host
 * memory, with a per-request hot buffer kept by least-recently-used replacement.
 *
 * Source: "GLM 5.3 Optimizations, Part 1: Hybrid HiSparse Offloading in vLLM",
 * section "How it works" (mixed residency: the block table holds real blocks and null
 * placeholders side by side; one fused kernel resolves the top-K: resident tokens are
 * read in place, hot tokens are read and their LRU entry refreshed, and a miss copies a
 * single row from pinned host memory into an LRU slot; nothing on the decode path
 * waits on a CPU decision, so it stays CUDA-graph-capturable) and section "Composing
 * with the rest of vLLM" (hot buffers default to 2 x top-K rows per request).
 *
 * The pages sketch the policy; this library takes these readings. One call is one step
 * `step` of every request j = 0 .. rows - 1; request j's selected positions (distinct,
 * -1 padding; e.g. the out_pos of topk_select_paged) are resolved in output order:
 *   - page p / page_size of the request's table row holds a block b >= 0: resident,
 *     KV row b * page_size + p % page_size (the slot rule of topk_select_paged);
 *   - else token_to_hot[j][p] = h >= 0: a hit, KV row hot_rows[j][h], and
 *     hot_step[j][h] = step;
 *   - else a miss. Misses take victims in output order: the request's slots with
 *     hot_step < step (a slot used at this step is never evicted), least recently used
 *     first, ties to the lower slot index (never-used slots, hot_step -1, first). Miss
 *     i takes victim i: the victim's old position loses its mapping, the slot maps to
 *     p, hot_step = step, and host row host_base[j] + p is copied into KV row
 *     hot_rows[j][v], which is the resolved row.
 * Steps never decrease from call to call; the hot state starts all -1.
 *
 * Multi-token verify steps (section "Composing with the rest of vLLM": with speculative
 * decoding the hot buffers hold (num_speculative_tokens + 2) x top-K rows): a request's
 * query rows (the decoded token and its draft tokens, each with its own top-K) share
 * its hot state. hisparse_resolve_mtp resolves them one after another at the same
 * step, as consecutive hisparse_resolve calls with one step value would: a position
 * an earlier row brought in is a hit for a later row, and a slot any of them used at
 * this step is not a victim for the rest.
 */
#ifndef HISPARSE_RESOLVER_H
#define HISPARSE_RESOLVER_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* resolver_stream_t; /* identical to cudaStream_t */

/* Host-side return codes (negative: nothing was enqueued). */
enum {
  RESOLVER_OK = 0,
  RESOLVER_ERR_NULL = -1,  /* a required pointer is NULL (with rows > 0) */
  RESOLVER_ERR_SHAPE = -2, /* rows < 0, k outside [1, 2048], hot_size outside [1, 4096],
                              page_size < 1, table_ld < 1, map_ld < 1, step < 0,
                              row_bytes < 16 or not a multiple of 16, kv_rows or
                              host_rows < 0 */
  RESOLVER_ERR_ALIGN = -3, /* kv or host_kv not 16-byte aligned, host_base not 8-byte
                              aligned, an int32 array not 4-byte aligned */
  RESOLVER_ERR_CUDA = -4   /* the launch or an attribute call failed */
};

/* Device status bits, OR-ed into *status; each failing entry resolves to -1. */
enum {
  RESOLVER_STATUS_NO_VICTIM = 1, /* more misses than slots unused at this step */
  RESOLVER_STATUS_POSITION = 2,  /* position past the table row or the position map */
  RESOLVER_STATUS_HOST_ROW = 4,  /* host_base[j] + p outside [0, host_rows) */
  RESOLVER_STATUS_KV_ROW = 8     /* a victim's KV row outside [0, kv_rows) */
};

/* One launch on `stream`: one CTA per request owns its state; when the batch leaves
 * SMs free, each request is a cluster of 2, 4 or 8 CTAs that share its row copies.
 * Argument errors return before anything is enqueued.
 *   positions    device int32 [rows, k]: selected positions, -1 padding
 *   block_table  device int32 [rows, table_ld]: block id, or < 0 (host only)
 *   token_to_hot device int32 [rows, map_ld]: slot holding each position, -1 none
 *   hot_token    device int32 [rows, hot_size]: position each slot holds, -1 free
 *   hot_step     device int32 [rows, hot_size]: last step each slot was used, -1 never
 *   hot_rows     device int32 [rows, hot_size]: KV row of each slot
 *   host_kv      pinned host memory (device-accessible), [host_rows, row_bytes]
 *   host_base    device int64 [rows]: host row of position 0 of each request
 *   kv           device [kv_rows, row_bytes]: the KV tensor (missed rows written)
 *   out_rows     device int32 [rows, k]: resolved KV rows, -1 for padding / failures
 *   counts       device int32 [rows, 3] or NULL: resident, hits, misses copied
 *   status       device int32 [1] or NULL: RESOLVER_STATUS_* bits OR-ed in
 * The hot state arrays and kv are read and written in place. */
int hisparse_resolve(const int32_t* positions, int rows, int k, const int32_t* block_table,
                     int64_t table_ld, int page_size, int32_t* token_to_hot, int64_t map_ld,
                     int32_t* hot_token, int32_t* hot_step, const int32_t* hot_rows,
                     int hot_size, int step, const uint8_t* host_kv, const int64_t* host_base,
                     int64_t host_rows, uint8_t* kv, int64_t kv_rows, int row_bytes,
                     int32_t* out_rows, int32_t* counts, int32_t* status,
                     resolver_stream_t stream);

/* The same for q_rows query rows per request (q_rows >= 1): positions and out_rows
 * are [rows, q_rows, k]; request j's rows are resolved in order q = 0 .. q_rows - 1 at
 * step `step`, by the CTA that owns the request; counts sum over its rows. Other arguments,
 * return codes and status bits as hisparse_resolve (RESOLVER_ERR_SHAPE also for
 * q_rows < 1). */
int hisparse_resolve_mtp(const int32_t* positions, int rows, int q_rows, int k,
                         const int32_t* block_table, int64_t table_ld, int page_size,
                         int32_t* token_to_hot, int64_t map_ld, int32_t* hot_token,
                         int32_t* hot_step, const int32_t* hot_rows, int hot_size, int step,
                         const uint8_t* host_kv, const int64_t* host_base, int64_t host_rows,
                         uint8_t* kv, int64_t kv_rows, int row_bytes, int32_t* out_rows,
                         int32_t* counts, int32_t* status, resolver_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* HISPARSE_RESOLVER_H */
