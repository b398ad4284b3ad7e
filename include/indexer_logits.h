/* Indexer score producer ("MQA logits"): one fp32 score per (query row, key
 * position) from FP8 (e4m3) query heads, per-head gate weights and the FP8 keys of
 * the paged indexer KV cache with their per-token scales. Its output rows are the
 * score rows that topk_select_paged (topk_paged.h) selects from.
 *
 * Source: "Serving GLM5.2 NVFP4 Agentic Workload with SGLang". Section "Indexer
 * Prologue Fusion": the key side stores each key as FP8 codes with a per-token scale
 * in the paged indexer KV cache (what indexer_k_prologue writes); the query side
 * quantizes the query heads to FP8 and applies the head-gate scaling, the gates
 * coming from the weights projection (one gate per head). Section "What's next":
 * the indexer's MQA logits kernel consumes both. The pages give no formula; this
 * library computes
 *
 *   score(t, p) = sk(s) * sum_h g(t, h) * max(0, sum_d q(t, h, d) * k(s, d))
 *
 * with s = table[r][p / page_size] * page_size + p % page_size the slot of position
 * p (r the block-table row of t's group), q and k the e4m3 code values, sk(s) the
 * key scale and g(t, h) the gate (with the query's quantization scale folded in).
 * The per-head ReLU is a reading: with no non-linearity the gated sum over heads
 * would collapse to a single query vector.
 *
 * The query-key products run on the tensor cores (e4m3 x e4m3, fp32 accumulation),
 * so a score matches the exact value to within a few fp32 roundings of
 * sk(s) * sum_h |g(t, h)| * sum_d |q(t, h, d) k(s, d)|, not bit for bit.
 */
#ifndef INDEXER_LOGITS_H
#define INDEXER_LOGITS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* logits_stream_t; /* identical to cudaStream_t */

/* Host-side return codes (negative: nothing was enqueued). */
enum {
  LOGITS_OK = 0,
  LOGITS_ERR_NULL = -1,   /* a required pointer is NULL (with rows > 0) */
  LOGITS_ERR_SHAPE = -2,  /* rows < 0, heads != 64, dim != 128, group_rows outside
                             [1, 8], max_len < 0, n_tables < 1, table_ld < 1,
                             page_size not a positive multiple of 64, num_slots outside
                             [1, 2^31), ld < max_len, or ceil(rows / G) *
                             ceil(max_len / 128) >= 2^31 */
  LOGITS_ERR_ALIGN = -3,  /* q, w, cache or cache_scale not 16-byte aligned, or
                             another array not 4-byte aligned */
  LOGITS_ERR_CUDA = -4    /* a launch, the device query or the tensor-map encoding
                             failed */
};

/* Device status bits, OR-ed into *status. */
enum {
  LOGITS_STATUS_LEN = 1,          /* a row's length is < 0 or > max_len: row not scored */
  LOGITS_STATUS_TABLE_WIDTH = 2,  /* a row's pages do not fit table_ld: row not scored */
  LOGITS_STATUS_TABLE_ENTRY = 4,  /* a scored position's page entry is negative: -inf */
  LOGITS_STATUS_SLOT = 8,         /* a scored position's slot is >= num_slots: -inf */
  LOGITS_STATUS_TABLE_ROW = 16,   /* a group's table row is outside [0, n_tables): its
                                     rows are not scored */
  LOGITS_STATUS_TIMEOUT = 32      /* a bounded wait inside the kernel expired: the
                                     scores of this call are unreliable */
};

/* One launch on `stream`; every argument error is reported before anything is
 * enqueued.
 *   q            device uint8 [rows, heads, dim], 16-byte aligned: e4m3 codes of the
 *                query heads, row-major
 *   w            device float32 [rows, heads], 16-byte aligned: gate weights
 *   rows         query rows; 0 enqueues nothing
 *   heads, dim   64 and 128
 *   lens         device int32 [rows]: row t scores positions [0, lens[t])
 *   max_len      bound on every length (and on the work the launch plans for)
 *   group_rows   G in [1, 8]: rows g*G .. g*G + G - 1 form group g (the last group
 *                may be shorter) and share one block-table row; each group's keys
 *                are read once for all of its rows
 *   group_table  device int32 [ceil(rows / G)]: block-table row of each group, or
 *                NULL (group g uses row g)
 *   block_table  device int32 [n_tables, table_ld]: physical page ids (< 0: none)
 *   page_size    tokens per page: a positive multiple of 64
 *   cache        device uint8 [num_slots, dim], 16-byte aligned: e4m3 key codes
 *   cache_scale  device float32 [num_slots], 16-byte aligned: key scales
 *   scores       device float32 [rows, ld]: row t's positions [0, lens[t]) are
 *                written; nothing else is touched
 *   status       device int32 [1] or NULL: LOGITS_STATUS_* bits are OR-ed in (the
 *                caller clears it)
 * Codes must hold no NaN pattern (S.1111.111; the key-path prologue never writes
 * one): a product with one is undefined here. Each CTA of the launch holds all 512
 * tensor-memory columns of its SM while it runs. */
int indexer_mqa_logits(const uint8_t* q, const float* w, int rows, int heads, int dim,
                       const int32_t* lens, int max_len, int group_rows,
                       const int32_t* group_table, const int32_t* block_table, int n_tables,
                       int table_ld, int page_size, const uint8_t* cache,
                       const float* cache_scale, int64_t num_slots, float* scores, int64_t ld,
                       int32_t* status, logits_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* INDEXER_LOGITS_H */
