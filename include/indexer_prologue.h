/* Indexer key-path prologue: LayerNorm + RoPE + FP8 (e4m3) quantization + store into
 * the paged indexer KV cache, in one kernel.
 *
 * Source: "Serving GLM5.2 NVFP4 Agentic Workload with SGLang", section "Indexer
 * Prologue Fusion" (Figure 5): on the key side of the DSA indexer prologue, LayerNorm,
 * RoPE, FP8 quantization and the paged indexer-KV-cache store run as one fused kernel
 * on the key activations of the fused wk projection (a GEMM, not part of this call).
 * The pages fix none of the steps' parameters; this library takes these readings:
 *   - LayerNorm over the dim channels of a token: (x - mean) / sqrt(var + eps) * w + b,
 *     var the population variance;
 *   - RoPE on channels [0, rope_dim) in adjacent pairs (2i, 2i + 1):
 *     (a, b) -> (a cos - b sin, a sin + b cos), cos and sin from the caller's table
 *     row of the token's position; channels [rope_dim, dim) are not rotated;
 *   - one fp32 scale per token, scale = max |y| / 448 (1 when every y is 0), and codes
 *     e4m3(y / scale) rounded to nearest-even and saturated at +-448 ("fn" e4m3:
 *     exponent bias 7, 3 mantissa bits, no infinity);
 *   - the token at logical position p of the request whose block-table row is t goes
 *     to the physical slot table[t][p / page_size] * page_size + p % page_size (the
 *     slot rule of topk_select_paged's page translation): codes to
 *     cache[slot * dim .. + dim), the scale to cache_scale[slot].
 */
#ifndef INDEXER_PROLOGUE_H
#define INDEXER_PROLOGUE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* indexer_stream_t; /* identical to cudaStream_t */

/* Host-side return codes (negative: nothing was enqueued). */
enum {
  INDEXER_OK = 0,
  INDEXER_ERR_NULL = -1,   /* a required pointer is NULL (with tokens > 0) */
  INDEXER_ERR_SHAPE = -2,  /* tokens < 0, dim != 128, rope_dim odd or outside [0, dim],
                              max_pos < 1, page_size < 1, n_tables < 1, table_ld < 1,
                              num_slots < 0,
                              ld < dim or ld not a multiple of 8, eps negative or not finite */
  INDEXER_ERR_ALIGN = -3,  /* k, ln_w or ln_b not 16-byte aligned, cache not 8-byte
                              aligned, cos_sin or the int32 arrays not 4-byte aligned */
  INDEXER_ERR_CUDA = -4    /* the launch failed */
};

/* Device status bits, OR-ed into *status (a token with a set bit is not stored). */
enum {
  INDEXER_STATUS_POSITION = 1,     /* position < 0 or >= max_pos */
  INDEXER_STATUS_TABLE_WIDTH = 2,  /* position / page_size >= table_ld */
  INDEXER_STATUS_TABLE_ENTRY = 4,  /* the page entry is negative */
  INDEXER_STATUS_SLOT = 8,         /* the slot is >= num_slots */
  INDEXER_STATUS_TABLE_ROW = 16    /* token_table entry outside [0, n_tables) */
};

/* One launch on `stream`; every argument error is reported before anything is
 * enqueued.
 *   k           device bf16 bits (uint16) [tokens, ld], row-major; 16-byte aligned,
 *               ld a multiple of 8; channels [0, dim) of each row are read
 *   tokens      number of tokens (rows of k); 0 enqueues nothing
 *   dim         channels per token: 128 (the indexer head dimension)
 *   ln_w, ln_b  device float32 [dim], 16-byte aligned: LayerNorm weight and bias
 *   eps         LayerNorm epsilon (finite, >= 0)
 *   positions   device int32 [tokens]: logical position of each token in its request
 *   cos_sin     device float32 [max_pos, rope_dim], 4-byte aligned: row p holds
 *               cos(angle_i(p)) for i < rope_dim / 2, then sin(angle_i(p)); may be
 *               NULL when rope_dim is 0 (max_pos still bounds the positions)
 *   rope_dim    rotated channels (even, 0..dim)
 *   token_table device int32 [tokens]: block-table row of each token's request
 *   block_table device int32 [n_tables, table_ld]: physical page ids (< 0: no page)
 *   n_tables    rows of block_table (>= 1)
 *   page_size   tokens per page (>= 1)
 *   cache       device uint8 [num_slots, dim], 8-byte aligned: e4m3 codes (written)
 *   cache_scale device float32 [num_slots]: per-token scales (written)
 *   status      device int32 [1] or NULL: INDEXER_STATUS_* bits are OR-ed in (the
 *               caller clears it); slots of tokens with a status bit are not touched
 * Two tokens with the same slot race (one of them wins). Slots no token maps to are
 * not touched. */
int indexer_k_prologue(const uint16_t* k, int64_t ld, int tokens, int dim, const float* ln_w,
                       const float* ln_b, float eps, const int32_t* positions,
                       const float* cos_sin, int max_pos, int rope_dim,
                       const int32_t* token_table, const int32_t* block_table, int n_tables,
                       int64_t table_ld, int page_size, uint8_t* cache, float* cache_scale,
                       int64_t num_slots, int32_t* status, indexer_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* INDEXER_PROLOGUE_H */
