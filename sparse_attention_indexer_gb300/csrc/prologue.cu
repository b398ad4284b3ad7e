// Indexer key-path prologue: LayerNorm + RoPE + FP8 (e4m3) quantization + paged store,
// one kernel ("Serving GLM5.2 NVFP4 Agentic Workload with SGLang", section "Indexer
// Prologue Fusion", Figure 5). The readings of the steps' parameters are stated in
// include/indexer_prologue.h.
//
// HBM-bound elementwise work with three per-token reductions: one warp per token,
// lane l holding channels [4l, 4l + 4) of the 128. The key row is one coalesced
// 256-byte load (8 bytes per lane), the codes one coalesced 128-byte store (4 bytes
// per lane); LayerNorm's mean and variance and the absolute maximum are warp
// shuffles; RoPE's adjacent pairs (4l, 4l + 1) and (4l + 2, 4l + 3) sit inside one
// lane, so the rotation needs no exchange. The position, the block-table entry and
// the cos/sin row are loaded once per token and broadcast by the memory system.
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "indexer_prologue.h"

namespace {

constexpr int kDim = 128;
constexpr int kWarpsPerBlock = 8;
constexpr float kE4m3Max = 448.0f;

struct Params {
  const uint16_t* k;
  int64_t ld;
  int tokens;
  const float* ln_w;
  const float* ln_b;
  float eps;
  const int32_t* positions;
  const float* cos_sin;
  int max_pos;
  int rope_dim;
  const int32_t* token_table;
  const int32_t* block_table;
  int n_tables;
  int64_t table_ld;
  int page_size;
  uint8_t* cache;
  float* cache_scale;
  int64_t num_slots;
  int32_t* status;
};

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float bf16_bits_to_float(uint32_t bits16) {
  return __uint_as_float(bits16 << 16);
}

// (a, b) -> (a cos - b sin, a sin + b cos)
__device__ __forceinline__ void rotate(float& a, float& b, float c, float s) {
  const float x = a * c - b * s;
  const float y = a * s + b * c;
  a = x;
  b = y;
}

__global__ void __launch_bounds__(kWarpsPerBlock * 32) key_prologue_kernel(Params p) {
  const int t = (int)(((int64_t)blockIdx.x * kWarpsPerBlock) + (threadIdx.x >> 5));
  const int lane = threadIdx.x & 31;
  if (t >= p.tokens) return;  // whole warps leave together

  // independent loads first: the key row, the token's position and table row, the
  // LayerNorm parameters (L1/L2 resident across tokens)
  const uint2 kv = __ldg(reinterpret_cast<const uint2*>(p.k + (int64_t)t * p.ld) + lane);
  const int pos = __ldg(p.positions + t);
  const int tab = __ldg(p.token_table + t);
  const float4 w = __ldg(reinterpret_cast<const float4*>(p.ln_w) + lane);
  const float4 bb = __ldg(reinterpret_cast<const float4*>(p.ln_b) + lane);

  // the token's slot (warp-uniform decision)
  int err = 0;
  int64_t slot = -1;
  if (pos < 0 || pos >= p.max_pos) {
    err = INDEXER_STATUS_POSITION;
  } else if (tab < 0 || tab >= p.n_tables) {
    err = INDEXER_STATUS_TABLE_ROW;
  } else {
    const int pg = pos / p.page_size;
    if ((int64_t)pg >= p.table_ld) {
      err = INDEXER_STATUS_TABLE_WIDTH;
    } else {
      const int32_t page = __ldg(p.block_table + (int64_t)tab * p.table_ld + pg);
      if (page < 0) {
        err = INDEXER_STATUS_TABLE_ENTRY;
      } else {
        slot = (int64_t)page * p.page_size + (pos - pg * p.page_size);
        if (slot >= p.num_slots) err = INDEXER_STATUS_SLOT;
      }
    }
  }
  if (err) {
    if (lane == 0 && p.status) atomicOr(p.status, err);
    return;
  }

  // cos/sin of this lane's two pairs (pair i = 2l covers channels 4l, 4l + 1)
  const int half = p.rope_dim >> 1;
  float2 cs = make_float2(1.0f, 1.0f), sn = make_float2(0.0f, 0.0f);
  const bool rot0 = 4 * lane < p.rope_dim, rot1 = 4 * lane + 2 < p.rope_dim;
  if (rot0) {  // scalar loads: the sines start at rope_dim / 2, which may be odd
    const float* row = p.cos_sin + (int64_t)pos * p.rope_dim;
    cs.x = __ldg(row + 2 * lane);
    sn.x = __ldg(row + half + 2 * lane);
    if (rot1) {
      cs.y = __ldg(row + 2 * lane + 1);
      sn.y = __ldg(row + half + 2 * lane + 1);
    }
  }

  // LayerNorm (two-pass mean / population variance over the 128 channels)
  float x0 = bf16_bits_to_float(kv.x & 0xFFFFu), x1 = bf16_bits_to_float(kv.x >> 16);
  float x2 = bf16_bits_to_float(kv.y & 0xFFFFu), x3 = bf16_bits_to_float(kv.y >> 16);
  const float mean = warp_sum((x0 + x1) + (x2 + x3)) * (1.0f / kDim);
  x0 -= mean;
  x1 -= mean;
  x2 -= mean;
  x3 -= mean;
  const float var = warp_sum((x0 * x0 + x1 * x1) + (x2 * x2 + x3 * x3)) * (1.0f / kDim);
  const float rstd = 1.0f / sqrtf(var + p.eps);
  float y0 = fmaf(x0 * rstd, w.x, bb.x), y1 = fmaf(x1 * rstd, w.y, bb.y);
  float y2 = fmaf(x2 * rstd, w.z, bb.z), y3 = fmaf(x3 * rstd, w.w, bb.w);

  // RoPE on the lane's pairs inside [0, rope_dim)
  if (rot0) rotate(y0, y1, cs.x, sn.x);
  if (rot1) rotate(y2, y3, cs.y, sn.y);

  // per-token scale and e4m3 codes (round to nearest even, saturate at +-448)
  const float amax = warp_max(fmaxf(fmaxf(fabsf(y0), fabsf(y1)), fmaxf(fabsf(y2), fabsf(y3))));
  const float scale = amax > 0.0f ? amax / kE4m3Max : 1.0f;
  const __nv_fp8x2_storage_t lo =
      __nv_cvt_float2_to_fp8x2(make_float2(y0 / scale, y1 / scale), __NV_SATFINITE, __NV_E4M3);
  const __nv_fp8x2_storage_t hi =
      __nv_cvt_float2_to_fp8x2(make_float2(y2 / scale, y3 / scale), __NV_SATFINITE, __NV_E4M3);
  const uint32_t codes = (uint32_t)lo | ((uint32_t)hi << 16);
  reinterpret_cast<uint32_t*>(p.cache + slot * kDim)[lane] = codes;
  if (lane == 0) p.cache_scale[slot] = scale;
}

bool aligned(const void* q, uintptr_t a) { return (reinterpret_cast<uintptr_t>(q) % a) == 0; }

}  // namespace

extern "C" int indexer_k_prologue(const uint16_t* k, int64_t ld, int tokens, int dim,
                                  const float* ln_w, const float* ln_b, float eps,
                                  const int32_t* positions, const float* cos_sin, int max_pos,
                                  int rope_dim, const int32_t* token_table,
                                  const int32_t* block_table, int n_tables, int64_t table_ld,
                                  int page_size, uint8_t* cache, float* cache_scale,
                                  int64_t num_slots, int32_t* status, indexer_stream_t stream) {
  if (tokens < 0 || dim != kDim || rope_dim < 0 || rope_dim > dim || (rope_dim & 1) ||
      max_pos < 1 || page_size < 1 || n_tables < 1 || table_ld < 1 || num_slots < 0 || ld < dim ||
      (ld & 3) ||
      !(eps >= 0.0f) || !std::isfinite(eps))
    return INDEXER_ERR_SHAPE;
  if (tokens == 0) return INDEXER_OK;
  if (!k || !ln_w || !ln_b || !positions || (rope_dim > 0 && !cos_sin) || !token_table ||
      !block_table || !cache || !cache_scale)
    return INDEXER_ERR_NULL;
  if (!aligned(k, 8) || !aligned(cos_sin, 4) || !aligned(ln_w, 16) || !aligned(ln_b, 16) ||
      !aligned(cache, 4) || !aligned(cache_scale, 4) || !aligned(positions, 4) ||
      !aligned(token_table, 4) || !aligned(block_table, 4) || (status && !aligned(status, 4)))
    return INDEXER_ERR_ALIGN;
  Params p{k, ld, tokens, ln_w, ln_b, eps, positions, cos_sin, max_pos, rope_dim, token_table,
           block_table, n_tables, table_ld, page_size, cache, cache_scale, num_slots, status};
  const int64_t blocks = ((int64_t)tokens + kWarpsPerBlock - 1) / kWarpsPerBlock;
  key_prologue_kernel<<<(unsigned)blocks, kWarpsPerBlock * 32, 0, (cudaStream_t)stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? INDEXER_OK : INDEXER_ERR_CUDA;
}
