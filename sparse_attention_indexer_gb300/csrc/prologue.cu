// Indexer key-path prologue: LayerNorm + RoPE + FP8 (e4m3) quantization + paged store,
// one kernel ("Serving GLM5.2 NVFP4 Agentic Workload with SGLang", section "Indexer
// Prologue Fusion", Figure 5). The readings of the steps' parameters are stated in
// include/indexer_prologue.h.
//
// HBM-bound elementwise work with three per-token reductions. The key row of a token
// is one coalesced 256-byte load (16 bytes per lane of a half-warp) and its codes one
// coalesced 128-byte store; LayerNorm's mean and variance and the absolute maximum
// are shuffles inside the half-warp; RoPE's adjacent pairs sit inside one lane, so the
// rotation needs no exchange. An approximate reciprocal for the codes' scaling and
// rsqrtf keep the per-token instruction count low: the kernel is bound by instruction
// issue, not by memory (IEEE divisions per channel made it 1.5x slower). They move
// y / scale by a few fp32 ulps, far inside the tolerance a rounding-midpoint decision
// allows.
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
  int page_shift;  // log2(page_size) when it is a power of two, else -1
  uint8_t* cache;
  float* cache_scale;
  int64_t num_slots;
  int32_t* status;
};

// Sums / maxima over the 16 lanes of a half-warp (one token each half).
__device__ __forceinline__ float half_sum(float v) {
#pragma unroll
  for (int o = 8; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float half_max(float v) {
#pragma unroll
  for (int o = 8; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// (a, b) -> (a cos - b sin, a sin + b cos)
__device__ __forceinline__ void rotate(float& a, float& b, float c, float s) {
  const float x = a * c - b * s;
  const float y = a * s + b * c;
  a = x;
  b = y;
}

__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
  const __nv_fp8x2_storage_t lo =
      __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
  const __nv_fp8x2_storage_t hi =
      __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
  return (uint32_t)lo | ((uint32_t)hi << 16);
}

// Each half-warp takes one token at a time, lane h (0..15) holding channels
// [8h, 8h + 8): the key row is one 16-byte load per lane, the codes one 8-byte store,
// the three reductions four shuffle levels inside the half, and every scalar step
// (slot, scale, reciprocal) serves two tokens per warp instruction. A warp takes
// kTokensPerWarp consecutive tokens and issues all their loads before it waits on
// any: the key rows with the positions and table rows, then (they depend on the
// position) the page entries and cos/sin values.
constexpr int kTokensPerWarp = 4;
constexpr int kPairs = kTokensPerWarp / 2;

__global__ void __launch_bounds__(kWarpsPerBlock * 32) key_prologue_kernel(Params p) {
  const int64_t w0 =
      ((int64_t)blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5)) * kTokensPerWarp;
  const int lane = threadIdx.x & 31;
  const int h = lane & 15;       // lane within the half-warp
  const int side = lane >> 4;    // which token of a pair
  if (w0 >= p.tokens) return;    // whole warps leave together

  const float4* wv = reinterpret_cast<const float4*>(p.ln_w) + 2 * h;
  const float4* bv = reinterpret_cast<const float4*>(p.ln_b) + 2 * h;
  const float4 wa = __ldg(wv), wb = __ldg(wv + 1), ba = __ldg(bv), bb = __ldg(bv + 1);
  uint4 kv[kPairs];
  int pos[kPairs], tab[kPairs];
#pragma unroll
  for (int j = 0; j < kPairs; ++j) {
    const int64_t t = w0 + 2 * j + side;
    const bool in = t < p.tokens;
    kv[j] = in ? __ldg(reinterpret_cast<const uint4*>(p.k + t * p.ld) + h) : make_uint4(0, 0, 0, 0);
    pos[j] = in ? __ldg(p.positions + t) : -1;
    tab[j] = in ? __ldg(p.token_table + t) : 0;
  }

  // slots (uniform per half) and, for valid positions, this lane's cos/sin values:
  // pairs 4h .. 4h + 3 cover channels 8h .. 8h + 7
  const int half = p.rope_dim >> 1;
  const int nrot = min(4, max(0, (p.rope_dim - 8 * h) >> 1));  // rotated pairs of this lane
  int64_t slot[kPairs];
  float cs[kPairs][4], sn[kPairs][4];
  int err = 0;
#pragma unroll
  for (int j = 0; j < kPairs; ++j) {
    slot[j] = -1;
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      cs[j][m] = 1.0f;
      sn[j][m] = 0.0f;
    }
    if (w0 + 2 * j + side >= p.tokens) continue;
    const int ps = pos[j];
    if (ps < 0 || ps >= p.max_pos) {
      err |= INDEXER_STATUS_POSITION;
      continue;
    }
    if (tab[j] < 0 || tab[j] >= p.n_tables) {
      err |= INDEXER_STATUS_TABLE_ROW;
    } else {
      const int pg = p.page_shift >= 0 ? (ps >> p.page_shift) : ps / p.page_size;
      if ((int64_t)pg >= p.table_ld) {
        err |= INDEXER_STATUS_TABLE_WIDTH;
      } else {
        const int32_t page = __ldg(p.block_table + (int64_t)tab[j] * p.table_ld + pg);
        const int64_t sl = (int64_t)page * p.page_size + (ps - pg * p.page_size);
        if (page < 0) err |= INDEXER_STATUS_TABLE_ENTRY;
        else if (sl >= p.num_slots) err |= INDEXER_STATUS_SLOT;
        else slot[j] = sl;
      }
    }
    const float* row = p.cos_sin + (int64_t)ps * p.rope_dim;
#pragma unroll
    for (int m = 0; m < 4; ++m)
      if (m < nrot) {  // scalar loads: the sines start at rope_dim / 2, which may be odd
        cs[j][m] = __ldg(row + 4 * h + m);
        sn[j][m] = __ldg(row + half + 4 * h + m);
      }
  }
  if (err && h == 0 && p.status) atomicOr(p.status, err);

#pragma unroll
  for (int j = 0; j < kPairs; ++j) {
    // both halves run the shuffles; a half whose token is not stored skips the store
    float x[8] = {bf16_lo(kv[j].x), bf16_hi(kv[j].x), bf16_lo(kv[j].y), bf16_hi(kv[j].y),
                  bf16_lo(kv[j].z), bf16_hi(kv[j].z), bf16_lo(kv[j].w), bf16_hi(kv[j].w)};
    // LayerNorm (two-pass mean / population variance over the 128 channels)
    const float mean =
        half_sum(((x[0] + x[1]) + (x[2] + x[3])) + ((x[4] + x[5]) + (x[6] + x[7]))) *
        (1.0f / kDim);
    float ss = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      x[i] -= mean;
      ss = fmaf(x[i], x[i], ss);
    }
    const float rstd = rsqrtf(half_sum(ss) * (1.0f / kDim) + p.eps);
    const float wl[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
    const float bl[8] = {ba.x, ba.y, ba.z, ba.w, bb.x, bb.y, bb.z, bb.w};
    float y[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) y[i] = fmaf(x[i] * rstd, wl[i], bl[i]);
    // RoPE on the lane's pairs inside [0, rope_dim)
#pragma unroll
    for (int m = 0; m < 4; ++m)
      if (m < nrot) rotate(y[2 * m], y[2 * m + 1], cs[j][m], sn[j][m]);
    // per-token scale and e4m3 codes (round to nearest even, saturate at +-448)
    float a = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) a = fmaxf(a, fabsf(y[i]));
    const float amax = half_max(a);
    // the stored scale is amax / 448 to within one ulp (a product by the rounded
    // reciprocal of 448); the codes use an approximate reciprocal of it
    const float scale = amax > 0.0f ? amax * (1.0f / kE4m3Max) : 1.0f;
    const float inv = amax > 0.0f ? __fdividef(kE4m3Max, amax) : 1.0f;
    if (slot[j] < 0) continue;
    const uint2 codes = make_uint2(e4m3x4(y[0] * inv, y[1] * inv, y[2] * inv, y[3] * inv),
                                   e4m3x4(y[4] * inv, y[5] * inv, y[6] * inv, y[7] * inv));
    reinterpret_cast<uint2*>(p.cache + slot[j] * kDim)[h] = codes;
    if (h == 0) p.cache_scale[slot[j]] = scale;
  }
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
      (ld & 7) ||
      !(eps >= 0.0f) || !std::isfinite(eps))
    return INDEXER_ERR_SHAPE;
  if (tokens == 0) return INDEXER_OK;
  if (!k || !ln_w || !ln_b || !positions || (rope_dim > 0 && !cos_sin) || !token_table ||
      !block_table || !cache || !cache_scale)
    return INDEXER_ERR_NULL;
  if (!aligned(k, 16) || !aligned(cos_sin, 4) || !aligned(ln_w, 16) || !aligned(ln_b, 16) ||
      !aligned(cache, 8) || !aligned(cache_scale, 4) || !aligned(positions, 4) ||
      !aligned(token_table, 4) || !aligned(block_table, 4) || (status && !aligned(status, 4)))
    return INDEXER_ERR_ALIGN;
  int shift = -1;
  if ((page_size & (page_size - 1)) == 0)
    for (shift = 0; (1 << shift) < page_size; ++shift) {
    }
  Params p{k,           ld,          tokens,   ln_w,      ln_b,  eps,         positions,
           cos_sin,     max_pos,     rope_dim, token_table, block_table, n_tables, table_ld,
           page_size,   shift,       cache,    cache_scale, num_slots,   status};
  const int64_t per_block = (int64_t)kWarpsPerBlock * kTokensPerWarp;
  const int64_t blocks = ((int64_t)tokens + per_block - 1) / per_block;
  key_prologue_kernel<<<(unsigned)blocks, kWarpsPerBlock * 32, 0, (cudaStream_t)stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? INDEXER_OK : INDEXER_ERR_CUDA;
}
