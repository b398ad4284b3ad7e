// Planning decisions shared by the device planning kernel and its host reference.
//
// "Serving GLM5.2 NVFP4 Agentic Workload with SGLang", "Kernel Optimization >
// TopK-V2": a planning kernel picks the cutoff between the short-row paths and the
// multi-CTA path from the batch's length distribution, and builds a work list for a
// persistent grid; the plan is built once per forward and reused by every layer.
//
// Here the cutoff is a chunk size c (elements per CTA): rows with len <= c run on one
// CTA (their row stays resident in that CTA's shared memory); longer rows are split
// into G = ceil(len / c) CTAs that combine histograms through global memory. The
// automatic c is the smallest multiple of kChunkAlign, at least c0 = ceil(total /
// grid) (so the batch is spread evenly over the co-resident grid) and kMinAutoChunk,
// whose multi-CTA rows fit one wave of the grid (auto_chunk_ref). A forced c grows
// only while a hard limit is broken (next_chunk).
#pragma once

#include "common.cuh"

namespace topk {

struct PlanStats {
  int64_t slots;  // sum of G over multi-CTA rows
  int n_multi;    // rows with G >= 2
  int max_g;      // largest G
};

__host__ __device__ inline int round_chunk(int64_t c) {
  c = ceil_div64(c, kChunkAlign) * kChunkAlign;
  if (c < kChunkAlign) c = kChunkAlign;
  if (c > kChunkCap) c = kChunkCap;
  return (int)c;
}

__host__ __device__ inline int valid_len(int32_t L, int max_len) {
  return (L >= 0 && L <= max_len) ? L : 0;
}

// CTAs for a row of (valid) length L at chunk c (32-bit: L < 2^31, c <= kChunkCap).
__host__ __device__ inline int row_groups(int L, int c) {
  return L > c ? (int)(((uint32_t)L + (uint32_t)c - 1u) / (uint32_t)c) : 1;
}

__host__ __device__ inline int initial_chunk(int64_t total, int grid, int forced) {
  if (forced > 0) return round_chunk(forced);
  int64_t c = grid > 0 ? ceil_div64(total, grid) : total;
  if (c < kMinAutoChunk) c = kMinAutoChunk;
  return round_chunk(c);
}

// Packs multi-CTA groups (sizes g[0..n), in order) into waves of `grid` CTAs; a group
// never straddles two waves. Writes each group's wave and first CTA when the output
// arrays are non-null. Returns the number of waves.
__host__ __device__ inline int pack_waves(const int32_t* g, int n, int grid, int32_t* wave,
                                          int32_t* first_cta) {
  int w = 0, used = 0;
  for (int i = 0; i < n; ++i) {
    if (used + g[i] > grid) {
      ++w;
      used = 0;
    }
    if (wave) {
      wave[i] = w;
      first_cta[i] = used;
    }
    used += g[i];
  }
  return n > 0 ? w + 1 : 0;
}

// Decides whether chunk c is acceptable; if not, returns the next chunk to try
// (> c), or -1 when no chunk works.
__host__ __device__ inline int next_chunk(int c, const PlanStats& s, int waves, int grid,
                                          bool forced, int ngroups) {
  const bool hard_ok = s.max_g <= grid && s.n_multi <= ngroups && waves <= kMaxWaves;
  const bool soft_ok = forced || s.slots <= grid;
  if (hard_ok && soft_ok) return c;
  if (c >= kChunkCap) return hard_ok ? c : -1;
  int64_t nc = c + kChunkAlign;
  if (!soft_ok && grid > 0) {
    const int64_t scaled = ceil_div64((int64_t)c * s.slots, grid);
    if (scaled > nc) nc = scaled;
  }
  if (!hard_ok && 2 * (int64_t)c > nc) nc = 2 * (int64_t)c;
  return round_chunk(nc);
}

// Automatic chunk: the smallest multiple of kChunkAlign in [c0, kChunkCap] with
// slots_at(c) <= grid, where slots_at(c) counts the CTAs of the rows split at chunk c
// (sum of G over rows with G > 1; it never grows with c, so bisection finds the
// first pass). Returns false, with *c = kChunkCap, when not even kChunkCap fits.
template <class SlotsAt>
inline bool auto_chunk_ref(int c0, int grid, SlotsAt slots_at, int* c) {
  if (slots_at(c0) <= grid) {
    *c = c0;
    return true;
  }
  if (slots_at(kChunkCap) > grid) {
    *c = kChunkCap;
    return false;
  }
  int lo = c0, hi = kChunkCap;  // lo fails, hi passes
  while (hi - lo > kChunkAlign) {
    const int mid = lo + (hi - lo) / (2 * kChunkAlign) * kChunkAlign;
    if (slots_at(mid) <= grid) hi = mid;
    else lo = mid;
  }
  *c = hi;
  return true;
}

// Bucket of a single-CTA row for the longest-first claim order.
__host__ __device__ inline int len_bucket(int L) {
#ifdef __CUDA_ARCH__
  return L > 1 ? 31 - __clz(L) : 0;  // floor(log2 L): the loop below, without the loop
#else
  int b = 0;
  while (L > 1 && b < 31) {
    L >>= 1;
    ++b;
  }
  return b;
#endif
}

// The unit of chunk `rank` of a row split over G CTAs.
__host__ __device__ inline UnitDesc make_unit(int row, int L, int rank, int G, int group) {
  UnitDesc u;
  int b, e;
  chunk_range(L, G, rank, &b, &e);
  u.row = row;
  u.s0 = b;
  u.n = e - b;
  u.len = L;
  u.rank = rank;
  u.G = G;
  u.group = group;
  u.pad = 0;
  return u;
}

}  // namespace topk
