// Select + page-table kernel for batches of a few long rows (GB300, sm_103a).
//
// "Serving GLM5.2 NVFP4 Agentic Workload with SGLang", "Kernel Optimization > TopK-V2":
// rows are binned by length into a register path, a single-CTA path and a path where
// the CTAs of a thread-block cluster share a row and meet through distributed shared
// memory. Here a batch whose rows are all longer than one medium CTA holds
// (kMediumMaxLen) and at most kClusterMaxLen values, and whose clusters fit the GPU at
// once, runs one cluster of 2, 4 or 8 CTAs per row: the fewest that keep each CTA's
// share of the row at most 16384 values. CTA c of a row's cluster owns positions
// [c * chunk, (c + 1) * chunk), so the CTA ranks order the positions.
//
// Per row:
//  1. Each CTA loads its share (whole 16-byte vectors below max_len, eight per thread
//     in flight) as soon as it starts, before the row's length is read; once the length
//     is known it stores the row's values into shared memory and histograms their 12-bit
//     coarse digit.
//  2. Cluster barrier. Every CTA reads the peers' histograms through the cluster's
//     shared window and finds the same boundary bin: first over the 64 super-bin
//     totals, then over the 64 bins of the super-bin that holds it. The same reads
//     give each peer's count above the boundary and at it.
//  3. Each CTA stages its values above the boundary; their output range starts after
//     the lower-ranked peers' counts. Unless the boundary bin completes the row, its
//     values are written as (key, position) into every CTA's candidate list, at
//     offsets from the lower-ranked peers' counts at the boundary (into CTA 0's list
//     alone when there are more than kClRankMax of them).
//  4. A second cluster barrier. Each CTA translates its staged positions to slots and
//     writes them, and ranks its own candidates against the whole list by counting:
//     a rank below what the row still needs is the candidate's output index. (A longer
//     list is ranked by CTA 0 alone: radix levels over the composite key's bytes, then
//     one warp.)
// A boundary bin with more values than the candidate list holds (kClCap) is refined by
// the whole cluster, one key byte per level (a cluster barrier and a merged 256-bin
// histogram each), before step 3. Values whose keys are still all equal after the last
// byte are taken in position order: CTA by CTA, each CTA's first ones.
//
// Every decision that decides a barrier is taken from merged counts, so all CTAs of a
// cluster pass the same barriers. A CTA's shared memory is read by its peers only
// before the barrier that ends the row.
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"
#include "keys.cuh"

namespace topk {

namespace {

constexpr int kClThreads = 512;
constexpr int kClWarps = kClThreads / 32;
constexpr int kClPer = kClusterMaxLen / 8;        // values of one CTA's share, at most
constexpr int kClSteps = kClPer / kClThreads;     // value s * kClThreads + t is bit s of thread t
constexpr int kClVec = kClPer / 4 / kClThreads;  // 16-byte vectors of a share per thread
constexpr int kClCap = 4096;                      // boundary values gathered for the ranking
constexpr int kClRankMax = 1024;                  // up to this many: every CTA holds them all and ranks its own
constexpr int kClFinish = 256;                    // one warp ranks lists of at most this many
constexpr int kClLevels = 5;                      // coarse digit, then the 4 key bytes
constexpr int kClSegs = kClLevels + 1;            // staged output ranges: one per level, one for ties

static_assert(kClSteps == 32, "a thread's values of a share fit one 32-bit mask");
static_assert(kClVec * 4 * kClThreads == kClPer, "a share is whole vectors per thread");
static_assert(kClPer <= 65536, "local indices fit uint16");

struct __align__(16) ClShared {
  int hist[kBins0];             // coarse histogram; its first 256 bins serve the even key levels
  int hist_odd[256];            // odd key levels; CTA 0's candidate ranking
  int sup[64];                  // coarse super-bin totals (64 bins each), read by the peers
  uint32_t ckey[kClCap];        // the row's boundary values (keys; every CTA, or CTA 0) ...
  int32_t cpos[kClCap];         // ... and their positions
  int32_t tpos[TOPK_MAX_K];     // CTA 0: positions the candidate ranking selects
  uint16_t elist[TOPK_MAX_K];   // local indices of this CTA's staged values
  uint16_t tlist[2][kClCap];    // CTA 0: running candidate lists of the ranking
  int msum[256];                // merged counts of the bins a merge examines
  int peer_take[8];             // per peer: values taken at the current level
  int peer_at[8];               // per peer: values at the current boundary
  int seg_start[kClSegs + 1];   // staged output ranges: first elist index ...
  int seg_base[kClSegs];        // ... and first output index
  int warp_tot[kClWarps];
  int n_tpos, n_tlist;
  int bnd_d, bnd_above, bnd_at, bnd_ok;
  int len, trow, hdr_ok, status;
};
static_assert(sizeof(ClShared) % 16 == 0, "the share buffer after it is 16-byte aligned");

#ifdef TOPK_TRACE
// Per-CTA phase stamps (%globaltimer), trace builds only.
__device__ uint64_t g_cl_trace[kMaxGrid * 16];
#define CL_MARK(slot)                                                                  \
  do {                                                                                 \
    if (threadIdx.x == 0) g_cl_trace[blockIdx.x * 16 + (slot)] = global_timer_ns();    \
  } while (0)
#else
#define CL_MARK(slot) \
  do {                \
  } while (0)
#endif

__device__ __forceinline__ uint32_t cl_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// All threads of every CTA of the cluster; shared-memory writes before it (local or
// remote) are seen by the cluster's shared-memory reads after it.
__device__ __forceinline__ void cl_sync() {
  __syncwarp();
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

// Address of `p` (this CTA's shared memory) in CTA `rank` of the cluster's shared window.
__device__ __forceinline__ uint32_t cl_map(const void* p, int rank) {
  const uint32_t a = (uint32_t)__cvta_generic_to_shared(p);
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
  return r;
}

__device__ __forceinline__ int cl_ld(uint32_t a) {
  int v;
  asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
  return v;
}

__device__ __forceinline__ void cl_st(uint32_t a, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}

// Boundary bin of 64 counts (warp 0): the bin b with (counts above b) < need <=
// (counts at or above b). Lane l holds bins 2l and 2l + 1.
__device__ void cl_bnd64(ClShared& S, const int* cnt, int need, int base_above, int bin0) {
  const int lane = threadIdx.x & 31;
  const int lo = cnt[2 * lane], hi = cnt[2 * lane + 1];
  int incl = lo + hi;  // sum over lanes [lane, 31]
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_down_sync(0xffffffffu, incl, o);
    if (lane + o < 32) incl += y;
  }
  const int above = incl - lo - hi;
  if (above < need && above + hi >= need) {
    S.bnd_d = bin0 + 2 * lane + 1;
    S.bnd_above = base_above + above;
    S.bnd_at = hi;
    S.bnd_ok = 1;
  } else if (above + hi < need && above + hi + lo >= need) {
    S.bnd_d = bin0 + 2 * lane;
    S.bnd_above = base_above + above + hi;
    S.bnd_at = lo;
    S.bnd_ok = 1;
  }
}

// The same over 256 counts (warp 0): lane l holds bins [8l, 8l + 8).
__device__ void cl_bnd256(ClShared& S, const int* cnt, int need) {
  const int lane = threadIdx.x & 31;
  int c[8], mine = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    c[j] = cnt[8 * lane + ((j + lane) & 7)];  // rotated: one load touches distinct banks
    mine += c[j];
  }
  int incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_down_sync(0xffffffffu, incl, o);
    if (lane + o < 32) incl += y;
  }
  int above = incl - mine;
  if (above < need && above + mine >= need) {
    for (int b = 7; b >= 0; --b) {
      const int v = cnt[8 * lane + b];
      if (above + v >= need) {
        S.bnd_d = 8 * lane + b;
        S.bnd_above = above;
        S.bnd_at = v;
        S.bnd_ok = 1;
        break;
      }
      above += v;
    }
  }
}

// Offsets of this thread's taken and kept values among the CTA's (warp order, then
// lane, then bit): one block scan of both counts. *tt, *tk receive the CTA's totals.
__device__ __forceinline__ int2 cl_offsets(ClShared& S, int ct, int ck, int* tt, int* tk) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int it = warp_incl_scan(ct), ik = warp_incl_scan(ck);
  if (lane == 31) S.warp_tot[warp] = it | (ik << 16);  // at most 1024 each
  __syncthreads();
  int bt = 0, bk = 0, at = 0, ak = 0;
#pragma unroll
  for (int w = 0; w < kClWarps; ++w) {
    const int v = S.warp_tot[w];
    if (w < warp) {
      bt += v & 0xFFFF;
      bk += v >> 16;
    }
    at += v & 0xFFFF;
    ak += v >> 16;
  }
  *tt = at;
  *tk = ak;
  return make_int2(bt + it - ct, bk + ik - ck);
}

// Writes the local indices of the set bits of `m` (bit s = index s * kClThreads + t)
// to the staged list from index o on.
__device__ __forceinline__ void cl_stage(ClShared& S, uint32_t m, int o) {
  for (; m; m &= m - 1u, ++o) {
    const int s = __ffs(m) - 1;
    if (o < TOPK_MAX_K) S.elist[o] = (uint16_t)(s * kClThreads + (int)threadIdx.x);
  }
}

// Writes the set bits of `m` as (key, position) into the candidate list of CTAs
// [0, n_dst) from index o on.
__device__ __forceinline__ void cl_push(ClShared& S, const float* sx, uint32_t m, int o, int c0,
                                        int n_dst) {
  const uint32_t k0 = (uint32_t)__cvta_generic_to_shared(S.ckey);
  const uint32_t p0 = (uint32_t)__cvta_generic_to_shared(S.cpos);
  for (; m; m &= m - 1u, ++o) {
    const int i = (__ffs(m) - 1) * kClThreads + (int)threadIdx.x;
    if (o >= kClCap) break;
    const uint32_t key = f2key(sx[i]), pos = (uint32_t)(c0 + i);
    for (int q = 0; q < n_dst; ++q) {
      uint32_t ka, pa;
      asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ka) : "r"(k0 + 4u * (uint32_t)o), "r"(q));
      asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(pa) : "r"(p0 + 4u * (uint32_t)o), "r"(q));
      cl_st(ka, key);
      cl_st(pa, pos);
    }
  }
}

// Slot of position p, whose page's table entry is pg; sets status bits of bad entries.
__device__ __forceinline__ int32_t cl_slot(const SelectParams& P, int32_t pg, int p, int* st) {
  const int ps = P.page_size;
  const int in = (ps & (ps - 1)) == 0 ? (p & (ps - 1)) : p % ps;
  const int64_t sl = (int64_t)pg * ps + in;
  if (pg < 0) {
    *st |= TOPK_STATUS_TABLE_ENTRY;
    return -1;
  }
  if (sl > 0x7FFFFFFFll) {
    *st |= TOPK_STATUS_SLOT_OVERFLOW;
    return -1;
  }
  return (int32_t)sl;
}

__device__ __forceinline__ int cl_page(const SelectParams& P, int p) {
  const int ps = P.page_size;
  return (ps & (ps - 1)) == 0 ? p >> (__ffs(ps) - 1) : p / ps;
}

// One warp selects the `need` best of the n candidates list[0 .. n) (all of
// [0, n) when list is null; n <= 32 * kPer) by the 64-bit composite key << 32 |
// ~position (all distinct): a radix selection from the highest bit where they differ,
// one warp-wide count per bit. Appends the selected positions to S.tpos.
template <int kPer>
__device__ void cl_warp_rank(ClShared& S, const uint16_t* list, int n, int need) {
  const int lane = threadIdx.x & 31;
  uint64_t key[kPer];
  int pos[kPer];
  uint32_t cand = 0u;
  uint32_t an_hi = 0xFFFFFFFFu, an_lo = 0xFFFFFFFFu, or_hi = 0u, or_lo = 0u;
#pragma unroll
  for (int c = 0; c < kPer; ++c) {
    const int j = lane + 32 * c;
    key[c] = 0ull;
    pos[c] = 0;
    if (j < n) {
      const int e = list ? (int)list[j] : j;
      pos[c] = S.cpos[e];
      key[c] = ((uint64_t)S.ckey[e] << 32) | (uint64_t)(~(uint32_t)pos[c]);
      cand |= 1u << c;
      an_hi &= (uint32_t)(key[c] >> 32);
      an_lo &= (uint32_t)key[c];
      or_hi |= (uint32_t)(key[c] >> 32);
      or_lo |= (uint32_t)key[c];
    }
  }
  an_hi = __reduce_and_sync(0xffffffffu, an_hi);
  an_lo = __reduce_and_sync(0xffffffffu, an_lo);
  or_hi = __reduce_or_sync(0xffffffffu, or_hi);
  or_lo = __reduce_or_sync(0xffffffffu, or_lo);
  const uint64_t diff = ((uint64_t)(an_hi ^ or_hi) << 32) | (uint64_t)(an_lo ^ or_lo);
  uint32_t sel = 0u;
  if (diff == 0ull) {
    sel = cand;  // a single candidate: it is the one needed
  } else {
    for (int bit = 63 - __clzll((long long)diff); bit >= 0 && need > 0; --bit) {
      uint32_t m1 = 0u;
#pragma unroll
      for (int c = 0; c < kPer; ++c) m1 |= (uint32_t)((key[c] >> bit) & 1ull) << c;
      m1 &= cand;
      const int cnt = (int)__reduce_add_sync(0xffffffffu, (unsigned)__popc(m1));
      if (cnt >= need) {
        cand = m1;
        if (cnt == need) {
          sel |= m1;
          need = 0;
        }
      } else {
        sel |= m1;
        need -= cnt;
        cand &= ~m1;
      }
    }
    if (need > 0) sel |= cand;  // the last remaining candidate (the keys are distinct)
  }
  const unsigned lt = (1u << lane) - 1u;
  int base = S.n_tpos;
#pragma unroll
  for (int c = 0; c < kPer; ++c) {
    const bool s = (sel >> c) & 1u;
    const unsigned b = __ballot_sync(0xffffffffu, s);
    if (s) {
      const int o = base + __popc(b & lt);
      if (o < TOPK_MAX_K) S.tpos[o] = pos[c];
    }
    base += __popc(b);
  }
  if (lane == 0) S.n_tpos = base;
}

__device__ void cl_warp_rank_any(ClShared& S, const uint16_t* list, int n, int need) {
  if (n <= 64) cl_warp_rank<2>(S, list, n, need);
  else if (n <= 128) cl_warp_rank<4>(S, list, n, need);
  else cl_warp_rank<8>(S, list, n, need);
}

// CTA 0 after the row's last barrier: selects `need` of the n candidates S.ckey/S.cpos
// [0, n) into S.tpos. Lists longer than one warp ranks are first cut down by radix
// levels over the bytes of the composite key, from the top (the whole CTA).
__device__ __noinline__ void cl_rank_candidates(ClShared& S, int n, int need) {
  const int tid = threadIdx.x, lane = tid & 31;
  if (tid == 0) S.n_tpos = 0;
  __syncthreads();
  int src = -1;  // running list: S.tlist[src][0 .. n), or [0, n) when src < 0
  for (int byte = 7; byte >= 0 && need > 0 && n > kClFinish; --byte) {
    const int sh = 8 * byte;
    auto comp = [&](int e) {
      return ((uint64_t)S.ckey[e] << 32) | (uint64_t)(~(uint32_t)S.cpos[e]);
    };
    if (tid < 256) S.hist_odd[tid] = 0;
    if (tid == 0) {
      S.n_tlist = 0;
      S.bnd_ok = 0;
    }
    __syncthreads();
    for (int j = tid; j < n; j += kClThreads) {
      const int e = src >= 0 ? (int)S.tlist[src][j] : j;
      atomicAdd(&S.hist_odd[(uint32_t)(comp(e) >> sh) & 0xFFu], 1);
    }
    __syncthreads();
    if (tid < 32) cl_bnd256(S, S.hist_odd, need);
    __syncthreads();
    const uint32_t d = (uint32_t)S.bnd_d;
    const int above = S.bnd_above, at = S.bnd_at;
    const bool ends = above + at == need;
    const int dst = src == 0 ? 1 : 0;
    for (int j0 = 0; j0 < n; j0 += kClThreads) {
      const int j = j0 + tid;
      int e = 0;
      bool take = false, keep = false;
      if (j < n) {
        e = src >= 0 ? (int)S.tlist[src][j] : j;
        const uint32_t dg = (uint32_t)(comp(e) >> sh) & 0xFFu;
        take = dg > d || (ends && dg == d);
        keep = !ends && dg == d;
      }
      const unsigned bt = __ballot_sync(0xffffffffu, take), bk = __ballot_sync(0xffffffffu, keep);
      int ot = 0, ok = 0;
      if (lane == 0) {
        if (bt) ot = atomicAdd(&S.n_tpos, __popc(bt));
        if (bk) ok = atomicAdd(&S.n_tlist, __popc(bk));
      }
      ot = __shfl_sync(0xffffffffu, ot, 0) + __popc(bt & ((1u << lane) - 1u));
      ok = __shfl_sync(0xffffffffu, ok, 0) + __popc(bk & ((1u << lane) - 1u));
      if (take && ot < TOPK_MAX_K) S.tpos[ot] = S.cpos[e];
      if (keep && ok < kClCap) S.tlist[dst][ok] = (uint16_t)e;
    }
    __syncthreads();
    if (!S.bnd_ok) break;  // cannot happen: the counts hold `need`
    need = ends ? 0 : need - above;
    n = ends ? 0 : at;
    src = dst;
  }
  if (need > 0 && n > 0 && n <= kClFinish && tid < 32)
    cl_warp_rank_any(S, src >= 0 ? S.tlist[src] : nullptr, n, need);
  __syncthreads();
}

struct ClParams {
  SelectParams P;
  int csize;  // CTAs per row (the cluster size)
  int chunk;  // positions per CTA (a multiple of 4, at most kClPer)
};

__global__ void __launch_bounds__(kClThreads, 1) rowcluster_kernel(const __grid_constant__ ClParams A) {
  const SelectParams& P = A.P;
  extern __shared__ __align__(16) unsigned char cl_smem[];
  ClShared& S = *reinterpret_cast<ClShared*>(cl_smem);
  float* const sx = reinterpret_cast<float*>(cl_smem + sizeof(ClShared));
  Header* h = reinterpret_cast<Header*>(P.ws);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int cs = A.csize;
  const int crank = (int)cl_rank();
  const int r = (int)blockIdx.x / cs;
  const int c0 = crank * A.chunk;  // position of this CTA's local index 0
  const float* row = P.scores + (int64_t)r * P.ld;
  CL_MARK(0);

  // The share's whole vectors below max_len (inside the row's stride), eight per thread
  // in flight, before anything else; an unaligned row is read later with plain loads.
  int nv = min(c0 + A.chunk, P.max_len) - c0;
  nv = nv > 0 ? nv >> 2 : 0;
  if ((reinterpret_cast<uintptr_t>(row) & 15u) != 0) nv = 0;
  const float4* const row4 = reinterpret_cast<const float4*>(row + c0);
  float4 v[kClVec];
#pragma unroll
  for (int j = 0; j < kClVec; ++j) {
    const int vi = tid + j * kClThreads;
    if (vi < nv) v[j] = __ldg(row4 + vi);
  }
  if (tid == 0) {
    // the row's length, its table row and the plan header: one round trip
    const int4 h0 = __ldcg(reinterpret_cast<const int4*>(h));
    const int plan_error = __ldcg(&h->plan_error);
    const int L = P.lens[r];
    const int t = P.row_to_table ? P.row_to_table[r] : r;
    S.hdr_ok = ((uint32_t)h0.x == kMagic && h0.y == P.rows && h0.z == P.max_len && plan_error == 0) ? 1 : 0;
    S.len = L;
    S.trow = t;
    S.status = 0;
    S.seg_start[0] = 0;
  }
  for (int i = tid; i < kBins0 / 4; i += kClThreads)
    reinterpret_cast<int4*>(S.hist)[i] = make_int4(0, 0, 0, 0);
  __syncthreads();
  CL_MARK(1);

  const int L = S.len;
  int err = 0;
  if (!S.hdr_ok) err = TOPK_STATUS_PLAN_MISMATCH;
  else if (L < 0 || L > P.max_len) err = TOPK_STATUS_LEN;
  else if (ceil_div64(L, P.page_size) > P.table_ld) err = TOPK_STATUS_TABLE_WIDTH;
  const int kr = err ? 0 : min(P.k, L);
  int32_t* const os = P.out_slots + (int64_t)r * P.k;
  int32_t* const op = P.out_pos ? P.out_pos + (int64_t)r * P.k : nullptr;
  const int32_t* const trow = P.table + (int64_t)S.trow * P.table_ld;

  if (kr == 0 || L <= P.k) {
    // -1 padding, and every position when the row has no more than k: the scores are
    // not needed. The cluster's CTAs share the outputs.
    if (err && crank == 0 && tid == 0) atomicOr(&h->status, err);
    int st = 0;
    for (int o = crank * kClThreads + tid; o < P.k; o += cs * kClThreads) {
      int32_t v = -1, pv = -1;
      if (o < kr) {
        v = cl_slot(P, __ldg(trow + cl_page(P, o)), o, &st);
        pv = o;
      }
      os[o] = v;
      if (op) op[o] = pv;
    }
    if (st) atomicOr(&h->status, st);
    return;
  }

  // ---- 1. the share into shared memory, and its coarse histogram
  const int n_c = max(0, min(c0 + A.chunk, L) - c0);  // values of this CTA (positions c0 + i)
  const int nf = 4 * nv;                              // values the vector loads brought
#pragma unroll
  for (int j = 0; j < kClVec; ++j) {
    const int vi = tid + j * kClThreads;
    if (vi < nv && 4 * vi < n_c) {
      reinterpret_cast<float4*>(sx)[vi] = v[j];
      const float e[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
      for (int c = 0; c < 4; ++c)
        if (4 * vi + c < n_c) atomicAdd(&S.hist[coarse_digit(e[c])], 1);
    }
  }
  for (int s0 = 0; s0 < kClSteps; s0 += 8) {  // the rest (a short tail, or an unaligned row)
    float x[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int i = (s0 + j) * kClThreads + tid;
      if (i >= nf && i < n_c) x[j] = __ldg(row + c0 + i);
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int i = (s0 + j) * kClThreads + tid;
      if (i >= nf && i < n_c) {
        sx[i] = x[j];
        atomicAdd(&S.hist[coarse_digit(x[j])], 1);
      }
    }
  }
  __syncthreads();
  CL_MARK(2);
  {
    int v = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) v += S.hist[8 * tid + ((j + tid) & 7)];
    v += __shfl_xor_sync(0xffffffffu, v, 1);
    v += __shfl_xor_sync(0xffffffffu, v, 2);
    v += __shfl_xor_sync(0xffffffffu, v, 4);
    if ((lane & 7) == 0) S.sup[tid >> 3] = v;
  }

  // ---- 2./3. levels: merged boundary, staging, and the push into CTA 0's list
  int need = kr;     // values the row still needs
  int emitted = 0;   // values taken so far by the whole row
  int n_elist = 0;   // values this CTA has staged
  uint32_t running = 0u;
  bool pushed = false;
  int n_push = 0, nseg = 0;
  int before = 0, at_before = 0, at_mine = 0;
  for (int lv = 0; lv < kClLevels; ++lv) {
    int* const hb = (lv & 1) ? S.hist_odd : S.hist;
    const int sh = 32 - 8 * lv;  // key byte of level lv >= 1: bits [sh, sh + 8)
    if (lv > 0) {
      // local histogram of the key byte over the running values; the buffer's last
      // remote reads were two levels ago, before the barrier of the previous level
      if (tid < 256) hb[tid] = 0;
      __syncthreads();
      for (uint32_t m = running; m; m &= m - 1u) {
        const int i = (__ffs(m) - 1) * kClThreads + tid;
        atomicAdd(&hb[(f2key(sx[i]) >> sh) & 0xFFu], 1);
      }
    }
    if (tid < 8) {
      S.peer_take[tid] = 0;
      S.peer_at[tid] = 0;
    }
    if (tid == 0) {
      S.bnd_d = 0;
      S.bnd_above = 0;
      S.bnd_at = 0;
      S.bnd_ok = 0;
    }
    cl_sync();  // every histogram of this level is complete
    if (lv == 0) CL_MARK(3);

    // merged counts, and each peer's count taken and at the boundary
    bool ends;
    int d, above, at;
    if (lv == 0) {
      const int mp = tid & 7, mj = tid >> 3;
      const int v1 = mp < cs ? cl_ld(cl_map(&S.sup[mj], mp)) : 0;
      int s1 = v1;
      s1 += __shfl_xor_sync(0xffffffffu, s1, 1);
      s1 += __shfl_xor_sync(0xffffffffu, s1, 2);
      s1 += __shfl_xor_sync(0xffffffffu, s1, 4);
      if (mp == 0) S.msum[mj] = s1;
      __syncthreads();
      if (warp == 0) cl_bnd64(S, S.msum, need, 0, 0);
      __syncthreads();
      const int sb = min(max(S.bnd_d, 0), 63), sabove = S.bnd_above;
      const int v2 = mp < cs ? cl_ld(cl_map(&S.hist[64 * sb + mj], mp)) : 0;
      __syncthreads();  // S.msum and S.bnd_* are read above
      int s2 = v2;
      s2 += __shfl_xor_sync(0xffffffffu, s2, 1);
      s2 += __shfl_xor_sync(0xffffffffu, s2, 2);
      s2 += __shfl_xor_sync(0xffffffffu, s2, 4);
      if (mp == 0) S.msum[mj] = s2;
      if (tid == 0) S.bnd_ok = 0;
      __syncthreads();
      if (warp == 0) cl_bnd64(S, S.msum, need - sabove, sabove, 64 * sb);
      __syncthreads();
      d = S.bnd_d;
      above = S.bnd_above;
      at = S.bnd_at;
      ends = above + at == need;
      const int bin = d - 64 * sb;
      // this thread's share of peer mp's taken count
      int take_p = (mj > sb ? v1 : 0) + ((mj > bin || (ends && mj == bin)) ? v2 : 0);
      if (mj == bin && mp < cs) S.peer_at[mp] = v2;
      // lanes p, p + 8, p + 16, p + 24 hold peer p
      take_p += __shfl_xor_sync(0xffffffffu, take_p, 8);
      take_p += __shfl_xor_sync(0xffffffffu, take_p, 16);
      if (lane < 8 && lane < cs && take_p) atomicAdd(&S.peer_take[lane], take_p);
    } else {
      const int b = tid >> 1, half = tid & 1;
      int v[4], sum = 0;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int p = 4 * half + q;
        v[q] = p < cs ? cl_ld(cl_map(&hb[b], p)) : 0;
        sum += v[q];
      }
      sum += __shfl_xor_sync(0xffffffffu, sum, 1);
      if (half == 0) S.msum[b] = sum;
      __syncthreads();
      if (warp == 0) cl_bnd256(S, S.msum, need);
      __syncthreads();
      d = S.bnd_d;
      above = S.bnd_above;
      at = S.bnd_at;
      ends = above + at == need;
      const bool tk = b > d || (ends && b == d);
      if (b == d)
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (4 * half + q < cs) S.peer_at[4 * half + q] = v[q];
      // lanes of the same parity hold the same four peers
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        int t = tk ? v[q] : 0;
        t += __shfl_xor_sync(0xffffffffu, t, 2);
        t += __shfl_xor_sync(0xffffffffu, t, 4);
        t += __shfl_xor_sync(0xffffffffu, t, 8);
        t += __shfl_xor_sync(0xffffffffu, t, 16);
        if (lane < 2 && 4 * lane + q < cs && t) atomicAdd(&S.peer_take[4 * lane + q], t);
      }
    }
    if (tid == 0 && !S.bnd_ok) atomicOr(&S.status, TOPK_STATUS_ORDER);  // cannot happen: the counts hold `need`
    __syncthreads();  // peer counts complete
    if (lv == 0) CL_MARK(4);

    // classify this CTA's running values: taken (above the boundary, or at it when
    // that completes the row) or kept (at it otherwise)
    uint32_t take = 0u, keep = 0u;
    if (lv == 0) {
      if (d >= 2048) {
        // positive side: the bin's float bounds are exact; NaN compares false, and the
        // top bin has nothing above it
        const float t_at = skip_below((uint32_t)d);
        const float t_above = d < 4095 ? skip_below((uint32_t)d + 1u) : __int_as_float(0x7FC00000);
        const int nsteps = (n_c + kClThreads - 1) / kClThreads;  // <= kClSteps
        for (int s0 = 0; s0 < nsteps; s0 += 4) {  // four steps' reads in flight; s0 + 3 < 32
          float x[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int i = (s0 + u) * kClThreads + tid;
            x[u] = __int_as_float(0x7FC00000);  // past the share: NaN is neither taken nor kept
            if (i < n_c) x[u] = sx[i];
          }
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const bool a = x[u] >= t_above, g = x[u] >= t_at;
            take |= (uint32_t)(a || (ends && g)) << (s0 + u);
            keep |= (uint32_t)(!ends && g && !a) << (s0 + u);
          }
        }
      } else {
        for (int s = 0; s * kClThreads < n_c; ++s) {
          const int i = s * kClThreads + tid;
          if (i >= n_c) break;
          const int dg = (int)coarse_digit(sx[i]);
          take |= (uint32_t)(dg > d || (ends && dg == d)) << s;
          keep |= (uint32_t)(!ends && dg == d) << s;
        }
      }
    } else {
      for (uint32_t m = running; m; m &= m - 1u) {
        const int s = __ffs(m) - 1;
        const int dg = (int)((f2key(sx[s * kClThreads + tid]) >> sh) & 0xFFu);
        take |= (uint32_t)(dg > d || (ends && dg == d)) << s;
        keep |= (uint32_t)(!ends && dg == d) << s;
      }
    }
    if (lv == 0) CL_MARK(11);
    before = 0;
    at_before = 0;  // lower-ranked peers' counts
    for (int p = 0; p < crank; ++p) {
      before += S.peer_take[p];
      at_before += S.peer_at[p];
    }
    at_mine = S.peer_at[crank];
    const bool push = !ends && at <= kClCap;
    int tot_t, tot_k;
    const int2 off = cl_offsets(S, __popc(take), push ? __popc(keep) : 0, &tot_t, &tot_k);
    if (lv == 0) CL_MARK(12);
    if (tid == 0) {
      S.seg_start[nseg] = n_elist;
      S.seg_base[nseg] = emitted + before;
    }
    cl_stage(S, take, n_elist + off.x);
    if (lv == 0) CL_MARK(13);
    n_elist += tot_t;
    ++nseg;
    if (ends) {
      emitted += need;
      need = 0;
      break;
    }
    emitted += above;
    need -= above;
    if (push) {
      // every CTA gets the list when it is short enough for each to rank its own
      // candidates against all of them; otherwise CTA 0 ranks them all
      cl_push(S, sx, keep, at_before + off.y, c0, at <= kClRankMax ? cs : 1);
      pushed = true;
      n_push = at;
      break;
    }
    running = keep;
    if (lv == kClLevels - 1) {
      // every key byte is fixed: the running values are equal, and the first `need`
      // of them in position order are taken (CTA by CTA, in local index order)
      const int mine = max(0, min(need - at_before, S.peer_at[crank]));
      if (tid == 0) S.seg_base[nseg] = emitted + min(need, at_before);
      int carry = 0;
      uint32_t tie_take = 0u;
      for (int s = 0; s < kClSteps; ++s) {
        const bool in = (running >> s) & 1u;
        const unsigned bl = __ballot_sync(0xffffffffu, in);
        __syncthreads();  // warp_tot of the previous step is read
        if (lane == 0) S.warp_tot[warp] = __popc(bl);
        __syncthreads();
        int rank = carry + __popc(bl & ((1u << lane) - 1u));
        for (int w = 0; w < warp; ++w) rank += S.warp_tot[w];
        for (int w = 0; w < kClWarps; ++w) carry += S.warp_tot[w];
        if (in && rank < mine) tie_take |= 1u << s;
      }
      __syncthreads();  // the last step's reads of warp_tot are done
      int tot_t, tot_k;
      const int2 off = cl_offsets(S, __popc(tie_take), 0, &tot_t, &tot_k);
      if (tid == 0) S.seg_start[nseg] = n_elist;
      cl_stage(S, tie_take, n_elist + off.x);
      n_elist += tot_t;
      ++nseg;
      emitted += need;
      need = 0;
    }
  }
  CL_MARK(5);
  cl_sync();  // 4. the candidates are in CTA 0; no peer reads this CTA's histograms any more
  CL_MARK(6);

  // ---- 4. staged values to slots (table reads of the whole CTA in flight together)
  int st = 0;
  const int ne = min(n_elist, TOPK_MAX_K);
  for (int e0 = 0; e0 < ne; e0 += 4 * kClThreads) {
    int pp[4], oo[4];
    int32_t pg[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = e0 + j * kClThreads + tid;
      pp[j] = -1;
      oo[j] = -1;
      if (e < ne) {
        int g = 0;
        while (g + 1 < nseg && S.seg_start[g + 1] <= e) ++g;
        oo[j] = S.seg_base[g] + (e - S.seg_start[g]);
        pp[j] = c0 + (int)S.elist[e];
      }
      pg[j] = pp[j] >= 0 ? __ldg(trow + cl_page(P, pp[j])) : 0;
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (pp[j] < 0 || oo[j] < 0 || oo[j] >= kr) continue;  // oo < kr by construction; guarded
      os[oo[j]] = cl_slot(P, pg[j], pp[j], &st);
      if (op) op[oo[j]] = pp[j];
    }
  }
  CL_MARK(7);
  if (pushed && n_push <= kClRankMax) {
    // this CTA's own candidates (list entries [at_before, at_before + at_mine)), each
    // ranked against all n_push by T lanes; a rank below `need` is its output index
    // after the values taken so far
    const int n = n_push, m = at_mine;
    int T = 1;
    while (T < 32 && m * T * 2 <= kClThreads) T *= 2;
    const int sub = tid & (T - 1);
    for (int i0 = 0; i0 < m * T; i0 += kClThreads) {
      const int gi = (i0 + tid) / T;
      const bool act = gi < m;
      const int e = at_before + (act ? gi : 0);
      const uint64_t ci = ((uint64_t)S.ckey[e] << 32) | (uint64_t)(~(uint32_t)S.cpos[e]);
      int rank = 0;
      if (act)
        for (int j = sub; j < n; j += T) {
          const uint64_t cj = ((uint64_t)S.ckey[j] << 32) | (uint64_t)(~(uint32_t)S.cpos[j]);
          rank += cj > ci ? 1 : 0;
        }
      for (int o = 1; o < T; o <<= 1) rank += __shfl_xor_sync(0xffffffffu, rank, o);
      if (act && sub == 0 && rank < need) {
        const int p = S.cpos[e], o = emitted + rank;
        if (o < kr) {
          os[o] = cl_slot(P, __ldg(trow + cl_page(P, p)), p, &st);
          if (op) op[o] = p;
        }
      }
    }
    CL_MARK(8);
  } else if (pushed && crank == 0) {
    // the candidates the row still needs, at the end of its output
    cl_rank_candidates(S, min(n_push, kClCap), need);
    const int nt = min(S.n_tpos, need);
    for (int j0 = 0; j0 < nt; j0 += 4 * kClThreads) {
      int pp[4];
      int32_t pg[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int jj = j0 + j * kClThreads + tid;
        pp[j] = jj < nt ? S.tpos[jj] : -1;
        pg[j] = pp[j] >= 0 ? __ldg(trow + cl_page(P, pp[j])) : 0;
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int o = emitted + j0 + j * kClThreads + tid;
        if (pp[j] < 0 || o >= kr) continue;
        os[o] = cl_slot(P, pg[j], pp[j], &st);
        if (op) op[o] = pp[j];
      }
    }
    if (tid == 0 && S.n_tpos != need) atomicOr(&S.status, TOPK_STATUS_ORDER);  // cannot happen
    CL_MARK(8);
  }
  if (st) atomicOr(&S.status, st);
  __syncthreads();
  if (tid == 0) {
    const int s = S.status;
    if (s) atomicOr(&h->status, s);
  }
#ifdef TOPK_TRACE
  if (tid == 0) g_cl_trace[blockIdx.x * 16 + 10] = (uint64_t)nseg | ((uint64_t)n_push << 8);
#endif
  CL_MARK(9);
}

}  // namespace

#ifdef TOPK_TRACE
extern "C" int topk_trace_cluster(uint64_t* host, int n) {
  if (n > kMaxGrid * 16) n = kMaxGrid * 16;
  return cudaMemcpyFromSymbol(host, g_cl_trace, sizeof(uint64_t) * n) == cudaSuccess ? 0 : -9;
}
#endif

// Dynamic shared memory of a launch whose CTAs hold `chunk` values.
static size_t rowcluster_smem(int chunk) {
  return sizeof(ClShared) + (size_t)((chunk + 3) & ~3) * sizeof(float);
}

cudaError_t launch_rowcluster(const SelectParams& p, cudaStream_t stream) {
  static bool attr_set[64] = {};
  const int cs = cluster_size_for(p.max_len);
  if (cs < 2 || p.rows < 1) return cudaErrorInvalidValue;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    e = cudaFuncSetAttribute(rowcluster_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)rowcluster_smem(kClPer));
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  ClParams a;
  a.P = p;
  a.csize = cs;
  a.chunk = (int)((ceil_div64(p.max_len, cs) + 3) & ~3ll);  // <= kClPer
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3((unsigned)(p.rows * cs));
  cfg.blockDim = dim3(kClThreads);
  cfg.dynamicSmemBytes = rowcluster_smem(a.chunk);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, rowcluster_kernel, a);
}

}  // namespace topk
