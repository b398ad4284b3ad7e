// Fused top-K resolver with per-request LRU hot buffers ("GLM 5.3 Optimizations,
// Part 1: Hybrid HiSparse Offloading in vLLM", section "How it works"); the readings of
// the policy are stated in include/hisparse_resolver.h.
//
// One CTA per request. Its threads classify the selected positions (resident, hit with
// the slot's step refreshed, miss); a block scan ranks the misses in output order;
// when there are any, the CTA orders the slots unused at this step by (last step, slot)
// (a counting order over the eight oldest step values when the victims lie there, else
// a radix select of the victims and a bitonic sort of those), hands miss r victim r,
// updates the two maps, and copies the missed rows from pinned host memory
// (read directly by the kernel, eight 16-byte chunks per thread in flight) into the
// victims' KV rows. Every phase issues its independent loads together: one CTA per
// request leaves little other parallelism to hide their latency.
//
// The host reads of one SM do not go faster with more of them in flight, so a batch of
// few requests runs each request as a thread-block cluster: CTA 0 of the cluster owns
// the request's state and does everything above; once its copy list is complete (a
// cluster barrier), every CTA of the cluster copies a share of the rows, reading the
// list from CTA 0's shared memory, and a second cluster barrier ends the row's copies
// before the list is reused.
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "hisparse_resolver.h"

namespace {

constexpr int kThreads = 512;
constexpr int kMaxK = 2048;
constexpr int kMaxHot = 4096;
constexpr uint64_t kNone = ~0ull;

struct Params {
  const int32_t* positions;
  int rows, k;
  const int32_t* table;
  int64_t table_ld;
  int page_size;
  int32_t* t2h;
  int64_t map_ld;
  int32_t* hot_token;
  int32_t* hot_step;
  const int32_t* hot_rows;
  int hot;
  int step;
  const uint8_t* host;
  const int64_t* host_base;
  int64_t host_rows;
  uint8_t* kv;
  int64_t kv_rows;
  int row_bytes;
  int32_t* out;
  int32_t* counts;
  int32_t* status;
  int q_rows;  // query rows per request, resolved one after another at the same step
  int csize;   // CTAs per request (a cluster when > 1); CTA 0 owns the request
};

struct Smem {
  uint64_t keys[kMaxHot];     // victim order: (hot_step + 1) << 32 | slot, kNone excluded
  uint64_t vkeys[kMaxK];      // the victims' keys, sorted (selection path)
  uint32_t hist[256];
  int32_t sel[8];
  int32_t miss_entry[kMaxK];  // entry index of the miss of each rank
  uint8_t is_miss[kMaxK];
  uint8_t hit_slot[kMaxHot];  // slots refreshed by a hit of this step
  int64_t copy_src[kMaxK];    // host row of each assigned miss (by rank), -1 none
  int32_t copy_dst[kMaxK];    // KV row
  int32_t n_list;             // entries of copy_src / copy_dst for this query row
  int32_t wsum[kThreads / 32];
  uint64_t wsum2[2][kThreads / 32];
  int32_t red[4][kThreads / 32];
};

static_assert(offsetof(Smem, hit_slot) % 8 == 0, "hit bitmap zeroed with 8-byte stores");

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// All threads of every CTA of the cluster: shared-memory writes before it are seen by
// the cluster's shared-memory reads after it.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

// Address in the cluster's shared window of `p` (this CTA's shared memory) in CTA 0.
__device__ __forceinline__ uint32_t in_rank0(const void* p) {
  uint32_t a = (uint32_t)__cvta_generic_to_shared(p), r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, 0;" : "=r"(r) : "r"(a));
  return r;
}

__device__ __forceinline__ int64_t ld_cluster_s64(uint32_t a) {
  int64_t v;
  asm volatile("ld.shared::cluster.s64 %0, [%1];" : "=l"(v) : "r"(a) : "memory");
  return v;
}

__device__ __forceinline__ int32_t ld_cluster_s32(uint32_t a) {
  int32_t v;
  asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
  return v;
}

// The row copies of one query row, shared among the request's csize CTAs (crank = this
// CTA's rank): (miss, 16-byte chunk) pairs, eight per thread in flight, loads first and
// then the stores. The list (n entries) is CTA 0's; other CTAs read it through the
// cluster's shared window.
__device__ __noinline__ void copy_rows(const Params& p, Smem& s, int crank, int n) {
  const int chunks = p.row_bytes >> 4;
  const int64_t total = (int64_t)n * chunks;
  const int64_t stride = (int64_t)p.csize * kThreads;
  const uint32_t src0 = crank > 0 ? in_rank0(&s.copy_src[0]) : 0u;
  const uint32_t dst0 = crank > 0 ? in_rank0(&s.copy_dst[0]) : 0u;
  constexpr int kC = 8;
  for (int64_t c0 = (int64_t)crank * kThreads + threadIdx.x; c0 < total; c0 += kC * stride) {
    uint4 v[kC];
    int64_t dst[kC];
#pragma unroll
    for (int e = 0; e < kC; ++e) {
      const int64_t c = c0 + e * stride;
      dst[e] = -1;
      if (c < total) {
        const int rr = (int)(c / chunks), cq = (int)(c - (int64_t)rr * chunks);
        const int64_t src = crank > 0 ? ld_cluster_s64(src0 + 8u * rr) : s.copy_src[rr];
        if (src >= 0) {
          const int32_t kr = crank > 0 ? ld_cluster_s32(dst0 + 4u * rr) : s.copy_dst[rr];
          v[e] = *reinterpret_cast<const uint4*>(p.host + src * p.row_bytes + 16 * cq);
          dst[e] = (int64_t)kr * p.row_bytes + 16 * cq;
        }
      }
    }
#pragma unroll
    for (int e = 0; e < kC; ++e)
      if (dst[e] >= 0) *reinterpret_cast<uint4*>(p.kv + dst[e]) = v[e];
  }
}

__device__ int block_excl_scan(int v, int* total, Smem& s) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s.wsum[w] = x;
  __syncthreads();
  int before = 0, tot = 0;
#pragma unroll
  for (int i = 0; i < kThreads / 32; ++i) {
    if (i < w) before += s.wsum[i];
    tot += s.wsum[i];
  }
  __syncthreads();
  *total = tot;
  return before + x - v;
}

// kRows: the request has several query rows (a loop over them); else exactly one, and
// the body compiles without the loop (the loop costs the one-row step registers).
template <bool kRows>
__global__ void __launch_bounds__(kThreads) resolve_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  Smem& s = *reinterpret_cast<Smem*>(smem_raw);
  const int j = blockIdx.x / p.csize;
  const int n_rows = kRows ? p.q_rows : 1;
  if (p.csize > 1 && cluster_rank() != 0) {
    // A copying CTA of the request: its share of each query row's copies.
    const int crank = (int)cluster_rank();
    const uint32_t nl = in_rank0(&s.n_list);
    for (int qr = 0; qr < n_rows; ++qr) {
      cluster_sync();  // CTA 0's list for this row is complete
      copy_rows(p, s, crank, ld_cluster_s32(nl));
      cluster_sync();  // every CTA is done with the list
    }
    return;
  }
  const int32_t* tab = p.table + (int64_t)j * p.table_ld;
  int32_t* t2h = p.t2h + (int64_t)j * p.map_ld;
  int32_t* htok = p.hot_token + (int64_t)j * p.hot;
  int32_t* hstep = p.hot_step + (int64_t)j * p.hot;
  const int32_t* hrows = p.hot_rows + (int64_t)j * p.hot;
  int err = 0, n_res = 0, n_hit = 0, n_copy = 0;
  // The request's query rows, one after another: a later row sees the state an earlier
  // one left (its misses are hits now, and the slots it used, at this step, are not
  // victims). Global writes of the block are visible to it after each row's barrier.
  for (int qr = 0; qr < n_rows; ++qr) {
  const int32_t* pos = p.positions + ((int64_t)j * p.q_rows + qr) * p.k;
  int32_t* out = p.out + ((int64_t)j * p.q_rows + qr) * p.k;

  // The slots' last steps (for the victim order) do not depend on the classification:
  // thread t reads those of slots 8t .. 8t + 7 now, and the hits found below are
  // marked in a shared bitmap instead of being read back.
  constexpr int kV = kMaxHot / kThreads;
  static_assert(kV == 8, "8 slots per thread: 4-bit counters, 8 counted offsets");
  const int h0 = threadIdx.x * kV;
  __syncthreads();  // the previous row's shared state is no longer read
  reinterpret_cast<uint2*>(s.hit_slot)[threadIdx.x] = make_uint2(0u, 0u);
  __syncthreads();
  int sv[kV];
#pragma unroll
  for (int e = 0; e < kV; ++e) sv[e] = h0 + e < p.hot ? hstep[h0 + e] : p.step;

  // 1. classify; hits refresh their slot (distinct positions -> distinct slots). Each
  // thread takes entries t, t + 512, t + 1024, t + 1536 and issues each level of its
  // dependent loads for all four before it waits on any: the position; its page entry
  // and its position-map entry together (the map is read for resident positions too,
  // so that it does not wait on the page entry); the hot row of a hit.
  constexpr int kE = kMaxK / kThreads;
  int q[kE], pg[kE], b[kE], h[kE], hr[kE];
#pragma unroll
  for (int e = 0; e < kE; ++e) {
    const int i = threadIdx.x + e * kThreads;
    q[e] = i < p.k ? pos[i] : -1;
  }
#pragma unroll
  for (int e = 0; e < kE; ++e) {
    pg[e] = q[e] >= 0 ? q[e] / p.page_size : 0;
    const bool ok = q[e] >= 0 && (int64_t)pg[e] < p.table_ld && (int64_t)q[e] < p.map_ld;
    if (q[e] >= 0 && !ok) {
      err |= RESOLVER_STATUS_POSITION;
      q[e] = -2;  // resolved to -1, not a miss
    }
    b[e] = ok ? tab[pg[e]] : -1;
    h[e] = ok ? t2h[q[e]] : -1;
  }
#pragma unroll
  for (int e = 0; e < kE; ++e) {
    const bool hit = q[e] >= 0 && b[e] < 0 && h[e] >= 0 && h[e] < p.hot;
    if (!hit) h[e] = -1;
    hr[e] = hit ? hrows[h[e]] : -1;
  }
#pragma unroll
  for (int e = 0; e < kE; ++e) {
    const int i = threadIdx.x + e * kThreads;
    if (i >= p.k) continue;
    uint8_t miss = 0;
    int row = -1;
    if (q[e] >= 0) {
      if (b[e] >= 0) {
        row = (int)((int64_t)b[e] * p.page_size + (q[e] - pg[e] * p.page_size));
        ++n_res;
      } else if (h[e] >= 0) {
        row = hr[e];
        hstep[h[e]] = p.step;
        s.hit_slot[h[e]] = 1;
        ++n_hit;
      } else {
        miss = 1;
      }
    }
    out[i] = row;
    s.is_miss[i] = miss;
  }
  __syncthreads();

  // 2. miss ranks in output order: thread t scans entries [4t, 4t + 4)
  int local = 0;
  for (int i = 4 * threadIdx.x; i < 4 * threadIdx.x + 4 && i < p.k; ++i) local += s.is_miss[i];
  int m = 0;
  int r = block_excl_scan(local, &m, s);
  for (int i = 4 * threadIdx.x; i < 4 * threadIdx.x + 4 && i < p.k; ++i)
    if (s.is_miss[i]) s.miss_entry[r++] = i;

  if (m > 0) {
    int want = 0;
    uint64_t* victims = s.vkeys;
    // 3. victim order: the slots unused at this step, by (last step, slot). Thread t
    // holds slots 8t .. 8t + 7. Keyed by d = last step + 1 - (oldest such value), the
    // order is a stable counting sort on d in slot order: a slot's rank is the number
    // of candidates with a smaller d, plus those with its d in lower slots. One block
    // scan of per-thread counts for d < 8 gives every rank when the victims all lie
    // there (the usual LRU case: they come from the oldest few steps); otherwise the
    // general order below runs.
#pragma unroll
    for (int e = 0; e < kV; ++e)
      if (s.hit_slot[h0 + e]) sv[e] = p.step;  // used at this step: not a candidate
    uint32_t lo = 0xFFFFFFFFu;
    int ncand = 0;
#pragma unroll
    for (int e = 0; e < kV; ++e)
      if (sv[e] < p.step) {
        lo = min(lo, (uint32_t)(sv[e] + 1));
        ++ncand;
      }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
      ncand += __shfl_xor_sync(0xffffffffu, ncand, o);
    }
    if ((threadIdx.x & 31) == 0) {
      s.red[0][threadIdx.x >> 5] = (int)lo;
      s.red[2][threadIdx.x >> 5] = ncand;
    }
    __syncthreads();
    lo = 0xFFFFFFFFu;
    int cand = 0;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) {
      lo = min(lo, (uint32_t)s.red[0][w]);
      cand += s.red[2][w];
    }
    want = min(m, cand);
    // per-thread counts of d = 0 .. 7 (4 bits each), widened to 16-bit fields of two
    // words for the block scan (totals <= 4096)
    uint32_t c4 = 0u;
#pragma unroll
    for (int e = 0; e < kV; ++e) {
      const uint32_t d = (uint32_t)(sv[e] + 1) - lo;
      if (sv[e] < p.step && d < 8u) c4 += 1u << (4u * d);
    }
    uint64_t wa = 0ull, wb = 0ull;
#pragma unroll
    for (int d = 0; d < 4; ++d) {
      wa |= (uint64_t)((c4 >> (4 * d)) & 15u) << (16 * d);
      wb |= (uint64_t)((c4 >> (4 * d + 16)) & 15u) << (16 * d);
    }
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    uint64_t xa = wa, xb = wb;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint64_t ya = __shfl_up_sync(0xffffffffu, xa, o);
      const uint64_t yb = __shfl_up_sync(0xffffffffu, xb, o);
      if (lane >= o) {
        xa += ya;
        xb += yb;
      }
    }
    if (lane == 31) {
      s.wsum2[0][w] = xa;
      s.wsum2[1][w] = xb;
    }
    __syncthreads();
    uint64_t ba = xa - wa, bb = xb - wb, ta = 0ull, tb = 0ull;
#pragma unroll
    for (int i = 0; i < kThreads / 32; ++i) {
      if (i < w) {
        ba += s.wsum2[0][i];
        bb += s.wsum2[1][i];
      }
      ta += s.wsum2[0][i];
      tb += s.wsum2[1][i];
    }
    // first rank of offset d (the totals of the offsets below it) plus this thread's
    // exclusive prefix, per 16-bit field: exclusive prefix sums inside a word by
    // shifted adds (no field exceeds 2 * 4096)
    constexpr uint64_t kOnes = 0x0001000100010001ull;
    const uint64_t total_a = ((ta * kOnes) >> 48) & 0xFFFFull;
    const int run = (int)(total_a + (((tb * kOnes) >> 48) & 0xFFFFull));
    const uint64_t fa = (ta << 16) + (ta << 32) + (ta << 48) + ba;
    const uint64_t fb = total_a * kOnes + (tb << 16) + (tb << 32) + (tb << 48) + bb;
    const bool fast = run >= want;  // the same in every thread
    if (fast) {
      uint32_t seen = 0u;  // this thread's earlier candidates per offset (4 bits each)
#pragma unroll
      for (int e = 0; e < kV; ++e) {
        const uint32_t d = (uint32_t)(sv[e] + 1) - lo;
        if (sv[e] < p.step && d < 8u) {
          const int rank = (int)(((d < 4u ? fa : fb) >> (16u * (d & 3u))) & 0xFFFFull) +
                           (int)((seen >> (4u * d)) & 15u);
          seen += 1u << (4u * d);
          if (rank < want)
            s.vkeys[rank] = ((uint64_t)(uint32_t)(sv[e] + 1) << 32) | (uint32_t)(h0 + e);
        }
      }
      victims = s.vkeys;
      __syncthreads();
    } else {
      // General order: slots unused at this step by (last step, slot), padded to 2^n
      int n = 1;
      while (n < p.hot) n <<= 1;
      constexpr int kS = kMaxHot / kThreads;
      int st[kS];
  #pragma unroll
      for (int e = 0; e < kS; ++e) {  // hits of this step are written above (same block)
        const int hh = threadIdx.x + e * kThreads;
        st[e] = hh < p.hot ? hstep[hh] : p.step;
      }
  #pragma unroll
      for (int e = 0; e < kS; ++e) {
        const int hh = threadIdx.x + e * kThreads;
        if (hh < n)
          s.keys[hh] = st[e] < p.step ? ((uint64_t)(uint32_t)(st[e] + 1) << 32) | (uint32_t)hh
                                      : kNone;
      }
      __syncthreads();
      // The misses need only the m oldest keys. When the candidates' steps span less than
      // 2^20, each key fits 32 bits ((step - oldest step) << 12 | slot, unique): a radix
      // select in four 8-bit passes finds the m-th smallest, the keys up to it are
      // compacted (exactly min(m, candidates) of them) and only those are sorted. Else
      // every key is sorted.
      uint32_t lo = 0xFFFFFFFFu, hi = 0u;
      int ncand = 0;
  #pragma unroll
      for (int e = 0; e < kS; ++e) {
        const int hh = threadIdx.x + e * kThreads;
        if (hh < n && s.keys[hh] != kNone) {
          const uint32_t stp = (uint32_t)(s.keys[hh] >> 32);
          lo = min(lo, stp);
          hi = max(hi, stp);
          ++ncand;
        }
      }
  #pragma unroll
      for (int o = 16; o; o >>= 1) {
        lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
        hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
        ncand += __shfl_xor_sync(0xffffffffu, ncand, o);
      }
      if ((threadIdx.x & 31) == 0) {
        s.red[0][threadIdx.x >> 5] = (int)lo;
        s.red[1][threadIdx.x >> 5] = (int)hi;
        s.red[2][threadIdx.x >> 5] = ncand;
      }
      __syncthreads();
      if (threadIdx.x == 0) {
        uint32_t l = 0xFFFFFFFFu, h2 = 0u;
        int c = 0;
        for (int w = 0; w < kThreads / 32; ++w) {
          l = min(l, (uint32_t)s.red[0][w]);
          h2 = max(h2, (uint32_t)s.red[1][w]);
          c += s.red[2][w];
        }
        s.sel[0] = (int)l;
        s.sel[1] = (int)h2;
        s.sel[2] = c;
      }
      __syncthreads();
      const uint32_t base = (uint32_t)s.sel[0];
      const int cand = s.sel[2];
      want = min(m, cand);  // victims to hand out
      const bool small = cand > 0 && (uint32_t)s.sel[1] - base < (1u << 20);
      victims = s.keys;  // sorted victim keys, victims[0 .. want)
      if (small && want > 0) {
        auto key32 = [&](uint64_t k64) -> uint32_t {
          return (((uint32_t)(k64 >> 32) - base) << 12) | ((uint32_t)k64 & 0xFFFu);
        };
        uint32_t prefix = 0u, mask = 0u;
        int need = want;
        for (int shift = 24; shift >= 0; shift -= 8) {
          for (int i = threadIdx.x; i < 256; i += kThreads) s.hist[i] = 0u;
          __syncthreads();
  #pragma unroll
          for (int e = 0; e < kS; ++e) {
            const int hh = threadIdx.x + e * kThreads;
            if (hh < n && s.keys[hh] != kNone) {
              const uint32_t k = key32(s.keys[hh]);
              if ((k & mask) == prefix) atomicAdd(&s.hist[(k >> shift) & 255u], 1u);
            }
          }
          __syncthreads();
          if (threadIdx.x < 32) {  // digit where the running count reaches `need`
            const int lane = threadIdx.x;
            int c[8], tot = 0;
  #pragma unroll
            for (int q = 0; q < 8; ++q) {
              c[q] = (int)s.hist[8 * lane + q];
              tot += c[q];
            }
            int incl = tot;
  #pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
              const int y = __shfl_up_sync(0xffffffffu, incl, o);
              if (lane >= o) incl += y;
            }
            int before = incl - tot;
            if (before < need && need <= incl) {
  #pragma unroll
              for (int q = 0; q < 8; ++q) {
                if (before + c[q] >= need) {
                  s.sel[3] = 8 * lane + q;
                  s.sel[4] = need - before;
                  break;
                }
                before += c[q];
              }
            }
          }
          __syncthreads();
          prefix |= (uint32_t)s.sel[3] << shift;
          mask |= 255u << shift;
          need = s.sel[4];
          __syncthreads();
        }
        // compact the victims (key32 <= prefix: exactly `want` keys), then sort them
        if (threadIdx.x == 0) s.sel[5] = 0;
        __syncthreads();
  #pragma unroll
        for (int e = 0; e < kS; ++e) {
          const int hh = threadIdx.x + e * kThreads;
          if (hh < n && s.keys[hh] != kNone && key32(s.keys[hh]) <= prefix)
            s.vkeys[atomicAdd(&s.sel[5], 1)] = s.keys[hh];
        }
        __syncthreads();
        int nv = 1;
        while (nv < want) nv <<= 1;
        for (int i = want + threadIdx.x; i < nv; i += kThreads) s.vkeys[i] = kNone;
        __syncthreads();
        victims = s.vkeys;
        n = nv;
      }
      // Bitonic sort by pairs of victims[0 .. n): stage (k2, j2) compares keys i and
      // i + j2 for every i whose bit j2 is clear, ascending where bit k2 of i is clear.
      // Each thread takes pairs t, t + 512, ... and loads all of them before it stores.
      constexpr int kP = kMaxHot / 2 / kThreads;
      const int pairs = n >> 1;
      for (int k2 = 2; k2 <= n; k2 <<= 1) {
        for (int j2 = k2 >> 1; j2 > 0; j2 >>= 1) {
          uint64_t a[kP], b[kP];
          int ia[kP];
  #pragma unroll
          for (int e = 0; e < kP; ++e) {
            const int pi = threadIdx.x + e * kThreads;
            ia[e] = -1;
            if (pi < pairs) {
              const int i = ((pi & ~(j2 - 1)) << 1) | (pi & (j2 - 1));
              ia[e] = i;
              a[e] = victims[i];
              b[e] = victims[i + j2];
            }
          }
  #pragma unroll
          for (int e = 0; e < kP; ++e) {
            if (ia[e] < 0) continue;
            const bool up = (ia[e] & k2) == 0;
            if ((a[e] > b[e]) == up) {
              victims[ia[e]] = b[e];
              victims[ia[e] + j2] = a[e];
            }
          }
          __syncthreads();
        }
      }

    }
    // 4. miss rank r takes victim r: maps, step, output row, the copy to make
    const int64_t hb = p.host_base[j];
    for (int rr = threadIdx.x; rr < m; rr += kThreads) {
      const int i = s.miss_entry[rr];
      const int q = pos[i];
      s.copy_src[rr] = -1;
      s.copy_dst[rr] = -1;
      const uint64_t key = rr < want ? victims[rr] : kNone;
      if (key == kNone) {
        err |= RESOLVER_STATUS_NO_VICTIM;
        continue;
      }
      const int64_t hr = hb + q;
      if (hr < 0 || hr >= p.host_rows) {
        err |= RESOLVER_STATUS_HOST_ROW;
        continue;
      }
      const int v = (int)(uint32_t)key;
      const int32_t kr = hrows[v];
      if (kr < 0 || (int64_t)kr >= p.kv_rows) {
        err |= RESOLVER_STATUS_KV_ROW;
        continue;
      }
      const int old = htok[v];
      if (old >= 0 && (int64_t)old < p.map_ld) t2h[old] = -1;  // not selected this step
      htok[v] = q;
      t2h[q] = v;
      hstep[v] = p.step;
      out[i] = kr;
      s.copy_src[rr] = hr;
      s.copy_dst[rr] = kr;
    }
    __syncthreads();

    for (int rr = threadIdx.x; rr < m; rr += kThreads) n_copy += s.copy_src[rr] >= 0 ? 1 : 0;
  }
  // 5. copies of this row's misses, over the request's CTAs
  if (threadIdx.x == 0) s.n_list = m;
  if (p.csize > 1) {
    cluster_sync();
    copy_rows(p, s, 0, m);
    cluster_sync();
  } else {
    __syncthreads();
    copy_rows(p, s, 0, m);
  }
  __syncthreads();  // this row's state writes are seen by the next row
  }  // query rows

  // 6. counts and status (misses copied = assigned copies), over all query rows
  if (p.counts || p.status) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    int v0 = n_res, v1 = n_hit, v2 = n_copy, v3 = err;
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      v0 += __shfl_xor_sync(0xffffffffu, v0, o);
      v1 += __shfl_xor_sync(0xffffffffu, v1, o);
      v2 += __shfl_xor_sync(0xffffffffu, v2, o);
      v3 |= __shfl_xor_sync(0xffffffffu, v3, o);
    }
    if (lane == 0) {
      s.red[0][w] = v0;
      s.red[1][w] = v1;
      s.red[2][w] = v2;
      s.red[3][w] = v3;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      int a = 0, b = 0, c = 0, e = 0;
      for (int i = 0; i < kThreads / 32; ++i) {
        a += s.red[0][i];
        b += s.red[1][i];
        c += s.red[2][i];
        e |= s.red[3][i];
      }
      if (p.counts) {
        p.counts[3 * j + 0] = a;
        p.counts[3 * j + 1] = b;
        p.counts[3 * j + 2] = c;
      }
      if (e && p.status) atomicOr(p.status, e);
    }
  }
}

bool aligned(const void* q, uintptr_t a) { return (reinterpret_cast<uintptr_t>(q) % a) == 0; }

int resolve_launch(const int32_t* positions, int rows, int q_rows, int k, const int32_t* block_table,
                   int64_t table_ld, int page_size, int32_t* token_to_hot, int64_t map_ld,
                   int32_t* hot_token, int32_t* hot_step, const int32_t* hot_rows, int hot_size,
                   int step, const uint8_t* host_kv, const int64_t* host_base, int64_t host_rows,
                   uint8_t* kv, int64_t kv_rows, int row_bytes, int32_t* out_rows, int32_t* counts,
                   int32_t* status, resolver_stream_t stream) {
  if (rows < 0 || q_rows < 1 || k < 1 || k > kMaxK || hot_size < 1 || hot_size > kMaxHot || page_size < 1 ||
      table_ld < 1 || map_ld < 1 || step < 0 || row_bytes < 16 || (row_bytes & 15) ||
      kv_rows < 0 || host_rows < 0)
    return RESOLVER_ERR_SHAPE;
  if (rows == 0) return RESOLVER_OK;
  if (!positions || !block_table || !token_to_hot || !hot_token || !hot_step || !hot_rows ||
      !host_kv || !host_base || !kv || !out_rows)
    return RESOLVER_ERR_NULL;
  if (!aligned(kv, 16) || !aligned(host_kv, 16) || !aligned(host_base, 8) ||
      !aligned(positions, 4) || !aligned(block_table, 4) || !aligned(token_to_hot, 4) ||
      !aligned(hot_token, 4) || !aligned(hot_step, 4) || !aligned(hot_rows, 4) ||
      !aligned(out_rows, 4) || (counts && !aligned(counts, 4)) || (status && !aligned(status, 4)))
    return RESOLVER_ERR_ALIGN;
  static bool attr_set = false;  // the attribute is per function, process-wide
  if (!attr_set) {
    if (cudaFuncSetAttribute(resolve_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)sizeof(Smem)) != cudaSuccess ||
        cudaFuncSetAttribute(resolve_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)sizeof(Smem)) != cudaSuccess)
      return RESOLVER_ERR_CUDA;
    attr_set = true;
  }
  // CTAs per request: the largest cluster size (8, 4, 2) that keeps every request's
  // cluster resident at once (one CTA per SM), else 1.
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return RESOLVER_ERR_CUDA;
  int csize = 8;
  while (csize > 1 && (int64_t)rows * csize > sms) csize >>= 1;
  Params p{positions, rows,     k,        block_table, table_ld,  page_size, token_to_hot,
           map_ld,    hot_token, hot_step, hot_rows,    hot_size,  step,      host_kv,
           host_base, host_rows, kv,       kv_rows,     row_bytes, out_rows,  counts,
           status,    q_rows,    csize};
  void (*fn)(Params) = q_rows == 1 ? resolve_kernel<false> : resolve_kernel<true>;
  if (csize > 1) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)csize;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3((unsigned)(rows * csize));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = sizeof(Smem);
    cfg.stream = (cudaStream_t)stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, fn, p) == cudaSuccess) return RESOLVER_OK;
    (void)cudaGetLastError();  // clusters refused: one CTA per request
    p.csize = 1;
  }
  fn<<<rows, kThreads, sizeof(Smem), (cudaStream_t)stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? RESOLVER_OK : RESOLVER_ERR_CUDA;
}

}  // namespace

extern "C" int hisparse_resolve(const int32_t* positions, int rows, int k,
                                const int32_t* block_table, int64_t table_ld, int page_size,
                                int32_t* token_to_hot, int64_t map_ld, int32_t* hot_token,
                                int32_t* hot_step, const int32_t* hot_rows, int hot_size, int step,
                                const uint8_t* host_kv, const int64_t* host_base,
                                int64_t host_rows, uint8_t* kv, int64_t kv_rows, int row_bytes,
                                int32_t* out_rows, int32_t* counts, int32_t* status,
                                resolver_stream_t stream) {
  return resolve_launch(positions, rows, 1, k, block_table, table_ld, page_size, token_to_hot,
                        map_ld, hot_token, hot_step, hot_rows, hot_size, step, host_kv, host_base,
                        host_rows, kv, kv_rows, row_bytes, out_rows, counts, status, stream);
}

extern "C" int hisparse_resolve_mtp(const int32_t* positions, int rows, int q_rows, int k,
                                    const int32_t* block_table, int64_t table_ld, int page_size,
                                    int32_t* token_to_hot, int64_t map_ld, int32_t* hot_token,
                                    int32_t* hot_step, const int32_t* hot_rows, int hot_size,
                                    int step, const uint8_t* host_kv, const int64_t* host_base,
                                    int64_t host_rows, uint8_t* kv, int64_t kv_rows, int row_bytes,
                                    int32_t* out_rows, int32_t* counts, int32_t* status,
                                    resolver_stream_t stream) {
  return resolve_launch(positions, rows, q_rows, k, block_table, table_ld, page_size, token_to_hot,
                        map_ld, hot_token, hot_step, hot_rows, hot_size, step, host_kv, host_base,
                        host_rows, kv, kv_rows, row_bytes, out_rows, counts, status, stream);
}
