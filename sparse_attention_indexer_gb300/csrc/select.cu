// Select + page-table kernel for GB300 (sm_103a).
//
// "Serving GLM5.2 NVFP4 Agentic Workload with SGLang", "Kernel Optimization >
// TopK-V2" (Figs. 2-3): each row's scores are binned by an order-preserving unsigned
// key into a coarse radix histogram; the histograms of the CTAs sharing a row are
// reduced to find the bin holding the k-th largest score; values above that bin are
// emitted directly, the boundary bin is refined exactly on the fp32 key with a radix
// tie-break, and every selected logical position is translated to a physical
// indexer KV-cache slot in the same kernel.
//
// One persistent, co-resident grid (one 512-thread CTA per SM). Each CTA first runs
// its static multi-CTA units (wave order), then single-CTA rows: one handed to it by
// the plan, then more claimed from a ticket counter. A unit's chunk of scores is
// brought into shared memory by bulk async copies (one mbarrier per 16 KB piece) and
// stays resident for every later pass, so HBM is read once.
//
// Multi-CTA rows publish the histogram bins at or above each CTA's own local
// threshold bin (the row's threshold cannot lie lower) and meet at a bounded spin
// barrier (co-residency is guaranteed by the cooperative launch). The row's last CTA
// to finish ranks the boundary candidates exactly and clears the row's counters.
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"

namespace topk {

namespace {

#ifdef TOPK_TRACE
__device__ uint64_t g_select_trace[kMaxGrid * 16];
// Per-CTA event log: (row + 1) << 44 | event << 40 | low 40 bits of %globaltimer.
__device__ uint64_t g_select_log[kMaxGrid * 64];
__device__ int g_select_log_n[kMaxGrid];
#define TOPK_LOG(row, ev)                                                              \
  do {                                                                                 \
    if (threadIdx.x == 0) {                                                            \
      const int n_ = g_select_log_n[blockIdx.x];                                       \
      if (n_ < 64)                                                                     \
        g_select_log[blockIdx.x * 64 + n_] = ((uint64_t)((row) + 1) << 44) |           \
                                             ((uint64_t)(ev) << 40) |                  \
                                             (global_timer_ns() & 0xFFFFFFFFFFull);    \
      g_select_log_n[blockIdx.x] = n_ + 1;                                             \
    }                                                                                  \
  } while (0)
#else
#define TOPK_LOG(row, ev) \
  do {                    \
  } while (0)
#endif

enum : uint8_t { kRej = 0, kActive = 1, kSel = 2 };

// Shared memory. After the coarse threshold is known the histogram region is reused
// for the unit's staging lists (emitted positions, boundary candidates).
struct __align__(16) Smem {
  float buf[kBufFloats];
  union {
    uint32_t hist[kBins0];
    struct {
      int32_t elist[TOPK_MAX_K];  // positions to emit (above the threshold bin)
      uint32_t ckey[kListCap];    // boundary candidates: key
      uint32_t cpos[kListCap];    //                      position
    } l;
  } u;
  uint8_t cst[kGroupCap];         // list-selection state
  uint32_t hist8[kListBins];
  uint64_t mbar[kPieces];
  int wsum[kWarps];
  int wsum2[kWarps];
  uint32_t wand[kWarps];
  uint32_t wor[kWarps];
  int bc[32];
  UnitDesc ud;
};
static_assert(sizeof(int32_t) * TOPK_MAX_K + 2 * sizeof(uint32_t) * kListCap <=
                  sizeof(uint32_t) * kBins0,
              "staging lists must fit the histogram region");

// ------------------------------------------------------------- keys and digits

// Order-preserving 32-bit key: larger key <=> larger score. -0.0 is folded onto
// +0.0; every NaN maps to 0, below -inf (0x007FFFFF).
__device__ __forceinline__ uint32_t f2key(float x) {
  const uint32_t u = __float_as_uint(x);
  const uint32_t a = u & 0x7FFFFFFFu;
  if (a > 0x7F800000u) return 0u;
  if (a == 0u) return 0x80000000u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Coarse 12-bit digit, monotone non-decreasing in the score: sign, a 5-bit exponent
// window (|x| in [2^-15, 2^17)) and 6 mantissa bits, clamped at both ends. Equal
// scores share a digit (-0 is folded onto +0 by adding +0); NaN is first mapped to
// -inf, which together with every score at or below -2^17 lands in bin 0.
__device__ __forceinline__ uint32_t coarse_digit(float x) {
  const float xc = __fadd_rn(fmaxf(x, __int_as_float(0xFF800000)), 0.0f);
  const float ax = fminf(fmaxf(fabsf(xc), 3.0517578125e-05f), 131071.99f);
  const uint32_t m = (__float_as_uint(ax) >> 17) - 7168u;  // in [0, 2047]
  const uint32_t s = (uint32_t)((int32_t)__float_as_uint(xc) >> 31);
  return ((m ^ s) ^ 0x800u) & 0xFFFu;
}

// A float t such that x < t implies coarse_digit(x) < b (a conservative filter used
// to skip vectors without computing digits). NaN never satisfies x < t.
__device__ __forceinline__ float skip_below(uint32_t b) {
  if (b == 0u) return __uint_as_float(0xFF800000u);  // -inf: nothing is skipped
  if (b < 2048u) {
    const uint32_t j = 2048u - b;  // (2047 - b) + 1, in [1, 2047]
    return -__uint_as_float((j + 7168u) << 17);
  }
  if (b == 2048u) return 0.0f;
  return __uint_as_float(((b - 2048u) + 7168u) << 17);
}

// ------------------------------------------------------------- block helpers

__device__ __forceinline__ int warp_incl_scan(int x) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  return x;
}

// Exclusive scan over the CTA in thread order; *total gets the CTA sum.
__device__ int block_excl_scan(int v, int* total, Smem& s) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int incl = warp_incl_scan(v);
  if (lane == 31) s.wsum[w] = incl;
  __syncthreads();
  if (w == 0) {
    const int x = lane < kWarps ? s.wsum[lane] : 0;
    const int y = warp_incl_scan(x);
    if (lane < kWarps) s.wsum2[lane] = y;
  }
  __syncthreads();
  const int before = w > 0 ? s.wsum2[w - 1] : 0;
  *total = s.wsum2[kWarps - 1];
  __syncthreads();
  return before + incl - v;
}

__device__ int block_sum(int v, Smem& s) {
  int t;
  block_excl_scan(v, &t, s);
  return t;
}

__device__ void block_and_or(uint32_t& a, uint32_t& o, Smem& s) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
  for (int d = 16; d; d >>= 1) {
    a &= __shfl_xor_sync(0xffffffffu, a, d);
    o |= __shfl_xor_sync(0xffffffffu, o, d);
  }
  if (lane == 0) {
    s.wand[w] = a;
    s.wor[w] = o;
  }
  __syncthreads();
  uint32_t ta = 0xFFFFFFFFu, to = 0u;
#pragma unroll
  for (int i = 0; i < kWarps; ++i) {
    ta &= s.wand[i];
    to |= s.wor[i];
  }
  __syncthreads();
  a = ta;
  o = to;
}

// Warp-aggregated append: every lane with `pred` gets a distinct slot of `counter`
// (one shared atomic per warp). All 32 lanes must call it.
__device__ __forceinline__ int warp_append(bool pred, int* counter) {
  const unsigned m = __ballot_sync(0xffffffffu, pred);
  if (m == 0u) return -1;
  const int lane = threadIdx.x & 31;
  const int leader = __ffs(m) - 1;
  int base = 0;
  if (lane == leader) base = atomicAdd(counter, __popc(m));
  base = __shfl_sync(0xffffffffu, base, leader);
  return pred ? base + __popc(m & ((1u << lane) - 1u)) : -1;
}

__device__ __forceinline__ void set_status(Header* h, int bits) { atomicOr(&h->status, bits); }

// Records the first expired wait of this plan (thread 0 only).
__device__ void record_timeout(Header* h, int kind, int row, int rank, int seq, int seen,
                               int target) {
  if (atomicCAS(&h->diag[0], 0, kind) == 0) {
    h->diag[1] = row;
    h->diag[2] = rank;
    h->diag[3] = seq;
    h->diag[4] = seen;
    h->diag[5] = target;
    h->diag[6] = (int)blockIdx.x;
  }
}

// ------------------------------------------------------------- per-unit context

struct Unit {
  int r, rank, G, L, kr, t, s0, n, head, nvec, npieces;
  GroupState* gs;
  uint32_t bar_seq;  // barriers passed in this unit
};

struct Ctx {
  const SelectParams& p;
  Header* h;
  Smem& s;
  uint32_t mphase;  // parity bits of the piece mbarriers
};

// Writes one selected position p at output index idx of the unit's row.
__device__ __forceinline__ void emit(const Ctx& c, const Unit& u, int idx, int p) {
  const SelectParams& P = c.p;
  if ((unsigned)idx >= (unsigned)P.k || (unsigned)p >= (unsigned)u.L) return;  // never taken
  const int32_t page = __ldg(P.table + (int64_t)u.t * P.table_ld + p / P.page_size);
  int32_t slot;
  if (page < 0) {
    set_status(c.h, TOPK_STATUS_TABLE_ENTRY);
    slot = -1;
  } else {
    const int64_t sl = (int64_t)page * P.page_size + p % P.page_size;
    if (sl > 0x7FFFFFFFll) {
      set_status(c.h, TOPK_STATUS_SLOT_OVERFLOW);
      slot = -1;
    } else {
      slot = (int32_t)sl;
    }
  }
  const int64_t o = (int64_t)u.r * P.k + idx;
  P.out_slots[o] = slot;
  if (P.out_pos) P.out_pos[o] = p;
}

__device__ void fill_row(const Ctx& c, int r, int from, int to) {
  const SelectParams& P = c.p;
  for (int i = from + threadIdx.x; i < to; i += kThreads) {
    const int64_t o = (int64_t)r * P.k + i;
    P.out_slots[o] = -1;
    if (P.out_pos) P.out_pos[o] = -1;
  }
}

// Group barrier among the G CTAs of a row. All threads call it; a thread that wrote
// row state to global memory (histogram reductions, candidates, counts) passes
// wrote = true and fences its own writes first, so that they are performed before
// thread 0 releases the arrival (a release by one thread does not order other
// warps' writes still in flight). The waiting side acquires. Returns false if the
// bounded wait expired (status set).
__device__ bool group_barrier(Ctx& c, Unit& u, bool wrote) {
  if (wrote) __threadfence();
  __syncthreads();
  u.bar_seq += 1;
  if (threadIdx.x == 0) {
    const uint32_t target = (uint32_t)u.G * u.bar_seq;
    red_release_add_u32(&u.gs->bar, 1u);
    bool ok = ld_acquire_u32(&u.gs->bar) >= target;
    if (!ok) {
      const uint64_t t0 = global_timer_ns();
      while (true) {
        if (ld_acquire_u32(&u.gs->bar) >= target) {
          ok = true;
          break;
        }
        if (global_timer_ns() - t0 > kWaitNs) break;
      }
    }
    c.s.bc[15] = ok ? 1 : 0;
    if (!ok) {
      set_status(c.h, TOPK_STATUS_TIMEOUT);
      record_timeout(c.h, 1, u.r, u.rank, (int)u.bar_seq, (int)ld_acquire_u32(&u.gs->bar),
                     (int)target);
    }
  }
  __syncthreads();
  return c.s.bc[15] != 0;
}

// Finds bin b of a 4096-bin histogram (8 bins per thread, counts in v[]) with
// above(b) < need <= above(b) + hist[b]; above(b) counts bins > b. Results land in
// s.bc[0..2] = (b, above, eq). Requires 1 <= need <= total.
__device__ void find_threshold(const uint32_t (&v)[8], int need, Smem& s) {
  int sum = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) sum += (int)v[j];
  int total;
  const int excl = block_excl_scan(sum, &total, s);
  const int above_t = total - excl - sum;  // bins owned by higher threads
  if (above_t < need && need <= above_t + sum) {
    int cum = above_t;
#pragma unroll
    for (int j = 7; j >= 0; --j) {
      if (cum + (int)v[j] >= need) {
        s.bc[0] = threadIdx.x * 8 + j;
        s.bc[1] = cum;
        s.bc[2] = (int)v[j];
        break;
      }
      cum += (int)v[j];
    }
  }
  __syncthreads();
}

__device__ __forceinline__ void load8(const uint32_t* p, uint32_t (&v)[8]) {
  const uint4 x = *reinterpret_cast<const uint4*>(p);
  const uint4 y = *reinterpret_cast<const uint4*>(p + 4);
  v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
  v[4] = y.x; v[5] = y.y; v[6] = y.z; v[7] = y.w;
}

__device__ __forceinline__ void load8_cg(const uint32_t* p, uint32_t (&v)[8]) {
  const uint4 x = __ldcg(reinterpret_cast<const uint4*>(p));
  const uint4 y = __ldcg(reinterpret_cast<const uint4*>(p + 4));
  v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
  v[4] = y.x; v[5] = y.y; v[6] = y.z; v[7] = y.w;
}

// Threshold of the unit's row from the local histogram in s.u.hist. For G > 1 a CTA
// whose chunk holds at least `need` values first finds its own threshold bin for
// `need` values; the row's threshold cannot lie below it (the row has at least as
// many values at or above it), so the CTA publishes only the bins at or above it to
// `ghist` and reads back only those. A CTA with fewer values publishes and reads
// every bin. Every bin at or above the row threshold is then complete in `ghist`.
// `sparse` = false publishes every nonzero bin.
// Outputs b, above, eq (row-wide) and local_above, local_eq. False on timeout.
__device__ bool reduce_and_find(Ctx& c, Unit& u, uint32_t* ghist, int need, int local_n,
                                bool sparse, int& b, int& above, int& eq, int& local_above,
                                int& local_eq) {
  Smem& s = c.s;
  uint32_t loc[8], glob[8];
  const int b0 = threadIdx.x * 8;
  load8(&s.u.hist[b0], loc);
  if (u.G > 1) {
    // Own threshold bin: only meaningful when this chunk alone holds `need` values;
    // then the row's threshold cannot lie below it. Otherwise every bin counts.
    int blocal = 0;
    if (sparse && local_n >= need) {
      find_threshold(loc, need, s);
      blocal = s.bc[0];
    }
    bool wrote = false;
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (loc[j] && b0 + j >= blocal) {
        red_add_u32(&ghist[b0 + j], loc[j]);
        wrote = true;
      }
    if (!group_barrier(c, u, wrote)) return false;
    if (b0 + 7 >= blocal) {
      load8_cg(&ghist[b0], glob);
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) glob[j] = 0u;
    }
  } else {
#pragma unroll
    for (int j = 0; j < 8; ++j) glob[j] = loc[j];
  }
  find_threshold(glob, need, s);
  b = s.bc[0];
  above = s.bc[1];
  eq = s.bc[2];
  int la = 0, le = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    if (b0 + j > b) la += (int)loc[j];
    if (b0 + j == b) le = (int)loc[j];
  }
  if (b >= b0 && b < b0 + 8) s.bc[3] = le;
  local_above = block_sum(la, s);  // its CTA barriers also publish bc[3]
  local_eq = s.bc[3];
  __syncthreads();
  return true;
}

// ------------------------------------------------------------- chunk loading

// Thread 0 issues the bulk copies of the unit's chunk [s0, s0 + n) of row r.
__device__ void issue_chunk(Ctx& c, Unit& u) {
  Smem& s = c.s;
  const SelectParams& P = c.p;
  const float* src = P.scores + (int64_t)u.r * P.ld + u.s0;
  const uintptr_t A = reinterpret_cast<uintptr_t>(src);
  const uintptr_t A0 = A & ~uintptr_t(15);
  const uintptr_t A1 = (A + 4ull * (uint64_t)u.n + 15ull) & ~uintptr_t(15);
  const uint32_t bytes = u.n > 0 ? (uint32_t)(A1 - A0) : 0u;
  u.head = (int)((A - A0) >> 2);
  u.nvec = (int)(bytes >> 4);
  u.npieces = (int)((bytes + kPieceBytes - 1) / kPieceBytes);
  if (threadIdx.x == 0) {
    fence_proxy_async_smem();
    for (int i = 0; i < u.npieces; ++i) {
      const uint32_t off = (uint32_t)i * kPieceBytes;
      const uint32_t sz = min((uint32_t)kPieceBytes, bytes - off);
      mbar_arrive_expect_tx(&s.mbar[i], sz);
      bulk_g2s(reinterpret_cast<char*>(s.buf) + off, reinterpret_cast<const char*>(A0) + off, sz,
               &s.mbar[i]);
    }
  }
}

__device__ __forceinline__ void wait_piece(Ctx& c, int i) {
  const uint32_t par = (c.mphase >> i) & 1u;
  if (!mbar_wait_bounded(&c.s.mbar[i], par)) {
    if (threadIdx.x == 0) {
      set_status(c.h, TOPK_STATUS_TIMEOUT);
      record_timeout(c.h, 2, -1, i, (int)par, 0, 0);
    }
    mbar_wait_bounded(&c.s.mbar[i], par);
  }
  c.mphase ^= (1u << i);
}

// Waits for every piece of the unit (used when a unit is abandoned after its copies
// were issued: shared memory must not be reused while copies are in flight).
__device__ void drain_chunk(Ctx& c, Unit& u) {
  for (int i = 0; i < u.npieces; ++i) wait_piece(c, i);
  __syncthreads();
}

// Adds a full float4's digits. A warp whose 128 values share one digit adds them
// with one atomic (all-equal rows, -inf tails); otherwise one atomic per value.
// All 32 lanes must call it.
__device__ __forceinline__ void hist_add4(Smem& s, uint32_t d0, uint32_t d1, uint32_t d2,
                                          uint32_t d3, bool full) {
  const int lane = threadIdx.x & 31;
  const bool uni = full && d0 == d1 && d1 == d2 && d2 == d3;
  const uint32_t dl = __shfl_sync(0xffffffffu, d0, 0);
  if (__all_sync(0xffffffffu, uni && d0 == dl)) {
    if (lane == 0) atomicAdd(&s.u.hist[d0], 128u);
  } else if (full) {
    atomicAdd(&s.u.hist[d0], 1u);
    atomicAdd(&s.u.hist[d1], 1u);
    atomicAdd(&s.u.hist[d2], 1u);
    atomicAdd(&s.u.hist[d3], 1u);
  }
}

// Waits for the pieces as they land and builds the coarse histogram of the chunk in
// s.u.hist (zeroed by the caller before the CTA barrier that precedes this call).
__device__ void histogram_chunk(Ctx& c, Unit& u) {
  Smem& s = c.s;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const float4* b4 = reinterpret_cast<const float4*>(s.buf);
  constexpr int kVecPerPiece = kPieceBytes / 16;
  // Vectors [vfull0, vfull1) hold only chunk elements; the first and last vectors may
  // be partial.
  const int vfull0 = (u.head + 3) >> 2;
  const int vfull1 = (u.head + u.n) >> 2;
#ifdef TOPK_TRACE
  uint64_t waited = 0;
#endif
  for (int i = 0; i < u.npieces; ++i) {
#ifdef TOPK_TRACE
    const uint64_t w0 = global_timer_ns();
#endif
    wait_piece(c, i);
#ifdef TOPK_TRACE
    waited += global_timer_ns() - w0;
    if (threadIdx.x == 0 && i == u.npieces - 1)
      g_select_trace[blockIdx.x * 16 + 11] = global_timer_ns();
#endif
    const int vbeg = i * kVecPerPiece;
    const int vend = min(vbeg + kVecPerPiece, u.nvec);
    for (int vb = vbeg + warp * 32; vb < vend; vb += kThreads) {
      const int v = vb + lane;
      if (vb + 32 <= vend && vb >= vfull0 && vb + 32 <= vfull1) {
        const float4 x = b4[v];
        hist_add4(s, coarse_digit(x.x), coarse_digit(x.y), coarse_digit(x.z),
                  coarse_digit(x.w), true);
      } else {
        const bool act = v < vend;
        float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
        if (act) x = b4[v];
        const int e0 = 4 * v - u.head;
        const bool full = act && e0 >= 0 && e0 + 3 < u.n;
        const uint32_t d0 = coarse_digit(x.x), d1 = coarse_digit(x.y);
        const uint32_t d2 = coarse_digit(x.z), d3 = coarse_digit(x.w);
        hist_add4(s, d0, d1, d2, d3, full);
        if (act && !full) {
          if (e0 >= 0 && e0 < u.n) atomicAdd(&s.u.hist[d0], 1u);
          if (e0 + 1 >= 0 && e0 + 1 < u.n) atomicAdd(&s.u.hist[d1], 1u);
          if (e0 + 2 >= 0 && e0 + 2 < u.n) atomicAdd(&s.u.hist[d2], 1u);
          if (e0 + 3 >= 0 && e0 + 3 < u.n) atomicAdd(&s.u.hist[d3], 1u);
        }
      }
    }
  }
#ifdef TOPK_TRACE
  if (threadIdx.x == 0) g_select_trace[blockIdx.x * 16 + 10] = waited;
#endif
  __syncthreads();
}

// ------------------------------------------------------------- boundary selection

// Exact selection among n <= kRankMax candidates: candidate i is taken iff fewer
// than `need` candidates rank before it (larger key, or equal key and smaller
// position); it goes to output index base + its rank (deterministic order).
__device__ void rank_select_emit(Ctx& c, const Unit& u, const uint32_t* key, const uint32_t* pos,
                                 int n, int need, int base) {
  for (int i = threadIdx.x; i < n; i += kThreads) {
    const uint32_t ki = key[i], pi = pos[i];
    int rank = 0;
    for (int j = 0; j < n; ++j) {
      const uint32_t kj = key[j], pj = pos[j];
      rank += (kj > ki || (kj == ki && pj < pi)) ? 1 : 0;
    }
    if (rank < need) emit(c, u, base + rank, (int)pi);
  }
}

// Among list entries [0, n) marks exactly `need` entries kSel: the largest keys, ties
// to the smaller position. Radix passes of 8 bits start at the highest bit where the
// active entries differ.
__device__ void list_select(Smem& s, const uint32_t* key, const uint32_t* pos, uint8_t* st,
                            int n, int need) {
  for (int i = threadIdx.x; i < n; i += kThreads) st[i] = kActive;
  __syncthreads();
  for (int phase = 0; phase < 2 && need > 0; ++phase) {
    uint32_t a = 0xFFFFFFFFu, o = 0u;
    for (int i = threadIdx.x; i < n; i += kThreads)
      if (st[i] == kActive) {
        const uint32_t v = phase == 0 ? key[i] : ~pos[i];
        a &= v;
        o |= v;
      }
    block_and_or(a, o, s);
    if (a == o) continue;  // all active equal: decided by the next phase
    int hb = 31 - __clz(a ^ o);
    while (true) {
      const int shift = max(hb - 7, 0);
      const uint32_t dmask = (1u << (hb - shift + 1)) - 1u;
      for (int i = threadIdx.x; i < kListBins; i += kThreads) s.hist8[i] = 0u;
      __syncthreads();
      for (int i = threadIdx.x; i < n; i += kThreads)
        if (st[i] == kActive) {
          const uint32_t v = phase == 0 ? key[i] : ~pos[i];
          atomicAdd(&s.hist8[(v >> shift) & dmask], 1u);
        }
      __syncthreads();
      if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        uint32_t cnt[8];
        int sum = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          cnt[j] = s.hist8[lane * 8 + j];
          sum += (int)cnt[j];
        }
        const int incl = warp_incl_scan(sum);
        const int total = __shfl_sync(0xffffffffu, incl, 31);
        const int above_t = total - incl;
        if (above_t < need && need <= above_t + sum) {
          int cum = above_t;
#pragma unroll
          for (int j = 7; j >= 0; --j) {
            if (cum + (int)cnt[j] >= need) {
              s.bc[4] = lane * 8 + j;
              s.bc[5] = cum;
              s.bc[6] = (int)cnt[j];
              break;
            }
            cum += (int)cnt[j];
          }
        }
      }
      __syncthreads();
      const uint32_t b = (uint32_t)s.bc[4];
      const int above = s.bc[5], eq = s.bc[6];
      need -= above;
      const bool take_eq = (eq == need);
      for (int i = threadIdx.x; i < n; i += kThreads)
        if (st[i] == kActive) {
          const uint32_t v = phase == 0 ? key[i] : ~pos[i];
          const uint32_t d = (v >> shift) & dmask;
          if (d > b || (take_eq && d == b))
            st[i] = kSel;
          else if (d < b)
            st[i] = kRej;
        }
      __syncthreads();
      if (take_eq) {
        need = 0;
        break;
      }
      if (shift == 0) break;
      hb = shift - 1;
    }
  }
  __syncthreads();
}

// Emits the kSel entries of a list at output indices base, base+1, ... Entries are
// dealt round-robin so that the table lookups of one CTA run in parallel.
__device__ void list_emit(Ctx& c, const Unit& u, const uint32_t* pos, const uint8_t* st, int n,
                          int base) {
  if (threadIdx.x == 0) c.s.bc[16] = 0;
  __syncthreads();
  for (int i0 = 0; i0 < n; i0 += kThreads) {
    const int i = i0 + threadIdx.x;
    const bool sel = i < n && st[i] == kSel;
    const int slot = warp_append(sel, &c.s.bc[16]);
    if (sel) emit(c, u, base + slot, (int)pos[i]);
  }
}

// Selects `need` of the n boundary candidates (keys/positions in shared memory, st
// scratch) and emits them from output index `base`.
__device__ void select_boundary(Ctx& c, const Unit& u, const uint32_t* key, const uint32_t* pos,
                                uint8_t* st, int n, int need, int base) {
  if (n <= kRankMax) {
    rank_select_emit(c, u, key, pos, n, need, base);
  } else {
    list_select(c.s, key, pos, st, n, need);
    list_emit(c, u, pos, st, n, base);
  }
}

// ------------------------------------------------------------- in-place fallback

// Boundary bin too large for a compact list (massive ties): refine in place on the
// full key, then take tied values in position order. fa/fo: AND/OR of the boundary
// keys over the row. `need` values remain to be chosen among coarse digit b0.
__device__ bool refine_in_place(Ctx& c, Unit& u, int b0, int need, int above0, uint32_t fa,
                                uint32_t fo, int local_eq0) {
  Smem& s = c.s;
  const float4* b4 = reinterpret_cast<const float4*>(s.buf);
  int emitted = above0;  // G == 1: running output index
  uint32_t pmask = 0u, pval = 0u;
  int local_tie = local_eq0;
  bool done = false;
  if (fa != fo) {
    int hb = 31 - __clz(fa ^ fo);
    pmask = hb == 31 ? 0u : ~((2u << hb) - 1u);
    pval = fa & pmask;
    for (int lev = 0; lev < 3 && !done; ++lev) {
      const int shift = max(hb - (kLevelBits - 1), 0);
      const uint32_t dmask = (1u << (hb - shift + 1)) - 1u;
      __syncthreads();
      for (int i = threadIdx.x; i < kBins0; i += kThreads) s.u.hist[i] = 0u;
      __syncthreads();
      for (int v = threadIdx.x; v < u.nvec; v += kThreads) {
        const float4 x = b4[v];
        const float xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int e = 4 * v - u.head + j;
          if (e < 0 || e >= u.n) continue;
          if (coarse_digit(xs[j]) != (uint32_t)b0) continue;
          const uint32_t key = f2key(xs[j]);
          if ((key & pmask) != pval) continue;
          atomicAdd(&s.u.hist[(key >> shift) & dmask], 1u);
        }
      }
      __syncthreads();
      if (u.G > 1 && threadIdx.x == 0) u.gs->levels = (uint32_t)(lev + 1);
      int bl, abl, eql, lal, lel;
      if (!reduce_and_find(c, u, u.G > 1 ? u.gs->hlev[lev] : nullptr, need, 0, false, bl, abl,
                           eql, lal, lel))
        return false;
      need -= abl;
      const bool take = (eql == need);
      if (threadIdx.x == 0) {
        const int cnt = lal + (take ? lel : 0);
        s.bc[7] = u.G > 1 ? (int)atomicAdd(&u.gs->out_ctr, (uint32_t)cnt) : emitted;
        s.bc[9] = 0;
      }
      __syncthreads();
      const int ob = s.bc[7];
      for (int v = threadIdx.x; v < u.nvec; v += kThreads) {
        const float4 x = b4[v];
        const float xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int e = 4 * v - u.head + j;
          if (e < 0 || e >= u.n) continue;
          if (coarse_digit(xs[j]) != (uint32_t)b0) continue;
          const uint32_t key = f2key(xs[j]);
          if ((key & pmask) != pval) continue;
          const uint32_t d = (key >> shift) & dmask;
          if (d > (uint32_t)bl || (take && d == (uint32_t)bl)) {
            const int idx = atomicAdd(&s.bc[9], 1);
            emit(c, u, ob + idx, u.s0 + e);
          }
        }
      }
      __syncthreads();
      emitted += abl + (take ? eql : 0);
      pmask |= dmask << shift;
      pval |= (uint32_t)bl << shift;
      local_tie = lel;
      if (take) done = true;
      else if (shift == 0) break;
      else hb = shift - 1;
    }
  } else {
    pmask = 0xFFFFFFFFu;
    pval = fa;
  }
  if (done) return true;
  // Every remaining candidate has key == pval. Take the `need` smallest positions
  // among them, across the row's chunks in position order.
  const uint32_t T = pval;
  int prefix = 0;
  if (u.G > 1) {
    if (threadIdx.x == 0) u.gs->tie_cnt[u.rank] = (uint32_t)local_tie;
    if (!group_barrier(c, u, threadIdx.x == 0)) return false;
    int acc = 0;
    for (int j = threadIdx.x; j < u.rank; j += kThreads) acc += (int)__ldcg(&u.gs->tie_cnt[j]);
    prefix = block_sum(acc, s);
  }
  const int tie_base = u.kr - need;  // every other entry fills [0, kr - need)
  int running = prefix;
  for (int t0 = 0; t0 < u.n && running < need; t0 += 4 * kThreads) {
    int cnt = 0;
    bool is_tie[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = t0 + 4 * threadIdx.x + j;
      is_tie[j] = e < u.n && f2key(s.buf[u.head + e]) == T;
      cnt += is_tie[j] ? 1 : 0;
    }
    int total;
    int rk = running + block_excl_scan(cnt, &total, s);
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (is_tie[j]) {
        if (rk < need) emit(c, u, tie_base + rk, u.s0 + t0 + 4 * threadIdx.x + j);
        ++rk;
      }
    running += total;
  }
  return true;
}

// ------------------------------------------------------------- the unit

__device__ void process_unit(Ctx& c, const UnitDesc& d) {
  const SelectParams& P = c.p;
  Smem& s = c.s;
  Unit u;
  u.r = d.row;
  u.rank = d.rank;
  u.G = d.G;
  u.s0 = d.s0;
  u.n = d.n;
  u.L = d.len;
  u.bar_seq = 0;
  u.head = 0;
  u.nvec = 0;
  u.npieces = 0;
  u.gs = (u.G > 1 && d.group >= 0)
             ? reinterpret_cast<GroupState*>(P.ws + make_layout(P.rows).groups) + d.group
             : nullptr;
  const bool valid_plan_len = u.L >= 0 && u.L <= P.max_len;
  const bool copy_all = valid_plan_len && u.L <= P.k;

  __syncthreads();  // the previous unit no longer uses shared memory
  TOPK_LOG(u.r, 1);
  // Issue the chunk's copies first: [s0, s0 + n) lies inside the row by construction
  // of the plan, which the kernel validated against rows / max_len.
  if (!copy_all && valid_plan_len && (u.G == 1 || u.gs != nullptr)) issue_chunk(c, u);
  for (int i = threadIdx.x; i < kBins0; i += kThreads) s.u.hist[i] = 0u;
  TOPK_MARK(g_select_trace, 1);

  // Row-level checks against the call: every CTA of the row decides the same way.
  const int Lcall = P.lens[u.r];
  int err = 0;
  if (Lcall != u.L || (u.G > 1 && u.gs == nullptr)) err = TOPK_STATUS_PLAN_MISMATCH;
  else if (!valid_plan_len) err = TOPK_STATUS_LEN;
  else if (ceil_div64(u.L, P.page_size) > P.table_ld) err = TOPK_STATUS_TABLE_WIDTH;
  if (err) {
    TOPK_LOG(u.r, 14);
    drain_chunk(c, u);
    if (u.rank == 0) {
      if (threadIdx.x == 0) set_status(c.h, err);
      fill_row(c, u.r, 0, P.k);
    }
    return;
  }
  u.t = P.row_to_table ? P.row_to_table[u.r] : u.r;
  u.kr = min(P.k, u.L);
  if (u.rank == 0) fill_row(c, u.r, u.kr, P.k);

  // Short row: every position is selected, in position order.
  if (copy_all) {
    TOPK_LOG(u.r, 13);
    for (int i = threadIdx.x; i < u.n; i += kThreads) emit(c, u, u.s0 + i, u.s0 + i);
    return;
  }

  __syncthreads();  // histogram zeroed
  histogram_chunk(c, u);
  TOPK_MARK(g_select_trace, 2);
  TOPK_LOG(u.r, 2);

  int b0, above0, eq0, la0, le0;
  if (!reduce_and_find(c, u, u.G > 1 ? u.gs->hist0 : nullptr, u.kr, u.n, true, b0, above0, eq0,
                       la0, le0))
    return;
  TOPK_MARK(g_select_trace, 3);
  TOPK_LOG(u.r, 3);
  const int need = u.kr - above0;
  const bool all_eq = (eq0 == need);
  const bool compact = !all_eq && eq0 <= (u.G > 1 ? kGroupCap : kListCap);
  const bool fallback = !all_eq && !compact;
  const bool stage_cand = compact && le0 <= kListCap;  // else written straight to global

  // Reserve output and candidate space for this CTA with one atomic (thread 0); its
  // latency overlaps the classification pass, the result is read after it.
  unsigned long long resv = 0ull;
  if (u.G > 1 && threadIdx.x == 0) {
    const unsigned long long cnt_out = (unsigned long long)(la0 + (all_eq ? le0 : 0));
    const unsigned long long cnt_cand = compact ? (unsigned long long)le0 : 0ull;
    resv = atomicAdd(reinterpret_cast<unsigned long long*>(&u.gs->out_ctr),
                     cnt_out | (cnt_cand << 32));
  }
  if (threadIdx.x == 0) {
    s.bc[9] = 0;   // staged emissions
    s.bc[10] = 0;  // staged candidates
  }
  __syncthreads();  // histogram region is free: reused for the staging lists

  // Pass 2 over the resident chunk (warp-synchronous): stage positions above the
  // threshold bin and boundary candidates, or fold the boundary keys (fallback).
  const float tlo = skip_below((uint32_t)b0);
  const float4* b4 = reinterpret_cast<const float4*>(s.buf);
  uint32_t fa = 0xFFFFFFFFu, fo = 0u;
  {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int vb = warp * 32; vb < u.nvec; vb += kThreads) {
      const int v = vb + lane;
      float4 x = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
      if (v < u.nvec) x = b4[v];
      const float m = fmaxf(fmaxf(x.x, x.y), fmaxf(x.z, x.w));
      const bool hit = v < u.nvec && !(m < tlo);
      if (!__any_sync(0xffffffffu, hit)) continue;
      const float xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int e = 4 * v - u.head + j;
        const bool in = hit && e >= 0 && e < u.n;
        const uint32_t dg = coarse_digit(xs[j]);
        const bool above = in && (dg > (uint32_t)b0 || (all_eq && dg == (uint32_t)b0));
        const bool cand = in && !all_eq && dg == (uint32_t)b0;
        const int slot = warp_append(above, &s.bc[9]);
        if (above && slot < TOPK_MAX_K) s.u.l.elist[slot] = u.s0 + e;
        if (stage_cand) {
          const int ci = warp_append(cand, &s.bc[10]);
          if (cand && ci < kListCap) {
            s.u.l.ckey[ci] = f2key(xs[j]);
            s.u.l.cpos[ci] = (uint32_t)(u.s0 + e);
          }
        } else if (fallback && cand) {
          const uint32_t key = f2key(xs[j]);
          fa &= key;
          fo |= key;
        }
      }
    }
  }
  if (threadIdx.x == 0) {
    s.bc[7] = (int)(uint32_t)(resv & 0xFFFFFFFFull);
    s.bc[8] = (int)(uint32_t)(resv >> 32);
  }
  __syncthreads();
  TOPK_MARK(g_select_trace, 4);
  const int out_base = u.G > 1 ? s.bc[7] : 0;
  const int cand_base = s.bc[8];
  const int n_emit = min(s.bc[9], TOPK_MAX_K);

  // Emit the staged positions (table lookups of the whole CTA in parallel).
  for (int i = threadIdx.x; i < n_emit; i += kThreads) emit(c, u, out_base + i, s.u.l.elist[i]);

  bool wrote_cand = false;  // this thread stored candidates that the last CTA reads
  if (compact && u.G > 1) {
    if (stage_cand) {
      const int nc = min(s.bc[10], kListCap);
      for (int i = threadIdx.x; i < nc; i += kThreads) {
        if (cand_base + i < kGroupCap) {
          u.gs->cand_key[cand_base + i] = s.u.l.ckey[i];
          u.gs->cand_pos[cand_base + i] = s.u.l.cpos[i];
          wrote_cand = true;
        }
      }
    } else {
      // Too many local candidates to stage: a second pass writes them to global.
      if (threadIdx.x == 0) s.bc[10] = 0;
      __syncthreads();
      for (int v = threadIdx.x; v < u.nvec; v += kThreads) {
        const float4 x = b4[v];
        const float xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int e = 4 * v - u.head + j;
          if (e < 0 || e >= u.n || coarse_digit(xs[j]) != (uint32_t)b0) continue;
          const int gi = cand_base + atomicAdd(&s.bc[10], 1);
          if (gi < kGroupCap) {
            u.gs->cand_key[gi] = f2key(xs[j]);
            u.gs->cand_pos[gi] = (uint32_t)(u.s0 + e);
            wrote_cand = true;
          }
        }
      }
    }
  }

  if (compact && u.G == 1) {
    __syncthreads();
    select_boundary(c, u, s.u.l.ckey, s.u.l.cpos, s.cst, min(eq0, kListCap), need, above0);
  }

  if (fallback) {
    block_and_or(fa, fo, s);
    if (u.G > 1) {
      if (threadIdx.x == 0) {
        atomicOr(&u.gs->and_key, ~fa);  // stored inverted so the reset value is 0
        atomicOr(&u.gs->or_key, fo);
      }
      if (!group_barrier(c, u, threadIdx.x == 0)) return;
      if (threadIdx.x == 0) {
        s.bc[11] = (int)~__ldcg(&u.gs->and_key);
        s.bc[12] = (int)__ldcg(&u.gs->or_key);
      }
      __syncthreads();
      fa = (uint32_t)s.bc[11];
      fo = (uint32_t)s.bc[12];
      __syncthreads();
    }
    if (!refine_in_place(c, u, b0, need, above0, fa, fo, le0)) return;
  }

  if (u.G > 1) {
    // End of the row for this CTA. The last one finishes the compact selection and
    // clears the row's counters for the next call.
    TOPK_MARK(g_select_trace, 5);
    if (wrote_cand) __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
      __threadfence();
      const uint32_t old = atomicAdd(&u.gs->fin, 1u);
      s.bc[13] = (old + 1u == (uint32_t)u.G) ? 1 : 0;
      __threadfence();
    }
    __syncthreads();
    TOPK_MARK(g_select_trace, 6);
    TOPK_LOG(u.r, s.bc[13] ? 7 : 6);
    if (s.bc[13]) {
      if (compact) {
        uint32_t* lkey = reinterpret_cast<uint32_t*>(s.buf);
        uint32_t* lpos = lkey + kGroupCap;
        const int n = min(eq0, kGroupCap);
        for (int i = threadIdx.x; i < n; i += kThreads) {
          lkey[i] = __ldcg(&u.gs->cand_key[i]);
          lpos[i] = __ldcg(&u.gs->cand_pos[i]);
        }
        __syncthreads();
        select_boundary(c, u, lkey, lpos, s.cst, n, need, above0);
      }
      TOPK_MARK(g_select_trace, 7);
      const uint32_t levels = __ldcg(&u.gs->levels);
      for (int i = threadIdx.x; i < kBins0; i += kThreads) {
        u.gs->hist0[i] = 0u;
        for (uint32_t l = 0; l < levels && l < 3; ++l) u.gs->hlev[l][i] = 0u;
      }
      if (threadIdx.x == 0) {
        u.gs->bar = 0u;
        u.gs->fin = 0u;
        u.gs->out_ctr = 0u;
        u.gs->cand_ctr = 0u;
        u.gs->and_key = 0u;
        u.gs->or_key = 0u;
        u.gs->levels = 0u;
      }
      TOPK_MARK(g_select_trace, 8);
    }
  }
}

__global__ void __launch_bounds__(kThreads, 1) select_kernel(SelectParams p) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  Smem& s = *reinterpret_cast<Smem*>(smem_raw);
  const Layout lay = make_layout(p.rows);
  Header* h = reinterpret_cast<Header*>(p.ws + lay.header);
  const UnitDesc* units = reinterpret_cast<const UnitDesc*>(p.ws + lay.units);
  TOPK_MARK(g_select_trace, 0);

  if (threadIdx.x == 0) {
    // Header and this CTA's first static unit: independent loads, one round trip.
    const int4 h0 = *reinterpret_cast<const int4*>(h);
    const int4 h1 = *reinterpret_cast<const int4*>(reinterpret_cast<const char*>(h) + 16);
    const int4 h2 = *reinterpret_cast<const int4*>(reinterpret_cast<const char*>(h) + 32);
    s.ud = units[blockIdx.x];
    s.bc[20] = h0.x;  // magic
    s.bc[21] = h0.y;  // rows
    s.bc[22] = h0.z;  // max_len
    s.bc[23] = h0.w;  // grid
    s.bc[24] = h1.y;  // waves
    s.bc[25] = h1.z;  // n_single
    s.bc[26] = h2.y;  // plan_error
    s.bc[27] = h2.z;  // n_implicit
    s.bc[28] = h2.w;  // dyn_period
    for (int i = 0; i < kPieces; ++i) mbar_init(&s.mbar[i], 1);
    fence_mbar_init();
  }
  __syncthreads();
  const bool bad = (uint32_t)s.bc[20] != kMagic || s.bc[21] != p.rows || s.bc[22] != p.max_len ||
                   s.bc[23] != (int)gridDim.x || s.bc[26] != 0;
  if (bad) {
    if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(&h->status, TOPK_STATUS_PLAN_MISMATCH);
    const int64_t total = (int64_t)p.rows * p.k;
    for (int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * kThreads) {
      p.out_slots[i] = -1;
      if (p.out_pos) p.out_pos[i] = -1;
    }
    return;
  }
  const int waves = s.bc[24], n_single = s.bc[25], n_implicit = s.bc[27];
  const int dyn_period = s.bc[28];
#ifdef TOPK_TRACE
  if (threadIdx.x == 0) g_select_log_n[blockIdx.x] = 0;
  TOPK_LOG(-1, 0);
#endif

  Ctx c{p, h, s, 0u};
  for (int w = 0; w < waves; ++w) {
    UnitDesc d;
    if (w == 0) {
      d = s.ud;
    } else {
      __syncthreads();
      if (threadIdx.x == 0) s.ud = units[(int64_t)w * kMaxGrid + blockIdx.x];
      __syncthreads();
      d = s.ud;
    }
    TOPK_LOG(d.row, 15);
    if (d.row >= 0) process_unit(c, d);
  }

  const int2* singles = reinterpret_cast<const int2*>(p.ws + lay.singles);
  const int32_t* first_single = reinterpret_cast<const int32_t*>(p.ws + lay.first_single);
  int idx = first_single[blockIdx.x];
  bool implicit = idx >= 0;
  while (true) {
    if (!implicit) {
      __syncthreads();
      if (threadIdx.x == 0) {
        const unsigned long long t = atomicAdd(&h->steal, 1ull);
        s.bc[14] = n_implicit + (int)(t % (unsigned long long)dyn_period);
      }
      __syncthreads();
      idx = s.bc[14];
    }
    implicit = false;
    if (idx >= n_single) break;
    const int2 sr = singles[idx];
    UnitDesc d;
    d.row = sr.x;
    d.s0 = 0;
    d.len = sr.y;
    d.n = (sr.y >= 0 && sr.y <= p.max_len) ? sr.y : 0;
    d.rank = 0;
    d.G = 1;
    d.group = -1;
    d.pad = 0;
    process_unit(c, d);
  }
  TOPK_MARK(g_select_trace, 9);
}

}  // namespace

#ifdef TOPK_TRACE
extern "C" int topk_trace_log(uint64_t* host, int* counts) {
  if (cudaMemcpyFromSymbol(host, g_select_log, sizeof(uint64_t) * kMaxGrid * 64) != cudaSuccess)
    return -9;
  return cudaMemcpyFromSymbol(counts, g_select_log_n, sizeof(int) * kMaxGrid) == cudaSuccess ? 0 : -9;
}
extern "C" int topk_trace_select(uint64_t* host, int n) {
  if (n > kMaxGrid * 16) n = kMaxGrid * 16;
  return cudaMemcpyFromSymbol(host, g_select_trace, sizeof(uint64_t) * n) == cudaSuccess ? 0 : -9;
}
#endif

size_t select_smem_bytes() { return sizeof(Smem); }

const void* select_kernel_ptr() { return reinterpret_cast<const void*>(&select_kernel); }

cudaError_t launch_select(const SelectParams& p, int grid, cudaStream_t stream) {
  SelectParams q = p;
  void* args[] = {&q};
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = sizeof(Smem);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelExC(&cfg, reinterpret_cast<const void*>(&select_kernel), args);
}

}  // namespace topk
