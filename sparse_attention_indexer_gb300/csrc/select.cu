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
// barrier (co-residency is guaranteed by the cooperative launch); while it propagates
// each CTA marks the vectors that reach its own bin. A second barrier delivers every
// CTA's counts and boundary candidates: each CTA then writes its staged positions at
// its row offset, ranks its own candidates against all of the row's, and clears the
// histogram bins it published. Rarely taken paths (general pass 2, large boundary
// sets, massive ties) are out-of-line functions, so that the common path's code stays
// compact when it is fetched cold.
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"
#include "keys.cuh"

namespace topk {

namespace {

#ifdef TOPK_TRACE
__device__ uint64_t g_select_trace[kMaxGrid * 32];
// Per-CTA event log: (row + 1) << 44 | event << 40 | low 40 bits of %globaltimer.
__device__ uint64_t g_select_log[kMaxGrid * 256];
__device__ int g_select_log_n[kMaxGrid];
__device__ __forceinline__ int& trace_log_n() {
  __shared__ int n;  // events logged by this CTA (written out at the end)
  return n;
}
#define TOPK_LOG(row, ev)                                                              \
  do {                                                                                 \
    if (threadIdx.x == 0) {                                                            \
      const int n_ = trace_log_n();                                                    \
      if (n_ < 256)                                                                    \
        g_select_log[blockIdx.x * 256 + n_] = ((uint64_t)((row) + 1) << 44) |          \
                                              ((uint64_t)(ev) << 40) |                 \
                                              (global_timer_ns() & 0xFFFFFFFFFFull);   \
      trace_log_n() = n_ + 1;                                                          \
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
  uint32_t pay[kMaxGrid];         // per-rank payloads delivered by the last row barrier
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

// ------------------------------------------------------------- block helpers

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
  int blocal;  // lowest coarse bin this CTA published to the row histogram
  int issued;  // pieces of the chunk whose copies were issued
  const char* src;  // the chunk's aligned source and its size in bytes
  uint32_t bytes;
  GroupState* gs;
  uint32_t bar_seq;    // barriers passed in this unit
  uint32_t flag_base;  // barriers this rank had passed before this unit
};

struct Ctx {
  const SelectParams& p;
  Header* h;
  Smem& s;
  uint32_t mphase;  // parity bits of the piece mbarriers
};

// Physical slot of logical position p of the unit's row (-1 with a status bit for a
// negative table entry or a slot above INT32_MAX).
__device__ __forceinline__ int32_t lookup_slot(const Ctx& c, const Unit& u, int p) {
  const SelectParams& P = c.p;
  const int32_t page = __ldg(P.table + (int64_t)u.t * P.table_ld + p / P.page_size);
  if (page < 0) {
    set_status(c.h, TOPK_STATUS_TABLE_ENTRY);
    return -1;
  }
  const int64_t sl = (int64_t)page * P.page_size + p % P.page_size;
  if (sl > 0x7FFFFFFFll) {
    set_status(c.h, TOPK_STATUS_SLOT_OVERFLOW);
    return -1;
  }
  return (int32_t)sl;
}

// Writes position p with its slot at output index idx of the unit's row.
__device__ __forceinline__ void put(const Ctx& c, const Unit& u, int idx, int p, int32_t slot) {
  const SelectParams& P = c.p;
  if ((unsigned)idx >= (unsigned)P.k) return;  // never taken
  const int64_t o = (int64_t)u.r * P.k + idx;
  P.out_slots[o] = slot;
  if (P.out_pos) P.out_pos[o] = p;
}

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

// Row barriers among the G CTAs of a row, as an arrival and a wait (a CTA can work
// in between). All threads call both. At arrival the CTA barrier orders every
// thread's earlier global writes (histogram reductions, candidates) before thread 0's
// gpu-scope release store of its rank's flag, (barriers passed) << 32 | payload. A
// release is cumulative in the PTX memory model, so that one store publishes the
// whole CTA's writes to a rank that acquires the flag; no thread needs its own fence.
// The wait has the lanes of warp 0 acquire every rank's flag, then a CTA barrier
// passes the ordering on; afterwards s.pay[j] holds rank j's payload, *prefix (if
// non-null) the sum of the payloads of ranks below this one and s.bc[18] the largest
// payload. group_wait returns false if a bounded wait expired (status set). Test hook:
// CTA p.skip_cta never arrives at the first row barrier of its units, so that the
// waits of the row it serves run out (the call then reports TOPK_STATUS_TIMEOUT).
__device__ uint32_t group_arrive(const Ctx& c, Unit& u, uint32_t payload) {
  __syncthreads();
#ifdef TOPK_TRACE
  if (threadIdx.x == 0 && u.bar_seq == 0) g_select_trace[blockIdx.x * 32 + 26] = global_timer_ns();
#endif
  const bool skip = u.bar_seq == 0 && (int)blockIdx.x == c.p.skip_cta;
  u.bar_seq += 1;
  const uint32_t my = u.flag_base + u.bar_seq;
  if (threadIdx.x == 0 && !skip) {
    st_release_u64(&u.gs->flag[u.rank], ((unsigned long long)my << 32) | payload);
    // The payload history is read only by a waiter that finds this flag one barrier
    // ahead; the next release orders this store before that flag. Storing it after
    // the release keeps it off this barrier's critical path.
    __stcg(&u.gs->pay2[my & 1u][u.rank], payload);
  }
  return my;
}

__device__ bool group_wait(Ctx& c, Unit& u, uint32_t my, int* prefix) {
  if (threadIdx.x < 32) {
    __syncwarp();
    int acc = 0;
    uint32_t mx = 0u;
    bool ok = true, overrun = false;
    int stuck = -1;
    for (int j = threadIdx.x; j < u.G && ok; j += 32) {
      unsigned long long v = ld_acquire_u64(&u.gs->flag[j]);
      if ((uint32_t)(v >> 32) < my) {
        const uint64_t t0 = global_timer_ns();
        while ((uint32_t)((v = ld_acquire_u64(&u.gs->flag[j])) >> 32) < my) {
          if (global_timer_ns() - t0 > c.p.wait_ns) {
            ok = false;
            stuck = j;
            break;
          }
        }
      }
      // A rank one barrier ahead (it passed this one while this waiter was still
      // reading other flags) has replaced the flag's payload; its pay2 entry of this
      // barrier's parity still holds it. Two barriers ahead cannot happen (the rank
      // would have passed a barrier this CTA has not arrived at): reported.
      uint32_t pv = (uint32_t)v;
      const uint32_t seen = (uint32_t)(v >> 32);
      if (seen != my) {
        if (seen == my + 1u) pv = __ldcg(&u.gs->pay2[my & 1u][j]);
        else overrun = true;
      }
      c.s.pay[j] = pv;
      if (j < u.rank) acc += (int)pv;
      mx = max(mx, pv);
    }
    const bool all_ok = __all_sync(0xffffffffu, ok);
    if (__any_sync(0xffffffffu, overrun) && threadIdx.x == 0) set_status(c.h, TOPK_STATUS_ORDER);
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      acc += __shfl_xor_sync(0xffffffffu, acc, o);
      mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    }
    if (!ok) {
      set_status(c.h, TOPK_STATUS_TIMEOUT);
      record_timeout(c.h, 1, u.r, u.rank, (int)(my - u.flag_base), stuck, (int)my);
    }
    if (threadIdx.x == 0) {
      c.s.bc[15] = all_ok ? 1 : 0;
      c.s.bc[17] = acc;
      c.s.bc[18] = (int)mx;
    }
  }
  __syncthreads();
  if (prefix) *prefix = c.s.bc[17];
  return c.s.bc[15] != 0;
}

__device__ bool group_sync(Ctx& c, Unit& u, uint32_t payload, int* prefix) {
  return group_wait(c, u, group_arrive(c, u, payload), prefix);
}

// Finds bin b of a 4096-bin histogram (8 bins per thread: row-wide counts g[], this
// CTA's counts l[]) with above(b) < need <= above(b) + g[b], above(b) counting bins
// > b. Writes s.bc[0..4] = (b, above, g[b], this CTA's count above b, l[b]); nothing
// is written when the histogram holds fewer than `need` values.
__device__ void find_threshold(const uint32_t (&g)[8], const uint32_t (&l)[8], int need, Smem& s) {
  // Two 32-bit scans (counts never exceed a row's length, < 2^31).
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int gs = 0, ls = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    gs += (int)g[j];
    ls += (int)l[j];
  }
  const int ig = warp_incl_scan(gs), il = warp_incl_scan(ls);
  if (lane == 31) {
    s.wsum[w] = ig;
    s.wsum2[w] = il;
  }
  __syncthreads();
  int bg = 0, tg = 0, bl = 0, tl = 0;
#pragma unroll
  for (int i = 0; i < kWarps; ++i) {
    const int xg = s.wsum[i], xl = s.wsum2[i];
    if (i < w) {
      bg += xg;
      bl += xl;
    }
    tg += xg;
    tl += xl;
  }
  // counts owned by higher threads
  const int g_above = tg - (bg + ig);
  const int l_above = tl - (bl + il);
  if (g_above < need && need <= g_above + gs) {
    int cg = g_above, cl = l_above;
#pragma unroll
    for (int j = 7; j >= 0; --j) {
      if (cg + (int)g[j] >= need) {
        s.bc[0] = threadIdx.x * 8 + j;
        s.bc[1] = cg;
        s.bc[2] = (int)g[j];
        s.bc[3] = cl;
        s.bc[4] = (int)l[j];
        break;
      }
      cg += (int)g[j];
      cl += (int)l[j];
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

__device__ __forceinline__ float vmax4(const float4& x) {
  return fmaxf(fmaxf(x.x, x.y), fmaxf(x.z, x.w));
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
    int blocal = 0;
    if (sparse && local_n >= need) {
      find_threshold(loc, loc, need, s);
      blocal = s.bc[0];
    }
    u.blocal = blocal;
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (loc[j] && b0 + j >= blocal) red_add_u32(&ghist[b0 + j], loc[j]);
    if (!group_sync(c, u, 0u, nullptr)) return false;
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
  find_threshold(glob, loc, need, s);
  b = s.bc[0];
  above = s.bc[1];
  eq = s.bc[2];
  local_above = s.bc[3];
  local_eq = s.bc[4];
  __syncthreads();
  return true;
}

// Level-0 threshold of the unit's row from the coarse histogram in s.u.hist (complete
// for the chunk). A single-CTA row searches it directly. A CTA of a multi-CTA row
// publishes only the bins at or above its own bin for `est` values, est = 4k/G (the
// row's k values spread over G chunks), and sends that bin as its barrier payload.
// The row histogram is then complete at bins >= the highest payload, B; if at least
// `need` values lie there, the row's threshold is found exactly. Otherwise every CTA
// publishes the bins it held back and the row meets once more. Outputs as
// reduce_and_find; false on timeout.
//
// While the first barrier propagates, a CTA whose own bin lies on the positive side
// (where a bin's lower float bound is exact) marks in *pre bit i each of its vectors
// v = threadIdx.x + i * kThreads that reaches that bound. When the first round is
// complete the row's threshold bin is at or above the CTA's own bin, so every vector
// holding a value at or above the row's threshold is marked; *pre_ok says so.
__device__ bool coarse_reduce(Ctx& c, Unit& u, int& b, int& above, int& eq, int& local_above,
                              int& local_eq, uint32_t& pre, bool& pre_ok) {
  Smem& s = c.s;
  const int need = u.kr;
  const int t = threadIdx.x * 8;
  uint32_t loc[8], glob[8];
  load8(&s.u.hist[t], loc);
  if (u.G == 1) {
    find_threshold(loc, loc, need, s);
  } else {
    const int est = min(need, (int)((4ll * need + u.G - 1) / u.G));
    int blocal = 0;
    if (u.n >= est) {
      find_threshold(loc, loc, est, s);
      blocal = s.bc[0];
      __syncthreads();
    }
    u.blocal = blocal;
    TOPK_MARK(g_select_trace, 24);
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (loc[j] && t + j >= blocal) red_add_u32(&u.gs->hist0[t + j], loc[j]);
#ifdef TOPK_TRACE
    {
      int nw = 0;
      for (int j = 0; j < 8; ++j) nw += (loc[j] && t + j >= blocal) ? 1 : 0;
      nw = __reduce_add_sync(0xffffffffu, nw);
      if ((threadIdx.x & 31) == 0) atomicAdd(&s.bc[30], nw);
    }
#endif
    const uint32_t seq = group_arrive(c, u, (uint32_t)blocal);
    if (blocal >= 2048) {
      const float tl = skip_below((uint32_t)blocal);
      const float4* b4 = reinterpret_cast<const float4*>(s.buf);
      uint32_t m = 0u;
      for (int i = 0, v = threadIdx.x; v < u.nvec; ++i, v += kThreads)
        m |= vmax4(b4[v]) >= tl ? (1u << i) : 0u;
      pre = m;
      pre_ok = true;
    }
    if (!group_wait(c, u, seq, nullptr)) return false;
    TOPK_MARK(g_select_trace, 25);
    const int top = s.bc[18];
    if (t + 7 >= blocal) {
      load8_cg(&u.gs->hist0[t], glob);
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) glob[j] = 0u;
    }
    if (threadIdx.x == 0) s.bc[0] = -1;
    find_threshold(glob, loc, need, s);  // leaves s.bc[0] = -1 when not found
    const bool complete = s.bc[0] >= top;
    __syncthreads();
    if (!complete) {
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (loc[j] && t + j < blocal) red_add_u32(&u.gs->hist0[t + j], loc[j]);
      u.blocal = 0;
      pre_ok = false;
      if (!group_sync(c, u, 0u, nullptr)) return false;
      load8_cg(&u.gs->hist0[t], glob);
      find_threshold(glob, loc, need, s);
    }
  }
  b = s.bc[0];
  above = s.bc[1];
  eq = s.bc[2];
  local_above = s.bc[3];
  local_eq = s.bc[4];
  __syncthreads();
  return true;
}

// ------------------------------------------------------------- chunk loading

// Geometry of the unit's chunk [s0, s0 + n) of row r in shared memory: the copy
// covers the aligned 16-byte vectors holding the chunk; element 0 sits at float
// index `head`.
__device__ __forceinline__ uint32_t chunk_geometry(const SelectParams& P, Unit& u,
                                                    const char** src_aligned) {
  const float* src = P.scores + (int64_t)u.r * P.ld + u.s0;
  const uintptr_t A = reinterpret_cast<uintptr_t>(src);
  const uintptr_t A0 = A & ~uintptr_t(15);
  const uintptr_t A1 = (A + 4ull * (uint64_t)u.n + 15ull) & ~uintptr_t(15);
  const uint32_t bytes = u.n > 0 ? (uint32_t)(A1 - A0) : 0u;
  u.head = (int)((A - A0) >> 2);
  u.nvec = (int)(bytes >> 4);
  u.npieces = (int)((bytes + kPieceBytes - 1) / kPieceBytes);
  u.src = reinterpret_cast<const char*>(A0);
  u.bytes = bytes;
  *src_aligned = u.src;
  return bytes;
}

// Bulk copies of pieces [first, first + count) of the chunk, one per 16 KB piece,
// each completing on its mbarrier. Called by one thread; the first call of a unit
// comes after the previous unit's shared-memory accesses completed. At most kWindow
// pieces are in flight: the copy engine interleaves outstanding copies, so with every
// piece issued at once they all complete near the end; a window makes them land in
// order, and pass 1 follows them.
constexpr int kWindow = 4;

__device__ void issue_copies(Smem& s, const char* src, uint32_t bytes, int first, int count) {
  if (first == 0) fence_proxy_async_smem();
  for (int i = first; i < first + count; ++i) {
    const uint32_t off = (uint32_t)i * kPieceBytes;
    const uint32_t sz = min((uint32_t)kPieceBytes, bytes - off);
    mbar_arrive_expect_tx(&s.mbar[i], sz);
    bulk_g2s(reinterpret_cast<char*>(s.buf) + off, src + off, sz, &s.mbar[i]);
  }
}

__device__ void issue_chunk(Ctx& c, Unit& u) {
  const char* src;
  const uint32_t bytes = chunk_geometry(c.p, u, &src);
  u.issued = min(kWindow, u.npieces);
  if (threadIdx.x == 0) issue_copies(c.s, src, bytes, 0, u.issued);
}

// Bounded wait for piece i. A wait that runs out sets the status and waits once more
// (bounded); if the copy still has not landed, the CTA is marked aborting (s.bc[7],
// with the piece and its phase in s.bc[8], s.bc[13]): it takes no further units, and
// before it exits it waits (bounded) for that copy once more, so that no copy it
// issued is left writing into shared memory it no longer owns.
__device__ __forceinline__ void wait_piece(Ctx& c, int i) {
  const uint32_t par = (c.mphase >> i) & 1u;
  if (!mbar_wait_bounded(&c.s.mbar[i], par, c.p.wait_ns)) {
    if (threadIdx.x == 0) {
      set_status(c.h, TOPK_STATUS_TIMEOUT);
      record_timeout(c.h, 2, -1, i, (int)par, 0, 0);
    }
    if (!mbar_wait_bounded(&c.s.mbar[i], par, c.p.wait_ns) && atomicExch(&c.s.bc[7], 1) == 0) {
      c.s.bc[8] = i;
      c.s.bc[13] = (int)par;
    }
  }
  c.mphase ^= (1u << i);
}

// Waits for every piece of the unit (used when a unit is abandoned after its copies
// were issued: shared memory must not be reused while copies are in flight).
__device__ void drain_chunk(Ctx& c, Unit& u) {
  for (int i = 0; i < u.issued; ++i) wait_piece(c, i);
  __syncthreads();
}

// Builds the coarse histogram of the chunk in s.u.hist (zeroed by the caller before
// the CTA barrier that precedes this call) piece by piece as the pieces land: every
// thread waits on piece p, thread 0 then issues piece p + kWindow, and each thread
// counts its (at most two) vectors of piece p.
__device__ void histogram_chunk(Ctx& c, Unit& u) {
  Smem& s = c.s;
  const float4* b4 = reinterpret_cast<const float4*>(s.buf);
  constexpr int kVecPerPiece = kPieceBytes / 16;
  const int vfull0 = (u.head + 3) >> 2;  // first vector holding only chunk elements
  const int vfull1 = (u.head + u.n) >> 2;
  for (int p = 0; p < u.npieces; ++p) {
    wait_piece(c, p);
    if (p == u.npieces - 1) TOPK_LOG(u.r, 10);
    if (threadIdx.x == 0 && p + kWindow < u.npieces) issue_copies(s, u.src, u.bytes, p + kWindow, 1);
    const int vend = min((p + 1) * kVecPerPiece, u.nvec);
    for (int v = p * kVecPerPiece + threadIdx.x; v < vend; v += kThreads) {
      const float4 x = b4[v];
      if (v >= vfull0 && v < vfull1) {
        atomicAdd(&s.u.hist[coarse_digit(x.x)], 1u);
        atomicAdd(&s.u.hist[coarse_digit(x.y)], 1u);
        atomicAdd(&s.u.hist[coarse_digit(x.z)], 1u);
        atomicAdd(&s.u.hist[coarse_digit(x.w)], 1u);
      } else {  // first or last vector of the chunk
        const int e0 = 4 * v - u.head;
        const float xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (e0 + j >= 0 && e0 + j < u.n) atomicAdd(&s.u.hist[coarse_digit(xs[j])], 1u);
      }
    }
  }
  u.issued = u.npieces;
#ifdef TOPK_TRACE
  if (threadIdx.x == 0) g_select_trace[blockIdx.x * 32 + 11] = global_timer_ns();
#endif
  __syncthreads();
}

// ------------------------------------------------------------- boundary selection

// Exact selection among n <= kRankMax candidates: candidate i is taken iff fewer
// than `need` candidates rank before it (larger key, or equal key and smaller
// position); it goes to output index base + its rank (deterministic order). A group
// of T lanes shares each candidate's comparisons.
__device__ void rank_select_emit(Ctx& c, const Unit& u, const uint32_t* key, const uint32_t* pos,
                                 int n, int need, int base) {
  int T = 1;
  while (T < 8 && n * (T * 2) <= kThreads) T *= 2;  // lanes per candidate (1..8)
  const int sub = threadIdx.x & (T - 1);
  for (int i0 = 0; i0 < n * T; i0 += kThreads) {
    const int i = (i0 + threadIdx.x) / T;  // groups never straddle a warp (T divides 32)
    const bool act = i < n;
    const uint32_t ki = act ? key[i] : 0u, pi = act ? pos[i] : 0u;
    int rank = 0;
    if (act) {
      int j = sub;
      for (; j + 3 * T < n; j += 4 * T) {
        const uint32_t k0 = key[j], k1 = key[j + T], k2 = key[j + 2 * T], k3 = key[j + 3 * T];
        const uint32_t p0 = pos[j], p1 = pos[j + T], p2 = pos[j + 2 * T], p3 = pos[j + 3 * T];
        rank += (k0 > ki || (k0 == ki && p0 < pi)) ? 1 : 0;
        rank += (k1 > ki || (k1 == ki && p1 < pi)) ? 1 : 0;
        rank += (k2 > ki || (k2 == ki && p2 < pi)) ? 1 : 0;
        rank += (k3 > ki || (k3 == ki && p3 < pi)) ? 1 : 0;
      }
      for (; j < n; j += T) {
        const uint32_t kj = key[j], pj = pos[j];
        rank += (kj > ki || (kj == ki && pj < pi)) ? 1 : 0;
      }
    }
    for (int o = 1; o < T; o <<= 1) rank += __shfl_xor_sync(0xffffffffu, rank, o);
    if (act && sub == 0 && rank < need) emit(c, u, base + rank, (int)pi);
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

// Emits, in a fixed order (thread, then vector), every chunk value whose index e and
// value x satisfy pred(e, x), at output indices base, base + 1, ... Two passes over
// the resident chunk: count, CTA scan, write.
template <class Pred>
__device__ void emit_ordered(Ctx& c, const Unit& u, int base, Pred pred) {
  const float4* b4 = reinterpret_cast<const float4*>(c.s.buf);
  int cnt = 0;
  for (int v = threadIdx.x; v < u.nvec; v += kThreads) {
    const float4 x = b4[v];
    const float xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = 4 * v - u.head + j;
      if (e >= 0 && e < u.n && pred(e, xs[j])) ++cnt;
    }
  }
  int total;
  int o = base + block_excl_scan(cnt, &total, c.s);
  if (cnt == 0) return;
  for (int v = threadIdx.x; v < u.nvec; v += kThreads) {
    const float4 x = b4[v];
    const float xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = 4 * v - u.head + j;
      if (e >= 0 && e < u.n && pred(e, xs[j])) emit(c, u, o++, u.s0 + e);
    }
  }
}

// Boundary bin too large for a compact list (massive ties): refine in place on the
// full key, then take tied values in position order. fa/fo: AND/OR of the boundary
// keys over the row; `need` values remain to be chosen among coarse digit b0, after
// `emitted` row entries (all values above the threshold bin). For G > 1 every level
// exchanges per-rank counts so that output offsets are deterministic, and each CTA
// clears the level histogram once the next barrier shows it has been read.
__device__ __noinline__ bool refine_in_place(Ctx c, Unit u, int b0, int need, int emitted,
                                             uint32_t fa, uint32_t fo, int local_eq0) {
  Smem& s = c.s;
  const float4* b4 = reinterpret_cast<const float4*>(s.buf);
  bool reset_and_or = u.G > 1;  // cleared by rank 0 after the next barrier
  auto passed_barrier = [&]() {
    if (reset_and_or && u.rank == 0 && threadIdx.x == 0) {
      u.gs->and_key = 0u;
      u.gs->or_key = 0u;
    }
    reset_and_or = false;
  };
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
      int bl, abl, eql, lal, lel;
      if (!reduce_and_find(c, u, u.G > 1 ? u.gs->hlev[lev] : nullptr, need, 0, false, bl, abl,
                           eql, lal, lel))
        return false;
      if (u.G > 1) passed_barrier();
      need -= abl;
      const bool take = (eql == need);
      int ob = emitted;
      if (u.G > 1) {
        int pre;
        if (!group_sync(c, u, (uint32_t)(lal + (take ? lel : 0)), &pre)) return false;
        for (int i = threadIdx.x; i < kBins0; i += kThreads) u.gs->hlev[lev][i] = 0u;
        ob += pre;
      }
      const uint32_t pm = pmask, pv = pval;
      emit_ordered(c, u, ob, [&](int e, float x) {
        (void)e;
        if (coarse_digit(x) != (uint32_t)b0) return false;
        const uint32_t key = f2key(x);
        if ((key & pm) != pv) return false;
        const uint32_t d = (key >> shift) & dmask;
        return d > (uint32_t)bl || (take && d == (uint32_t)bl);
      });
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
    if (!group_sync(c, u, (uint32_t)local_tie, &prefix)) return false;
    passed_barrier();
  }
  const int tie_base = emitted;  // every other entry fills [0, emitted)
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

// ------------------------------------------------------------- out-of-line paths
//
// Paths that the common rows never take live in out-of-line functions, so that the
// common path's instructions stay compact: a kernel whose code was evicted fetches it
// from memory phase by phase, and interleaved rare code lengthens every such fetch.
// They take the context and the unit by value so that callers keep theirs in
// registers.

// Pass 2 when the threshold bin's float bounds are not exact (negative side, the top
// bin) or the boundary bin is too large for a compact list: every value is classified
// by its coarse digit. Counts, scans and writes the staging lists like the exact
// path, leaves the staged counts in s.bc[9] (positions) and s.bc[10] (candidates) and
// returns this thread's AND / OR of the boundary keys (x, y).
__device__ __noinline__ uint2 pass2_general(Ctx c, Unit u, int b0, bool all_eq, bool fallback,
                                            bool stage_cand) {
  Smem& s = c.s;
  const float4* b4 = reinterpret_cast<const float4*>(s.buf);
  const float tlo = skip_below((uint32_t)b0);
  // classify one value: 0 below, 1 above (staged position), 2 boundary
  auto klass = [&](float x) -> int {
    const uint32_t dg = coarse_digit(x);
    if (dg < (uint32_t)b0) return 0;
    return (dg > (uint32_t)b0 || all_eq) ? 1 : 2;
  };
  uint32_t fa = 0xFFFFFFFFu, fo = 0u, hm = 0u;
  int na = 0, nc = 0;
  for (int i = 0, v = threadIdx.x; v < u.nvec; ++i, v += kThreads) {
    const float4 x = b4[v];
    if (vmax4(x) < tlo) continue;
    const int e0 = 4 * v - u.head;
    const float xs[4] = {x.x, x.y, x.z, x.w};
    int a = 0, cd = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = e0 + j;
      if (e < 0 || e >= u.n) continue;
      const int k = klass(xs[j]);
      if (k == 1) {
        ++a;
      } else if (k == 2) {
        ++cd;
        if (fallback) {
          const uint32_t key = f2key(xs[j]);
          fa &= key;
          fo |= key;
        }
      }
    }
    if (!stage_cand) cd = 0;
    na += a;
    nc += cd;
    hm |= (a + cd) ? (1u << i) : 0u;
  }
  int tot_ac;
  const int off_ac = block_excl_scan(na | (nc << 16), &tot_ac, s);
  if (threadIdx.x == 0) {
    s.bc[9] = tot_ac & 0xFFFF;
    s.bc[10] = tot_ac >> 16;
  }
  int oa = off_ac & 0xFFFF, oc = off_ac >> 16;
  while (hm) {
    const int i = __ffs(hm) - 1;
    hm &= hm - 1u;
    const int v = threadIdx.x + i * kThreads;
    const float4 x = b4[v];
    const int p0 = u.s0 + 4 * v - u.head;
    const float xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = 4 * v - u.head + j;
      if (e < 0 || e >= u.n) continue;
      const int k = klass(xs[j]);
      if (k == 1) {
        if (oa < TOPK_MAX_K) s.u.l.elist[oa] = p0 + j;
        ++oa;
      } else if (k == 2 && stage_cand) {
        if (oc < kListCap) {
          s.u.l.ckey[oc] = f2key(xs[j]);
          s.u.l.cpos[oc] = (uint32_t)(p0 + j);
        }
        ++oc;
      }
    }
  }
  return make_uint2(fa, fo);
}

// A multi-CTA row's boundary candidates of coarse digit b0 that did not fit the
// staging list: written in chunk order to the row's candidate list from index base.
__device__ __noinline__ void write_candidates_ordered(Ctx c, Unit u, int b0, int base) {
  Smem& s = c.s;
  const float4* b4 = reinterpret_cast<const float4*>(s.buf);
  int cnt = 0;
  for (int v = threadIdx.x; v < u.nvec; v += kThreads) {
    const float4 x = b4[v];
    const float xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = 4 * v - u.head + j;
      if (e >= 0 && e < u.n && coarse_digit(xs[j]) == (uint32_t)b0) ++cnt;
    }
  }
  int total;
  int gi = base + block_excl_scan(cnt, &total, s);
  for (int v = threadIdx.x; v < u.nvec && cnt > 0; v += kThreads) {
    const float4 x = b4[v];
    const float xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = 4 * v - u.head + j;
      if (e >= 0 && e < u.n && coarse_digit(xs[j]) == (uint32_t)b0) {
        if (gi < kGroupCap) {
          u.gs->cand_key[gi] = f2key(xs[j]);
          u.gs->cand_pos[gi] = (uint32_t)(u.s0 + e);
        }
        ++gi;
      }
    }
  }
}

// A single-CTA row's boundary: `need` of its n staged candidates, emitted from `base`.
__device__ __noinline__ void select_boundary_single(Ctx c, Unit u, int n, int need, int base) {
  select_boundary(c, u, c.s.u.l.ckey, c.s.u.l.cpos, c.s.cst, n, need, base);
}

// A multi-CTA row with more than kRankOwnMax boundary candidates (gathered in lkey /
// lpos, the same list in every CTA of the row): radix-select `need` of them (the same
// marks in every CTA), then each CTA emits its own marked candidates, own0..own1, at
// their position among the marked ones after the `above` values above the bin.
__device__ __noinline__ void emit_listed(Ctx c, Unit u, const uint32_t* lkey,
                                        const uint32_t* lpos, int n, int need, int own0,
                                        int own1, int above) {
  Smem& s = c.s;
  list_select(s, lkey, lpos, s.cst, n, need);
  int cnt = 0, before = 0;
  for (int i = threadIdx.x; i < own0; i += kThreads)
    if (s.cst[i] == kSel) ++before;
  before = block_sum(before, s);
  for (int i0 = own0; i0 < own1; i0 += kThreads) {
    const int i = i0 + threadIdx.x;
    const bool sel = i < own1 && s.cst[i] == kSel;
    int total;
    const int off = block_excl_scan(sel ? 1 : 0, &total, s);
    if (sel) emit(c, u, above + before + cnt + off, (int)lpos[i]);
    cnt += total;
  }
}

// ------------------------------------------------------------- the unit

__device__ void process_unit(Ctx& c, const UnitDesc& d, bool pre_issued) {
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
  u.issued = 0;
  u.gs = (u.G > 1 && d.group >= 0)
             ? reinterpret_cast<GroupState*>(P.ws + make_layout(P.rows).groups) + d.group
             : nullptr;
  const bool valid_plan_len = u.L >= 0 && u.L <= P.max_len;
  const bool copy_all = valid_plan_len && u.L <= P.k;

  __syncthreads();  // the previous unit no longer uses shared memory
  TOPK_LOG(u.r, 1);
  // Issue the chunk's copies first: [s0, s0 + n) lies inside the row by construction
  // of the plan, which the kernel validated against rows / max_len. The first static
  // unit's copies were issued in the kernel prologue.
  if (!copy_all && valid_plan_len && (u.G == 1 || u.gs != nullptr)) {
    if (pre_issued) {
      const char* src;
      chunk_geometry(P, u, &src);
      u.issued = min(kWindow, u.npieces);
    } else {
      issue_chunk(c, u);
    }
  }
  for (int i = threadIdx.x; i < kBins0; i += kThreads) s.u.hist[i] = 0u;
#ifdef TOPK_TRACE
  if (threadIdx.x == 0) s.bc[30] = 0;
#endif
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
  u.flag_base = u.G > 1 ? (uint32_t)(__ldcg(&u.gs->flag[u.rank]) >> 32) : 0u;
  if (u.rank == 0) fill_row(c, u.r, u.kr, P.k);
  if (!copy_all && u.n > 0 && threadIdx.x >= kThreads - 32) {
    // Bring this chunk's page-table entries into L2 for the emission step.
    const int32_t* t0 = P.table + (int64_t)u.t * P.table_ld + u.s0 / P.page_size;
    const int32_t* t1 = P.table + (int64_t)u.t * P.table_ld + (u.s0 + u.n - 1) / P.page_size;
    const uintptr_t l0 = reinterpret_cast<uintptr_t>(t0) & ~uintptr_t(127);
    const uintptr_t l1 = reinterpret_cast<uintptr_t>(t1) & ~uintptr_t(127);
    for (uintptr_t a = l0 + 128u * (threadIdx.x - (kThreads - 32)); a <= l1; a += 128u * 32u)
      asm volatile("prefetch.global.L2 [%0];" ::"l"(a));
  }

  // Short row: every position is selected, in position order.
  if (copy_all) {
    TOPK_LOG(u.r, 13);
    for (int i = threadIdx.x; i < u.n; i += kThreads) emit(c, u, u.s0 + i, u.s0 + i);
    return;
  }

  __syncthreads();  // histogram zeroed
  TOPK_LOG(u.r, 9);
  histogram_chunk(c, u);
  if (s.bc[7]) return;  // a copy never landed: this CTA aborts (histogram_chunk ended in a CTA barrier)
  TOPK_MARK(g_select_trace, 2);
  TOPK_LOG(u.r, 2);

  int b0, above0, eq0, la0, le0;
  u.blocal = 0;
  uint32_t pre = 0u;
  bool pre_ok = false;
  if (!coarse_reduce(c, u, b0, above0, eq0, la0, le0, pre, pre_ok)) return;
  TOPK_MARK(g_select_trace, 3);
#ifdef TOPK_TRACE
  if (threadIdx.x == 0) g_select_trace[blockIdx.x * 32 + 28] = (uint64_t)s.bc[30] << 32;
#endif
  TOPK_LOG(u.r, 3);
  const int need = u.kr - above0;
  const bool all_eq = (eq0 == need);
  const bool compact = !all_eq && eq0 <= (u.G > 1 ? kGroupCap : kListCap);
  const bool fallback = !all_eq && !compact;
  const bool stage_cand = compact && le0 <= kListCap;  // else written straight to global
  // Per-rank counts for the row's output offsets: staged emissions, candidates.
  const int my_emit = la0 + (all_eq ? le0 : 0);
  const int my_cand = compact ? le0 : 0;
  TOPK_MARK(g_select_trace, 16);
  __syncthreads();  // histogram region is free: reused for the staging lists
  TOPK_MARK(g_select_trace, 17);

  // Pass 2 over the resident chunk, in two steps with a CTA scan between them. Count:
  // each thread reads its vectors (v = threadIdx.x + i * kThreads), skips those whose
  // largest value lies below the threshold bin (nearly all of a long row), counts the
  // values it will stage (positions above the threshold bin, boundary candidates) or
  // folds the boundary keys (fallback), and sets bit i of a mask for each vector that
  // held a value to stage. Write: after the scan turns the counts into offsets, each
  // thread revisits only its masked vectors. No shared atomics; the staging order is
  // deterministic. For a threshold bin on the positive side the bin's float bounds
  // are exact, so values are classified by compares alone and each vector's values go
  // to their slots by popcounts of its compare masks, without branches. Other bins
  // classify by digit, out of line (pass2_general).
  static_assert((kBufFloats / 4 + kThreads - 1) / kThreads <= 32,
                "a thread's vectors of one chunk fit the 32-bit hit mask");
  const float tlo = skip_below((uint32_t)b0);
  const bool exact = b0 >= 2048 && b0 < 4095 && !fallback;
  const float thi = exact ? skip_below((uint32_t)b0 + 1u) : 0.0f;
  const float4* b4 = reinterpret_cast<const float4*>(s.buf);
  uint32_t fa = 0xFFFFFFFFu, fo = 0u;  // AND / OR of the boundary keys (fallback)
  // The chunk's first and last vectors may hold values of the neighbouring chunks:
  // those become -inf, below tlo (exact mode has tlo >= +0).
  const int vfull0 = (u.head + 3) >> 2, vfull1 = (u.head + u.n) >> 2;
  auto clip = [&](int v, float4& x) {
    if (v < vfull0 || v >= vfull1) {
      const int e0 = 4 * v - u.head;
      const float ninf = __int_as_float(0xFF800000);
      if (e0 < 0 || e0 >= u.n) x.x = ninf;
      if (e0 + 1 < 0 || e0 + 1 >= u.n) x.y = ninf;
      if (e0 + 2 < 0 || e0 + 2 >= u.n) x.z = ninf;
      if (e0 + 3 < 0 || e0 + 3 >= u.n) x.w = ninf;
    }
  };
  // bit j set iff component j of x is >= t
  auto ge_mask = [](const float4& x, float t) -> uint32_t {
    return (x.x >= t ? 1u : 0u) | (x.y >= t ? 2u : 0u) | (x.z >= t ? 4u : 0u) |
           (x.w >= t ? 8u : 0u);
  };
  if (exact) {
    int na = 0, nc = 0;
    uint32_t hm = 0u;  // bit i: this thread's i-th vector holds a value to stage
    auto count = [&](int i, int v, float4 x) {
      clip(v, x);
      const uint32_t mg = ge_mask(x, tlo);
      const uint32_t ma = all_eq ? mg : ge_mask(x, thi);
      const uint32_t mc = stage_cand ? (mg & ~ma) : 0u;
      na += __popc(ma);
      nc += __popc(mc);
      hm |= (ma | mc) ? (1u << i) : 0u;
    };
    // This CTA holds la0 + le0 values at or above the threshold bin. Sparse (under
    // one per 16 vectors, the usual case on long rows): most warps' vectors are all
    // below tlo, so a max filter skips them. Dense: every warp would take the branch,
    // so every vector is classified without one.
    if (pre_ok) {
      // only the vectors marked while the first barrier propagated
      for (uint32_t m = pre; m; m &= m - 1u) {
        const int i = __ffs(m) - 1;
        const int v = threadIdx.x + i * kThreads;
        const float4 x = b4[v];
        if (vmax4(x) >= tlo) count(i, v, x);
      }
    } else if ((int64_t)(la0 + le0) * 16 < u.nvec) {
      for (int i = 0, v = threadIdx.x; v < u.nvec; ++i, v += kThreads) {
        const float4 x = b4[v];
        if (vmax4(x) >= tlo) count(i, v, x);
      }
    } else {
      for (int i = 0, v = threadIdx.x; v < u.nvec; ++i, v += kThreads) count(i, v, b4[v]);
    }
    TOPK_LOG(u.r, 6);
#ifdef TOPK_TRACE_DETAIL  // block-wide timing; distorts the phases it brackets
    if (threadIdx.x == 0) g_select_trace[blockIdx.x * 32 + 18] = global_timer_ns();
    {
      // slowest thread of the count pass
      __shared__ unsigned long long tmax;
      if (threadIdx.x == 0) tmax = 0;
      __syncthreads();
      atomicMax(&tmax, (unsigned long long)global_timer_ns());
      __syncthreads();
      if (threadIdx.x == 0) g_select_trace[blockIdx.x * 32 + 20] = tmax;
      if (threadIdx.x == 0) g_select_trace[blockIdx.x * 32 + 21] = __popc(hm);
    }
#endif
    int tot_ac;
    const int off_ac = block_excl_scan(na | (nc << 16), &tot_ac, s);
    if (threadIdx.x == 0) {
      s.bc[9] = tot_ac & 0xFFFF;  // staged emissions
      s.bc[10] = tot_ac >> 16;    // staged candidates
    }
    TOPK_LOG(u.r, 7);
#ifdef TOPK_TRACE
    if (threadIdx.x == 0) g_select_trace[blockIdx.x * 32 + 19] = global_timer_ns();
#endif
    int oa = off_ac & 0xFFFF, oc = off_ac >> 16;
    while (hm) {
      const int i = __ffs(hm) - 1;
      hm &= hm - 1u;
      const int v = threadIdx.x + i * kThreads;
      float4 x = b4[v];
      const int p0 = u.s0 + 4 * v - u.head;  // position of component 0
      clip(v, x);
      const uint32_t mg = ge_mask(x, tlo);
      const uint32_t ma = all_eq ? mg : ge_mask(x, thi);
      const uint32_t mc = stage_cand ? (mg & ~ma) : 0u;
      const float xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t below = (1u << j) - 1u;
        const int o = oa + __popc(ma & below);
        if (((ma >> j) & 1u) && o < TOPK_MAX_K) s.u.l.elist[o] = p0 + j;
        const int q = oc + __popc(mc & below);
        if (((mc >> j) & 1u) && q < kListCap) {
          s.u.l.ckey[q] = f2key(xs[j]);
          s.u.l.cpos[q] = (uint32_t)(p0 + j);
        }
      }
      oa += __popc(ma);
      oc += __popc(mc);
    }
  } else {
    const uint2 f = pass2_general(c, u, b0, all_eq, fallback, stage_cand);
    fa = f.x;
    fo = f.y;
  }
#ifdef TOPK_TRACE_DETAIL  // block-wide timing; distorts the phases it brackets
  {
    __shared__ unsigned long long wmax;
    if (threadIdx.x == 0) wmax = 0;
    const unsigned long long tnow = global_timer_ns();
    __syncthreads();
    atomicMax(&wmax, tnow);
    __syncthreads();
    if (threadIdx.x == 0) g_select_trace[blockIdx.x * 32 + 22] = wmax;
  }
#endif
  __syncthreads();  // staging lists and counts complete
  TOPK_MARK(g_select_trace, 4);
  TOPK_LOG(u.r, 4);
  if (fallback) block_and_or(fa, fo, s);

  // Multi-CTA rows: per-rank candidate slots let one barrier carry both the counts
  // (in the flags) and the candidates when the row's boundary bin is small enough
  // for every rank to fit its slot; otherwise candidates wait for the offsets.
  const int slot_cap = u.G > 1 ? kGroupCap / u.G : 0;
  const bool slots = compact && u.G > 1 && eq0 <= slot_cap;
  auto write_candidates = [&](int base) {
    // staged list, or an ordered second pass straight to global
    if (stage_cand) {
      const int nc = min(s.bc[10], kListCap);
      for (int i = threadIdx.x; i < nc; i += kThreads)
        if (base + i < kGroupCap) {
          u.gs->cand_key[base + i] = s.u.l.ckey[i];
          u.gs->cand_pos[base + i] = s.u.l.cpos[i];
        }
    } else {
      write_candidates_ordered(c, u, b0, base);
    }
  };
  if (slots) write_candidates(u.rank * slot_cap);

  // Row-wide offsets (G > 1) come with one barrier that delivers every rank's counts;
  // each CTA then clears the histogram bins it published. On the common path the
  // slots of the staged positions and of this CTA's own candidates are looked up
  // between its arrival and the wait (into the chunk buffer, free once pass 2 is
  // done: the candidate gather below uses its first 2 * kGroupCap words), so that
  // emitting after the barrier is stores only. The fallback's barrier also carries
  // the boundary keys' AND/OR.
  const uint32_t counts = (uint32_t)my_emit | ((uint32_t)my_cand << 16);
  const int n_emit = min(s.bc[9], TOPK_MAX_K);
  const int n_own = stage_cand ? min(s.bc[10], kListCap) : 0;
  int32_t* slot_e = reinterpret_cast<int32_t*>(s.buf) + 2 * kGroupCap;  // [TOPK_MAX_K]
  int32_t* slot_c = slot_e + TOPK_MAX_K;                                // [kListCap]
  const bool overlap = u.G > 1 && !fallback && !(compact && !slots && !stage_cand);
  int out_base = 0, cand_base = 0;
  if (overlap) {
    const uint32_t seq = group_arrive(c, u, counts);
    for (int i = threadIdx.x; i < n_emit; i += kThreads)
      slot_e[i] = lookup_slot(c, u, s.u.l.elist[i]);
    for (int i = threadIdx.x; i < n_own; i += kThreads)
      slot_c[i] = lookup_slot(c, u, (int)s.u.l.cpos[i]);
    int pre;
#ifdef TOPK_TRACE
    const long long qa = clock64();
#endif
    if (!group_wait(c, u, seq, &pre)) return;
#ifdef TOPK_TRACE
    const long long qb = clock64();
#endif
    out_base = pre & 0xFFFF;
    cand_base = pre >> 16;
    TOPK_MARK(g_select_trace, 5);
    for (int i = threadIdx.x; i < n_emit; i += kThreads)
      put(c, u, out_base + i, s.u.l.elist[i], slot_e[i]);
#ifdef TOPK_TRACE
    const long long qc = clock64();
    if (threadIdx.x == 0) {
      g_select_trace[blockIdx.x * 32 + 13] = (uint64_t)(qb - qa);
      g_select_trace[blockIdx.x * 32 + 14] = (uint64_t)(qc - qb);
    }
#endif
  } else {
    if (u.G > 1) {
      if (fallback && threadIdx.x == 0) {
        atomicOr(&u.gs->and_key, ~fa);  // stored inverted so the reset value is 0
        atomicOr(&u.gs->or_key, fo);
      }
      int pre;
      if (!group_sync(c, u, counts, &pre)) return;
      for (int i = u.blocal + threadIdx.x; i < kBins0; i += kThreads) u.gs->hist0[i] = 0u;
      out_base = pre & 0xFFFF;
      cand_base = pre >> 16;
      if (fallback) {
        if (threadIdx.x == 0) {
          s.bc[11] = (int)~__ldcg(&u.gs->and_key);
          s.bc[12] = (int)__ldcg(&u.gs->or_key);
        }
        __syncthreads();
        fa = (uint32_t)s.bc[11];
        fo = (uint32_t)s.bc[12];
      }
    }
    TOPK_MARK(g_select_trace, 5);
    // Emit the staged positions (table lookups of the whole CTA in parallel).
    for (int i = threadIdx.x; i < n_emit; i += kThreads) emit(c, u, out_base + i, s.u.l.elist[i]);
  }

  TOPK_LOG(u.r, 5);
  if (compact && u.G == 1) {
    __syncthreads();
    select_boundary_single(c, u, min(eq0, kListCap), need, above0);
  }

  if (compact && u.G > 1) {
    // Every CTA gathers all candidates (in rank order) and selects among them;
    // each emits its own selected candidates.
    const int n = min(eq0, kGroupCap);
    uint32_t* lkey = reinterpret_cast<uint32_t*>(s.buf);
    uint32_t* lpos = lkey + kGroupCap;
    __syncthreads();  // staged candidates (in the histogram region) no longer needed
    if (slots) {
      // s.pay[j] := exclusive prefix of the ranks' candidate counts (warp 0), then
      // every thread fetches its share of candidates with independent loads.
      if (threadIdx.x < 32) {
        int carry = 0;
        for (int j0 = 0; j0 < u.G; j0 += 32) {
          const int j = j0 + threadIdx.x;
          const int lj = j < u.G ? (int)(s.pay[j] >> 16) : 0;
          const int incl = warp_incl_scan(lj);
          if (j < u.G) s.pay[j] = (uint32_t)(carry + incl - lj);
          carry += __shfl_sync(0xffffffffu, incl, 31);
        }
      }
      __syncthreads();
      for (int i = threadIdx.x; i < n; i += kThreads) {
        int lo = 0, hi = u.G - 1;  // last rank whose prefix <= i
        while (lo < hi) {
          const int mid = (lo + hi + 1) >> 1;
          if ((int)s.pay[mid] <= i) lo = mid;
          else hi = mid - 1;
        }
        const int src = lo * slot_cap + (i - (int)s.pay[lo]);
        lkey[i] = __ldcg(&u.gs->cand_key[src]);
        lpos[i] = __ldcg(&u.gs->cand_pos[src]);
      }
    } else {
      write_candidates(cand_base);
      if (!group_sync(c, u, 0u, nullptr)) return;
      for (int i = threadIdx.x; i < n; i += kThreads) {
        lkey[i] = __ldcg(&u.gs->cand_key[i]);
        lpos[i] = __ldcg(&u.gs->cand_pos[i]);
      }
    }
    __syncthreads();
    TOPK_MARK(g_select_trace, 6);
#ifdef TOPK_TRACE
    const long long qd = clock64();
#endif
    const int own0 = min(cand_base, n), own1 = min(cand_base + le0, n);
    // The method must be the same in every CTA of the row (output index schemes
    // differ), so it depends on the row-wide count only.
    if (n <= kRankOwnMax) {
      // Rank this CTA's own candidates against all of them, T lanes per candidate
      // (groups of T never straddle a warp); the own staged candidates' slots were
      // looked up before the barrier.
      const int m = own1 - own0;
      const bool have_slots = overlap && stage_cand;
      int T = 1;
      while (T < 32 && m * (T * 2) <= kThreads) T *= 2;
      const int sub = threadIdx.x & (T - 1);
      for (int i0 = 0; i0 < m * T; i0 += kThreads) {
        const int gi = (i0 + threadIdx.x) / T;
        const bool act = gi < m;
        const uint32_t ki = act ? lkey[own0 + gi] : 0u, pi = act ? lpos[own0 + gi] : 0u;
        int rank = 0;
        if (act)
          for (int j = sub; j < n; j += T) {
            const uint32_t kj = lkey[j], pj = lpos[j];
            rank += (kj > ki || (kj == ki && pj < pi)) ? 1 : 0;
          }
        for (int o = 1; o < T; o <<= 1) rank += __shfl_xor_sync(0xffffffffu, rank, o);
        if (act && sub == 0 && rank < need) {
          if (have_slots) put(c, u, above0 + rank, (int)pi, slot_c[gi]);
          else emit(c, u, above0 + rank, (int)pi);
        }
      }
#ifdef TOPK_TRACE_DETAIL  // block-wide timing; distorts the phases it brackets
      {
        const long long qe = clock64();
        __shared__ unsigned long long qmx;
        if (threadIdx.x == 0) qmx = 0;
        __syncthreads();
        atomicMax(&qmx, (unsigned long long)(qe - qd));
        __syncthreads();
        if (threadIdx.x == 0) {
          g_select_trace[blockIdx.x * 32 + 15] = qmx;
          g_select_trace[blockIdx.x * 32 + 31] = (uint64_t)m | ((uint64_t)T << 16) | ((uint64_t)n << 32);
        }
      }
#endif
    } else {
      emit_listed(c, u, lkey, lpos, n, need, own0, own1, above0);
    }
    TOPK_MARK(g_select_trace, 7);
  }

  if (fallback) {
    if (!refine_in_place(c, u, b0, need, above0, fa, fo, le0)) return;
  }
  // The row histogram bins this CTA published are read by every CTA of the row before
  // its barrier-2 arrival; clear them for the next call (off the critical path).
  if (overlap)
    for (int i = u.blocal + threadIdx.x; i < kBins0; i += kThreads) u.gs->hist0[i] = 0u;
  TOPK_MARK(g_select_trace, 8);
  TOPK_LOG(u.r, 8);
}

__global__ void __launch_bounds__(kThreads, 1) select_kernel(const __grid_constant__ SelectParams p) {
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
    s.bc[29] = reinterpret_cast<const int32_t*>(p.ws + lay.first_single)[blockIdx.x];
    s.bc[20] = h0.x;  // magic
    s.bc[21] = h0.y;  // rows
    s.bc[22] = h0.z;  // max_len
    s.bc[23] = h0.w;  // grid
    s.bc[24] = h1.y;  // waves
    s.bc[25] = h1.z;  // n_single
    s.bc[26] = h2.y;  // plan_error
    s.bc[27] = h2.z;  // n_implicit
    s.bc[28] = h2.w;  // dyn_period
    s.bc[7] = 0;      // no aborting copy
    for (int i = 0; i < kPieces; ++i) mbar_init(&s.mbar[i], 1);
    fence_mbar_init();
    // Start the first static unit's copies right away when the plan is valid.
    const UnitDesc d = s.ud;
    const bool ok = (uint32_t)h0.x == kMagic && h0.y == p.rows && h0.z == p.max_len &&
                    h0.w == (int)gridDim.x && h2.y == 0 && h1.y > 0;
    s.bc[19] = 0;
    if (ok && d.row >= 0 && d.len >= 0 && d.len <= p.max_len && d.len > p.k &&
        (d.G == 1 || d.group >= 0)) {
      Unit u;
      u.r = d.row;
      u.s0 = d.s0;
      u.n = d.n;
      const char* src;
      const uint32_t bytes = chunk_geometry(p, u, &src);
      issue_copies(s, src, bytes, 0, min(kWindow, u.npieces));
      s.bc[19] = 1;
    }
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
  if (threadIdx.x == 0) trace_log_n() = 0;
  TOPK_LOG(-1, 0);
#endif

  const bool pre_issued = s.bc[19] != 0;
  Ctx c{p, h, s, 0u};
  bool ran = false;  // a unit ran: s.bc[7] (aborting) is read after a CTA barrier
  // Units in one loop (one call site keeps the unit body inlined once): the static
  // multi-CTA units of every wave, then the single row the plan hands this CTA (read
  // in the prologue), then tickets. When the plan hands out every single row, no CTA
  // claims one (each call then advances the ticket counter by 0, a multiple of its
  // period, as the modular claims need).
  const int2* singles = reinterpret_cast<const int2*>(p.ws + lay.singles);
  int idx = s.bc[29];
  bool implicit = idx >= 0;
  const bool tickets = n_single > n_implicit;
  for (int w = 0;;) {
    UnitDesc d;
    bool pre = false;
    if (w < waves) {
      if (w == 0) {
        d = s.ud;
        pre = pre_issued;
      } else {
        __syncthreads();
        if (ran && s.bc[7]) break;
        if (threadIdx.x == 0) s.ud = units[(int64_t)w * kMaxGrid + blockIdx.x];
        __syncthreads();
        d = s.ud;
      }
      ++w;
      TOPK_LOG(d.row, 15);
      if (d.row < 0) continue;
    } else {
      if (!implicit && !tickets) break;
      if (ran) {
        __syncthreads();
        if (s.bc[7]) break;
      }
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
      d.row = sr.x;
      d.s0 = 0;
      d.len = sr.y;
      d.n = (sr.y >= 0 && sr.y <= p.max_len) ? sr.y : 0;
      d.rank = 0;
      d.G = 1;
      d.group = -1;
      d.pad = 0;
    }
    process_unit(c, d, pre);
    ran = true;
  }
  if (ran) {
    __syncthreads();
    if (s.bc[7] && threadIdx.x == 0)  // the copy that never landed: one more bounded wait
      mbar_wait_bounded(&s.mbar[s.bc[8]], (uint32_t)s.bc[13], p.wait_ns);
  }
  TOPK_MARK(g_select_trace, 9);
#ifdef TOPK_TRACE
  if (threadIdx.x == 0) g_select_log_n[blockIdx.x] = trace_log_n();
#endif
}

}  // namespace

#ifdef TOPK_TRACE
extern "C" int topk_trace_log(uint64_t* host, int* counts) {
  if (cudaMemcpyFromSymbol(host, g_select_log, sizeof(uint64_t) * kMaxGrid * 256) != cudaSuccess)
    return -9;
  return cudaMemcpyFromSymbol(counts, g_select_log_n, sizeof(int) * kMaxGrid) == cudaSuccess ? 0 : -9;
}
extern "C" int topk_trace_select(uint64_t* host, int n) {
  if (n > kMaxGrid * 32) n = kMaxGrid * 32;
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
