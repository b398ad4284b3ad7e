// Planning kernel: bins the batch's rows into single-CTA and multi-CTA paths and
// builds the persistent grid's work list ("Serving GLM5.2 NVFP4 Agentic Workload
// with SGLang", "Kernel Optimization > TopK-V2": the planning kernel chooses the
// cluster cutoff from the sequence-length distribution and builds the work list).
//
// Block 0 plans; the other blocks clear the per-row group state so the select
// kernel's counters start at zero. Reads only device-resident lengths: no host sync.
//
// Output (see common.cuh): per-row info; a static unit table (one 32-byte
// descriptor per wave and CTA, multi-CTA rows only); the single-CTA rows longest
// bucket first; for each CTA without static work, the index of one single row it
// takes without claiming a ticket.
#include <cuda_runtime.h>

#include <climits>
#include <cstddef>

#include "common.cuh"
#include "plan_logic.cuh"

namespace topk {

namespace {

#ifdef TOPK_TRACE
__device__ uint64_t g_plan_trace[kMaxGrid * 32];
#endif

constexpr int kPlanThreads = 256;
constexpr int kPlanWarps = kPlanThreads / 32;
constexpr int kLensCache = 4096;     // batches up to this many rows plan from shared memory
constexpr int kCandidateRows = 64;   // chunk search by parallel candidates up to this many rows
constexpr int kZeroPerThread = 4;    // 16-byte stores per thread of a zeroing block

struct PlanSmem {
  long long red64[kPlanWarps];
  int red[3][kPlanWarps];
  int bcast[8];
  int32_t multi_rows[kMaxGroups];
  int32_t multi_g[kMaxGroups];
  int32_t multi_wave[kMaxGroups];
  int32_t multi_cta[kMaxGroups];
  uint8_t busy[kMaxGrid];  // CTAs with static units
  unsigned bucket_mask;
  int32_t wcnt[kPlanWarps][32];  // one-pass ranking: a round's single rows per warp, bucket
  int32_t bbase[32];             // first rank of each bucket (longer buckets first)
  int32_t bcarry[32];            // single rows of each bucket in the earlier rounds
  int32_t lens[kLensCache];
};

// row_groups(L, c) for 0 <= L < 2^31 and 1 <= c < 2^16 with a reciprocal instead of
// a division (division by an invariant integer: m = floor((2^32 - 1) / c) makes
// floor(n * m / 2^32) low by at most one, which one compare corrects).
struct Divider {
  uint32_t d, m;
  __device__ explicit Divider(int c) : d((uint32_t)c), m(0xFFFFFFFFu / (uint32_t)c) {}
  __device__ int groups(int L) const {
    if (L <= (int)d) return 1;
    const uint32_t n = (uint32_t)L + d - 1u;  // ceil(L / d) = floor(n / d)
    uint32_t q = __umulhi(n, m);
    if (n - q * d >= d) ++q;
    return (int)q;
  }
};

// The block-wide helpers stay out of line: the planner runs once per batch from a cold
// instruction cache, so one shared copy of each costs less than inlined copies.
__device__ __noinline__ void block_stats(long long& a, int& b, int& c, PlanSmem& s) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  long long aa = a;
  int bb = b, cc = c;
  for (int o = 16; o; o >>= 1) {
    aa += __shfl_xor_sync(0xffffffffu, aa, o);
    bb += __shfl_xor_sync(0xffffffffu, bb, o);
    cc = max(cc, __shfl_xor_sync(0xffffffffu, cc, o));
  }
  if (lane == 0) {
    s.red64[w] = aa;
    s.red[0][w] = bb;
    s.red[1][w] = cc;
  }
  __syncthreads();
  long long ta = 0;
  int tb = 0, tc = 0;
#pragma unroll
  for (int i = 0; i < kPlanWarps; ++i) {
    ta += s.red64[i];
    tb += s.red[0][i];
    tc = max(tc, s.red[1][i]);
  }
  __syncthreads();
  a = ta;
  b = tb;
  c = tc;
}

__device__ __noinline__ int block_min(int v, PlanSmem& s) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  for (int o = 16; o; o >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
  if (lane == 0) s.red[2][w] = v;
  __syncthreads();
  int m = s.red[2][0];
#pragma unroll
  for (int i = 1; i < kPlanWarps; ++i) m = min(m, s.red[2][i]);
  __syncthreads();
  return m;
}

// Exclusive scan of one int per thread; the block total goes to *total.
__device__ __noinline__ int block_scan(int v, int* total, PlanSmem& s) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int x = v;
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s.red[2][w] = x;
  __syncthreads();
  int before = 0, tot = 0;
#pragma unroll
  for (int i = 0; i < kPlanWarps; ++i) {
    if (i < w) before += s.red[2][i];
    tot += s.red[2][i];
  }
  __syncthreads();
  *total = tot;
  return before + x - v;
}

// CTAs of the multi-CTA rows at chunk c, one thread over every row (small batches).
__device__ long long slots_serial(const int32_t* L_, int rows, int max_len, int c) {
  const Divider dv(c);
  long long n = 0;
  for (int r = 0; r < rows; ++r) {
    const int G = dv.groups(valid_len(L_[r], max_len));
    if (G > 1) n += G;
  }
  return n;
}

// The same, rows spread over the block.
__device__ long long slots_block(const int32_t* L_, int rows, int max_len, int c, PlanSmem& s) {
  const Divider dv(c);
  long long n = 0;
  int b = 0, m = 0;
  for (int r = threadIdx.x; r < rows; r += kPlanThreads) {
    const int G = dv.groups(valid_len(L_[r], max_len));
    if (G > 1) n += G;
  }
  block_stats(n, b, m, s);
  return n;
}

// Automatic chunk (plan_logic.cuh, auto_chunk_ref): the smallest multiple of
// kChunkAlign >= c0 whose multi-CTA rows fit the grid; kChunkCap when none does
// (*fits = false). The CTA count only falls as c grows, so the first passing
// candidate is the answer: up to kCandidateRows rows, 256 candidates spanning
// [c0, kChunkCap] are tried at once and the step before the first pass is refined;
// larger batches bisect.
__device__ int auto_chunk(const int32_t* L_, int rows, int max_len, int grid, long long total,
                          bool* fits, PlanSmem& s) {
  const int c0 = initial_chunk(total, grid, 0);
  const int tid = threadIdx.x;
  *fits = true;
  if (rows <= kCandidateRows) {
    int step = (kChunkCap - c0 + kPlanThreads - 2) / (kPlanThreads - 1);
    step = max(kChunkAlign, (step + kChunkAlign - 1) / kChunkAlign * kChunkAlign);
    const int ct = min(c0 + step * tid, kChunkCap);
    const int first = block_min(slots_serial(L_, rows, max_len, ct) <= grid ? tid : INT_MAX, s);
    if (first == INT_MAX) {
      *fits = false;
      return kChunkCap;
    }
    if (first == 0) return c0;
    const int lo = c0 + step * (first - 1);          // fails
    const int hi = min(c0 + step * first, kChunkCap);  // passes
    const int n2 = (hi - lo) / kChunkAlign;            // lo + 16, ..., hi
    const int c2 = lo + kChunkAlign * (tid + 1);
    const bool ok2 = tid < n2 && slots_serial(L_, rows, max_len, c2) <= grid;
    const int f2 = block_min(ok2 ? tid : INT_MAX, s);
    return lo + kChunkAlign * (f2 + 1);
  }
  if (slots_block(L_, rows, max_len, c0, s) <= grid) return c0;
  if (slots_block(L_, rows, max_len, kChunkCap, s) > grid) {
    *fits = false;
    return kChunkCap;
  }
  int lo = c0, hi = kChunkCap;  // lo fails, hi passes
  while (hi - lo > kChunkAlign) {
    const int mid = lo + (hi - lo) / (2 * kChunkAlign) * kChunkAlign;
    if (slots_block(L_, rows, max_len, mid, s) <= grid) hi = mid;
    else lo = mid;
  }
  return hi;
}

// Plan of a batch of at most 64 rows without a forced chunk: warp 0 decides (lane l
// holds rows l and l + 32: the chunk search tries 32 candidates per round, a ballot
// picks the first that fits; group indices and first CTAs are warp scans), then the
// block writes the tables. Same plan as the general path below (auto_chunk_ref's rule, one wave).
// Returns false, with nothing written, when the rows do not fit one wave even at
// kChunkCap (the general path then packs several waves).
constexpr int kSmallRows = 64;
constexpr int kRowsPerLane = kSmallRows / 32;  // lane l holds rows l and l + 32

__device__ bool plan_small(const int32_t* __restrict__ lens, int rows, int max_len, int grid,
                           char* ws, const Layout& lay, PlanSmem& s) {
  Header* h = reinterpret_cast<Header*>(ws + lay.header);
  RowInfo* ri = reinterpret_cast<RowInfo*>(ws + lay.rowinfo);
  int2* singles = reinterpret_cast<int2*>(ws + lay.singles);
  int32_t* first_single = reinterpret_cast<int32_t*>(ws + lay.first_single);
  UnitDesc* units = reinterpret_cast<UnitDesc*>(ws + lay.units);
  const int tid = threadIdx.x, lane = tid & 31;
  constexpr unsigned kAll = 0xffffffffu;
  constexpr int kR = kRowsPerLane;
  if (tid < 32) {
    int Lraw[kR], L[kR];
#pragma unroll
    for (int q = 0; q < kR; ++q) {
      const int r = lane + 32 * q;
      Lraw[q] = r < rows ? lens[r] : 0;
      L[q] = r < rows ? valid_len(Lraw[q], max_len) : 0;
    }
    long long tot = 0;
    int mx = 0;
#pragma unroll
    for (int q = 0; q < kR; ++q) {
      tot += L[q];
      mx = max(mx, L[q]);
    }
    for (int o = 16; o; o >>= 1) {
      tot += __shfl_xor_sync(kAll, tot, o);
      mx = max(mx, __shfl_xor_sync(kAll, mx, o));
    }
    // CTAs of the split rows at chunk cc (every lane evaluates its own cc)
    auto slots_at = [&](int cc) {
      const Divider dv(cc);
      int n = 0;
#pragma unroll
      for (int q = 0; q < kR; ++q)
        for (int j = 0; j < 32 && 32 * q + j < rows; ++j) {
          const int G = dv.groups(__shfl_sync(kAll, L[q], j));
          n += G > 1 ? G : 0;
        }
      return n;
    };
#pragma unroll
    for (int q = 0; q < kR; ++q)
      if (lane + 32 * q < rows) s.lens[lane + 32 * q] = L[q];
    const int c0 = initial_chunk(tot, grid, 0);
    // a fails (c0 may pass). b: with grid / rows CTAs for every row, chunk
    // ceil(max length / (grid / rows)) fits whatever the lengths, so b is that chunk
    // (at least c0) when it is below kChunkCap; else kChunkCap, which passes unless no
    // chunk fits. The first round always runs, and its lane 31 evaluates b.
    int a = c0 - kChunkAlign, b = kChunkCap;
    const int per_row = rows > 0 ? grid / rows : 0;
    if (per_row > 0) {
      const uint32_t hi = ((uint32_t)mx + (uint32_t)per_row - 1u) / (uint32_t)per_row;
      if (hi < (uint32_t)kChunkCap) b = max(c0, round_chunk(hi));
    }
    bool fits = true;
    do {
      // 32 increasing candidates in (a, b], b among them. A wide bracket gets 16 spread
      // over (a, b - 256] and 16 at steps of 16 up to b: equal lengths put the answer
      // at or just below b, which one round then settles.
      int cand;
      if (b - a <= 32 * kChunkAlign) {
        cand = min(a + kChunkAlign * (lane + 1), b);
      } else if (lane >= 16) {
        cand = b - kChunkAlign * (31 - lane);
      } else {
        int step = (b - 16 * kChunkAlign - a + 15) / 16;
        step = (step + kChunkAlign - 1) / kChunkAlign * kChunkAlign;
        cand = min(a + step * (lane + 1), b - 16 * kChunkAlign);
      }
      const unsigned m = __ballot_sync(kAll, slots_at(cand) <= grid);
      if (m == 0u) {
        fits = false;
        break;
      }
      const int first = __ffs(m) - 1;
      const int nb = __shfl_sync(kAll, cand, first);
      const int na = __shfl_sync(kAll, cand, max(first - 1, 0));
      a = first == 0 ? a : na;
      b = nb;
    } while (b - a > kChunkAlign);
    const int c = b;
    if (lane == 0) s.bcast[4] = fits ? 1 : 0;
    if (fits) {
      // Rows in row order: all of the first set (lanes' rows 0..31), then the second.
      const Divider dv(c);
      const unsigned lt = (1u << lane) - 1u;
      int G[kR], gi[kR];
      bool multi[kR], single[kR];
      unsigned mm[kR], sm[kR];
      int bucket[kR];
      int before_m = 0, before_g = 0;  // multi rows and their CTAs in the earlier sets
#pragma unroll
      for (int q = 0; q < kR; ++q) {
        const int r = lane + 32 * q;
        G[q] = r < rows ? dv.groups(L[q]) : 1;
        multi[q] = G[q] > 1;
        mm[q] = __ballot_sync(kAll, multi[q]);
        gi[q] = before_m + __popc(mm[q] & lt);
        int incl = multi[q] ? G[q] : 0;
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(kAll, incl, o);
          if (lane >= o) incl += y;
        }
        if (multi[q]) {
          s.multi_rows[gi[q]] = r;
          s.multi_g[gi[q]] = G[q];
          s.multi_wave[gi[q]] = 0;
          s.multi_cta[gi[q]] = before_g + incl - G[q];
        }
        if (r < rows) {
          RowInfo x;
          x.len = Lraw[q];
          x.G = G[q];
          x.group = multi[q] ? gi[q] : -1;
          x.pad = 0;
          ri[r] = x;
        }
        before_m += __popc(mm[q]);
        before_g += __shfl_sync(kAll, incl, 31);
        single[q] = r < rows && !multi[q];
        bucket[q] = L[q] > 0 ? 31 - __clz(L[q]) : 0;
        sm[q] = __ballot_sync(kAll, single[q]);
      }
      const int total_slots = before_g;
      // single rows: longest length bucket first, row order inside a bucket. A row's
      // rank counts the single rows of a larger bucket and those of its bucket in lower
      // rows: the 5-bit buckets are compared bit by bit from the top on ballots.
      unsigned ones[kR][5];
#pragma unroll
      for (int p = 0; p < kR; ++p)
#pragma unroll
        for (int bit = 0; bit < 5; ++bit)
          ones[p][bit] = __ballot_sync(kAll, single[p] && ((bucket[p] >> bit) & 1));
      int n_single = 0;
#pragma unroll
      for (int p = 0; p < kR; ++p) n_single += __popc(sm[p]);
#pragma unroll
      for (int q = 0; q < kR; ++q) {
        int rank = 0;
#pragma unroll
        for (int p = 0; p < kR; ++p) {
          unsigned eq = sm[p], gt = 0u;
#pragma unroll
          for (int bit = 4; bit >= 0; --bit) {
            if ((bucket[q] >> bit) & 1) {
              eq &= ones[p][bit];
            } else {
              gt |= eq & ones[p][bit];
              eq &= ~ones[p][bit];
            }
          }
          rank += __popc(gt) + (p < q ? __popc(eq) : p == q ? __popc(eq & lt) : 0);
        }
        if (single[q]) singles[rank] = make_int2(lane + 32 * q, Lraw[q]);
      }
      int n_multi = 0;
#pragma unroll
      for (int q = 0; q < kR; ++q) n_multi += __popc(mm[q]);
      if (lane == 0) {
        const int n_implicit = min(grid - total_slots, n_single);
        h->magic = kMagic;
        h->rows = rows;
        h->max_len = max_len;
        h->grid = grid;
        h->chunk = c;
        h->waves = n_multi > 0 ? 1 : 0;
        h->n_single = n_single;
        h->n_multi = n_multi;
        h->status = 0;
        h->plan_error = 0;
        h->n_implicit = n_implicit;
        h->dyn_period = n_single - n_implicit + grid;
        h->steal = 0ull;
        h->med_ticket = 0ull;
        for (int i = 0; i < 8; ++i) h->diag[i] = 0;
        s.bcast[0] = n_multi;
        s.bcast[1] = total_slots;
        s.bcast[2] = n_single;
      }
    }
  }
  __syncthreads();
  if (!s.bcast[4]) return false;
  const int n_multi = s.bcast[0], total_slots = s.bcast[1], n_single = s.bcast[2];
  // Unit table of wave 0 (one thread per CTA, its descriptor as two 16-byte stores)
  // and the first-single table in closed form (busy CTAs are [0, total_slots)).
  for (int b = tid; b < grid; b += kPlanThreads) {
    UnitDesc u{-1, 0, 0, 0, 0, 0, 0, 0};
    if (n_multi > 0 && b < total_slots) {
      int lo = 0, hi = n_multi - 1;  // last group whose first CTA <= b
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s.multi_cta[mid] <= b) lo = mid;
        else hi = mid - 1;
      }
      const int row = s.multi_rows[lo];
      u = make_unit(row, s.lens[row], b - s.multi_cta[lo], s.multi_g[lo], lo);
    }
    uint4* d = reinterpret_cast<uint4*>(units + b);
    d[0] = make_uint4(u.row, u.s0, u.n, u.len);
    d[1] = make_uint4(u.rank, u.G, u.group, u.pad);
    first_single[b] = (b >= total_slots && b - total_slots < n_single) ? b - total_slots : -1;
  }
  return true;
}

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(const int32_t* __restrict__ lens,
                                                            int rows, int max_len, int grid,
                                                            int chunk_force, char* ws) {
  const Layout lay = make_layout(rows);
  Header* h = reinterpret_cast<Header*>(ws + lay.header);
  RowInfo* ri = reinterpret_cast<RowInfo*>(ws + lay.rowinfo);
  int2* singles = reinterpret_cast<int2*>(ws + lay.singles);
  int32_t* first_single = reinterpret_cast<int32_t*>(ws + lay.first_single);
  UnitDesc* units = reinterpret_cast<UnitDesc*>(ws + lay.units);

  TOPK_MARK(g_plan_trace, 0);
  if (blockIdx.x > 0) {
    // Clear what the select kernel needs at zero in every group state: barrier
    // flags, boundary-key AND/OR and histograms (the candidate lists are always
    // written before they are read).
    constexpr size_t kZeroBytes = offsetof(GroupState, cand_key);
    static_assert(kZeroBytes % 16 == 0 && sizeof(GroupState) % 16 == 0, "zeroing granularity");
    char* g = ws + lay.groups;
    constexpr uint32_t per = (uint32_t)(kZeroBytes / 16);
    const uint32_t n16 = per * (uint32_t)lay.ngroups;  // < 2^23
    const uint4 z = make_uint4(0, 0, 0, 0);
    for (uint32_t i = (blockIdx.x - 1) * blockDim.x + threadIdx.x; i < n16;
         i += (gridDim.x - 1) * blockDim.x) {
      const uint32_t grp = i / per, off = i - grp * per;
      reinterpret_cast<uint4*>(g + (size_t)grp * sizeof(GroupState))[off] = z;
    }
    TOPK_MARK(g_plan_trace, 9);
    return;
  }

  __shared__ PlanSmem s;
  const int tid = threadIdx.x;
  if (chunk_force <= 0 && rows <= kSmallRows && plan_small(lens, rows, max_len, grid, ws, lay, s)) {
    TOPK_MARK(g_plan_trace, 5);
    return;
  }

  // Lengths are read many times below: keep them in shared memory when they fit.
  const bool cached = rows <= kLensCache;
  if (cached) {
    // eight independent loads per thread in flight: the lengths come from cold memory
    for (int r0 = 0; r0 < rows; r0 += 8 * kPlanThreads) {
      int v[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int r = r0 + e * kPlanThreads + tid;
        v[e] = r < rows ? lens[r] : 0;
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int r = r0 + e * kPlanThreads + tid;
        if (r < rows) s.lens[r] = v[e];
      }
    }
  }
  __syncthreads();
  const int32_t* L_ = cached ? s.lens : lens;

  long long total = 0;
  int dummy_b = 0, dummy_c = 0;
  for (int r = tid; r < rows; r += kPlanThreads) total += valid_len(L_[r], max_len);
  block_stats(total, dummy_b, dummy_c, s);
  TOPK_MARK(g_plan_trace, 1);

  const bool forced = chunk_force > 0;
  bool fits = false;
  int c = forced ? initial_chunk(total, grid, chunk_force)
                 : auto_chunk(L_, rows, max_len, grid, total, &fits, s);
  TOPK_MARK(g_plan_trace, 2);

  int waves = 0, plan_error = 0, n_multi = 0;
  if (!forced && fits) {
    // One wave: a row's group index and first CTA are exclusive prefixes over the
    // rows (at most grid CTAs in total, so both fit 16 bits). Thread t takes a
    // contiguous range of rows, so one block scan of its (count, CTAs) orders them.
    const Divider dv(c);
    const int per = (rows + kPlanThreads - 1) / kPlanThreads;
    const int rb = min(rows, tid * per), re = min(rows, rb + per);
    int mine = 0;
    for (int r = rb; r < re; ++r) {
      const int G = dv.groups(valid_len(L_[r], max_len));
      if (G > 1) mine += (1 << 16) | G;
    }
    int tot;
    int off = block_scan(mine, &tot, s);
    for (int r = rb; r < re && mine; ++r) {
      const int G = dv.groups(valid_len(L_[r], max_len));
      if (G > 1) {
        const int i = off >> 16;
        s.multi_rows[i] = r;
        s.multi_g[i] = G;
        s.multi_wave[i] = 0;
        s.multi_cta[i] = off & 0xFFFF;
        off += (1 << 16) | G;
      }
    }
    n_multi = tot >> 16;
    waves = n_multi > 0 ? 1 : 0;
  } else {
    // Forced chunk, or rows that do not fit one wave even at kChunkCap: grow the
    // chunk while the groups break a hard limit (next_chunk), packing the groups
    // into waves greedily.
    PlanStats st{0, 0, 0};
    for (int iter = 0; iter < 64; ++iter) {
      long long slots = 0;
      int nm = 0, mg = 0;
      const Divider dv(c);
      for (int r = tid; r < rows; r += kPlanThreads) {
        const int G = dv.groups(valid_len(L_[r], max_len));
        if (G > 1) {
          slots += G;
          nm += 1;
          mg = max(mg, G);
        }
      }
      block_stats(slots, nm, mg, s);
      st = PlanStats{slots, nm, mg};
      if (nm <= lay.ngroups && mg <= grid) {
        int base = 0;
        for (int r0 = 0; r0 < rows; r0 += kPlanThreads) {
          const int r = r0 + tid;
          const int G = r < rows ? dv.groups(valid_len(L_[r], max_len)) : 1;
          int tot;
          const int off = block_scan(G > 1 ? 1 : 0, &tot, s);
          if (G > 1) {
            s.multi_rows[base + off] = r;
            s.multi_g[base + off] = G;
          }
          base += tot;
        }
        __syncthreads();
        if (tid == 0) s.bcast[0] = pack_waves(s.multi_g, nm, grid, s.multi_wave, s.multi_cta);
        __syncthreads();
        waves = s.bcast[0];
      } else {
        waves = kMaxWaves + 1;
      }
      const int nc = next_chunk(c, st, waves, grid, forced, lay.ngroups);
      if (nc == c) break;
      if (nc < 0) {
        plan_error = 1;
        break;
      }
      c = nc;
    }
    n_multi = plan_error ? 0 : st.n_multi;
  }
  __syncthreads();
  TOPK_MARK(g_plan_trace, 3);

  // Static unit table for the grid's CTAs, one pass: CTA b of wave w runs the group
  // whose CTA range holds it (groups are ordered by wave, then first CTA), else
  // nothing. Two threads write the two 16-byte halves of one descriptor, so each
  // warp stores 512 contiguous bytes.
  const int wv = plan_error ? 0 : waves;
  for (int i = tid; i < 2 * kMaxGrid; i += kPlanThreads) {
    const int b = i >> 1;
    if (b >= grid) break;
    bool busy = false;
    for (int w = 0; w < wv; ++w) {
      int lo = 0, hi = n_multi - 1, f = -1;
      while (lo <= hi) {
        const int mid = (lo + hi) >> 1;
        if (s.multi_wave[mid] < w || (s.multi_wave[mid] == w && s.multi_cta[mid] <= b)) {
          f = mid;
          lo = mid + 1;
        } else {
          hi = mid - 1;
        }
      }
      UnitDesc u{-1, 0, 0, 0, 0, 0, 0, 0};
      if (f >= 0 && s.multi_wave[f] == w && b < s.multi_cta[f] + s.multi_g[f]) {
        const int row = s.multi_rows[f];
        u = make_unit(row, valid_len(L_[row], max_len), b - s.multi_cta[f], s.multi_g[f], f);
        busy = true;
      }
      const uint4 half = (i & 1) ? make_uint4(u.rank, u.G, u.group, u.pad)
                                 : make_uint4(u.row, u.s0, u.n, u.len);
      reinterpret_cast<uint4*>(units + (int64_t)w * kMaxGrid + b)[i & 1] = half;
    }
    if ((i & 1) == 0) s.busy[b] = busy ? 1 : 0;
  }
  TOPK_MARK(g_plan_trace, 10);
  __syncthreads();
  TOPK_MARK(g_plan_trace, 4);

  // Row info.
  const Divider dvc(c);
  for (int r = tid; r < rows; r += kPlanThreads) {
    RowInfo x;
    x.len = L_[r];
    x.G = plan_error ? 1 : dvc.groups(valid_len(L_[r], max_len));
    x.group = -1;
    x.pad = 0;
    ri[r] = x;
  }
  __syncthreads();
  TOPK_MARK(g_plan_trace, 6);
  for (int i = tid; i < n_multi; i += kPlanThreads) ri[s.multi_rows[i]].group = i;

  // Single-CTA rows, longest bucket first, row order inside a bucket.
  if (tid == 0) s.bucket_mask = 0u;
  __syncthreads();
  {
    // each thread ORs its rows' buckets, a warp reduction, one shared atomic per warp
    unsigned bm = 0u;
    for (int r = tid; r < rows; r += kPlanThreads) {
      const int L = valid_len(L_[r], max_len);
      if (plan_error || dvc.groups(L) == 1) bm |= 1u << len_bucket(L);
    }
    bm = __reduce_or_sync(0xffffffffu, bm);
    if ((tid & 31) == 0 && bm) atomicOr(&s.bucket_mask, bm);
  }
  __syncthreads();
  TOPK_MARK(g_plan_trace, 7);
#ifdef TOPK_TRACE
  const long long ck0 = clock64();
#endif
  const unsigned mask = s.bucket_mask;
  int n_single = 0;
  const int rounds = (rows + kPlanThreads - 1) / kPlanThreads;
  if (__popc(mask) > 2 * rounds) {
    // Many buckets, few rows: one pass in rounds of kPlanThreads rows (row r0 + tid).
    // A row's rank is its bucket's first rank, plus the bucket's single rows in earlier
    // rounds, in lower warps of this round and in lower lanes of its warp (peers by
    // __match_any_sync on the bucket). Two sweeps: bucket totals, then the ranks.
    const int lane = tid & 31, w = tid >> 5;
    const unsigned lt = (1u << lane) - 1u;
    if (tid < 32) {
      s.bbase[tid] = 0;
      s.bcarry[tid] = 0;
    }
    __syncthreads();
    for (int r0 = 0; r0 < rows; r0 += kPlanThreads) {  // totals per bucket
      const int r = r0 + tid;
      int key = 64 + lane;  // unique: matches no bucket
      if (r < rows) {
        const int L = valid_len(L_[r], max_len);
        if (plan_error || dvc.groups(L) == 1) key = len_bucket(L);
      }
      const unsigned peers = __match_any_sync(0xffffffffu, key);
      if (key < 32 && (peers & lt) == 0u) atomicAdd(&s.bbase[key], __popc(peers));
    }
    __syncthreads();
    if (tid < 32) {  // bbase[b] := single rows in buckets above b (longer first)
      const int t = s.bbase[tid];
      int incl = t;  // inclusive suffix sum: buckets >= tid
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_down_sync(0xffffffffu, incl, o);
        if (lane + o < 32) incl += y;
      }
      s.bbase[tid] = incl - t;
      if (tid == 0) s.bcast[5] = incl;  // all single rows
    }
    __syncthreads();
    n_single = s.bcast[5];
    for (int r0 = 0; r0 < rows; r0 += kPlanThreads) {  // ranks
      const int r = r0 + tid;
      int key = 64 + lane, Lraw = 0;
      if (r < rows) {
        Lraw = L_[r];
        const int L = valid_len(Lraw, max_len);
        if (plan_error || dvc.groups(L) == 1) key = len_bucket(L);
      }
      const unsigned peers = __match_any_sync(0xffffffffu, key);
      s.wcnt[w][lane] = 0;
      __syncwarp();
      if (key < 32 && (peers & lt) == 0u) s.wcnt[w][key] = __popc(peers);
      __syncthreads();
      if (key < 32) {
        int rank = s.bbase[key] + s.bcarry[key] + __popc(peers & lt);
        for (int v = 0; v < w; ++v) rank += s.wcnt[v][key];
        singles[rank] = make_int2(r, Lraw);
      }
      __syncthreads();
      if (tid < 32) {
        int add = 0;
#pragma unroll
        for (int v = 0; v < kPlanWarps; ++v) add += s.wcnt[v][tid];
        s.bcarry[tid] += add;
      }
      __syncthreads();
    }
  } else {
    // thread t takes a contiguous range of rows: one block scan per present bucket
    const int per = (rows + kPlanThreads - 1) / kPlanThreads;
    const int rb = min(rows, tid * per), re = min(rows, rb + per);
#pragma unroll 1
    for (unsigned m = mask; m != 0u; m &= ~(1u << (31 - __clz(m)))) {
      const int b = 31 - __clz(m);  // present buckets, longest first
      int cnt = 0;
      for (int r = rb; r < re; ++r) {
        const int L = valid_len(L_[r], max_len);
        cnt += ((plan_error || dvc.groups(L) == 1) && len_bucket(L) == b) ? 1 : 0;
      }
      int tot;
      int off = n_single + block_scan(cnt, &tot, s);
      for (int r = rb; r < re && cnt; ++r) {
        const int Lraw = L_[r];
        const int L = valid_len(Lraw, max_len);
        if ((plan_error || dvc.groups(L) == 1) && len_bucket(L) == b) {
          singles[off++] = make_int2(r, Lraw);
          --cnt;
        }
      }
      n_single += tot;
    }
  }

  // One single row per CTA without static units, in CTA order.
#ifdef TOPK_TRACE
  const long long ck1 = clock64();
  long long ck2 = 0, ck3 = 0;
#endif
  int ordinal_base = 0;
  for (int c0 = 0; c0 < grid; c0 += kPlanThreads) {
    const int cta = c0 + tid;
    const bool free_cta = cta < grid && !s.busy[cta];
    int tot;
    const int ord = ordinal_base + block_scan(free_cta ? 1 : 0, &tot, s);
#ifdef TOPK_TRACE
    ck2 = clock64();
#endif
    if (cta < grid) first_single[cta] = (free_cta && ord < n_single) ? ord : -1;
    ordinal_base += tot;
#ifdef TOPK_TRACE
    ck3 = clock64();
#endif
  }
#ifdef TOPK_TRACE
  if (tid == 0) {
    g_plan_trace[11] = (uint64_t)(ck1 - ck0);
    g_plan_trace[12] = (uint64_t)(ck2 - ck1);
    g_plan_trace[13] = (uint64_t)(ck3 - ck2);
    g_plan_trace[14] = (uint64_t)mask;
  }
#endif
  const int n_implicit = min(ordinal_base, n_single);
  TOPK_MARK(g_plan_trace, 8);

  if (tid == 0) {
    h->magic = kMagic;
    h->rows = rows;
    h->max_len = max_len;
    h->grid = grid;
    h->chunk = c;
    h->waves = wv;
    h->n_single = n_single;
    h->n_multi = n_multi;
    h->status = plan_error ? TOPK_STATUS_PLAN_MISMATCH : 0;
    h->plan_error = plan_error;
    h->n_implicit = n_implicit;
    h->dyn_period = n_single - n_implicit + grid;
    h->steal = 0ull;
    h->med_ticket = 0ull;
    for (int i = 0; i < 8; ++i) h->diag[i] = 0;
  }
  TOPK_MARK(g_plan_trace, 5);
}

}  // namespace

#ifdef TOPK_TRACE
extern "C" int topk_trace_plan(uint64_t* host, int n) {
  if (n > kMaxGrid * 32) n = kMaxGrid * 32;
  return cudaMemcpyFromSymbol(host, g_plan_trace, sizeof(uint64_t) * n) == cudaSuccess ? 0 : -9;
}
#endif

// Plan of a batch of short or medium rows (max_len <= kMediumMaxLen: the register path,
// one warp per row, or the medium path, one CTA per row), or of a few long rows (the
// cluster path, one thread-block cluster per row); no work list: the header alone,
// which the select kernels check, with the medium path's row tickets at 0.
__global__ void short_plan_kernel(int rows, int max_len, int grid, char* ws) {
  if (threadIdx.x != 0) return;
  Header* h = reinterpret_cast<Header*>(ws);
  h->magic = kMagic;
  h->rows = rows;
  h->max_len = max_len;
  h->grid = grid;
  h->chunk = 0;
  h->waves = 0;
  h->n_single = rows;
  h->n_multi = 0;
  h->status = 0;
  h->plan_error = 0;
  h->n_implicit = 0;
  h->dyn_period = 0;
  h->steal = 0ull;
  h->med_ticket = 0ull;
  for (int i = 0; i < 8; ++i) h->diag[i] = 0;
}

cudaError_t launch_plan(const int32_t* lens, int rows, int max_len, int grid, int chunk_force,
                        void* ws, cudaStream_t stream) {
  if ((max_len <= kMediumMaxLen || cluster_batch(rows, max_len, grid)) && chunk_force == 0) {
    short_plan_kernel<<<1, 32, 0, stream>>>(rows, max_len, grid, static_cast<char*>(ws));
    return cudaGetLastError();
  }
  const Layout lay = make_layout(rows);
  const size_t n16 = offsetof(GroupState, cand_key) / 16 * (size_t)lay.ngroups;
  const size_t per_block = (size_t)kPlanThreads * kZeroPerThread;
  int zero_blocks = (int)((n16 + per_block - 1) / per_block);
  if (zero_blocks < 1) zero_blocks = 1;
  if (zero_blocks > 512) zero_blocks = 512;
  plan_kernel<<<1 + zero_blocks, kPlanThreads, 0, stream>>>(lens, rows, max_len, grid,
                                                            chunk_force, static_cast<char*>(ws));
  return cudaGetLastError();
}

// Host reference of the same plan (sequential). Fills a workspace image in host
// memory (header, row info, singles, first-single table, unit table; group state is
// left untouched).
int plan_host(const int32_t* lens, int rows, int max_len, int grid, int chunk_force, char* ws) {
  const Layout lay = make_layout(rows);
  Header* h = reinterpret_cast<Header*>(ws + lay.header);
  if ((max_len <= kMediumMaxLen || cluster_batch(rows, max_len, grid)) && chunk_force == 0) {
    // register, medium or cluster path: header only
    *h = Header{};
    h->magic = kMagic;
    h->rows = rows;
    h->max_len = max_len;
    h->grid = grid;
    h->n_single = rows;
    return 0;
  }
  RowInfo* ri = reinterpret_cast<RowInfo*>(ws + lay.rowinfo);
  int2* singles = reinterpret_cast<int2*>(ws + lay.singles);
  int32_t* first_single = reinterpret_cast<int32_t*>(ws + lay.first_single);
  UnitDesc* units = reinterpret_cast<UnitDesc*>(ws + lay.units);

  long long total = 0;
  for (int r = 0; r < rows; ++r) total += valid_len(lens[r], max_len);
  const bool forced = chunk_force > 0;
  auto slots_at = [&](int c) {
    long long n = 0;
    for (int r = 0; r < rows; ++r) {
      const int G = row_groups(valid_len(lens[r], max_len), c);
      if (G > 1) n += G;
    }
    return n;
  };
  int c = initial_chunk(total, grid, chunk_force);
  const bool fits = !forced && auto_chunk_ref(c, grid, slots_at, &c);
  int waves = 0, plan_error = 0, n_multi = 0;
  static thread_local int32_t mr[kMaxGroups], mg[kMaxGroups], mw[kMaxGroups], mc[kMaxGroups];
  if (fits) {
    int cta = 0;
    for (int r = 0; r < rows; ++r) {
      const int G = row_groups(valid_len(lens[r], max_len), c);
      if (G > 1) {
        mr[n_multi] = r;
        mg[n_multi] = G;
        mw[n_multi] = 0;
        mc[n_multi] = cta;
        cta += G;
        ++n_multi;
      }
    }
    waves = n_multi > 0 ? 1 : 0;
  } else {
    PlanStats st{0, 0, 0};
    for (int iter = 0; iter < 64; ++iter) {
      st = PlanStats{0, 0, 0};
      for (int r = 0; r < rows; ++r) {
        const int G = row_groups(valid_len(lens[r], max_len), c);
        if (G > 1) {
          st.slots += G;
          st.n_multi += 1;
          if (G > st.max_g) st.max_g = G;
        }
      }
      if (st.n_multi <= lay.ngroups && st.max_g <= grid) {
        int n = 0;
        for (int r = 0; r < rows; ++r) {
          const int G = row_groups(valid_len(lens[r], max_len), c);
          if (G > 1) {
            mr[n] = r;
            mg[n] = G;
            ++n;
          }
        }
        waves = pack_waves(mg, n, grid, mw, mc);
      } else {
        waves = kMaxWaves + 1;
      }
      const int nc = next_chunk(c, st, waves, grid, forced, lay.ngroups);
      if (nc == c) break;
      if (nc < 0) {
        plan_error = 1;
        break;
      }
      c = nc;
    }
    n_multi = plan_error ? 0 : st.n_multi;
  }
  const int wv = plan_error ? 0 : waves;
  for (int i = 0; i < wv * kMaxGrid; ++i) units[i] = UnitDesc{-1, 0, 0, 0, 0, 0, 0, 0};
  static thread_local uint8_t busy[kMaxGrid];
  for (int i = 0; i < kMaxGrid; ++i) busy[i] = 0;
  for (int i = 0; i < n_multi; ++i) {
    const int L = valid_len(lens[mr[i]], max_len);
    for (int j = 0; j < mg[i]; ++j) {
      units[(int64_t)mw[i] * kMaxGrid + mc[i] + j] = make_unit(mr[i], L, j, mg[i], i);
      busy[mc[i] + j] = 1;
    }
  }
  for (int r = 0; r < rows; ++r) {
    const int L = valid_len(lens[r], max_len);
    ri[r].len = lens[r];
    ri[r].G = plan_error ? 1 : row_groups(L, c);
    ri[r].group = -1;
    ri[r].pad = 0;
  }
  for (int i = 0; i < n_multi; ++i) ri[mr[i]].group = i;
  int n_single = 0;
  for (int b = 31; b >= 0; --b)
    for (int r = 0; r < rows; ++r) {
      const int L = valid_len(lens[r], max_len);
      if ((plan_error || row_groups(L, c) == 1) && len_bucket(L) == b) {
        singles[n_single].x = r;
        singles[n_single].y = lens[r];
        ++n_single;
      }
    }
  int ord = 0;
  for (int cta = 0; cta < kMaxGrid; ++cta) {
    const bool free_cta = cta < grid && !busy[cta];
    first_single[cta] = (free_cta && ord < n_single) ? ord : -1;
    if (free_cta) ++ord;
  }
  const int n_implicit = ord < n_single ? ord : n_single;
  h->magic = kMagic;
  h->rows = rows;
  h->max_len = max_len;
  h->grid = grid;
  h->chunk = c;
  h->waves = wv;
  h->n_single = n_single;
  h->n_multi = n_multi;
  h->status = plan_error ? TOPK_STATUS_PLAN_MISMATCH : 0;
  h->plan_error = plan_error;
  h->n_implicit = n_implicit;
  h->dyn_period = n_single - n_implicit + grid;
  h->steal = 0ull;
  h->med_ticket = 0ull;
  for (int i = 0; i < 8; ++i) h->diag[i] = 0;
  return plan_error;
}

}  // namespace topk
