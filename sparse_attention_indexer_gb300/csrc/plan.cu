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

#include "common.cuh"
#include "plan_logic.cuh"

namespace topk {

namespace {

#ifdef TOPK_TRACE
__device__ uint64_t g_plan_trace[kMaxGrid * 32];
#endif

constexpr int kPlanThreads = 256;
constexpr int kPlanWarps = kPlanThreads / 32;
constexpr int kLensCache = 4096;  // batches up to this many rows plan from shared memory

struct PlanSmem {
  long long red64[kPlanWarps];
  int red[3][kPlanWarps];
  int bcast[8];
  int32_t multi_rows[kMaxGroups];
  int32_t multi_g[kMaxGroups];
  int32_t multi_wave[kMaxGroups];
  int32_t multi_cta[kMaxGroups];
  uint32_t busy[kMaxGrid / 32];  // CTAs with static units
  unsigned bucket_mask;
  int32_t lens[kLensCache];
};

__device__ void block_stats(long long& a, int& b, int& c, PlanSmem& s) {
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

// Exclusive scan of one int per thread; the block total goes to *total.
__device__ int block_scan(int v, int* total, PlanSmem& s) {
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
    // Clear every group state (the select kernel's counters and histograms).
    uint4* g = reinterpret_cast<uint4*>(ws + lay.groups);
    const size_t n16 = sizeof(GroupState) * (size_t)lay.ngroups / 16;
    const uint4 z = make_uint4(0, 0, 0, 0);
    for (size_t i = (size_t)(blockIdx.x - 1) * blockDim.x + threadIdx.x; i < n16;
         i += (size_t)(gridDim.x - 1) * blockDim.x)
      g[i] = z;
    TOPK_MARK(g_plan_trace, 9);
    return;
  }

  __shared__ PlanSmem s;
  const int tid = threadIdx.x;

  // Lengths are read many times below: keep them in shared memory when they fit.
  const bool cached = rows <= kLensCache;
  if (cached)
    for (int r = tid; r < rows; r += kPlanThreads) s.lens[r] = lens[r];
  __syncthreads();
  const int32_t* L_ = cached ? s.lens : lens;

  long long total = 0;
  int dummy_b = 0, dummy_c = 0;
  for (int r = tid; r < rows; r += kPlanThreads) total += valid_len(L_[r], max_len);
  block_stats(total, dummy_b, dummy_c, s);
  TOPK_MARK(g_plan_trace, 1);

  const bool forced = chunk_force > 0;
  int c = initial_chunk(total, grid, chunk_force);
  int waves = 0, plan_error = 0;
  PlanStats st{0, 0, 0};
  for (int iter = 0; iter < 64; ++iter) {
    long long slots = 0;
    int nm = 0, mg = 0;
    for (int r = tid; r < rows; r += kPlanThreads) {
      const int G = row_groups(valid_len(L_[r], max_len), c);
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
        const int G = r < rows ? row_groups(valid_len(L_[r], max_len), c) : 1;
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
  TOPK_MARK(g_plan_trace, 2);

  // Static unit table: clear the used waves, then one descriptor per multi-CTA chunk.
  const int wv = plan_error ? 0 : waves;
  for (int i = tid; i < wv * kMaxGrid; i += kPlanThreads) units[i].row = -1;
  for (int i = tid; i < kMaxGrid / 32; i += kPlanThreads) s.busy[i] = 0u;
  __syncthreads();
  if (!plan_error) {
    for (int i = 0; i < st.n_multi; ++i) {
      const int G = s.multi_g[i];
      const int row = s.multi_rows[i];
      const int L = valid_len(L_[row], max_len);
      for (int j = tid; j < G; j += kPlanThreads) {
        const int cta = s.multi_cta[i] + j;
        units[(int64_t)s.multi_wave[i] * kMaxGrid + cta] = make_unit(row, L, j, G, i);
        atomicOr(&s.busy[cta >> 5], 1u << (cta & 31));
      }
    }
  }
  TOPK_MARK(g_plan_trace, 3);

  // Row info.
  for (int r = tid; r < rows; r += kPlanThreads) {
    const int L = valid_len(L_[r], max_len);
    RowInfo x;
    x.len = L_[r];
    x.G = plan_error ? 1 : row_groups(L, c);
    x.group = -1;
    x.pad = 0;
    ri[r] = x;
  }
  __syncthreads();
  if (!plan_error)
    for (int i = tid; i < st.n_multi; i += kPlanThreads) ri[s.multi_rows[i]].group = i;
  TOPK_MARK(g_plan_trace, 4);

  // Single-CTA rows, longest bucket first, row order inside a bucket.
  if (tid == 0) s.bucket_mask = 0u;
  __syncthreads();
  for (int r = tid; r < rows; r += kPlanThreads) {
    const int L = valid_len(L_[r], max_len);
    if (plan_error || row_groups(L, c) == 1) atomicOr(&s.bucket_mask, 1u << len_bucket(L));
  }
  __syncthreads();
  const unsigned mask = s.bucket_mask;
  int n_single = 0;
  for (int b = 31; b >= 0; --b) {
    if (!(mask & (1u << b))) continue;
    for (int r0 = 0; r0 < rows; r0 += kPlanThreads) {
      const int r = r0 + tid;
      bool take = false;
      int Lraw = 0;
      if (r < rows) {
        Lraw = L_[r];
        const int L = valid_len(Lraw, max_len);
        take = (plan_error || row_groups(L, c) == 1) && len_bucket(L) == b;
      }
      int tot;
      const int off = block_scan(take ? 1 : 0, &tot, s);
      if (take) singles[n_single + off] = make_int2(r, Lraw);
      n_single += tot;
    }
  }

  // One single row per CTA without static units, in CTA order.
  int ordinal_base = 0;
  for (int c0 = 0; c0 < grid; c0 += kPlanThreads) {
    const int cta = c0 + tid;
    const bool free_cta = cta < grid && !((s.busy[cta >> 5] >> (cta & 31)) & 1u);
    int tot;
    const int ord = ordinal_base + block_scan(free_cta ? 1 : 0, &tot, s);
    if (cta < kMaxGrid) first_single[cta] = (free_cta && ord < n_single) ? ord : -1;
    ordinal_base += tot;
  }
  const int n_implicit = min(ordinal_base, n_single);

  if (tid == 0) {
    h->magic = kMagic;
    h->rows = rows;
    h->max_len = max_len;
    h->grid = grid;
    h->chunk = c;
    h->waves = wv;
    h->n_single = n_single;
    h->n_multi = plan_error ? 0 : st.n_multi;
    h->status = plan_error ? TOPK_STATUS_PLAN_MISMATCH : 0;
    h->plan_error = plan_error;
    h->n_implicit = n_implicit;
    h->dyn_period = n_single - n_implicit + grid;
    h->steal = 0ull;
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

cudaError_t launch_plan(const int32_t* lens, int rows, int max_len, int grid, int chunk_force,
                        void* ws, cudaStream_t stream) {
  const Layout lay = make_layout(rows);
  const size_t bytes = sizeof(GroupState) * (size_t)lay.ngroups;
  int zero_blocks = (int)((bytes / 16 + kPlanThreads * 16 - 1) / (kPlanThreads * 16));
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
  RowInfo* ri = reinterpret_cast<RowInfo*>(ws + lay.rowinfo);
  int2* singles = reinterpret_cast<int2*>(ws + lay.singles);
  int32_t* first_single = reinterpret_cast<int32_t*>(ws + lay.first_single);
  UnitDesc* units = reinterpret_cast<UnitDesc*>(ws + lay.units);

  long long total = 0;
  for (int r = 0; r < rows; ++r) total += valid_len(lens[r], max_len);
  const bool forced = chunk_force > 0;
  int c = initial_chunk(total, grid, chunk_force);
  int waves = 0, plan_error = 0;
  static thread_local int32_t mr[kMaxGroups], mg[kMaxGroups], mw[kMaxGroups], mc[kMaxGroups];
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
  const int wv = plan_error ? 0 : waves;
  for (int i = 0; i < wv * kMaxGrid; ++i) units[i].row = -1;
  static thread_local uint8_t busy[kMaxGrid];
  for (int i = 0; i < kMaxGrid; ++i) busy[i] = 0;
  if (!plan_error)
    for (int i = 0; i < st.n_multi; ++i) {
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
  if (!plan_error)
    for (int i = 0; i < st.n_multi; ++i) ri[mr[i]].group = i;
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
  h->n_multi = plan_error ? 0 : st.n_multi;
  h->status = plan_error ? TOPK_STATUS_PLAN_MISMATCH : 0;
  h->plan_error = plan_error;
  h->n_implicit = n_implicit;
  h->dyn_period = n_single - n_implicit + grid;
  h->steal = 0ull;
  for (int i = 0; i < 8; ++i) h->diag[i] = 0;
  return plan_error;
}

}  // namespace topk
