// Planning kernel: bins the batch's rows into single-CTA and multi-CTA paths and
// builds the persistent grid's work list ("Serving GLM5.2 NVFP4 Agentic Workload
// with SGLang", "Kernel Optimization > TopK-V2": the planning kernel chooses the
// cluster cutoff from the sequence-length distribution and builds the work list).
//
// Block 0 plans; the other blocks clear the per-row group state so the select
// kernel's counters start at zero. Reads only device-resident lengths: no host sync.
#include <cuda_runtime.h>

#include "common.cuh"
#include "plan_logic.cuh"

namespace topk {

namespace {

constexpr int kPlanThreads = 1024;

struct PlanSmem {
  long long red64[kPlanThreads / 32];
  int red[3][kPlanThreads / 32];
  int bcast[8];
  int multi_rows[kMaxGroups];
  int multi_g[kMaxGroups];
  unsigned bucket_mask;
};

__device__ long long block_sum64(long long v, PlanSmem& s) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if (lane == 0) s.red64[w] = v;
  __syncthreads();
  long long t = 0;
  for (int i = 0; i < kPlanThreads / 32; ++i) t += s.red64[i];
  __syncthreads();
  return t;
}

// Returns (sum a, sum b, max c) over the block.
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
  for (int i = 0; i < kPlanThreads / 32; ++i) {
    ta += s.red64[i];
    tb += s.red[0][i];
    tc = max(tc, s.red[1][i]);
  }
  __syncthreads();
  a = ta;
  b = tb;
  c = tc;
}

// Exclusive scan of one int per thread; returns the block total in *total.
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
  for (int i = 0; i < kPlanThreads / 32; ++i) {
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
  int32_t* singles = reinterpret_cast<int32_t*>(ws + lay.singles);
  int32_t* units = reinterpret_cast<int32_t*>(ws + lay.units);

  if (blockIdx.x > 0) {
    // Clear every group state (the select kernel's counters and histograms).
    uint4* g = reinterpret_cast<uint4*>(ws + lay.groups);
    const size_t n16 = sizeof(GroupState) * (size_t)lay.ngroups / 16;
    const uint4 z = make_uint4(0, 0, 0, 0);
    for (size_t i = (size_t)(blockIdx.x - 1) * blockDim.x + threadIdx.x; i < n16;
         i += (size_t)(gridDim.x - 1) * blockDim.x)
      g[i] = z;
    return;
  }

  __shared__ PlanSmem s;
  const int tid = threadIdx.x;

  // Total valid length.
  long long part = 0;
  for (int r = tid; r < rows; r += kPlanThreads) part += valid_len(lens[r], max_len);
  const long long total = block_sum64(part, s);

  const bool forced = chunk_force > 0;
  int c = initial_chunk(total, grid, chunk_force);
  int waves = 0, plan_error = 0;
  PlanStats st{0, 0, 0};
  for (int iter = 0; iter < 64; ++iter) {
    long long slots = 0;
    int nm = 0, mg = 0;
    for (int r = tid; r < rows; r += kPlanThreads) {
      const int G = row_groups(valid_len(lens[r], max_len), c);
      if (G > 1) {
        slots += G;
        nm += 1;
        mg = max(mg, G);
      }
    }
    block_stats(slots, nm, mg, s);
    st = PlanStats{slots, nm, mg};
    // Multi-CTA rows in row order (only when they fit the group-state table).
    if (nm <= kMaxGroups && mg <= grid) {
      int base = 0;
      for (int r0 = 0; r0 < rows; r0 += kPlanThreads) {
        const int r = r0 + tid;
        const int G = r < rows ? row_groups(valid_len(lens[r], max_len), c) : 1;
        int tot;
        const int off = block_scan(G > 1 ? 1 : 0, &tot, s);
        if (G > 1) {
          s.multi_rows[base + off] = r;
          s.multi_g[base + off] = G;
        }
        base += tot;
      }
      __syncthreads();
      if (tid == 0) s.bcast[0] = pack_waves(s.multi_rows, s.multi_g, nm, grid, nullptr);
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

  // Unit table: clear the used waves, then pack.
  const int wv = plan_error ? 0 : waves;
  for (int i = tid; i < wv * kMaxGrid; i += kPlanThreads) units[i] = -1;
  __syncthreads();
  if (tid == 0 && !plan_error) pack_waves(s.multi_rows, s.multi_g, st.n_multi, grid, units);

  // Row info.
  for (int r = tid; r < rows; r += kPlanThreads) {
    const int L = valid_len(lens[r], max_len);
    const int G = plan_error ? 1 : row_groups(L, c);
    RowInfo x;
    x.len = lens[r];
    x.G = G;
    x.group = -1;
    x.pad = 0;
    ri[r] = x;
  }
  __syncthreads();
  if (!plan_error)
    for (int i = tid; i < st.n_multi; i += kPlanThreads) ri[s.multi_rows[i]].group = i;

  // Single-CTA rows, longest bucket first, row order inside a bucket.
  if (tid == 0) s.bucket_mask = 0u;
  __syncthreads();
  for (int r = tid; r < rows; r += kPlanThreads) {
    const int L = valid_len(lens[r], max_len);
    if (plan_error || row_groups(L, c) == 1) atomicOr(&s.bucket_mask, 1u << len_bucket(L));
  }
  __syncthreads();
  const unsigned mask = s.bucket_mask;
  int base = 0;
  for (int b = 31; b >= 0; --b) {
    if (!(mask & (1u << b))) continue;
    for (int r0 = 0; r0 < rows; r0 += kPlanThreads) {
      const int r = r0 + tid;
      bool take = false;
      if (r < rows) {
        const int L = valid_len(lens[r], max_len);
        take = (plan_error || row_groups(L, c) == 1) && len_bucket(L) == b;
      }
      int tot;
      const int off = block_scan(take ? 1 : 0, &tot, s);
      if (take) singles[base + off] = r;
      base += tot;
    }
  }

  if (tid == 0) {
    h->magic = kMagic;
    h->rows = rows;
    h->max_len = max_len;
    h->grid = grid;
    h->chunk = c;
    h->waves = wv;
    h->n_single = base;
    h->n_multi = plan_error ? 0 : st.n_multi;
    h->status = plan_error ? TOPK_STATUS_PLAN_MISMATCH : 0;
    h->plan_error = plan_error;
    h->steal = 0ull;
  }
}

}  // namespace

cudaError_t launch_plan(const int32_t* lens, int rows, int max_len, int grid, int chunk_force,
                        void* ws, cudaStream_t stream) {
  const Layout lay = make_layout(rows);
  const size_t bytes = sizeof(GroupState) * (size_t)lay.ngroups;
  int zero_blocks = (int)((bytes / 16 + kPlanThreads * 8 - 1) / (kPlanThreads * 8));
  if (zero_blocks < 1) zero_blocks = 1;
  if (zero_blocks > 256) zero_blocks = 256;
  plan_kernel<<<1 + zero_blocks, kPlanThreads, 0, stream>>>(lens, rows, max_len, grid,
                                                            chunk_force, static_cast<char*>(ws));
  return cudaGetLastError();
}

// Host reference of the same plan (sequential). Fills a workspace image in host
// memory (header, row info, singles, unit table; group state is left untouched).
int plan_host(const int32_t* lens, int rows, int max_len, int grid, int chunk_force, char* ws) {
  const Layout lay = make_layout(rows);
  Header* h = reinterpret_cast<Header*>(ws + lay.header);
  RowInfo* ri = reinterpret_cast<RowInfo*>(ws + lay.rowinfo);
  int32_t* singles = reinterpret_cast<int32_t*>(ws + lay.singles);
  int32_t* units = reinterpret_cast<int32_t*>(ws + lay.units);

  long long total = 0;
  for (int r = 0; r < rows; ++r) total += valid_len(lens[r], max_len);
  const bool forced = chunk_force > 0;
  int c = initial_chunk(total, grid, chunk_force);
  int waves = 0, plan_error = 0;
  static thread_local int32_t mr[kMaxGroups], mgs[kMaxGroups];
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
    if (st.n_multi <= kMaxGroups && st.max_g <= grid) {
      int n = 0;
      for (int r = 0; r < rows; ++r) {
        const int G = row_groups(valid_len(lens[r], max_len), c);
        if (G > 1) {
          mr[n] = r;
          mgs[n] = G;
          ++n;
        }
      }
      waves = pack_waves(mr, mgs, n, grid, nullptr);
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
  for (int i = 0; i < wv * kMaxGrid; ++i) units[i] = -1;
  if (!plan_error) pack_waves(mr, mgs, st.n_multi, grid, units);
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
      if ((plan_error || row_groups(L, c) == 1) && len_bucket(L) == b) singles[n_single++] = r;
    }
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
  h->steal = 0ull;
  return plan_error;
}

}  // namespace topk
