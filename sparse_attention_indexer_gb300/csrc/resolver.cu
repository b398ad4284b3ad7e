// Fused top-K resolver with per-request LRU hot buffers ("GLM 5.3 Optimizations,
// Part 1: Hybrid HiSparse Offloading in vLLM", section "How it works"); the readings of
// the policy are stated in include/hisparse_resolver.h.
//
// One CTA per request. Its threads classify the selected positions (resident, hit with
// the slot's step refreshed, miss); a block scan ranks the misses in output order;
// when there are any, the CTA sorts the (last step, slot) keys of the slots unused at
// this step in shared memory (bitonic sort, at most 4096 keys), hands miss r victim r,
// updates the two maps, and copies the missed rows from pinned host memory (read
// directly by the kernel, 16 bytes per thread per chunk) into the victims' KV rows.
#include <cuda_runtime.h>

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
};

struct Smem {
  uint64_t keys[kMaxHot];     // victim order: (hot_step + 1) << 32 | slot, kNone excluded
  int32_t miss_entry[kMaxK];  // entry index of the miss of each rank
  uint8_t is_miss[kMaxK];
  int64_t copy_src[kMaxK];    // host row of each assigned miss (by rank), -1 none
  int32_t copy_dst[kMaxK];    // KV row
  int32_t wsum[kThreads / 32];
  int32_t red[4][kThreads / 32];
};

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

__global__ void __launch_bounds__(kThreads) resolve_kernel(Params p) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  Smem& s = *reinterpret_cast<Smem*>(smem_raw);
  const int j = blockIdx.x;
  const int32_t* pos = p.positions + (int64_t)j * p.k;
  int32_t* out = p.out + (int64_t)j * p.k;
  const int32_t* tab = p.table + (int64_t)j * p.table_ld;
  int32_t* t2h = p.t2h + (int64_t)j * p.map_ld;
  int32_t* htok = p.hot_token + (int64_t)j * p.hot;
  int32_t* hstep = p.hot_step + (int64_t)j * p.hot;
  const int32_t* hrows = p.hot_rows + (int64_t)j * p.hot;
  int err = 0, n_res = 0, n_hit = 0;

  // 1. classify; hits refresh their slot (distinct positions -> distinct slots)
  for (int i = threadIdx.x; i < p.k; i += kThreads) {
    const int q = pos[i];
    uint8_t miss = 0;
    int row = -1;
    if (q >= 0) {
      const int pg = q / p.page_size;
      if ((int64_t)pg >= p.table_ld || (int64_t)q >= p.map_ld) {
        err |= RESOLVER_STATUS_POSITION;
      } else {
        const int32_t b = tab[pg];
        if (b >= 0) {
          row = (int)((int64_t)b * p.page_size + (q - pg * p.page_size));
          ++n_res;
        } else {
          const int32_t h = t2h[q];
          if (h >= 0 && h < p.hot) {
            row = hrows[h];
            hstep[h] = p.step;
            ++n_hit;
          } else {
            miss = 1;
          }
        }
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
    // 3. victim order: slots unused at this step by (last step, slot), padded to 2^n
    int n = 1;
    while (n < p.hot) n <<= 1;
    for (int h = threadIdx.x; h < n; h += kThreads) {
      uint64_t key = kNone;
      if (h < p.hot) {
        const int st = hstep[h];  // hits of this step are written above (same block)
        if (st < p.step) key = ((uint64_t)(uint32_t)(st + 1) << 32) | (uint32_t)h;
      }
      s.keys[h] = key;
    }
    __syncthreads();
    for (int k2 = 2; k2 <= n; k2 <<= 1) {
      for (int j2 = k2 >> 1; j2 > 0; j2 >>= 1) {
        for (int i = threadIdx.x; i < n; i += kThreads) {
          const int ixj = i ^ j2;
          if (ixj > i) {
            const uint64_t a = s.keys[i], b = s.keys[ixj];
            const bool up = (i & k2) == 0;
            if ((a > b) == up) {
              s.keys[i] = b;
              s.keys[ixj] = a;
            }
          }
        }
        __syncthreads();
      }
    }

    // 4. miss rank r takes victim r: maps, step, output row, the copy to make
    const int64_t hb = p.host_base[j];
    for (int rr = threadIdx.x; rr < m; rr += kThreads) {
      const int i = s.miss_entry[rr];
      const int q = pos[i];
      s.copy_src[rr] = -1;
      s.copy_dst[rr] = -1;
      const uint64_t key = rr < n ? s.keys[rr] : kNone;
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

    // 5. copies: (miss, 16-byte chunk) pairs spread over the block
    const int chunks = p.row_bytes >> 4;
    const int64_t total = (int64_t)m * chunks;
    for (int64_t c = threadIdx.x; c < total; c += kThreads) {
      const int rr = (int)(c / chunks), q = (int)(c - (int64_t)rr * chunks);
      const int64_t src = s.copy_src[rr];
      if (src < 0) continue;
      const uint4 v = *reinterpret_cast<const uint4*>(p.host + src * p.row_bytes + 16 * q);
      *reinterpret_cast<uint4*>(p.kv + (int64_t)s.copy_dst[rr] * p.row_bytes + 16 * q) = v;
    }
  }

  // 6. counts and status (misses copied = assigned copies)
  if (p.counts || p.status) {
    int n_copy = 0;
    for (int rr = threadIdx.x; rr < m; rr += kThreads) n_copy += s.copy_src[rr] >= 0 ? 1 : 0;
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

}  // namespace

extern "C" int hisparse_resolve(const int32_t* positions, int rows, int k,
                                const int32_t* block_table, int64_t table_ld, int page_size,
                                int32_t* token_to_hot, int64_t map_ld, int32_t* hot_token,
                                int32_t* hot_step, const int32_t* hot_rows, int hot_size, int step,
                                const uint8_t* host_kv, const int64_t* host_base,
                                int64_t host_rows, uint8_t* kv, int64_t kv_rows, int row_bytes,
                                int32_t* out_rows, int32_t* counts, int32_t* status,
                                resolver_stream_t stream) {
  if (rows < 0 || k < 1 || k > kMaxK || hot_size < 1 || hot_size > kMaxHot || page_size < 1 ||
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
    if (cudaFuncSetAttribute(resolve_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)sizeof(Smem)) != cudaSuccess)
      return RESOLVER_ERR_CUDA;
    attr_set = true;
  }
  Params p{positions, rows,     k,        block_table, table_ld,  page_size, token_to_hot,
           map_ld,    hot_token, hot_step, hot_rows,    hot_size,  step,      host_kv,
           host_base, host_rows, kv,       kv_rows,     row_bytes, out_rows,  counts,
           status};
  resolve_kernel<<<rows, kThreads, sizeof(Smem), (cudaStream_t)stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? RESOLVER_OK : RESOLVER_ERR_CUDA;
}
