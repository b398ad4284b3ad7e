// Register-resident select + page-table kernel for batches of short rows (GB300,
// sm_103a).
//
// "Serving GLM5.2 NVFP4 Agentic Workload with SGLang", "Kernel Optimization > TopK-V2":
// short rows take a register-resident path, medium rows a single-CTA streaming path
// and long rows a multi-CTA path. Here a batch whose rows are all at most kShortMax
// values long (the host knows max_len at launch) runs one warp per row: lane l holds
// positions l, l + 32, ... of its row in registers, and the exact top k comes from a
// most-significant-bit-first radix selection over a 40-bit composite key (the
// order-preserving 32-bit score key, then the inverted 8-bit position, so that equal
// scores rank by the smaller position), one warp-wide ballot count per bit. Selected
// positions are translated to slots and written in position order.
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"
#include "keys.cuh"

namespace topk {

namespace {

constexpr int kShortWarps = 8;  // rows per CTA

__device__ __forceinline__ int32_t short_slot(const SelectParams& P, Header* h, int t, int p) {
  const int32_t page = __ldg(P.table + (int64_t)t * P.table_ld + p / P.page_size);
  const int64_t sl = (int64_t)page * P.page_size + p % P.page_size;
  if (page < 0) {
    atomicOr(&h->status, TOPK_STATUS_TABLE_ENTRY);
    return -1;
  }
  if (sl > 0x7FFFFFFFll) {
    atomicOr(&h->status, TOPK_STATUS_SLOT_OVERFLOW);
    return -1;
  }
  return (int32_t)sl;
}

// PER values per lane: rows of at most 32 * PER values.
template <int PER>
__global__ void __launch_bounds__(kShortWarps * 32) short_kernel(const __grid_constant__ SelectParams P) {
  __shared__ int hdr_ok;
  Header* h = reinterpret_cast<Header*>(P.ws);
  if (threadIdx.x == 0) {
    const int4 h0 = __ldcg(reinterpret_cast<const int4*>(h));
    const int plan_error = __ldcg(&h->plan_error);
    hdr_ok = ((uint32_t)h0.x == kMagic && h0.y == P.rows && h0.z == P.max_len && plan_error == 0)
                 ? 1
                 : 0;
  }
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int r = (int)blockIdx.x * kShortWarps + (int)(threadIdx.x >> 5);
  if (r >= P.rows) return;
  int32_t* os = P.out_slots + (int64_t)r * P.k;
  int32_t* op = P.out_pos ? P.out_pos + (int64_t)r * P.k : nullptr;
  const int L = P.lens[r];
  int err = 0;
  if (!hdr_ok) err = TOPK_STATUS_PLAN_MISMATCH;
  else if (L < 0 || L > P.max_len) err = TOPK_STATUS_LEN;
  else if (ceil_div64(L, P.page_size) > P.table_ld) err = TOPK_STATUS_TABLE_WIDTH;
  const int kr = err ? 0 : min(P.k, L);
  if (err && lane == 0) atomicOr(&h->status, err);
  for (int i = kr + lane; i < P.k; i += 32) {  // -1 padding (the whole row on an error)
    os[i] = -1;
    if (op) op[i] = -1;
  }
  if (kr == 0) return;
  const int t = P.row_to_table ? P.row_to_table[r] : r;

  // Load: component i of lane l is position l + 32 i (coalesced).
  const float* row = P.scores + (int64_t)r * P.ld;
  uint64_t key[PER];
  uint32_t valid = 0u;
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int p = lane + 32 * i;
    key[i] = 0ull;
    if (p < L) {
      key[i] = ((uint64_t)f2key(__ldg(row + p)) << 8) | (uint64_t)(255 - p);
      valid |= 1u << i;
    }
  }
  uint32_t sel = 0u;
  if (L <= P.k) {
    sel = valid;  // every position is taken
  } else {
    // Radix selection from the highest bit where the candidates differ: at each bit,
    // if at least `need` candidates have it set, the others drop out; otherwise all
    // of those are selected and the rest stay candidates for what is still needed.
    uint32_t cand = valid;
    int need = P.k;
    uint32_t an_hi = 0xFFFFFFFFu, an_lo = 0xFFFFFFFFu, or_hi = 0u, or_lo = 0u;
#pragma unroll
    for (int i = 0; i < PER; ++i)
      if ((cand >> i) & 1u) {
        an_hi &= (uint32_t)(key[i] >> 32);
        an_lo &= (uint32_t)key[i];
        or_hi |= (uint32_t)(key[i] >> 32);
        or_lo |= (uint32_t)key[i];
      }
    an_hi = __reduce_and_sync(0xffffffffu, an_hi);
    an_lo = __reduce_and_sync(0xffffffffu, an_lo);
    or_hi = __reduce_or_sync(0xffffffffu, or_hi);
    or_lo = __reduce_or_sync(0xffffffffu, or_lo);
    const uint64_t diff = ((uint64_t)(an_hi ^ or_hi) << 32) | (uint64_t)(an_lo ^ or_lo);
    // composite keys are unique (distinct positions), so some bit differs
    for (int bit = 63 - __clzll((long long)diff); bit >= 0 && need > 0; --bit) {
      uint32_t m1 = 0u;
#pragma unroll
      for (int i = 0; i < PER; ++i) m1 |= (uint32_t)((key[i] >> bit) & 1ull) << i;
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
    if (need > 0) sel |= cand;  // the last remaining candidate (unique keys)
  }

  // Emit in position order: component i of every lane comes before component i + 1.
  const unsigned lt = (1u << lane) - 1u;
  int base = 0;
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const bool s = (sel >> i) & 1u;
    const unsigned b = __ballot_sync(0xffffffffu, s);
    if (s) {
      const int p = lane + 32 * i;
      const int idx = base + __popc(b & lt);
      os[idx] = short_slot(P, h, t, p);
      if (op) op[idx] = p;
    }
    base += __popc(b);
  }
}

}  // namespace

static_assert(kShortMaxLen == 32 * 8, "rows of the register path fit 8 values per lane");

// Largest max_len the register path takes.
int short_max_len() { return kShortMaxLen; }

cudaError_t launch_short(const SelectParams& p, cudaStream_t stream) {
  const int blocks = (p.rows + kShortWarps - 1) / kShortWarps;
  if (p.max_len <= 64)
    short_kernel<2><<<blocks, kShortWarps * 32, 0, stream>>>(p);
  else
    short_kernel<8><<<blocks, kShortWarps * 32, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace topk
