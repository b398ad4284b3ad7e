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
// its static multi-CTA units (wave order), then claims single-CTA rows from a ticket
// counter. A unit's chunk of scores is brought into shared memory by bulk async
// copies (one mbarrier per 16 KB piece) and stays resident for every later pass.
//
// Multi-CTA rows combine their histograms in global memory and meet at bounded
// spin barriers (co-residency is guaranteed by the cooperative launch). The last CTA
// of a row to finish gathers the boundary candidates, finishes the exact selection
// and clears the row's counters for the next call.
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"

namespace topk {

namespace {

enum : uint8_t { kRej = 0, kActive = 1, kSel = 2 };

struct __align__(16) Smem {
  float buf[kBufFloats];
  uint32_t hist[kBins0];
  uint32_t lkey[kListCap];
  uint32_t lpos[kListCap];
  uint8_t lst[kListCap];
  uint32_t hist8[kListBins];
  uint64_t mbar[kPieces];
  int wsum[kWarps];
  int wsum2[kWarps];
  uint32_t wand[kWarps];
  uint32_t wor[kWarps];
  int bc[16];
};

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

// Coarse 12-bit digit, monotone non-decreasing in the key: sign, a 5-bit exponent
// window (|x| in [2^-15, 2^17)) and 6 mantissa bits, clamped at both ends. Integer
// only; equal scores (including +/-0) share a digit; NaN and -inf land in bin 0.
__device__ __forceinline__ uint32_t coarse_digit(float x) {
  const uint32_t u = __float_as_uint(x);
  const uint32_t a = u & 0x7FFFFFFFu;
  int m = (int)(a >> 17) - 7168;
  m = min(max(m, 0), 2047);
  const uint32_t d = ((u >> 31) && a) ? (uint32_t)(2047 - m) : (uint32_t)(2048 + m);
  return a > 0x7F800000u ? 0u : d;
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

__device__ __forceinline__ void set_status(Header* h, int bits) { atomicOr(&h->status, bits); }

// ------------------------------------------------------------- per-unit context

struct Unit {
  int r, rank, G, L, kr, t, s0, n, head, nvec;
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

// Group barrier among the G CTAs of a row. All threads call it. Returns false if
// the bounded wait expired (status set).
__device__ bool group_barrier(Ctx& c, Unit& u) {
  __threadfence();
  __syncthreads();
  u.bar_seq += 1;
  if (threadIdx.x == 0) {
    const uint32_t target = (uint32_t)u.G * u.bar_seq;
    atomicAdd(&u.gs->bar, 1u);
    bool ok = ld_acquire_u32(&u.gs->bar) >= target;
    if (!ok) {
      const uint64_t t0 = global_timer_ns();
      while (true) {
        if (ld_acquire_u32(&u.gs->bar) >= target) {
          ok = true;
          break;
        }
        if (global_timer_ns() - t0 > kWaitNs) break;
        __nanosleep(64);
      }
    }
    __threadfence();
    c.s.bc[15] = ok ? 1 : 0;
    if (!ok) set_status(c.h, TOPK_STATUS_TIMEOUT);
  }
  __syncthreads();
  return c.s.bc[15] != 0;
}

// Finds bin b of a 4096-bin histogram (owned 8 bins per thread, counts in v[])
// with above(b) < need <= above(b) + hist[b]; above(b) counts bins > b. Results
// land in s.bc[0..2] = (b, above, eq).
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

// Reduces the unit's local histogram in s.hist (4096 bins) with the row's other
// CTAs through `ghist` (when G > 1), then finds the threshold bin. Returns false on
// timeout. Outputs: b, above, eq (row-wide) and local_above, local_eq.
__device__ bool reduce_and_find(Ctx& c, Unit& u, uint32_t* ghist, int need, int& b, int& above,
                                int& eq, int& local_above, int& local_eq) {
  Smem& s = c.s;
  uint32_t loc[8], glob[8];
  const int b0 = threadIdx.x * 8;
  {
    const uint4 x = *reinterpret_cast<const uint4*>(&s.hist[b0]);
    const uint4 y = *reinterpret_cast<const uint4*>(&s.hist[b0 + 4]);
    loc[0] = x.x; loc[1] = x.y; loc[2] = x.z; loc[3] = x.w;
    loc[4] = y.x; loc[5] = y.y; loc[6] = y.z; loc[7] = y.w;
  }
  if (u.G > 1) {
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (loc[j]) red_add_u32(&ghist[b0 + j], loc[j]);
    if (!group_barrier(c, u)) return false;
    const uint4 x = __ldcg(reinterpret_cast<const uint4*>(&ghist[b0]));
    const uint4 y = __ldcg(reinterpret_cast<const uint4*>(&ghist[b0 + 4]));
    glob[0] = x.x; glob[1] = x.y; glob[2] = x.z; glob[3] = x.w;
    glob[4] = y.x; glob[5] = y.y; glob[6] = y.z; glob[7] = y.w;
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
  __syncthreads();
  local_above = block_sum(la, s);
  if (b >= b0 && b < b0 + 8) s.bc[3] = le;
  __syncthreads();
  local_eq = s.bc[3];
  __syncthreads();
  return true;
}

// ------------------------------------------------------------- chunk loading

// Issues the bulk copies of the unit's chunk (thread 0) and returns after every
// thread has built the coarse histogram of the chunk in s.hist.
__device__ void load_and_histogram(Ctx& c, Unit& u) {
  Smem& s = c.s;
  const SelectParams& P = c.p;
  const float* src = P.scores + (int64_t)u.r * P.ld + u.s0;
  const uintptr_t A = reinterpret_cast<uintptr_t>(src);
  const uintptr_t A0 = A & ~uintptr_t(15);
  const uintptr_t A1 = (A + 4ull * (uint64_t)u.n + 15ull) & ~uintptr_t(15);
  const uint32_t bytes = u.n > 0 ? (uint32_t)(A1 - A0) : 0u;
  u.head = (int)((A - A0) >> 2);
  u.nvec = (int)(bytes >> 4);
  const int npieces = (int)((bytes + kPieceBytes - 1) / kPieceBytes);

  // Previous generic-proxy accesses to buf are complete (caller synchronized).
  if (threadIdx.x == 0) {
    fence_proxy_async_smem();
    for (int i = 0; i < npieces; ++i) {
      const uint32_t off = (uint32_t)i * kPieceBytes;
      const uint32_t sz = min((uint32_t)kPieceBytes, bytes - off);
      mbar_arrive_expect_tx(&s.mbar[i], sz);
      bulk_g2s(reinterpret_cast<char*>(s.buf) + off, reinterpret_cast<const char*>(A0) + off, sz,
               &s.mbar[i]);
    }
  }
  for (int i = threadIdx.x; i < kBins0; i += kThreads) s.hist[i] = 0u;
  __syncthreads();

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const float4* b4 = reinterpret_cast<const float4*>(s.buf);
  constexpr int kVecPerPiece = kPieceBytes / 16;
  for (int i = 0; i < npieces; ++i) {
    const uint32_t par = (c.mphase >> i) & 1u;
    if (!mbar_wait_bounded(&s.mbar[i], par)) {
      if (threadIdx.x == 0) set_status(c.h, TOPK_STATUS_TIMEOUT);
      mbar_wait_bounded(&s.mbar[i], par);
    }
    c.mphase ^= (1u << i);
    const int vend = min((i + 1) * kVecPerPiece, u.nvec);
    for (int vb = i * kVecPerPiece + warp * 32; vb < vend; vb += kThreads) {
      const int v = vb + lane;
      const bool act = v < vend;
      float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
      if (act) x = b4[v];
      const int e0 = 4 * v - u.head;  // chunk index of x.x
      const bool full = act && e0 >= 0 && e0 + 3 < u.n;
      const uint32_t d0 = coarse_digit(x.x), d1 = coarse_digit(x.y);
      const uint32_t d2 = coarse_digit(x.z), d3 = coarse_digit(x.w);
      const bool uni = full && d0 == d1 && d1 == d2 && d2 == d3;
      const uint32_t dl = __shfl_sync(0xffffffffu, d0, 0);
      if (__all_sync(0xffffffffu, uni && d0 == dl)) {
        if (lane == 0) atomicAdd(&s.hist[d0], 128u);
      } else if (act) {
        if (full) {
          atomicAdd(&s.hist[d0], 1u);
          atomicAdd(&s.hist[d1], 1u);
          atomicAdd(&s.hist[d2], 1u);
          atomicAdd(&s.hist[d3], 1u);
        } else {
          if (e0 >= 0 && e0 < u.n) atomicAdd(&s.hist[d0], 1u);
          if (e0 + 1 >= 0 && e0 + 1 < u.n) atomicAdd(&s.hist[d1], 1u);
          if (e0 + 2 >= 0 && e0 + 2 < u.n) atomicAdd(&s.hist[d2], 1u);
          if (e0 + 3 >= 0 && e0 + 3 < u.n) atomicAdd(&s.hist[d3], 1u);
        }
      }
    }
  }
  __syncthreads();
}

// ------------------------------------------------------------- list selection

// Among list entries [0, n) (keys, positions, state bytes in shared memory) marks
// exactly `need` entries kSel: the largest keys, ties to the smaller position.
// Radix passes of 8 bits start at the highest bit where the active entries differ.
__device__ void list_select(Smem& s, const uint32_t* key, const uint32_t* pos, uint8_t* st,
                            int n, int need) {
  for (int i = threadIdx.x; i < n; i += kThreads) st[i] = kActive;
  __syncthreads();
  for (int phase = 0; phase < 2 && need > 0; ++phase) {
    // Value compared in this phase: the key, then the inverted position.
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

// Emits the kSel entries of a list at output indices base, base+1, ... (in list order).
__device__ void list_emit(Ctx& c, const Unit& u, const uint32_t* pos, const uint8_t* st, int n,
                          int base) {
  constexpr int kPer = (kGroupCap + kThreads - 1) / kThreads;  // 8 entries per thread
  const int i0 = threadIdx.x * kPer;
  int cnt = 0;
#pragma unroll
  for (int j = 0; j < kPer; ++j)
    if (i0 + j < n && st[i0 + j] == kSel) ++cnt;
  int total;
  int off = block_excl_scan(cnt, &total, c.s);
#pragma unroll
  for (int j = 0; j < kPer; ++j)
    if (i0 + j < n && st[i0 + j] == kSel) emit(c, u, base + off++, (int)pos[i0 + j]);
}

// ------------------------------------------------------------- the unit

__device__ void process_unit(Ctx& c, int r, int rank) {
  const SelectParams& P = c.p;
  Smem& s = c.s;
  const Layout lay = make_layout(P.rows);
  const RowInfo ri = reinterpret_cast<const RowInfo*>(P.ws + lay.rowinfo)[r];
  Unit u;
  u.r = r;
  u.rank = rank;
  u.G = ri.G;
  u.L = P.lens[r];
  u.bar_seq = 0;
  u.gs = ri.group >= 0 ? reinterpret_cast<GroupState*>(P.ws + lay.groups) + ri.group : nullptr;
  if (u.G > 1 && u.gs == nullptr) u.G = 1;  // defensive: never wait without state

  // Row-level checks: every CTA of the row takes the same decision.
  int err = 0;
  if (u.L != ri.len) err = TOPK_STATUS_PLAN_MISMATCH;
  else if (u.L < 0 || u.L > P.max_len) err = TOPK_STATUS_LEN;
  else if (ceil_div64(u.L, P.page_size) > P.table_ld) err = TOPK_STATUS_TABLE_WIDTH;
  if (err) {
    if (rank == 0) {
      if (threadIdx.x == 0) set_status(c.h, err);
      fill_row(c, r, 0, P.k);
    }
    return;
  }
  u.t = P.row_to_table ? P.row_to_table[r] : r;
  u.kr = min(P.k, u.L);
  chunk_range(u.L, u.G, rank, &u.s0, &u.n);
  u.n -= u.s0;
  if (rank == 0) fill_row(c, r, u.kr, P.k);

  // Short row: every position is selected, in position order.
  if (u.L <= P.k) {
    for (int i = threadIdx.x; i < u.n; i += kThreads) emit(c, u, u.s0 + i, u.s0 + i);
    return;
  }

  __syncthreads();  // buf / hist / list of the previous unit are no longer in use
  load_and_histogram(c, u);

  int b0, above0, eq0, la0, le0;
  if (!reduce_and_find(c, u, u.G > 1 ? u.gs->hist0 : nullptr, u.kr, b0, above0, eq0, la0, le0))
    return;
  int need = u.kr - above0;
  const bool all_eq = (eq0 == need);
  const bool compact = !all_eq && eq0 <= (u.G > 1 ? kGroupCap : kListCap);
  const bool fallback = !all_eq && !compact;

  // Reserve output (and candidate) space.
  if (threadIdx.x == 0) {
    const int cnt = la0 + (all_eq ? le0 : 0);
    int ob = 0, cb = 0;
    if (u.G > 1) {
      ob = (int)atomicAdd(&u.gs->out_ctr, (uint32_t)cnt);
      if (compact) cb = (int)atomicAdd(&u.gs->cand_ctr, (uint32_t)le0);
    }
    s.bc[7] = ob;
    s.bc[8] = cb;
    s.bc[9] = 0;   // emitted in this pass
    s.bc[10] = 0;  // candidates gathered in this pass
  }
  __syncthreads();
  const int out_base = s.bc[7], cand_base = s.bc[8];

  // Pass 2 over the resident chunk: emit above the threshold bin, gather or fold
  // the boundary bin.
  {
    const float tlo = skip_below((uint32_t)b0);
    const float4* b4 = reinterpret_cast<const float4*>(s.buf);
    uint32_t fa = 0xFFFFFFFFu, fo = 0u;
    for (int v = threadIdx.x; v < u.nvec; v += kThreads) {
      const float4 x = b4[v];
      const float m = fmaxf(fmaxf(x.x, x.y), fmaxf(x.z, x.w));
      if (m < tlo) continue;
      const float xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int e = 4 * v - u.head + j;
        if (e < 0 || e >= u.n) continue;
        const uint32_t d = coarse_digit(xs[j]);
        if (d < (uint32_t)b0) continue;
        const int p = u.s0 + e;
        if (d > (uint32_t)b0 || all_eq) {
          const int idx = atomicAdd(&s.bc[9], 1);
          emit(c, u, out_base + idx, p);
        } else if (compact) {
          const int ci = atomicAdd(&s.bc[10], 1);
          const uint32_t key = f2key(xs[j]);
          if (u.G > 1) {
            if (cand_base + ci < kGroupCap) {
              u.gs->cand_key[cand_base + ci] = key;
              u.gs->cand_pos[cand_base + ci] = (uint32_t)p;
            }
          } else if (ci < kListCap) {
            s.lkey[ci] = key;
            s.lpos[ci] = (uint32_t)p;
          }
        } else {
          const uint32_t key = f2key(xs[j]);
          fa &= key;
          fo |= key;
        }
      }
    }
    if (fallback) block_and_or(fa, fo, s);
    __syncthreads();
    if (fallback) {
      if (u.G > 1) {
        if (threadIdx.x == 0) {
          atomicOr(&u.gs->and_key, ~fa);  // stored inverted so the reset value is 0
          atomicOr(&u.gs->or_key, fo);
        }
        if (!group_barrier(c, u)) return;
        if (threadIdx.x == 0) {
          s.bc[11] = (int)~__ldcg(&u.gs->and_key);
          s.bc[12] = (int)__ldcg(&u.gs->or_key);
        }
        __syncthreads();
        fa = (uint32_t)s.bc[11];
        fo = (uint32_t)s.bc[12];
        __syncthreads();
      }
    }

    if (fallback) {
      // ---------------- in-place refinement on the full key, then ordered ties
      int emitted = above0;  // G == 1 running output index
      uint32_t pmask = 0u, pval = 0u;
      int local_tie = le0;
      bool done = false;
      if (fa != fo) {
        int hb = 31 - __clz(fa ^ fo);
        pmask = hb == 31 ? 0u : ~((2u << hb) - 1u);
        pval = fa & pmask;
        for (int lev = 0; lev < 3 && !done; ++lev) {
          const int shift = max(hb - (kLevelBits - 1), 0);
          const uint32_t dmask = (1u << (hb - shift + 1)) - 1u;
          for (int i = threadIdx.x; i < kBins0; i += kThreads) s.hist[i] = 0u;
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
              atomicAdd(&s.hist[(key >> shift) & dmask], 1u);
            }
          }
          __syncthreads();
          if (u.G > 1 && threadIdx.x == 0) u.gs->levels = (uint32_t)(lev + 1);
          int bl, abl, eql, lal, lel;
          if (!reduce_and_find(c, u, u.G > 1 ? u.gs->hlev[lev] : nullptr, need, bl, abl, eql,
                               lal, lel))
            return;
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
      if (!done) {
        // Every remaining candidate has key == pval. Take the `need` smallest
        // positions among them, across the row's chunks in position order.
        const uint32_t T = pval;
        int prefix = 0;
        if (u.G > 1) {
          if (threadIdx.x == 0) u.gs->tie_cnt[u.rank] = (uint32_t)local_tie;
          if (!group_barrier(c, u)) return;
          int acc = 0;
          for (int j = threadIdx.x; j < u.rank; j += kThreads) acc += (int)__ldcg(&u.gs->tie_cnt[j]);
          prefix = block_sum(acc, s);
        }
        const int tie_base = u.kr - need;  // all other entries fill [0, kr - need)
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
      }
    }
  }

  if (compact && u.G == 1) {
    __syncthreads();
    list_select(s, s.lkey, s.lpos, s.lst, eq0, need);
    list_emit(c, u, s.lpos, s.lst, eq0, above0);
  }

  if (u.G > 1) {
    // End of the row for this CTA. The last one finishes compact selection and
    // clears the row's counters for the next call.
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
      const uint32_t old = atomicAdd(&u.gs->fin, 1u);
      s.bc[13] = ((old + 1u) % (uint32_t)u.G) == 0u ? 1 : 0;
      __threadfence();
    }
    __syncthreads();
    if (s.bc[13]) {
      if (compact) {
        uint32_t* lkey = reinterpret_cast<uint32_t*>(s.buf);
        uint32_t* lpos = lkey + kGroupCap;
        uint8_t* lst = reinterpret_cast<uint8_t*>(lpos + kGroupCap);
        for (int i = threadIdx.x; i < eq0; i += kThreads) {
          lkey[i] = __ldcg(&u.gs->cand_key[i]);
          lpos[i] = __ldcg(&u.gs->cand_pos[i]);
        }
        __syncthreads();
        list_select(s, lkey, lpos, lst, eq0, need);
        list_emit(c, u, lpos, lst, eq0, above0);
      }
      const uint32_t levels = __ldcg(&u.gs->levels);
      for (int i = threadIdx.x; i < kBins0; i += kThreads) {
        u.gs->hist0[i] = 0u;
        for (uint32_t l = 0; l < levels && l < 3; ++l) u.gs->hlev[l][i] = 0u;
      }
      if (threadIdx.x == 0) {
        u.gs->bar = 0u;
        u.gs->out_ctr = 0u;
        u.gs->cand_ctr = 0u;
        u.gs->and_key = 0u;
        u.gs->or_key = 0u;
        u.gs->levels = 0u;
      }
    }
  }
}

__global__ void __launch_bounds__(kThreads, 1) select_kernel(SelectParams p) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  Smem& s = *reinterpret_cast<Smem*>(smem_raw);
  const Layout lay = make_layout(p.rows);
  Header* h = reinterpret_cast<Header*>(p.ws + lay.header);

  // Plan checks (uniform over the grid).
  const bool bad = h->magic != kMagic || h->rows != p.rows || h->max_len != p.max_len ||
                   h->grid != (int)gridDim.x || h->plan_error != 0;
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

  if (threadIdx.x == 0) {
    for (int i = 0; i < kPieces; ++i) mbar_init(&s.mbar[i], 1);
    fence_mbar_init();
  }
  __syncthreads();

  Ctx c{p, h, s, 0u};
  const int32_t* units = reinterpret_cast<const int32_t*>(p.ws + lay.units);
  const int waves = h->waves;
  for (int w = 0; w < waves; ++w) {
    const int32_t id = units[(int64_t)w * kMaxGrid + blockIdx.x];
    if (id >= 0) process_unit(c, id / kMaxGrid, id % kMaxGrid);
  }

  const int32_t* singles = reinterpret_cast<const int32_t*>(p.ws + lay.singles);
  const unsigned long long P = (unsigned long long)h->n_single + gridDim.x;
  const int n_single = h->n_single;
  while (true) {
    __syncthreads();
    if (threadIdx.x == 0) {
      const unsigned long long t = atomicAdd(&h->steal, 1ull);
      s.bc[14] = (int)(t % P);
    }
    __syncthreads();
    const int idx = s.bc[14];
    if (idx >= n_single) break;
    process_unit(c, singles[idx], 0);
  }
}

}  // namespace

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
