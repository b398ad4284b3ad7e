// Select + page-table kernel for batches of medium rows (GB300, sm_103a).
//
// "Serving GLM5.2 NVFP4 Agentic Workload with SGLang", "Kernel Optimization > TopK-V2":
// rows are binned by length into a register-resident path, a single-CTA streaming
// path and a multi-CTA path; "What's next" names ragged top-k for prefill, where
// thousands of query rows of a few thousand keys each come in one batch. A batch whose
// rows are all at most kMediumMaxLen values runs here: one 256-thread CTA per row, the
// row's scores in shared memory, and several CTAs per SM (three for rows of 12K
// values), so that the latency chains of different rows overlap on one SM.
//
// Per row, an exact radix selection over levels of digits, most significant first:
// the 12-bit coarse digit of the score, then the four bytes of the order-preserving
// 32-bit key, then the position in two 7-bit halves (smaller positions rank first).
// At each level the CTA histograms the digit over the values still in the running,
// finds the boundary digit (fewer than `need` values above it, at least `need` at or
// above it), emits every value above it, and keeps the boundary digit's values for
// the next level; a level whose boundary digit holds exactly what is still needed
// emits them too and ends the row. Key bytes on which every value of the row agrees
// are skipped. Once few values remain they are kept in a position list, so later
// levels do not rescan the row. Values are emitted through warp-aggregated shared
// counters (the order of a row's entries is unspecified) and translated to slots on
// the way out. While a row's slots are translated, the CTA's next row is already
// being copied into the row buffer by one bulk copy (its scores were prefetched into
// L2 earlier in the row), so the next row starts on data in shared memory.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "common.cuh"
#include "keys.cuh"

namespace topk {

namespace {

constexpr int kMedThreads = 256;
constexpr int kMedWarps = kMedThreads / 32;
constexpr int kCoarseBins = 4096;
constexpr int kCandCap = 2048;  // running positions kept in a list once this few remain
constexpr int kLevels = 7;      // coarse digit, 4 key bytes, 2 position halves
constexpr int kFinishPer = 8;   // values per lane of the one-warp finish (256 in all)

// The histogram of levels after the first uses hist[0, 256); the two running-position
// lists live in hist[256, ...), which the coarse level no longer needs once its
// boundary is known. Emitted positions are staged in outp and translated to slots in
// one pass at the end of the row, so that their table reads are in flight together.
struct MedShared {
  int hist[kCoarseBins];
  uint16_t outp[TOPK_MAX_K];
  int emitted;    // entries written to the row's output
  int listed;     // positions appended to the next list
  int bnd_digit;  // boundary digit of the current level
  int bnd_above;  // running values above it
  int bnd_at;     // running values at it
  int status;     // slot errors of the row
  unsigned key_and, key_or;
  int warp_tot[kMedWarps];
};
static_assert(sizeof(MedShared) % 16 == 0, "the row buffer after it is 16-byte aligned");
static_assert((kCoarseBins - 256) * sizeof(int) >= 2 * kCandCap * sizeof(uint16_t),
              "the position lists fit the coarse histogram's upper bins");

__device__ __forceinline__ uint16_t* med_list(MedShared& S, int which) {
  return reinterpret_cast<uint16_t*>(S.hist + 256) + which * kCandCap;
}

static_assert(kMediumMaxLen <= 1 << 14, "positions fit the two 7-bit position levels and uint16 lists");
static_assert(kMediumMaxLen <= 64 * kMedThreads, "a thread's entries of a row fit one 64-bit mask");

// Slots of the row's kr staged positions (outp, or the positions 0 .. kr - 1 when
// `identity`), written with the positions; eight table reads per thread in flight.
__device__ __forceinline__ void med_translate(const SelectParams& P, MedShared& S, int32_t* os,
                                              int32_t* op, int t, int kr, bool identity) {
  // a page size that is a power of two divides by a shift (the usual case, 64)
  const int ps = P.page_size;
  const bool pow2 = (ps & (ps - 1)) == 0;
  const int sh = __ffs(ps) - 1;
  const int32_t* trow = P.table + (int64_t)t * P.table_ld;
  for (int o0 = 0; o0 < kr; o0 += 8 * kMedThreads) {
    int pp[8];
    int32_t pg[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int o = o0 + j * kMedThreads + (int)threadIdx.x;
      pp[j] = o < kr ? (identity ? o : (int)S.outp[o]) : -1;
      pg[j] = pp[j] >= 0 ? __ldg(trow + (pow2 ? pp[j] >> sh : pp[j] / ps)) : 0;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int o = o0 + j * kMedThreads + (int)threadIdx.x;
      if (pp[j] < 0) continue;
      const int in = pow2 ? pp[j] & (ps - 1) : pp[j] % ps;
      const int64_t sl = (int64_t)pg[j] * ps + in;
      int32_t v = (int32_t)sl;
      if (pg[j] < 0) {
        atomicOr(&S.status, TOPK_STATUS_TABLE_ENTRY);
        v = -1;
      } else if (sl > 0x7FFFFFFFll) {
        atomicOr(&S.status, TOPK_STATUS_SLOT_OVERFLOW);
        v = -1;
      }
      os[o] = v;
      if (op) op[o] = pp[j];
    }
  }
}

// Digit of level lv: 0 = coarse (4096 bins), 1..4 = key bytes from the top (256
// bins), 5..6 = position bits 13..7 and 6..0, inverted so that smaller positions rank
// higher (128 bins).
__device__ __forceinline__ uint32_t med_digit(int lv, float x, uint32_t key, int p) {
  if (lv == 0) return coarse_digit(x);
  if (lv <= 4) return (key >> (32 - 8 * lv)) & 0xFFu;
  return 127u - (((uint32_t)p >> (lv == 5 ? 7 : 0)) & 127u);
}

__device__ __forceinline__ int med_bins(int lv) { return lv == 0 ? kCoarseBins : lv <= 4 ? 256 : 128; }

// Boundary digit of the histogram S.hist[0, nb): the digit d with (running values
// above d) < need <= (values at or above d). Thread t scans bins [t * per, ...) from
// the top; the block adds up the ranges above each thread.
__device__ void med_boundary(MedShared& S, int nb, int need) {
  // nb is 4096, 256 or 128: a thread's range is 16 bins or 1 (or empty past nb)
  const int per = (nb + kMedThreads - 1) / kMedThreads;
  const int lo = min(nb, (int)threadIdx.x * per), hi = min(nb, lo + per);
  int mine = 0;
  // lanes read their ranges in rotated order, so one load touches distinct banks
  if (hi - lo == per)
    for (int i = 0; i < per; ++i) mine += S.hist[lo + ((i + (int)threadIdx.x) & (per - 1))];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = mine;  // sum over lanes [lane, 31] of this warp
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_down_sync(0xffffffffu, incl, o);
    if (lane + o < 32) incl += y;
  }
  if (lane == 0) S.warp_tot[warp] = incl;
  __syncthreads();
  int above = incl - mine;
  for (int w = warp + 1; w < kMedWarps; ++w) above += S.warp_tot[w];
  if (above < need && above + mine >= need) {
    for (int i = hi - 1; i >= lo; --i) {
      const int c = S.hist[i];
      if (above + c >= need) {
        S.bnd_digit = i;
        S.bnd_above = above;
        S.bnd_at = c;
        break;
      }
      above += c;
    }
  }
  __syncthreads();
}

// One warp selects the `need` best of the n listed positions (n <= 32 * kPer):
// lane l holds positions list[l + 32 c] as 64-bit composite keys (score key << 14 |
// 16383 - position, all distinct), and a radix selection runs from the highest bit
// where they differ, one warp-wide count per bit. The selected positions are appended
// to S.outp after the S.emitted already there. kPer (values per lane) is the smallest
// that holds n, so each bit's step touches no more registers than needed.
template <int kPer>
__device__ void med_warp_finish(MedShared& S, const float* sx, const uint16_t* list, int n, int need,
                                int kr) {
  const int lane = threadIdx.x & 31;
  uint64_t key[kPer];
  int pos[kPer];
  uint32_t cand = 0u;
  uint32_t an_hi = 0xFFFFFFFFu, an_lo = 0xFFFFFFFFu, or_hi = 0u, or_lo = 0u;
#pragma unroll
  for (int c = 0; c < kPer; ++c) {
    const int i = lane + 32 * c;
    key[c] = 0ull;
    pos[c] = 0;
    if (i < n) {
      pos[c] = list[i];
      key[c] = ((uint64_t)f2key(sx[pos[c]]) << 14) | (uint64_t)(16383 - pos[c]);
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
    sel = cand;  // a single value: it is the one needed
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
    if (need > 0) sel |= cand;  // the last remaining value (the keys are distinct)
  }
  const unsigned lt = (1u << lane) - 1u;
  int base = S.emitted;
#pragma unroll
  for (int c = 0; c < kPer; ++c) {
    const bool s = (sel >> c) & 1u;
    const unsigned b = __ballot_sync(0xffffffffu, s);
    if (s) {
      const int o = base + __popc(b & lt);
      if (o < kr) S.outp[o] = (uint16_t)pos[c];  // o < kr by construction; guarded
    }
    base += __popc(b);
  }
  if (lane == 0) S.emitted = base;
}

// Bulk prefetch of row r's scores into L2: its first max_len values (inside the score
// array, whose rows are ld >= max_len apart), so that the row's length need not be read
// first; whole 16-byte units from an aligned start, an unaligned row not at all.
__device__ __forceinline__ void med_prefetch_row(const SelectParams& P, int r) {
  const float* row = P.scores + (int64_t)r * P.ld;
  const uint32_t bytes = (uint32_t)(P.max_len * 4) & ~15u;
  if ((reinterpret_cast<uintptr_t>(row) & 15u) != 0 || bytes == 0) return;
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(row), "r"(bytes) : "memory");
}

// Class of running-set entry i at level lv: 1 = emitted (above the boundary digit d,
// or at it when that ends the row), 2 = kept for the next level, 0 = neither or past
// the set. *pos receives its position.
__device__ __forceinline__ int med_class(MedShared& S, const float* sx, int src, int n_src, int i,
                                         int lv, const uint32_t (&chosen)[kLevels], uint32_t d,
                                         bool ends, bool list, int* pos) {
  if (i >= n_src) {
    *pos = 0;
    return 0;
  }
  const int p = src >= 0 ? (int)med_list(S, src)[i] : i;
  *pos = p;
  const float x = sx[p];
  const uint32_t key = f2key(x);
  if (src < 0)
    for (int l = 0; l < lv; ++l)
      if (med_digit(l, x, key, p) != chosen[l]) return 0;
  const uint32_t dg = med_digit(lv, x, key, p);
  if (dg > d || (ends && dg == d)) return 1;
  return list && dg == d ? 2 : 0;
}

__global__ void __launch_bounds__(kMedThreads, 3) medium_kernel(const __grid_constant__ SelectParams P) {
  extern __shared__ __align__(16) unsigned char med_smem[];
  MedShared& S = *reinterpret_cast<MedShared*>(med_smem);
  float* const sx = reinterpret_cast<float*>(med_smem + sizeof(MedShared));
  Header* h = reinterpret_cast<Header*>(P.ws);
  __shared__ int hdr_ok, row_sh;  // row_sh: the row this CTA works on
  if (threadIdx.x == 0) {
    const int4 h0 = __ldcg(reinterpret_cast<const int4*>(h));
    const int plan_error = __ldcg(&h->plan_error);
    hdr_ok = ((uint32_t)h0.x == kMagic && h0.y == P.rows && h0.z == P.max_len && plan_error == 0) ? 1 : 0;
  }
  const int lane = threadIdx.x & 31;
  // Rows by tickets. Every call takes exactly rows + gridDim.x of them (each CTA stops
  // at its first ticket past the rows), so ticket % period numbers the rows of every
  // call without a reset between calls; the plan sets the counter to 0.
  // Thread 0 claims the next row's ticket at the start of each row and reads it only
  // after the row's coarse level (then it prefetches that row into L2), so the claim's
  // round trip stays off the row's path.
  const unsigned long long period = (unsigned long long)P.rows + gridDim.x;
  unsigned long long pending = 0ull;  // thread 0: the claimed next ticket
  int nx = -1;                        // thread 0: its row, once computed
  int nx_len = -1;                    // thread 0: that row's length (read when nx is)
  // The next row's scores are copied into the row buffer (one bulk copy, completion on
  // row_bar) as soon as the current row no longer reads it, while the current row's
  // slots are translated; copy_sh tells the next row to wait for it.
  __shared__ __align__(8) uint64_t row_bar;
  __shared__ int copy_sh;
  uint32_t row_phase = 0u;
  if (threadIdx.x == 0) {
    mbar_init(&row_bar, 1);
    fence_mbar_init();
    copy_sh = 0;
  }
  // ticket -> row; a 32-bit remainder while the ticket counter fits (the 64-bit one is
  // a long software sequence on thread 0's path, which the CTA waits for)
  auto row_of = [&](unsigned long long tk) {
    return tk <= 0xFFFFFFFFull ? (int)((uint32_t)tk % (uint32_t)period) : (int)(tk % period);
  };
  if (threadIdx.x == 0) pending = atomicAdd(&h->med_ticket, 1ull);
  while (true) {
    __syncthreads();
    if (threadIdx.x == 0) {
      row_sh = nx >= 0 ? nx : row_of(pending);
      nx = -1;
      if (row_sh < P.rows) pending = atomicAdd(&h->med_ticket, 1ull);
      S.emitted = 0;
      S.status = 0;
      S.key_and = 0xFFFFFFFFu;
      S.key_or = 0u;
    }
    __syncthreads();
    const int r = row_sh;
    if (r >= P.rows) break;
    const bool copied = copy_sh != 0;
    if (copied) {
      // the copy lands in the row buffer whatever this row turns out to need
      bool ok = mbar_wait_bounded(&row_bar, row_phase, P.wait_ns);
      if (__syncthreads_or(!ok)) {
        if (threadIdx.x == 0) atomicOr(&h->status, TOPK_STATUS_TIMEOUT);
        ok = mbar_wait_bounded(&row_bar, row_phase, P.wait_ns);
        if (__syncthreads_or(!ok)) return;  // still in flight: leave the buffer alone
      }
      row_phase ^= 1u;
    }
    int32_t* os = P.out_slots + (int64_t)r * P.k;
    int32_t* op = P.out_pos ? P.out_pos + (int64_t)r * P.k : nullptr;
    const int L = P.lens[r];
    int err = 0;
    if (!hdr_ok) err = TOPK_STATUS_PLAN_MISMATCH;
    else if (L < 0 || L > P.max_len) err = TOPK_STATUS_LEN;
    else if (ceil_div64(L, P.page_size) > P.table_ld) err = TOPK_STATUS_TABLE_WIDTH;
    const int kr = err ? 0 : min(P.k, L);
    if (err && threadIdx.x == 0) atomicOr(&h->status, err);
    for (int i = kr + threadIdx.x; i < P.k; i += kMedThreads) {  // -1 padding
      os[i] = -1;
      if (op) op[i] = -1;
    }
    // A row that ends here drops the copy flag itself (the main path does so below):
    // every thread read it at the row's start, or it is already 0.
    if (kr == 0) {
      if (threadIdx.x == 0) copy_sh = 0;
      continue;
    }
    const int t = P.row_to_table ? P.row_to_table[r] : r;

    if (L <= P.k) {  // every position is taken: the scores are not read
      med_translate(P, S, os, op, t, kr, true);
      __syncthreads();
      if (threadIdx.x == 0) {
        if (S.status) atomicOr(&h->status, S.status);
        copy_sh = 0;
      }
      continue;
    }

    // Load the row into shared memory; histogram the coarse digit; AND / OR the keys.
    for (int i = threadIdx.x; i < kCoarseBins / 4; i += kMedThreads)
      reinterpret_cast<int4*>(S.hist)[i] = make_int4(0, 0, 0, 0);
    __syncthreads();
    if (threadIdx.x == 0) copy_sh = 0;  // read by every thread above
    const float* row = P.scores + (int64_t)r * P.ld;
    int head = 0;  // scalar positions start here
    if (copied) {
      // its 16-byte vectors were copied ahead: histogram them from shared memory
      const int nv = L >> 2;
      for (int i = threadIdx.x; i < nv; i += kMedThreads) {
        const float4 v = reinterpret_cast<const float4*>(sx)[i];
        atomicAdd(&S.hist[coarse_digit(v.x)], 1);
        atomicAdd(&S.hist[coarse_digit(v.y)], 1);
        atomicAdd(&S.hist[coarse_digit(v.z)], 1);
        atomicAdd(&S.hist[coarse_digit(v.w)], 1);
      }
      head = nv << 2;
    } else if ((reinterpret_cast<uintptr_t>(row) & 15u) == 0) {
      // 16-byte vectors, four per thread in flight before any is used
      const float4* r4 = reinterpret_cast<const float4*>(row);
      const int nv = L >> 2;
      for (int i0 = 0; i0 < nv; i0 += 4 * kMedThreads) {
        float4 v[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int i = i0 + j * kMedThreads + (int)threadIdx.x;
          if (i < nv) v[j] = __ldg(r4 + i);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int i = i0 + j * kMedThreads + (int)threadIdx.x;
          if (i >= nv) continue;
          reinterpret_cast<float4*>(sx)[i] = v[j];
          const float e[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            atomicAdd(&S.hist[coarse_digit(e[c])], 1);
          }
        }
      }
      head = nv << 2;
    }
    for (int p0 = head; p0 < L; p0 += 8 * kMedThreads) {  // the rest: scalars, 8 in flight
      float x[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int p = p0 + j * kMedThreads + (int)threadIdx.x;
        if (p < L) x[j] = __ldg(row + p);
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int p = p0 + j * kMedThreads + (int)threadIdx.x;
        if (p >= L) continue;
        sx[p] = x[j];
        atomicAdd(&S.hist[coarse_digit(x[j])], 1);
      }
    }
    __syncthreads();
    // AND / OR of the keys of the coarse boundary bin's values (filled on the coarse
    // level): key bytes on which they all agree need no level of their own
    uint32_t key_and = 0u, key_diff = 0xFFFFFFFFu;

    // Levels. The running set is { p : digit_l(p) == chosen[l] for every level l before
    // the current one }; src >= 0 when it is listed in med_list(S, src)[0 .. n_src).
    uint32_t chosen[kLevels];
    int need = kr, src = -1, n_src = L;
    for (int lv = 0; lv < kLevels && need > 0; ++lv) {
      if (src >= 0 && n_src <= 32 * kFinishPer) {
        // few values left, listed: one warp selects `need` of them in registers
        if (threadIdx.x < 32) {
          const uint16_t* l = med_list(S, src);
          if (n_src <= 32) med_warp_finish<1>(S, sx, l, n_src, need, kr);
          else if (n_src <= 64) med_warp_finish<2>(S, sx, l, n_src, need, kr);
          else if (n_src <= 128) med_warp_finish<4>(S, sx, l, n_src, need, kr);
          else med_warp_finish<8>(S, sx, l, n_src, need, kr);
        }
        __syncthreads();
        need = 0;
        break;
      }
      if (lv >= 1 && lv <= 4 && ((key_diff >> (32 - 8 * lv)) & 0xFFu) == 0u) {
        chosen[lv] = (key_and >> (32 - 8 * lv)) & 0xFFu;  // every running value agrees here
        continue;
      }
      const int nb = med_bins(lv);
      if (lv > 0) {  // histogram of this level's digit over the running set
        for (int i = threadIdx.x; i < nb; i += kMedThreads) S.hist[i] = 0;
        __syncthreads();
        for (int i = threadIdx.x; i < n_src; i += kMedThreads) {
          const int p = src >= 0 ? (int)med_list(S, src)[i] : i;
          const float x = sx[p];
          const uint32_t key = f2key(x);
          bool run = true;
          if (src < 0)
            for (int l = 0; l < lv && run; ++l) run = med_digit(l, x, key, p) == chosen[l];
          if (run) atomicAdd(&S.hist[med_digit(lv, x, key, p)], 1);
        }
        __syncthreads();
      }
      med_boundary(S, nb, need);
      if (lv == 0 && threadIdx.x == 0) {
        nx = row_of(pending);
        if (nx < P.rows) {
          med_prefetch_row(P, nx);
          nx_len = __ldg(P.lens + nx);  // first used once this row's levels are done
        }
      }
      const uint32_t d = (uint32_t)S.bnd_digit;
      const int above = S.bnd_above, at = S.bnd_at;
      const bool ends = above + at == need;  // the boundary digit completes the row
      const bool list = !ends && at <= kCandCap;
      const int dst = src == 0 ? 1 : 0;
      if (threadIdx.x == 0) S.listed = 0;
      __syncthreads();
      // Emit the running values above the boundary (and at it when that ends the row);
      // list the values at it for the next level. The first walk classifies this
      // thread's entries into two bit masks and the warp claims its output ranges with
      // one shared atomic each (same-address shared atomics from many warps, one per
      // step, would serialise); the second walk writes at ballot-prefix offsets. On the
      // coarse level with the boundary on the positive side, the bin's float bounds are
      // exact and classification is two compares.
      const bool fast = lv == 0 && d >= 2048u;
      const float t_at = skip_below(d), t_above = d < 4095u ? skip_below(d + 1u) : 0.0f;
      uint64_t m_take = 0ull, m_keep = 0ull;
      uint32_t t_lo = 0u, t_hi = 0u, k_lo = 0u, k_hi = 0u;  // their 32-bit halves (coarse level)
      uint32_t kand = 0xFFFFFFFFu, kor = 0u;  // keys of the coarse boundary bin's values
      if (fast) {
        // coarse level, boundary on the positive side: four values per step, bit
        // 4 step + c of the masks for position 4 (step * threads + t) + c
        // 4-bit compare masks per vector: above the bin, at or above it (NaN compares
        // false; a NaN bound keeps the top bin's "above" empty, +inf included)
        const int nv = (L + 3) >> 2;
        const float ta = d < 4095u ? t_above : __int_as_float(0x7FC00000);
        int jb = 0;
        for (int v0 = 0; v0 < nv; v0 += kMedThreads, jb += 4) {
          const int v = v0 + (int)threadIdx.x;
          if (v >= nv) continue;
          const float4 q = reinterpret_cast<const float4*>(sx)[v];
          const uint32_t vm = 4 * v + 4 <= L ? 0xFu : (1u << (L - 4 * v)) - 1u;  // the row's tail
          const uint32_t a_n = ((q.x >= ta ? 1u : 0u) | (q.y >= ta ? 2u : 0u) |
                                (q.z >= ta ? 4u : 0u) | (q.w >= ta ? 8u : 0u)) & vm;
          const uint32_t g_n = ((q.x >= t_at ? 1u : 0u) | (q.y >= t_at ? 2u : 0u) |
                                (q.z >= t_at ? 4u : 0u) | (q.w >= t_at ? 8u : 0u)) & vm;
          const uint32_t at_n = g_n & ~a_n;
          if (at_n) {
            const float e[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int c = 0; c < 4; ++c)
              if ((at_n >> c) & 1u) {
                const uint32_t key = f2key(e[c]);
                kand &= key;
                kor |= key;
              }
          }
          const uint32_t tn = a_n | (ends ? at_n : 0u), kn = list ? at_n : 0u;
          if (jb < 32) {  // the same for the whole warp
            t_lo |= tn << jb;
            k_lo |= kn << jb;
          } else {
            t_hi |= tn << (jb - 32);
            k_hi |= kn << (jb - 32);
          }
        }
        m_take = (uint64_t)t_hi << 32 | t_lo;
        m_keep = (uint64_t)k_hi << 32 | k_lo;
      } else {
        int j = 0;
        for (int i0 = 0; i0 < n_src; i0 += kMedThreads, ++j) {
          int p;
          const int cls = med_class(S, sx, src, n_src, i0 + (int)threadIdx.x, lv, chosen, d, ends,
                                    list, &p);
          m_take |= (uint64_t)(cls == 1) << j;
          m_keep |= (uint64_t)(cls == 2) << j;
        }
      }
      if (fast) {
        kand = __reduce_and_sync(0xffffffffu, kand);
        kor = __reduce_or_sync(0xffffffffu, kor);
        if (lane == 0) {
          atomicAnd(&S.key_and, kand);
          atomicOr(&S.key_or, kor);
        }
      }
      // each thread writes its own entries at offsets from a warp scan and one shared
      // atomic per warp (order inside a row is free)
      const int c_take = __popcll(m_take), c_keep = __popcll(m_keep);
      const int s_take = warp_incl_scan(c_take), s_keep = warp_incl_scan(c_keep);
      int o_base = 0, c_base = 0;
      if (lane == 31) {
        if (s_take) o_base = atomicAdd(&S.emitted, s_take);
        if (s_keep) c_base = atomicAdd(&S.listed, s_keep);
      }
      int o = __shfl_sync(0xffffffffu, o_base, 31) + s_take - c_take;
      int c = __shfl_sync(0xffffffffu, c_base, 31) + s_keep - c_keep;
      if (fast) {
        // bit js of a mask is component js & 3 of the thread's vector js >> 2; each
        // mask half is walked on its own (32-bit steps, no test of which mask)
        const int p0 = 4 * (int)threadIdx.x;
        auto pos_of = [&](int js) { return p0 + 4 * kMedThreads * (js >> 2) + (js & 3); };
        for (uint32_t m = t_lo; m; m &= m - 1u) {
          const int p = pos_of(__ffs(m) - 1);
          if (o < kr) S.outp[o] = (uint16_t)p;  // o < kr by construction; guarded
          ++o;
        }
        for (uint32_t m = t_hi; m; m &= m - 1u) {
          const int p = pos_of(__ffs(m) + 31);
          if (o < kr) S.outp[o] = (uint16_t)p;
          ++o;
        }
        uint16_t* dl = med_list(S, dst);
        for (uint32_t m = k_lo; m; m &= m - 1u) dl[c++] = (uint16_t)pos_of(__ffs(m) - 1);
        for (uint32_t m = k_hi; m; m &= m - 1u) dl[c++] = (uint16_t)pos_of(__ffs(m) + 31);
      } else {
        for (uint64_t m = m_take | m_keep; m; m &= m - 1) {
          const int js = __ffsll((long long)m) - 1;
          const int i = js * kMedThreads + (int)threadIdx.x;
          const int p = src >= 0 ? (int)med_list(S, src)[i] : i;
          if ((m_take >> js) & 1ull) {
            if (o < kr) S.outp[o] = (uint16_t)p;  // o < kr by construction; guarded
            ++o;
          } else {
            med_list(S, dst)[c++] = (uint16_t)p;
          }
        }
      }
      if (fast) {
        __syncthreads();
        key_and = S.key_and;
        key_diff = S.key_and ^ S.key_or;
      }
      __syncthreads();
      chosen[lv] = d;
      need = ends ? 0 : need - above;
      if (list) {
        src = dst;
        n_src = at;
      } else {
        src = -1;
        n_src = L;
      }
    }
    __syncthreads();
    if (threadIdx.x == 0 && nx >= 0 && nx < P.rows && nx_len > P.k && nx_len <= P.max_len) {
      // the row buffer is free: copy the next row's whole 16-byte vectors into it
      const float* nrow = P.scores + (int64_t)nx * P.ld;
      const uint32_t bytes = (uint32_t)(nx_len >> 2) * 16u;
      if ((reinterpret_cast<uintptr_t>(nrow) & 15u) == 0 && bytes > 0) {
        fence_proxy_async_smem();  // after this CTA's reads and writes of the buffer
        mbar_arrive_expect_tx(&row_bar, bytes);
        bulk_g2s(sx, nrow, bytes, &row_bar);
        copy_sh = 1;
      }
    }
    med_translate(P, S, os, op, t, min(S.emitted, kr), false);
    __syncthreads();
    if (threadIdx.x == 0) {
      int st = S.status;
      if (S.emitted != kr) st |= TOPK_STATUS_ORDER;  // cannot happen: every position is distinct
      if (st) atomicOr(&h->status, st);
    }
  }
}

}  // namespace

int medium_max_len() { return kMediumMaxLen; }

// Dynamic shared memory of a launch for rows of at most max_len values.
static size_t medium_smem(int max_len) {
  return sizeof(MedShared) + (size_t)((max_len + 3) & ~3) * sizeof(float);
}

cudaError_t launch_medium(const SelectParams& p, int sms, cudaStream_t stream) {
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const size_t smem = medium_smem(p.max_len);
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    e = cudaFuncSetAttribute(medium_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)medium_smem(kMediumMaxLen));
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, medium_kernel, kMedThreads, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) per_sm = 1;
  const int grid = (int)std::min<int64_t>((int64_t)p.rows, (int64_t)per_sm * sms);
  if (grid < 1) return cudaSuccess;
  medium_kernel<<<grid, kMedThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace topk
