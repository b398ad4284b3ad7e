// CPU oracle for per-query top-k selection fused with paged slot translation.
//
// TEST INFRASTRUCTURE ONLY. Nothing in the product path (the CUDA library and its
// Python binding) may include, link, load or call this file. Only the tests, the
// smoke check and the benchmark's CPU-baseline arm use it.
//
// What it computes, written as the plain definition:
//
//   "Serving GLM5.2 NVFP4 Agentic Workload with SGLang", section "Kernel
//   Optimization > TopK-V2" (Figs. 2-3 and the paragraphs after them): each query
//   row holds one fp32 score per historical KV position; the kernel returns exactly
//   k of them (runtime k up to 2048), decided exactly in fp32 with a tie-break, and
//   translates each selected logical position into a physical indexer KV-cache slot
//   through the page table.
//
// The pages leave the tie rule, short rows and the slot formula open. Readings used:
//   * order: p before q iff s(p) > s(q), or s(p) == s(q) and p < q (IEEE equality,
//     so -0.0 == +0.0); every NaN ranks below -inf, NaNs tie among themselves and
//     fall back to position;
//   * a row of valid length L yields min(k, L) entries, sorted by that order, and
//     the remaining k - min(k, L) output entries are -1;
//   * slot(p) = table[t][p / page_size] * page_size + p % page_size, t the row's
//     table (row_to_table[r], identity when absent), computed in 64-bit;
//   * a row whose length lies outside [0, max_len] or whose pages exceed the
//     table width is written as all -1 and reported; a negative table entry or a
//     slot above INT32_MAX gives -1 for that entry and is reported.
//
// The method itself (radix histograms, refinement) reaches the same set faster;
// this oracle instead sorts each row's (score, position) pairs with std::sort and
// the comparator above and takes the prefix. A second entry point uses
// std::nth_element + std::sort as a library cross-check of the first.
//
// Parity status: pinned (brute-force rank counts on tiny rows, invariants, closed
// forms and hand-worked fixtures in the test suite).

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

namespace {

struct Entry {
  float s;
  int32_t p;
};

// p ranks before q (see the reading above). ORACLE_MUTANT selects a deliberately
// wrong variant, compiled only by the pin-strength tests.
inline bool ranks_before(const Entry& a, const Entry& b) {
  const bool na = std::isnan(a.s), nb = std::isnan(b.s);
#if ORACLE_MUTANT == 5
  // mutant: NaN not demoted (treated by raw comparison, which is never true)
  (void)na; (void)nb;
  if (a.s != b.s) return a.s > b.s;
  return a.p < b.p;
#else
  if (na != nb) return nb;         // the non-NaN one ranks first
  if (na) return a.p < b.p;        // both NaN: by position
#endif
#if ORACLE_MUTANT == 1
  if (a.s != b.s) return a.s > b.s;
  return a.p > b.p;                // mutant: ties to the larger position
#elif ORACLE_MUTANT == 2
  if (a.s != b.s) return a.s < b.s;  // mutant: smallest scores first
  return a.p < b.p;
#elif ORACLE_MUTANT == 6
  // mutant: compares bit patterns as signed integers (-0 != +0, negatives reversed)
  int32_t ia, ib;
  std::memcpy(&ia, &a.s, 4);
  std::memcpy(&ib, &b.s, 4);
  if (ia != ib) return ia > ib;
  return a.p < b.p;
#else
  if (a.s != b.s) return a.s > b.s;
  return a.p < b.p;
#endif
}

enum : int {
  kOk = 0,
  kErrLen = 1,
  kErrTableWidth = 2,
  kErrTableEntry = 4,
  kErrSlotOverflow = 8,
};

struct Args {
  const float* scores;
  int64_t ld;
  const int32_t* lens;
  int rows;
  int max_len;
  int k;
  const int32_t* table;
  int64_t table_ld;
  const int32_t* row_to_table;
  int page_size;
  int32_t* out_slots;
  int32_t* out_pos;
  int use_nth;
};

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// One row: returns the error bits it raised.
int one_row(const Args& a, int r) {
  int32_t* slots = a.out_slots + int64_t(r) * a.k;
  int32_t* pos = a.out_pos ? a.out_pos + int64_t(r) * a.k : nullptr;
  for (int i = 0; i < a.k; ++i) {
    slots[i] = -1;
    if (pos) pos[i] = -1;
  }
  const int32_t L = a.lens[r];
  if (L < 0 || L > a.max_len) return kErrLen;
  if (ceil_div(L, a.page_size) > a.table_ld) return kErrTableWidth;
  const int64_t t = a.row_to_table ? a.row_to_table[r] : r;

  std::vector<Entry> e(static_cast<size_t>(L));
  const float* row = a.scores + int64_t(r) * a.ld;
  for (int32_t p = 0; p < L; ++p) e[p] = Entry{row[p], p};

#if ORACLE_MUTANT == 4
  const int32_t m = std::min<int32_t>(a.k, L) - (L > 0 ? 1 : 0);  // mutant: one short
#else
  const int32_t m = std::min<int32_t>(a.k, L);
#endif
  if (a.use_nth && m < L) {
    std::nth_element(e.begin(), e.begin() + m, e.end(), ranks_before);
    std::sort(e.begin(), e.begin() + m, ranks_before);
  } else {
    std::sort(e.begin(), e.end(), ranks_before);
  }

  int err = kOk;
  const int32_t* trow = a.table + t * a.table_ld;
  for (int32_t i = 0; i < m; ++i) {
    const int32_t p = e[i].p;
    if (pos) pos[i] = p;
#if ORACLE_MUTANT == 3
    const int64_t page = trow[p / a.page_size];
    const int64_t slot = page * a.page_size;  // mutant: drops the in-page offset
#elif ORACLE_MUTANT == 7
    const int64_t page = (a.table + int64_t(r) * a.table_ld)[p / a.page_size];  // mutant: ignores row_to_table
    const int64_t slot = page * a.page_size + p % a.page_size;
#else
    const int64_t page = trow[p / a.page_size];
    const int64_t slot = page * a.page_size + p % a.page_size;
#endif
    if (page < 0) {
      err |= kErrTableEntry;
      continue;
    }
    if (slot > INT32_MAX) {
      err |= kErrSlotOverflow;
      continue;
    }
    slots[i] = static_cast<int32_t>(slot);
  }
  return err;
}

int run(const Args& a, int threads) {
  if (a.rows <= 0) return kOk;
  if (threads <= 1 || a.rows == 1) {
    int err = 0;
    for (int r = 0; r < a.rows; ++r) err |= one_row(a, r);
    return err;
  }
  threads = std::min(threads, a.rows);
  std::vector<int> errs(static_cast<size_t>(threads), 0);
  std::vector<std::thread> pool;
  for (int w = 0; w < threads; ++w) {
    pool.emplace_back([&, w] {
      for (int r = w; r < a.rows; r += threads) errs[w] |= one_row(a, r);
    });
  }
  int err = 0;
  for (int w = 0; w < threads; ++w) {
    pool[w].join();
    err |= errs[w];
  }
  return err;
}

}  // namespace

extern "C" {

// Returns a bit set of kErr* flags (0 when every row was well formed).
// scores: host float32 [rows, ld]; lens: host int32 [rows]; table: host int32
// [n_tables, table_ld]; row_to_table: host int32 [rows] or null (identity);
// out_slots (and out_pos when non-null): host int32 [rows, k], fully written.
int oracle_topk_paged(const float* scores, int64_t ld, const int32_t* lens, int rows,
                      int max_len, int k, const int32_t* table, int64_t table_ld,
                      const int32_t* row_to_table, int page_size, int32_t* out_slots,
                      int32_t* out_pos, int threads) {
  if (k < 1 || page_size < 1 || rows < 0) return -1;
  Args a{scores, ld, lens, rows, max_len, k, table, table_ld, row_to_table, page_size,
         out_slots, out_pos, 0};
  return run(a, threads);
}

// Library cross-check: the same result through std::nth_element + std::sort.
int oracle_topk_paged_nth(const float* scores, int64_t ld, const int32_t* lens, int rows,
                          int max_len, int k, const int32_t* table, int64_t table_ld,
                          const int32_t* row_to_table, int page_size, int32_t* out_slots,
                          int32_t* out_pos, int threads) {
  if (k < 1 || page_size < 1 || rows < 0) return -1;
  Args a{scores, ld, lens, rows, max_len, k, table, table_ld, row_to_table, page_size,
         out_slots, out_pos, 1};
  return run(a, threads);
}

int oracle_mutant_id(void) { return ORACLE_MUTANT; }

}  // extern "C"
