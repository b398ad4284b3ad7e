// Shared definitions of the top-k + paged-slot kernels for GB300 (sm_103a):
// tuning constants, the workspace layout written by the planner and read by the
// select kernel, and small inline-PTX helpers (bulk copies, mbarriers, timers).
#pragma once

#include <cstddef>
#include <cstdint>

#include "../../include/topk_paged.h"

namespace topk {

// ---------------------------------------------------------------- constants
constexpr int kThreads = 512;              // threads per select CTA (16 warps)
constexpr int kWarps = kThreads / 32;
constexpr int kMaxGrid = 1024;             // largest persistent grid the plan describes
constexpr int kMaxWaves = 16;              // waves of multi-CTA groups in one plan
constexpr int kMaxGroups = 512;            // multi-CTA rows with group state in one plan
constexpr int kChunkCap = 48128;           // elements one CTA keeps resident in smem
constexpr int kChunkAlign = 16;            // chunk boundaries are multiples of 16 elements
constexpr int kMinAutoChunk = 2048;        // automatic plans never split finer than this
constexpr int kPieceBytes = 16384;         // one bulk copy (and one mbarrier) per piece
constexpr int kBufFloats = kChunkCap + 8;  // resident buffer incl. alignment slack
constexpr int kPieces = (kBufFloats * 4 + kPieceBytes - 1) / kPieceBytes;
constexpr int kBins0 = 4096;               // coarse histogram (12-bit digit)
constexpr int kLevelBits = 12;             // in-place refinement digit width
constexpr int kListCap = 1024;             // single-CTA compact candidate list (smem)
constexpr int kRankMax = 192;              // boundary sets up to this size: rank counting
constexpr int kRankOwnMax = 1024;          // multi-CTA rows: each CTA ranks its own candidates
constexpr int kGroupCap = 8192;            // multi-CTA compact candidate list (global)
constexpr int kListBins = 256;             // digit width 8 for list refinement
constexpr uint32_t kMagic = 0x54504B32u;   // plan magic
constexpr uint64_t kWaitNs = 200ull * 1000ull * 1000ull;  // bounded waits: 200 ms
constexpr int kShortMaxLen = 256;          // batches with max_len <= this: register path
constexpr int kMediumMaxLen = 16384;       // batches with max_len <= this: one CTA per row, several per SM
constexpr int kClusterMaxLen = 131072;     // longer ones up to this: one cluster per row, when they fit

// ---------------------------------------------------------------- workspace
// All offsets are multiples of 256 bytes.
struct Header {
  uint32_t magic;
  int32_t rows;
  int32_t max_len;
  int32_t grid;
  int32_t chunk;        // chunk target chosen by the planner (elements)
  int32_t waves;        // waves of the static multi-CTA unit table
  int32_t n_single;     // rows processed by one CTA
  int32_t n_multi;      // rows split over several CTAs
  int32_t status;       // sticky device status bits (TOPK_STATUS_*)
  int32_t plan_error;   // nonzero when the plan could not be built
  int32_t n_implicit;   // single rows handed out statically (one per idle CTA)
  int32_t dyn_period;   // claims of the ticket counter per call
  unsigned long long med_ticket;  // row ticket counter of the medium-row path (0 after a plan)
  int32_t pad0[2];
  unsigned long long steal;  // single-row ticket counter (advances by dyn_period per call)
  int32_t pad1[14];
  // First expired bounded wait (written once per plan, for diagnosis): kind
  // (1 = row barrier, 2 = piece copy), row, rank, barrier sequence, observed count,
  // target count, CTA index, unit wave-or-single marker.
  int32_t diag[8];
  int32_t pad2[24];
};
static_assert(sizeof(Header) == 256, "header size");
static_assert(offsetof(Header, diag) == 128, "diagnostic record offset");

struct RowInfo {
  int32_t len;    // length the plan was built for
  int32_t G;      // CTAs sharing the row (1 = single-CTA path)
  int32_t group;  // group-state index for G > 1, else -1
  int32_t pad;
};

// One CTA's share of a row: positions [s0, s0 + n) of row `row` (plan length len),
// chunk `rank` of G; `group` indexes the row's GroupState (-1 when G == 1).
struct __align__(16) UnitDesc {
  int32_t row, s0, n, len;
  int32_t rank, G, group, pad;
};

// Per multi-CTA row. Row barriers use one flag word per rank: (barriers passed by
// that rank) << 32 | a 32-bit payload, written with release semantics; a waiter
// acquires every rank's flag, so a barrier also delivers each rank's payload (its
// counts). Each rank also keeps the payloads of its last two barriers (pay2, by
// barrier parity, stored right after the flag, so that the next flag's release
// orders it): a rank can run at most one barrier ahead of a waiter still reading its
// flag (it cannot pass the next barrier before that waiter arrives there), and the
// waiter, seeing that next flag, then takes the payload from pay2. Flags only
// grow and are never reset by the select kernel. The histograms are cleared by the
// CTAs that wrote them once a later barrier shows every CTA has read them; the
// candidate slots and pay2 are written before they are read in every call.
struct GroupState {
  unsigned long long flag[kMaxGrid];
  uint32_t and_key;  // ~AND of boundary keys (stored inverted: reset value 0)
  uint32_t or_key;   // OR of boundary keys
  uint32_t pad[62];
  uint32_t hist0[kBins0];
  uint32_t hlev[3][1 << kLevelBits];
  uint32_t cand_key[kGroupCap];
  uint32_t cand_pos[kGroupCap];
  uint32_t pay2[2][kMaxGrid];
};
static_assert(sizeof(GroupState) % 256 == 0, "group state alignment");

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct Layout {
  size_t header, rowinfo, singles, first_single, units, groups, total;
  int ngroups;
};

__host__ __device__ inline Layout make_layout(int rows) {
  Layout l;
  const size_t r = (size_t)(rows > 0 ? rows : 1);
  l.ngroups = rows < kMaxGroups ? rows : kMaxGroups;
  l.header = 0;
  l.rowinfo = align256(sizeof(Header));
  l.singles = l.rowinfo + align256(sizeof(RowInfo) * r);
  l.first_single = l.singles + align256(sizeof(int32_t) * 2 * r);
  l.units = l.first_single + align256(sizeof(int32_t) * (size_t)kMaxGrid);
  l.groups = l.units + align256(sizeof(UnitDesc) * (size_t)kMaxWaves * kMaxGrid);
  l.total = l.groups + sizeof(GroupState) * (size_t)l.ngroups;
  return l;
}

__host__ __device__ inline int64_t ceil_div64(int64_t a, int64_t b) { return (a + b - 1) / b; }

// CTAs of the thread-block cluster that runs one row of a batch with this max_len on
// the cluster path (2, 4 or 8: the fewest that keep a CTA's share at most
// kClusterMaxLen / 8 values), or 0 outside that path's lengths.
__host__ __device__ inline int cluster_size_for(int max_len) {
  if (max_len <= kMediumMaxLen || max_len > kClusterMaxLen) return 0;
  return max_len <= kClusterMaxLen / 4 ? 2 : max_len <= kClusterMaxLen / 2 ? 4 : 8;
}

// Whether an unforced plan of this batch sends it down the cluster path: its rows'
// clusters fit the grid (one CTA per SM) at once. The plan is then its header alone.
__host__ __device__ inline bool cluster_batch(int rows, int max_len, int grid) {
  const int cs = cluster_size_for(max_len);
  return cs > 0 && rows >= 1 && (int64_t)rows * cs <= (int64_t)grid;
}

// Chunk of `rank` among G CTAs of a row of length L: [begin, end).
__host__ __device__ inline void chunk_range(int L, int G, int rank, int* begin, int* end) {
  int64_t c = ceil_div64(L, G);
  c = ceil_div64(c, kChunkAlign) * kChunkAlign;
  int64_t b = (int64_t)rank * c;
  int64_t e = b + c;
  if (b > L) b = L;
  if (e > L) e = L;
  *begin = (int)b;
  *end = (int)e;
}

// Arguments of one select launch (see topk_select_paged in include/topk_paged.h).
struct SelectParams {
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
  char* ws;
  uint64_t wait_ns;  // limit of every bounded wait (kWaitNs unless a test shortens it)
  int skip_cta;      // test hook: this CTA never arrives at its first row barrier (-1: none)
};

// ---------------------------------------------------------------- PTX helpers
#if defined(__CUDACC__)

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile(
      "mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
      : "memory");
}

// Bulk (non-tensor) copy global -> shared, completion signalled on `bar`.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for phase `parity` of `bar` to complete, for at most wait_ns. Returns false
// on expiry.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  uint64_t wait_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 > wait_ns) return false;
  }
}

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void red_release_add_u32(uint32_t* p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void red_add_u32(uint32_t* p, uint32_t v) {
  asm volatile("red.relaxed.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t ld_cg_u32(const uint32_t* p) { return __ldcg(p); }

#endif  // __CUDACC__

// Optional phase trace (compiled in only with -DTOPK_TRACE): thread 0 of each CTA
// stamps %globaltimer at fixed points into a per-translation-unit device array.
#if defined(TOPK_TRACE) && defined(__CUDACC__)
#define TOPK_MARK(arr, slot)                                                       \
  do {                                                                             \
    if (threadIdx.x == 0 && (slot) < 32) arr[blockIdx.x * 32 + (slot)] = global_timer_ns(); \
  } while (0)
#else
#define TOPK_MARK(arr, slot) \
  do {                       \
  } while (0)
#endif

}  // namespace topk
