// Indexer score producer ("MQA logits") on the 5th-generation tensor cores (GB300,
// sm_103a): tcgen05.mma of e4m3 keys against e4m3 query heads with fp32 accumulators
// in tensor memory, operands staged by TMA tensor copies.
//
// "Serving GLM5.2 NVFP4 Agentic Workload with SGLang", sections "Indexer Prologue
// Fusion" (FP8 keys with per-token scales in the paged indexer KV cache, FP8 query
// heads, one gate per head) and "What's next" (the MQA logits kernel). The formula
// (a reading; the pages give none) is
//   score(t, p) = sk(s) * sum_h g(t, h) * max(0, q(t, h) . k(s)),
//   s = table[r][p / page_size] * page_size + p % page_size.
//
// Work split. Query rows come in groups of G <= 8 rows sharing one block-table row;
// a unit is (group, tile of 128 key positions), and the launch's CTAs (one per SM,
// persistent) take units round-robin. For one unit the product is
//   D[128 keys, G * 64 (row, head) pairs] = K[128 keys, 128] . Q[G * 64, 128]^T,
// a dense contraction over the 128 channels: M = 128 keys (A, from the cache), N =
// the group's (row, head) pairs (B, from the queries, resident in shared memory for
// the whole group), K = 128 e4m3 values = 4 MMAs of K = 32. Rows 0..3 of a group are
// one MMA chain of N = 256 into tensor-memory columns [0, 256), rows 4..7 a second
// chain of N <= 256 into [256, 512): the tensor cores run at full rate only with wide
// N (an N = 64 chain per row ran at a quarter of it), and the two halves let the
// epilogue drain one half while the MMAs fill the other.
//
// Warp roles (18 warps): warp 0 issues the TMA copies (a group's query tile once,
// then two 64-key boxes per unit, each inside one page, into a ring of kStages shared
// buffers); warp 1 allocates tensor memory and one of its lanes issues the MMAs;
// warps 2..17 are the epilogue, warp w serving row slot r = (w - 2) / 4 of each half
// (rows r and 4 + r) for tensor-memory lanes 32 (w % 4) .. + 31, i.e. keys
// 32 (w % 4) + lane. Per half it loads its row's 64 accumulators (tcgen05.ld),
// applies the ReLU and the gates, frees the half (all 16 warps arrive), then scales
// by the key's scale and stores the score (consecutive keys per warp: 128-byte
// stores). One row per warp per half keeps a half's drain to one row's latency.
//
// Every mbarrier wait is bounded (%globaltimer); a wait that expires sets
// LOGITS_STATUS_TIMEOUT and ends the role's loop. Before the CTA exits, the MMA lane
// waits (bounded) for its last MMAs and the copy lane for its copies in flight, and
// the tensor memory is freed.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "indexer_logits.h"

namespace logits {

namespace {

constexpr int kHeads = 64;
constexpr int kDim = 128;            // channels = bytes per e4m3 row = one 128-byte swizzle row
constexpr int kTileKeys = 128;       // MMA M
constexpr int kBoxRows = 64;         // rows per TMA box (keys or query heads)
constexpr int kBoxBytes = kBoxRows * kDim;            // 8 KB
constexpr int kMaxGroup = 8;
constexpr int kHalfRows = 4;         // rows per accumulator half (4 * 64 = 256 columns)
constexpr int kEpiWarps = 16;        // 4 row slots x 4 lane quadrants
constexpr int kStages = 6;
constexpr int kStageBytes = kTileKeys * kDim;         // 16 KB
constexpr int kQBytes = kMaxGroup * kBoxBytes;        // 64 KB
constexpr int kThreads = 64 + kEpiWarps * 32;
constexpr int kTmemCols = 512;
constexpr uint64_t kWaitNs = 200ull * 1000 * 1000;    // 200 ms

// shared memory, base aligned to 1024 bytes: [Q 64 KB][key stages 6 x 16 KB][key
// scales 6 x 512 B][box records 6 x 2 int32][barriers 256 B][gates: 512 B per
// epilogue warp]
constexpr int kScaleOffset = kQBytes + kStages * kStageBytes;
constexpr int kBoxOffset = kScaleOffset + kStages * kTileKeys * 4;
constexpr int kBarOffset = kBoxOffset + kStages * 16;
constexpr int kGateOffset = kBarOffset + 256;
constexpr int kSmemBytes = kGateOffset + kEpiWarps * 512 + 1024;  // + alignment slack

// Box record of a stage (one per 64-key box), written by the copy lane: the slot of
// the box's first key, or one of these codes.
constexpr int kBoxNoPage = -1;    // negative page entry
constexpr int kBoxNoSlot = -2;    // slot past the cache
constexpr int kBoxUnused = -3;    // past the group's longest row

struct Params {
  const float* w;
  const int32_t* lens;
  const int32_t* group_table;
  const int32_t* table;
  const float* cache_scale;
  float* scores;
  int32_t* status;
  int64_t ld;
  int64_t num_slots;
  int units;  // n_groups * tiles (< 2^31)
  int rows, max_len, G, n_groups, n_tables, table_ld, page_size, tiles;
  int step_g, step_t;  // gridDim.x = step_g * tiles + step_t: a CTA's stride in (group, tile)
  uint64_t wait_ns;
};

// ------------------------------------------------------------------ PTX wrappers
__device__ __forceinline__ uint32_t su32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t now_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void bar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void bar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void bar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// One try: the thread may sleep until the phase completes (for at most the hint,
// 1 ms), so waiting warps leave the issue slots to the working ones.
__device__ __forceinline__ bool bar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(1000000u)
      : "memory");
  return ok != 0;
}

// Waits for the phase of parity `parity` to complete, for at most wait_ns.
__device__ __forceinline__ bool bar_wait(uint32_t bar, uint32_t parity, uint64_t wait_ns) {
  if (bar_try(bar, parity)) return true;
  const uint64_t t0 = now_ns();
  while (!bar_try(bar, parity))
    if (now_ns() - t0 > wait_ns) return false;
  return true;
}

// 2-D tiled TMA load of one box into shared memory, completion counted on `bar`.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// 1-D bulk copy global -> shared (16-byte aligned, size a multiple of 16).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Arrives on `bar` once every tcgen05 operation this thread issued before has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}

// D[tmem] (+)= A[smem] . B[smem]^T, e4m3 x e4m3 -> fp32.
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Instruction descriptor of kind::f8f6f4: D fp32 (bits 4-5 = 1), A and B e4m3 (format
// 0 in bits 7-9 and 10-12), both K-major (bits 15, 16 = 0), N >> 3 in bits 17-22,
// M >> 4 in bits 24-28.
__host__ __device__ constexpr uint32_t idesc_e4m3(int m, int n) {
  return (1u << 4) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

// Shared-memory matrix descriptor of a K-major operand in the 128-byte swizzle layout
// that a TMA copy with CU_TENSOR_MAP_SWIZZLE_128B writes: rows of 128 bytes, groups of
// 8 rows 1024 bytes apart (stride byte offset), start address >> 4 in bits 0-13,
// leading byte offset (unused for this layout; 16 bytes) in bits 16-29, stride byte
// offset >> 4 in bits 32-45, the descriptor version 1 in bits 46-47, swizzle mode 2
// (128-byte) in bits 61-63. The tile base is 1024-byte aligned; stepping K by 32
// bytes inside the swizzle row advances the start address by 32 bytes.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// 32 lanes x 64 consecutive 32-bit columns from tensor memory, waited for.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, uint32_t (&v)[64]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, "
      "%32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, "
      "%48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%64];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]),
        "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]),
        "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31]),
        "=r"(v[32]), "=r"(v[33]), "=r"(v[34]), "=r"(v[35]), "=r"(v[36]), "=r"(v[37]),
        "=r"(v[38]), "=r"(v[39]), "=r"(v[40]), "=r"(v[41]), "=r"(v[42]), "=r"(v[43]),
        "=r"(v[44]), "=r"(v[45]), "=r"(v[46]), "=r"(v[47]), "=r"(v[48]), "=r"(v[49]),
        "=r"(v[50]), "=r"(v[51]), "=r"(v[52]), "=r"(v[53]), "=r"(v[54]), "=r"(v[55]),
        "=r"(v[56]), "=r"(v[57]), "=r"(v[58]), "=r"(v[59]), "=r"(v[60]), "=r"(v[61]),
        "=r"(v[62]), "=r"(v[63])
      : "r"(taddr)
      : "memory");
}

// sum_h g[h] * max(0, acc[h]) over the 64 heads of one row (gates in shared memory):
// four accumulators of two lanes each, updated by packed two-lane fp32 FMAs, so each
// dependent chain is 8 FMAs long.
__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}

__device__ __forceinline__ float2 unpack2(uint64_t x) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(x));
  return r;
}

__device__ __forceinline__ float gate_sum(const float4* g4, const uint32_t (&v)[64]) {
  uint64_t acc[4] = {pack2(0.0f, 0.0f), pack2(0.0f, 0.0f), pack2(0.0f, 0.0f), pack2(0.0f, 0.0f)};
#pragma unroll
  for (int i = 0; i < kHeads / 4; ++i) {
    const float4 gw = g4[i];
    const uint64_t x01 = pack2(fmaxf(__uint_as_float(v[4 * i + 0]), 0.0f),
                               fmaxf(__uint_as_float(v[4 * i + 1]), 0.0f));
    const uint64_t x23 = pack2(fmaxf(__uint_as_float(v[4 * i + 2]), 0.0f),
                               fmaxf(__uint_as_float(v[4 * i + 3]), 0.0f));
    uint64_t& a = acc[(2 * i) & 3];
    uint64_t& b = acc[(2 * i + 1) & 3];
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(a) : "l"(pack2(gw.x, gw.y)), "l"(x01));
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(b) : "l"(pack2(gw.z, gw.w)), "l"(x23));
  }
  const float2 a0 = unpack2(acc[0]), a1 = unpack2(acc[1]), a2 = unpack2(acc[2]), a3 = unpack2(acc[3]);
  return ((a0.x + a0.y) + (a1.x + a1.y)) + ((a2.x + a2.y) + (a3.x + a3.y));
}

// ------------------------------------------------------------------ groups
struct Group {
  int row0;        // first row
  int n;           // rows in the group
  int tab;         // block-table row (-1: none)
  int glen;        // longest scored length of its rows
  int len[kMaxGroup];  // scored length of each row (0 on a row-level error)
  int err;         // row-level status bits of the group
};

__device__ __forceinline__ Group group_info(const Params& P, int g) {
  Group gi;
  gi.row0 = g * P.G;
  gi.n = min(P.G, P.rows - gi.row0);
  const int r = P.group_table ? __ldg(P.group_table + g) : g;
  const bool tab_ok = r >= 0 && r < P.n_tables;
  gi.tab = tab_ok ? r : -1;
  gi.glen = 0;
  gi.err = tab_ok ? 0 : LOGITS_STATUS_TABLE_ROW;
#pragma unroll
  for (int j = 0; j < kMaxGroup; ++j) {
    int L = 0;
    if (j < gi.n) {
      L = __ldg(P.lens + gi.row0 + j);
      if (L < 0 || L > P.max_len) {
        gi.err |= LOGITS_STATUS_LEN;
        L = 0;
      } else if (((int64_t)L + P.page_size - 1) / P.page_size > P.table_ld) {
        gi.err |= LOGITS_STATUS_TABLE_WIDTH;
        L = 0;
      } else if (!tab_ok) {
        L = 0;
      }
    }
    gi.len[j] = L;
    gi.glen = max(gi.glen, L);
  }
  return gi;
}

// Scored length of row j of a group (0 on a row-level error), as group_info finds it.
__device__ __forceinline__ int row_len(const Params& P, const Group& gi, int j) {
  const int L = __ldg(P.lens + gi.row0 + j);
  if (gi.tab < 0 || L < 0 || L > P.max_len ||
      ((int64_t)L + P.page_size - 1) / P.page_size > P.table_ld)
    return 0;
  return L;
}

// This CTA's units in order: (group, tile) of unit blockIdx.x, then steps of gridDim.x
// units, without divisions.
struct Units {
  int g, tile;
  __device__ __forceinline__ explicit Units(const Params& P)
      : g((int)(blockIdx.x / (unsigned)P.tiles)), tile((int)(blockIdx.x % (unsigned)P.tiles)) {}
  __device__ __forceinline__ bool more(const Params& P) const { return g < P.n_groups; }
  __device__ __forceinline__ void next(const Params& P) {
    g += P.step_g;
    tile += P.step_t;
    if (tile >= P.tiles) {
      tile -= P.tiles;
      ++g;
    }
  }
};

__device__ __forceinline__ void set_status(const Params& P, int bits) {
  if (P.status && bits) atomicOr(P.status, bits);
}

// ------------------------------------------------------------------ the kernel
__global__ void __launch_bounds__(kThreads, 1)
    logits_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ Params P) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = su32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const sbase = smem_raw + (base - raw);
  const uint32_t sQ = base;
  const uint32_t sStage = base + kQBytes;
  const uint32_t sScale = base + kScaleOffset;
  const float* const scale_f = reinterpret_cast<const float*>(sbase + kScaleOffset);
  volatile int* const box_rec = reinterpret_cast<volatile int*>(sbase + kBoxOffset);
  const uint32_t bars = base + kBarOffset;
  // barrier i at bars + 8 i
  const uint32_t b_full = bars;                       // [kStages] copy -> MMA (tx)
  const uint32_t b_empty = bars + 8 * kStages;        // [kStages] MMA commit -> copy
  const uint32_t b_tfull = bars + 16 * kStages;       // [2] MMA commit -> epilogue (a half)
  const uint32_t b_tempty = b_tfull + 16;             // [2] epilogue (16 warps) -> MMA
  const uint32_t b_qfull = b_tempty + 16;             // copy -> MMA (tx)
  const uint32_t b_qempty = b_qfull + 8;              // MMA commit -> copy
  const uint32_t b_done = b_qempty + 8;               // MMA commit: every MMA finished
  volatile uint32_t* const tmem_slot = reinterpret_cast<volatile uint32_t*>(sbase + kBarOffset + 192);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      bar_init(b_full + 8 * i, 1);
      bar_init(b_empty + 8 * i, 1 + kEpiWarps);  // MMA commit + each epilogue warp
    }
    for (int h = 0; h < 2; ++h) {
      bar_init(b_tfull + 8 * h, 1);
      bar_init(b_tempty + 8 * h, kEpiWarps);
    }
    bar_init(b_qfull, 1);
    bar_init(b_qempty, 1);
    bar_init(b_done, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_q)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_k)) : "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     su32(const_cast<uint32_t*>(tmem_slot))),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int T = P.tiles;
  if (warp == 0) {
    // ---------------------------------------------------------------- copies
    // The 32 lanes look up the key boxes of this CTA's next 32 units together (lane l:
    // the l-th of them), so that their table reads are in flight at once; the copies
    // are then issued unit by unit by lane 0. Every lane takes part in the waits.
    int n = 0, qn = 0, qg = -1;
    bool ok = true;
    const int64_t stride = gridDim.x;
    for (int64_t ub = blockIdx.x; ub < P.units && ok; ub += 32 * stride) {
      const int64_t ul = ub + (int64_t)lane * stride;
      int my_g = -1, y0 = kBoxUnused, y1 = kBoxUnused;  // my_g < 0: no unit, or nothing to score
      if (ul < P.units) {
        const int g = (int)((uint32_t)ul / (uint32_t)T), tile = (int)((uint32_t)ul % (uint32_t)T);
        const Group gi = group_info(P, g);
        if (tile == 0) set_status(P, gi.err);
        if (tile * kTileKeys < gi.glen) {
          my_g = g;
#pragma unroll
          for (int b = 0; b < 2; ++b) {
            const int p0 = tile * kTileKeys + b * kBoxRows;
            int y = kBoxUnused;
            if (p0 < gi.glen) {
              const int32_t page = __ldg(P.table + (int64_t)gi.tab * P.table_ld + p0 / P.page_size);
              const int64_t slot0 = (int64_t)page * P.page_size + p0 % P.page_size;
              y = page < 0 ? kBoxNoPage : slot0 >= P.num_slots ? kBoxNoSlot : (int)slot0;
            }
            (b == 0 ? y0 : y1) = y;
          }
        }
      }
      for (int k = 0; k < 32 && ok; ++k) {
        if (ub + (int64_t)k * stride >= P.units) break;
        const int g = __shfl_sync(0xffffffffu, my_g, k);
        const int ya = __shfl_sync(0xffffffffu, y0, k);
        const int yb = __shfl_sync(0xffffffffu, y1, k);
        if (g < 0) continue;
        if (g != qg) {
          const int row0 = g * P.G, nq = min(P.G, P.rows - row0);
          if (qn > 0) {
            ok = __all_sync(0xffffffffu, bar_wait(b_qempty, (uint32_t)(qn - 1) & 1u, P.wait_ns));
            if (!ok) break;
          }
          if (lane == 0) {
            bar_expect_tx(b_qfull, (uint32_t)(nq * kBoxBytes));
            for (int j = 0; j < nq; ++j)
              tma_load_2d(sQ + j * kBoxBytes, &tm_q, 0, (row0 + j) * kHeads, b_qfull);
          }
          qg = g;
          ++qn;
        }
        const int s = n % kStages;
        ok = __all_sync(0xffffffffu,
                        bar_wait(b_empty + 8 * s, ((uint32_t)(n / kStages) & 1u) ^ 1u, P.wait_ns));
        if (!ok) break;
        if (lane == 0) {
          // a box's 64 scales come along when the whole box lies inside the cache
          const bool sa = ya >= 0 && (int64_t)ya + kBoxRows <= P.num_slots;
          const bool sb = yb >= 0 && (int64_t)yb + kBoxRows <= P.num_slots;
          box_rec[2 * s] = ya;
          box_rec[2 * s + 1] = yb;
          bar_expect_tx(b_full + 8 * s, (ya >= 0 ? kBoxBytes : 0) + (yb >= 0 ? kBoxBytes : 0) +
                                            (sa ? kBoxRows * 4 : 0) + (sb ? kBoxRows * 4 : 0));
          if (ya >= 0) tma_load_2d(sStage + s * kStageBytes, &tm_k, 0, ya, b_full + 8 * s);
          if (yb >= 0) tma_load_2d(sStage + s * kStageBytes + kBoxBytes, &tm_k, 0, yb, b_full + 8 * s);
          if (sa) bulk_load(sScale + s * kTileKeys * 4, P.cache_scale + ya, kBoxRows * 4, b_full + 8 * s);
          if (sb)
            bulk_load(sScale + s * kTileKeys * 4 + kBoxRows * 4, P.cache_scale + yb, kBoxRows * 4,
                      b_full + 8 * s);
        }
        ++n;
      }
    }
    if (lane == 0) {
      if (!ok) set_status(P, LOGITS_STATUS_TIMEOUT);
      // copies still in flight land before the CTA exits (bounded)
      for (int i = max(0, n - kStages); i < n; ++i)
        bar_wait(b_full + 8 * (i % kStages), (uint32_t)(i / kStages) & 1u, P.wait_ns);
      if (qn > 0) bar_wait(b_qfull, (uint32_t)(qn - 1) & 1u, P.wait_ns);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMAs
    if (lane == 0) {
      int n = 0, qn = 0, qg = -1, cg = -1;
      uint32_t nh[2] = {0u, 0u};  // uses of each half
      Group gi;
      bool ok = true;
      for (Units it(P); it.more(P) && ok; it.next(P)) {
        const int g = it.g, tile = it.tile;
        if (g != cg) {
          gi = group_info(P, g);
          cg = g;
        }
        if (tile * kTileKeys >= gi.glen) continue;
        if (g != qg) {
          if (qn > 0) tc_commit(b_qempty);  // the previous group's queries are free
          if (!(ok = bar_wait(b_qfull, (uint32_t)qn & 1u, P.wait_ns))) break;
          qg = g;
          ++qn;
        }
        const int s = n % kStages;
        if (!(ok = bar_wait(b_full + 8 * s, (uint32_t)(n / kStages) & 1u, P.wait_ns))) break;
        tc_fence_after();
        const uint32_t a0 = sStage + s * kStageBytes;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int rows_h = h == 0 ? min(gi.n, kHalfRows) : gi.n - kHalfRows;
          if (rows_h <= 0 || !ok) continue;
          if (!(ok = bar_wait(b_tempty + 8 * h, (nh[h] & 1u) ^ 1u, P.wait_ns))) break;
          tc_fence_after();
          const uint32_t id = idesc_e4m3(kTileKeys, rows_h * kHeads);
#pragma unroll
          for (int k = 0; k < kDim / 32; ++k)
            tc_mma(tmem + h * kHalfRows * kHeads, sdesc_sw128(a0 + 32 * k),
                   sdesc_sw128(sQ + h * kHalfRows * kBoxBytes + 32 * k), id, k > 0 ? 1u : 0u);
          tc_commit(b_tfull + 8 * h);
          ++nh[h];
        }
        if (!ok) break;
        tc_commit(b_empty + 8 * s);
        ++n;
      }
      if (!ok) set_status(P, LOGITS_STATUS_TIMEOUT);
      tc_commit(b_done);  // every MMA issued above has finished when this arrives
      bar_wait(b_done, 0u, P.wait_ns);
    }
  } else {
    // ---------------------------------------------------------------- epilogue
    const int r = (warp - 2) >> 2;  // row slot within a half
    const int quad = warp & 3;
    const uint32_t t_lane = tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(r * kHeads);
    float4* const sgate = reinterpret_cast<float4*>(sbase + kGateOffset + (warp - 2) * 512);
    int cg = -1, n = 0;  // n: units taken, as the copy and MMA lanes count them
    uint32_t nh[2] = {0u, 0u};
    int len[2] = {0, 0};  // scored lengths of rows r and 4 + r of the current group
    Group gi;
    bool ok = true;
    for (Units it(P); it.more(P) && ok; it.next(P)) {
      const int g = it.g, tile = it.tile;
      if (g != cg) {
        gi = group_info(P, g);
        cg = g;
        len[0] = r < gi.n ? row_len(P, gi, r) : 0;
        len[1] = kHalfRows + r < gi.n ? row_len(P, gi, kHalfRows + r) : 0;
        // this warp's gates (rows r and 4 + r: 32 float4) into its own shared slice
        __syncwarp();
        const int jr = (lane < 16 ? r : kHalfRows + r);
        if (jr < gi.n)
          sgate[lane] = __ldg(reinterpret_cast<const float4*>(P.w + (int64_t)(gi.row0 + jr) * kHeads) +
                              (lane & 15));
        __syncwarp();
      }
      if (tile * kTileKeys >= gi.glen) continue;
      const int p = tile * kTileKeys + quad * 32 + lane;
      // this key's scale and box record from the stage, which is then released
      const int s = n % kStages;
      ok = __all_sync(0xffffffffu, bar_wait(b_full + 8 * s, (uint32_t)(n / kStages) & 1u, P.wait_ns));
      if (!ok) break;
      const int rec = box_rec[2 * s + (quad >> 1)];
      const int kb = quad * 32 + lane;  // key within the tile
      float sk = 0.0f;
      bool bad = false;
      if (p < gi.glen) {
        const int64_t slot = (int64_t)rec + (kb & (kBoxRows - 1));
        if (rec == kBoxNoPage) {
          bad = true;
          if (r == 0) set_status(P, LOGITS_STATUS_TABLE_ENTRY);
        } else if (rec == kBoxNoSlot || slot >= P.num_slots) {
          bad = true;
          if (r == 0) set_status(P, LOGITS_STATUS_SLOT);
        } else {
          sk = (int64_t)rec + kBoxRows <= P.num_slots ? scale_f[s * kTileKeys + kb]
                                                      : __ldg(P.cache_scale + slot);
        }
      }
      __syncwarp();
      if (lane == 0) bar_arrive(b_empty + 8 * s);
      ++n;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int rows_h = h == 0 ? min(gi.n, kHalfRows) : gi.n - kHalfRows;
        if (rows_h <= 0) continue;
        // every warp of the epilogue waits and arrives, with or without a row here;
        // the warp leaves together if any lane's wait expired
        ok = __all_sync(0xffffffffu, bar_wait(b_tfull + 8 * h, nh[h] & 1u, P.wait_ns));
        if (!ok) break;
        ++nh[h];
        tc_fence_after();
        const int j = h * kHalfRows + r;  // row within the group
        float acc = 0.0f;
        if (r < rows_h) {
          uint32_t v[64];
          tmem_ld64(t_lane + h * kHalfRows * kHeads, v);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) bar_arrive(b_tempty + 8 * h);
          acc = gate_sum(sgate + h * (kHeads / 4), v);
          if (p < len[h]) P.scores[(int64_t)(gi.row0 + j) * P.ld + p] = bad ? -INFINITY : sk * acc;
        } else {
          __syncwarp();
          if (lane == 0) bar_arrive(b_tempty + 8 * h);
        }
      }
    }
    if (!ok && lane == 0) set_status(P, LOGITS_STATUS_TIMEOUT);
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols)
                 : "memory");
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// Rows of 128 bytes, boxes of 64 rows, 128-byte swizzle.
bool encode_rows(CUtensorMap* map, const void* base, uint64_t n_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)kDim, (cuuint64_t)n_rows};
  const cuuint64_t strides[1] = {(cuuint64_t)kDim};
  const cuuint32_t box[2] = {(cuuint32_t)kDim, (cuuint32_t)kBoxRows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct DevInfo {
  int sms = 0;
  bool attr = false;
};

int launch(const uint8_t* q, const float* w, int rows, int heads, int dim, const int32_t* lens,
           int max_len, int G, const int32_t* group_table, const int32_t* table, int n_tables,
           int table_ld, int page_size, const uint8_t* cache, const float* cache_scale,
           int64_t num_slots, float* scores, int64_t ld, int32_t* status, cudaStream_t stream,
           uint64_t wait_ns) {
  if (rows < 0 || heads != kHeads || dim != kDim || G < 1 || G > kMaxGroup || max_len < 0 ||
      n_tables < 1 || table_ld < 1 || page_size < kBoxRows || page_size % kBoxRows != 0 ||
      num_slots < 1 || num_slots >= (int64_t(1) << 31) || ld < max_len)
    return LOGITS_ERR_SHAPE;
  if (rows == 0) return LOGITS_OK;
  if (!q || !w || !lens || !table || !cache || !cache_scale || !scores) return LOGITS_ERR_NULL;
  auto a16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  auto a4 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; };
  if (!a16(q) || !a16(w) || !a16(cache) || !a16(cache_scale) || !a4(lens) || !a4(table) ||
      !a4(scores) || (group_table && !a4(group_table)) || (status && !a4(status)))
    return LOGITS_ERR_ALIGN;
  if ((int64_t)rows * kHeads >= (int64_t(1) << 31)) return LOGITS_ERR_SHAPE;

  static DevInfo info[64];
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return LOGITS_ERR_CUDA;
  int sms;
  {
    std::lock_guard<std::mutex> lk(mu);
    if (!info[dev].attr) {
      if (cudaDeviceGetAttribute(&info[dev].sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
          cudaFuncSetAttribute(logits_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) !=
              cudaSuccess)
        return LOGITS_ERR_CUDA;
      info[dev].attr = true;
    }
    sms = info[dev].sms;
  }
  CUtensorMap tq, tk;
  if (!encode_rows(&tq, q, (uint64_t)rows * kHeads) || !encode_rows(&tk, cache, (uint64_t)num_slots))
    return LOGITS_ERR_CUDA;

  Params P;
  P.w = w;
  P.lens = lens;
  P.group_table = group_table;
  P.table = table;
  P.cache_scale = cache_scale;
  P.scores = scores;
  P.status = status;
  P.ld = ld;
  P.num_slots = num_slots;
  P.rows = rows;
  P.max_len = max_len;
  P.G = G;
  P.n_tables = n_tables;
  P.table_ld = table_ld;
  P.page_size = page_size;
  P.tiles = max(1, (max_len + kTileKeys - 1) / kTileKeys);
  const int n_groups = (rows + G - 1) / G;
  if ((int64_t)n_groups * P.tiles >= (int64_t(1) << 31)) return LOGITS_ERR_SHAPE;
  P.n_groups = n_groups;
  P.units = n_groups * P.tiles;
  P.wait_ns = wait_ns;
  const int grid = std::min(P.units, sms);
  P.step_g = grid / P.tiles;
  P.step_t = grid % P.tiles;
  logits_kernel<<<grid, kThreads, kSmemBytes, stream>>>(tq, tk, P);
  return cudaGetLastError() == cudaSuccess ? LOGITS_OK : LOGITS_ERR_CUDA;
}

}  // namespace
}  // namespace logits

extern "C" int indexer_mqa_logits(const uint8_t* q, const float* w, int rows, int heads, int dim,
                                  const int32_t* lens, int max_len, int group_rows,
                                  const int32_t* group_table, const int32_t* block_table,
                                  int n_tables, int table_ld, int page_size, const uint8_t* cache,
                                  const float* cache_scale, int64_t num_slots, float* scores,
                                  int64_t ld, int32_t* status, logits_stream_t stream) {
  return logits::launch(q, w, rows, heads, dim, lens, max_len, group_rows, group_table, block_table,
                        n_tables, table_ld, page_size, cache, cache_scale, num_slots, scores, ld,
                        status, reinterpret_cast<cudaStream_t>(stream), logits::kWaitNs);
}
