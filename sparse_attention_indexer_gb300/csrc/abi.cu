// C ABI of the library: argument checks, launch configuration and the status word.
// Every entry point is declared (with its contract) in include/topk_paged.h.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "common.cuh"

namespace topk {
cudaError_t launch_plan(const int32_t* lens, int rows, int max_len, int grid, int chunk_force,
                        void* ws, cudaStream_t stream);
int plan_host(const int32_t* lens, int rows, int max_len, int grid, int chunk_force, char* ws);
cudaError_t launch_select(const SelectParams& p, int grid, cudaStream_t stream);
size_t select_smem_bytes();
const void* select_kernel_ptr();
int short_max_len();
cudaError_t launch_short(const SelectParams& p, cudaStream_t stream);
int medium_max_len();
cudaError_t launch_medium(const SelectParams& p, int sms, cudaStream_t stream);
cudaError_t launch_rowcluster(const SelectParams& p, cudaStream_t stream);
}  // namespace topk

using namespace topk;

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int g_grid[kMaxDevices];  // 0 = not yet queried, < 0 = error code

// Persistent grid of the current device: co-resident CTAs of the select kernel.
int device_grid(int* grid) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return TOPK_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_grid[dev] == 0) {
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return TOPK_ERR_CUDA;
    if (!(prop.major == 10 && prop.minor == 3) || !prop.cooperativeLaunch) {
      g_grid[dev] = TOPK_ERR_DEVICE;
    } else {
      const size_t smem = select_smem_bytes();
      if (cudaFuncSetAttribute(select_kernel_ptr(), cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)smem) != cudaSuccess)
        return TOPK_ERR_CUDA;
      int per_sm = 0;
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, select_kernel_ptr(), kThreads,
                                                        smem) != cudaSuccess)
        return TOPK_ERR_CUDA;
      int g = per_sm * prop.multiProcessorCount;
      if (g > kMaxGrid) g = kMaxGrid;
      g_grid[dev] = g > 0 ? g : TOPK_ERR_DEVICE;
    }
  }
  if (g_grid[dev] < 0) return g_grid[dev];
  *grid = g_grid[dev];
  return TOPK_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Workspaces whose latest plan had a forced chunk (topk_plan_ex). A select on one of
// them runs the work-list kernel where an unforced plan would take the cluster path,
// so that a forced chunk still drives the rows through the multi-CTA path. Results
// never depend on it: the cluster kernel needs only the plan's header, which every
// plan writes.
constexpr int kForcedSlots = 64;
std::mutex g_forced_mu;
const void* g_forced[kForcedSlots];
int g_forced_next;

void note_plan(const void* ws, bool forced) {
  std::lock_guard<std::mutex> lk(g_forced_mu);
  for (int i = 0; i < kForcedSlots; ++i)
    if (g_forced[i] == ws) {
      if (!forced) g_forced[i] = nullptr;
      return;
    }
  if (forced) {
    g_forced[g_forced_next] = ws;
    g_forced_next = (g_forced_next + 1) % kForcedSlots;
  }
}

bool plan_forced(const void* ws) {
  std::lock_guard<std::mutex> lk(g_forced_mu);
  for (int i = 0; i < kForcedSlots; ++i)
    if (g_forced[i] == ws) return true;
  return false;
}

int plan_common(const int32_t* lens, int rows, int max_len, int chunk, void* ws, size_t ws_bytes,
                cudaStream_t stream) {
  if (rows < 0) return TOPK_ERR_ROWS;
  if (!ws || (rows > 0 && !lens)) return TOPK_ERR_NULL;
  if (max_len < 0) return TOPK_ERR_MAX_LEN;
  if (chunk != 0 && (chunk < kChunkAlign || chunk > kChunkCap)) return TOPK_ERR_CHUNK;
  if (!aligned(ws, 256) || ws_bytes < topk_workspace_bytes(rows, max_len)) return TOPK_ERR_WORKSPACE;
  int grid = 0;
  const int e = device_grid(&grid);
  if (e != TOPK_OK) return e;
  if ((int64_t)max_len > (int64_t)grid * kChunkCap) return TOPK_ERR_MAX_LEN;
  if (launch_plan(lens, rows, max_len, grid, chunk, ws, stream) != cudaSuccess) return TOPK_ERR_CUDA;
  note_plan(ws, chunk != 0);
  return TOPK_OK;
}

int select_common(const float* scores, int64_t ld, const int32_t* lens, int rows, int max_len,
                  int k, const int32_t* block_table, int64_t table_ld,
                  const int32_t* row_to_table, int page_size, int32_t* out_slots,
                  int32_t* out_pos, void* workspace, cudaStream_t stream, uint64_t wait_ns,
                  int skip_cta) {
  if (rows < 0) return TOPK_ERR_ROWS;
  if (k < 1 || k > TOPK_MAX_K) return TOPK_ERR_K;
  if (page_size < 1) return TOPK_ERR_PAGE_SIZE;
  if (max_len < 0) return TOPK_ERR_MAX_LEN;
  if (ld < max_len || table_ld < 1) return TOPK_ERR_LD;
  if (!workspace) return TOPK_ERR_NULL;
  if (rows == 0) return TOPK_OK;
  if (!scores || !lens || !block_table || !out_slots) return TOPK_ERR_NULL;
  if (!aligned(scores, 4) || !aligned(out_slots, 4) || (out_pos && !aligned(out_pos, 4)) ||
      !aligned(lens, 4) || !aligned(block_table, 4) || (row_to_table && !aligned(row_to_table, 4)))
    return TOPK_ERR_ALIGN;
  if (!aligned(workspace, 256)) return TOPK_ERR_WORKSPACE;
  int grid = 0;
  const int e = device_grid(&grid);
  if (e != TOPK_OK) return e;
  if ((int64_t)max_len > (int64_t)grid * kChunkCap) return TOPK_ERR_MAX_LEN;
  SelectParams p;
  p.scores = scores;
  p.ld = ld;
  p.lens = lens;
  p.rows = rows;
  p.max_len = max_len;
  p.k = k;
  p.table = block_table;
  p.table_ld = table_ld;
  p.row_to_table = row_to_table;
  p.page_size = page_size;
  p.out_slots = out_slots;
  p.out_pos = out_pos;
  p.ws = static_cast<char*>(workspace);
  p.wait_ns = wait_ns;
  p.skip_cta = skip_cta;
  // Batches of short rows take the register-resident path (one warp per row), batches
  // of medium rows the medium path (one CTA per row, several per SM), and a few long
  // rows the cluster path (one thread-block cluster per row) unless the plan forced a
  // chunk; the plan's header is still checked there. `grid` is one CTA per SM.
  if (max_len <= short_max_len()) return launch_short(p, stream) == cudaSuccess ? TOPK_OK : TOPK_ERR_CUDA;
  if (max_len <= medium_max_len())
    return launch_medium(p, grid, stream) == cudaSuccess ? TOPK_OK : TOPK_ERR_CUDA;
  if (cluster_batch(rows, max_len, grid) && !plan_forced(workspace))
    return launch_rowcluster(p, stream) == cudaSuccess ? TOPK_OK : TOPK_ERR_CUDA;
  if (launch_select(p, grid, stream) != cudaSuccess) return TOPK_ERR_CUDA;
  return TOPK_OK;
}

}  // namespace

extern "C" {

size_t topk_workspace_bytes(int rows, int max_len) {
  if (rows < 0 || max_len < 0) return 0;
  return make_layout(rows).total;
}

int topk_chunk_capacity(void) { return kChunkCap; }

int topk_grid_size(void) {
  int grid = 0;
  const int e = device_grid(&grid);
  return e == TOPK_OK ? grid : e;
}

int64_t topk_max_row_len(void) {
  int grid = 0;
  const int e = device_grid(&grid);
  return e == TOPK_OK ? (int64_t)grid * kChunkCap : (int64_t)e;
}

int topk_plan(const int32_t* lens, int rows, int max_len, void* workspace, size_t ws_bytes,
              topk_stream_t stream) {
  return plan_common(lens, rows, max_len, 0, workspace, ws_bytes, (cudaStream_t)stream);
}

int topk_plan_ex(const int32_t* lens, int rows, int max_len, int chunk, void* workspace,
                 size_t ws_bytes, topk_stream_t stream) {
  return plan_common(lens, rows, max_len, chunk, workspace, ws_bytes, (cudaStream_t)stream);
}

int topk_select_paged(const float* scores, int64_t ld, const int32_t* lens, int rows, int max_len,
                      int k, const int32_t* block_table, int64_t table_ld,
                      const int32_t* row_to_table, int page_size, int32_t* out_slots,
                      int32_t* out_pos, void* workspace, topk_stream_t stream) {
  return select_common(scores, ld, lens, rows, max_len, k, block_table, table_ld, row_to_table,
                       page_size, out_slots, out_pos, workspace, (cudaStream_t)stream, kWaitNs, -1);
}

// Test entry: topk_select_paged with a bounded-wait limit in nanoseconds (0: the
// default 200 ms) and one CTA (skip_cta >= 0) that never arrives at its first row
// barrier, so that the waits of the row it serves run out.
int topk_select_paged_test(const float* scores, int64_t ld, const int32_t* lens, int rows,
                           int max_len, int k, const int32_t* block_table, int64_t table_ld,
                           const int32_t* row_to_table, int page_size, int32_t* out_slots,
                           int32_t* out_pos, void* workspace, topk_stream_t stream,
                           uint64_t wait_ns, int skip_cta) {
  return select_common(scores, ld, lens, rows, max_len, k, block_table, table_ld, row_to_table,
                       page_size, out_slots, out_pos, workspace, (cudaStream_t)stream,
                       wait_ns ? wait_ns : kWaitNs, skip_cta);
}

int topk_read_status(const void* workspace, topk_stream_t stream, int* status) {
  if (!workspace || !status) return TOPK_ERR_NULL;
  const Header* h = static_cast<const Header*>(workspace);
  int v = 0;
  if (cudaMemcpyAsync(&v, &h->status, sizeof(int), cudaMemcpyDeviceToHost,
                      (cudaStream_t)stream) != cudaSuccess)
    return TOPK_ERR_CUDA;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return TOPK_ERR_CUDA;
  *status = v;
  return TOPK_OK;
}

int topk_clear_status(void* workspace, topk_stream_t stream) {
  if (!workspace) return TOPK_ERR_NULL;
  Header* h = static_cast<Header*>(workspace);
  if (cudaMemsetAsync(&h->status, 0, sizeof(int), (cudaStream_t)stream) != cudaSuccess)
    return TOPK_ERR_CUDA;
  return TOPK_OK;
}

const char* topk_status_str(int code) {
  switch (code) {
    case TOPK_OK: return "ok";
    case TOPK_ERR_NULL: return "a required pointer is NULL";
    case TOPK_ERR_ROWS: return "rows < 0";
    case TOPK_ERR_K: return "k outside [1, 2048]";
    case TOPK_ERR_PAGE_SIZE: return "page_size < 1";
    case TOPK_ERR_LD: return "ld < max_len or table_ld < 1";
    case TOPK_ERR_WORKSPACE: return "workspace too small or not 256-byte aligned";
    case TOPK_ERR_MAX_LEN: return "max_len negative or above the supported row length";
    case TOPK_ERR_ALIGN: return "a pointer is not 4-byte aligned";
    case TOPK_ERR_CUDA: return "a CUDA runtime call failed";
    case TOPK_ERR_DEVICE: return "the current device cannot run the kernels (needs sm_103)";
    case TOPK_ERR_CHUNK: return "forced chunk outside [16, chunk capacity]";
    case TOPK_ERR_STATIC_ROWS: return "rows above TOPK_STATIC_MAX_ROWS (64) for the no-allocation entry point";
    default: break;
  }
  if (code > 0) {
    // Single bits get a name; combinations are described generically.
    switch (code) {
      case TOPK_STATUS_LEN: return "device: a row length is outside [0, max_len]";
      case TOPK_STATUS_TABLE_WIDTH: return "device: a row needs more pages than table_ld";
      case TOPK_STATUS_TABLE_ENTRY: return "device: a selected position maps to a negative page";
      case TOPK_STATUS_SLOT_OVERFLOW: return "device: a slot exceeds INT32_MAX";
      case TOPK_STATUS_TIMEOUT: return "device: a bounded cross-CTA wait expired";
      case TOPK_STATUS_PLAN_MISMATCH: return "device: the plan does not match the call";
      case TOPK_STATUS_ORDER: return "device: a row barrier found a CTA already past it";
      default: return "device: several status bits are set";
    }
  }
  return "unknown code";
}

// Host reference of the planner, for inspection and tests: writes the header, row
// info, single-row list and unit table of a plan for `grid` CTAs into `ws_image`
// (host memory of at least topk_workspace_bytes(rows, max_len) bytes). No CUDA call.
int topk_plan_host(const int32_t* lens, int rows, int max_len, int grid, int chunk,
                   void* ws_image, size_t ws_bytes) {
  if (rows < 0) return TOPK_ERR_ROWS;
  if (!ws_image || (rows > 0 && !lens)) return TOPK_ERR_NULL;
  if (max_len < 0) return TOPK_ERR_MAX_LEN;
  if (grid < 1 || grid > kMaxGrid) return TOPK_ERR_DEVICE;
  if (chunk != 0 && (chunk < kChunkAlign || chunk > kChunkCap)) return TOPK_ERR_CHUNK;
  if (ws_bytes < topk_workspace_bytes(rows, max_len)) return TOPK_ERR_WORKSPACE;
  if ((int64_t)max_len > (int64_t)grid * kChunkCap) return TOPK_ERR_MAX_LEN;
  plan_host(lens, rows, max_len, grid, chunk, static_cast<char*>(ws_image));
  return TOPK_OK;
}

// Layout constants of the workspace and kernels, for tools and tests:
// [0] kMaxGrid, [1] kMaxWaves, [2] kChunkCap, [3] header bytes, then byte offsets for
// `rows` rows of [4] row info, [5] single rows, [6] first-single table, [7] unit
// table, [8] group states; [9] threads per CTA, [10] kGroupCap, [11] kListCap.
int topk_layout_info(int rows, int64_t* out, int n) {
  if (!out || rows < 0) return TOPK_ERR_NULL;
  const Layout l = make_layout(rows);
  const int64_t v[12] = {kMaxGrid,
                         kMaxWaves,
                         kChunkCap,
                         (int64_t)sizeof(Header),
                         (int64_t)l.rowinfo,
                         (int64_t)l.singles,
                         (int64_t)l.first_single,
                         (int64_t)l.units,
                         (int64_t)l.groups,
                         kThreads,
                         kGroupCap,
                         kListCap};
  for (int i = 0; i < n && i < 12; ++i) out[i] = v[i];
  return TOPK_OK;
}

}  // extern "C"
