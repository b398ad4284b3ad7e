// Entry point that plans and selects with a scratch area of fixed size that lives in
// the library's own device image, for callers that cannot hand the library device
// memory. Two kinds of caller need it: a plain C host with no device allocator of
// its own, and a plug-in inside a serving engine that has already reserved all free
// device memory for its KV cache, where a cudaMalloc fails. Even where an
// allocation would succeed, cudaMalloc/cudaFree synchronize the device and would
// stall the other streams of a decode step. The scratch array is allocated when the
// module is loaded; this entry point performs no allocation of its own.
//
// The computation is the one of topk_plan followed by topk_select_paged on the same
// stream; the scratch array plays the workspace.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "common.cuh"
#include "topk_paged.h"

using namespace topk;

// Scratch for one planned batch: header, per-row info, single-row list, unit table
// and the group states of up to TOPK_STATIC_MAX_ROWS multi-CTA rows. Every file-
// scope __device__ object starts zeroed; what a call needs at zero (the group
// states' barrier flags, histograms and candidate counters, the ticket counter and
// the status word) is cleared again by the planning kernel on every call.
static __device__ __align__(256) unsigned char g_static_scratch[TOPK_STATIC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch[kMaxDevices];  // device address of g_static_scratch, per device

// Address of the scratch array on the current device, looked up once per device with
// that device current. cudaGetSymbolAddress may load the module on first use.
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return TOPK_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) return TOPK_ERR_CUDA;
    if (reinterpret_cast<uintptr_t>(p) % 256 != 0) return TOPK_ERR_WORKSPACE;
    g_scratch[dev] = p;
  }
  *out = g_scratch[dev];
  return TOPK_OK;
}

bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3) == 0; }

}  // namespace

extern "C" int topk_select_paged_noalloc(const float* scores, int64_t ld, const int32_t* lens,
                                         int rows, int max_len, int k,
                                         const int32_t* block_table, int64_t table_ld,
                                         const int32_t* row_to_table, int page_size,
                                         int32_t* out_slots, int32_t* out_pos, int32_t* status,
                                         topk_stream_t stream) {
  // Every argument error is found before anything is enqueued.
  if (rows < 0) return TOPK_ERR_ROWS;
  if (rows > TOPK_STATIC_MAX_ROWS) return TOPK_ERR_STATIC_ROWS;
  if (k < 1 || k > TOPK_MAX_K) return TOPK_ERR_K;
  if (page_size < 1) return TOPK_ERR_PAGE_SIZE;
  if (max_len < 0) return TOPK_ERR_MAX_LEN;
  if (ld < max_len || table_ld < 1) return TOPK_ERR_LD;
  if (rows > 0 && (!scores || !lens || !block_table || !out_slots)) return TOPK_ERR_NULL;
  if (!aligned4(scores) || !aligned4(lens) || !aligned4(block_table) || !aligned4(out_slots) ||
      !aligned4(out_pos) || !aligned4(row_to_table) || !aligned4(status))
    return TOPK_ERR_ALIGN;
  const size_t need = topk_workspace_bytes(rows, max_len);
  if (need == 0 || need > TOPK_STATIC_SCRATCH_BYTES) return TOPK_ERR_STATIC_ROWS;
  void* ws = nullptr;
  int e = scratch_address(&ws);
  if (e != TOPK_OK) return e;
  const int64_t max_row = topk_max_row_len();
  if (max_row <= 0) return (int)max_row;
  if ((int64_t)max_len > max_row) return TOPK_ERR_MAX_LEN;
  if (rows == 0) {
    if (status && cudaMemsetAsync(status, 0, sizeof(int32_t), (cudaStream_t)stream) != cudaSuccess)
      return TOPK_ERR_CUDA;
    return TOPK_OK;
  }
  e = topk_plan(lens, rows, max_len, ws, TOPK_STATIC_SCRATCH_BYTES, stream);
  if (e != TOPK_OK) return e;
  e = topk_select_paged(scores, ld, lens, rows, max_len, k, block_table, table_ld, row_to_table,
                        page_size, out_slots, out_pos, ws, stream);
  if (e != TOPK_OK) return e;
  if (status) {
    const Header* h = static_cast<const Header*>(ws);
    if (cudaMemcpyAsync(status, &h->status, sizeof(int32_t), cudaMemcpyDeviceToDevice,
                        (cudaStream_t)stream) != cudaSuccess)
      return TOPK_ERR_CUDA;
  }
  return TOPK_OK;
}
