// cpkv_plan_build_noalloc: the compose plan for callers that cannot allocate
// device memory.
//
// cpkv_plan_build takes its workspace from the caller.  Some callers have no
// way to provide one: a plugin or extension that runs inside a host
// framework whose caching allocator owns all device memory (a raw cudaMalloc
// there would bypass the framework's accounting, and cudaMalloc / cudaFree
// synchronise the device, stalling the pipeline the plugin runs in), or a
// serving process that reserved nearly all of HBM for its KV cache pool up
// front, so that any later allocation outside the pool can fail.  This entry
// point gives them the same plan without any allocation: its workspace is a
// fixed array in device memory that belongs to the library (64 KiB per GPU,
// held from the library's load until the process exits).
//
// Set-up: on its first call on a device, with that device current, the
// entry point looks up the array's device address (cudaGetSymbolAddress) and
// keeps it for that device; later calls on that device reuse it.  That first
// call should come before any stream capture on the device.
// Every call on a device shares the one array, which keeps what the last
// call left there.  Nothing in it has to start at zero (a call reads only
// entries it wrote itself), but two calls whose kernels overlap on the GPU
// (streams with no order between them) race on it and may build wrong plans.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "cpkv.h"

namespace {

constexpr int64_t kScratchBytes = 64 * 1024;  // the largest workspace this entry point takes
constexpr int kMaxDevices = 64;

// The shared workspace.  In host code this name is only a host-side stand-in
// for the device array: its device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) int32_t plan_scratch[kScratchBytes / sizeof(int32_t)];

std::mutex scratch_mutex;
void *scratch_ptr[kMaxDevices] = {};

// Device address of plan_scratch on the current device (looked up once per
// device), or nullptr when the device cannot be queried or the lookup fails.
void *scratch_address() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    (void)cudaGetLastError();
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(scratch_mutex);
  if (scratch_ptr[dev] == nullptr) {
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, plan_scratch) != cudaSuccess) {
      (void)cudaGetLastError();
      return nullptr;
    }
    scratch_ptr[dev] = ptr;
  }
  return scratch_ptr[dev];
}

}  // namespace

extern "C" int cpkv_plan_build_noalloc(int B, int page_size, int cp_size, int64_t num_pool_pages,
                                       const int32_t *h_prefix_lens, const int32_t *h_cur_lens,
                                       const int32_t *d_prefix_pages, const int32_t *d_cur_pages,
                                       const int32_t *d_writer, int64_t dense_cap_pages, int32_t *d_prefix_spans,
                                       int32_t *d_cur_spans, int32_t *d_owner, int32_t *d_src,
                                       int32_t *d_page_inverse, int32_t *d_staging_page_inverse,
                                       int64_t *d_mixed_locs, int64_t *d_staging_rows, int32_t *d_token_writer_row,
                                       int32_t *d_status, cpkv_stream_t stream) {
  int64_t need = 0;
  const int rc = cpkv_plan_workspace_bytes(B, page_size, cp_size, h_cur_lens, &need);
  if (rc != CPKV_OK) return rc;
  if (need > kScratchBytes) return CPKV_ERR_LIMIT;  // the batch needs more than the fixed workspace
  void *scratch = nullptr;
  if (need > 0) {
    scratch = scratch_address();
    if (scratch == nullptr) return CPKV_ERR_CUDA;
  }
  // Every workspace entry that the plan reads is written earlier in the same
  // call, so what a previous call left in the array needs no clearing.
  return cpkv_plan_build(B, page_size, cp_size, num_pool_pages, h_prefix_lens, h_cur_lens, d_prefix_pages,
                         d_cur_pages, d_writer, dense_cap_pages, d_prefix_spans, d_cur_spans, d_owner, d_src,
                         d_page_inverse, d_staging_page_inverse, d_mixed_locs, d_staging_rows, d_token_writer_row,
                         scratch, kScratchBytes, d_status, stream);
}
