// cpkv_selftest_ring_timeout: exercises the bounded wait of the bulk-copy
// ring (bulk_ring.cuh) on the GPU without a fault.  One warp arms stage 0 of
// a ring for a 16-byte load that is never issued (an mbarrier phase nothing
// completes) and drains the ring: consume() gives up after the ring's time
// limit, raises CPKV_STATUS_TIMEOUT and stores nothing; the kernel returns
// normally and the context stays usable.
#include <stdint.h>

#include "bulk_ring.cuh"

namespace cpkv {
namespace {

__global__ void __launch_bounds__(32) ring_timeout_kernel(uint8_t *dst, int32_t *status) {
  __shared__ __align__(128) uint8_t stages[4 * 16];
  __shared__ __align__(8) uint64_t full[4];
  __shared__ uint8_t *ring_dst[4];
  __shared__ uint32_t ring_bytes[4];
  __shared__ int ring_live[4];
  BulkRing<4, 2> ring;
  ring.init(stages, full, ring_dst, ring_bytes, ring_live, status, 16);
  if ((threadIdx.x & 31) == 0) {
    // stage 0 now waits for 16 bytes that no copy will deliver
    ring_dst[0] = dst;
    ring_bytes[0] = 16;
    ring_live[0] = 1;
    mbar_arrive_expect_tx(&full[0], 16);
  }
  __syncwarp();
  ring.tail = 1;  // as if one load had been pushed
  ring.drain();
}

}  // namespace
}  // namespace cpkv

extern "C" int cpkv_selftest_ring_timeout(void *d_dst16, int32_t *d_status, cpkv_stream_t stream) {
  using namespace cpkv;
  if (d_dst16 == nullptr || d_status == nullptr || !aligned16(d_dst16)) return CPKV_ERR_ARG;
  ring_timeout_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(static_cast<uint8_t *>(d_dst16),
                                                                           d_status);
  return launch_status();
}
