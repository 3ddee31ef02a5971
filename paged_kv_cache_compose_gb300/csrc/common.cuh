// Shared helpers of the cpkv CUDA library (sm_103a): status reporting,
// 16-byte streaming loads/stores, mbarrier + bulk-copy (TMA) wrappers,
// block scans and host-side launch plumbing.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "cpkv.h"

#define CPKV_DEV __device__ __forceinline__

namespace cpkv {

// ---------------------------------------------------------------------------
// status word
// ---------------------------------------------------------------------------
CPKV_DEV void raise_status(int32_t *status, int32_t bits) { atomicOr(status, bits); }

// ---------------------------------------------------------------------------
// 16-byte streaming memory ops
// ---------------------------------------------------------------------------
CPKV_DEV uint4 ld_stream16(const void *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

CPKV_DEV void st_stream16(void *p, uint4 v) {
  asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

// L2 eviction-priority policies (createpolicy) and 16-byte ops that carry one.
// Data read or written exactly once is marked evict_first so it does not push
// out lines that the next kernel still needs (the staging written by the fill
// and read by the gather).
CPKV_DEV uint64_t l2_policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

CPKV_DEV uint64_t l2_policy_evict_last() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

CPKV_DEV uint4 ld_stream16_hint(const void *p, uint64_t pol) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p), "l"(pol));
  return v;
}

CPKV_DEV void st16_hint(void *p, uint4 v, uint64_t pol) {
  asm volatile("st.global.L1::no_allocate.L2::cache_hint.v4.u32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(p), "r"(v.x),
               "r"(v.y), "r"(v.z), "r"(v.w), "l"(pol)
               : "memory");
}

// ---------------------------------------------------------------------------
// shared-memory addresses, mbarriers and bulk async copies (TMA, non-tensor)
// ---------------------------------------------------------------------------
CPKV_DEV uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

CPKV_DEV void mbar_init(uint64_t *bar, uint32_t arrivals) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(arrivals)
               : "memory");
}

// Make mbarrier initialisation visible to the async (TMA) proxy.
CPKV_DEV void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Make generic-proxy shared-memory writes visible to the async proxy.
CPKV_DEV void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

CPKV_DEV void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

CPKV_DEV bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

CPKV_DEV uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait on an mbarrier phase: gives up (returns false) once
// `limit_ns` nanoseconds have passed.
CPKV_DEV bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > limit_ns) return false;
  }
  return true;
}

// global -> shared bulk copy, completion signalled on `bar` (complete_tx).
CPKV_DEV void bulk_load_g2s(void *smem_dst, const void *gsrc, uint32_t bytes, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(smem_dst)),
      "l"(gsrc), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// shared -> global bulk copy, tracked by the bulk async-group mechanism.
CPKV_DEV void bulk_store_s2g(void *gdst, const void *smem_src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst),
               "r"(smem_addr(smem_src)), "r"(bytes)
               : "memory");
}

// The same two copies with an L2 cache policy.
CPKV_DEV void bulk_load_g2s_hint(void *smem_dst, const void *gsrc, uint32_t bytes, uint64_t *bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_addr(smem_dst)),
      "l"(gsrc), "r"(bytes), "r"(smem_addr(bar)), "l"(pol)
      : "memory");
}

CPKV_DEV void bulk_store_s2g_hint(void *gdst, const void *smem_src, uint32_t bytes, uint64_t pol) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group.L2::cache_hint [%0], [%1], %2, %3;" ::"l"(gdst),
               "r"(smem_addr(smem_src)), "r"(bytes), "l"(pol)
               : "memory");
}

CPKV_DEV void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Wait until at most N committed bulk groups still read shared memory.
template <int N>
CPKV_DEV void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

CPKV_DEV void bulk_wait_read_dyn(int n) {
  switch (n) {
    case 0: bulk_wait_read<0>(); break;
    case 1: bulk_wait_read<1>(); break;
    case 2: bulk_wait_read<2>(); break;
    case 3: bulk_wait_read<3>(); break;
    case 4: bulk_wait_read<4>(); break;
    case 5: bulk_wait_read<5>(); break;
    case 6: bulk_wait_read<6>(); break;
    default: bulk_wait_read<7>(); break;
  }
}

// Wait until every committed bulk group has completed (writes visible).
CPKV_DEV void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

CPKV_DEV int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }

// ---------------------------------------------------------------------------
// programmatic dependent launch
// ---------------------------------------------------------------------------
// A kernel launched with programmatic stream serialization (launch_kernel
// with dependent = true) may start before the previous kernel on the stream
// has finished: as soon as every CTA of that kernel has run
// release_dependents() or exited.  wait_prerequisite() returns once the
// previous kernel has completed and its memory writes are visible; in a
// kernel not launched that way it returns at once.
CPKV_DEV void release_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

CPKV_DEV void wait_prerequisite() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Once per thread (`open` starts false): wait_prerequisite() before the
// thread's first global store, so that an early-launched kernel orders every
// write after the previous kernel while its loads may run ahead.
CPKV_DEV void store_gate(bool *open) {
  if (!*open) {
    wait_prerequisite();
    *open = true;
  }
}

// ---------------------------------------------------------------------------
// scans
// ---------------------------------------------------------------------------
template <typename T>
CPKV_DEV T warp_inclusive_scan(T x) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    T y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  return x;
}

// Exclusive scan over the block (blockDim.x a multiple of 32, <= 1024).
// `scratch` is shared memory of >= 33 elements.  Returns the exclusive
// prefix of `v`; *total receives the block sum.  Contains __syncthreads().
template <typename T>
CPKV_DEV T block_exclusive_scan(T v, T *scratch, T *total) {
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int nwarps = blockDim.x >> 5;
  T inc = warp_inclusive_scan(v);
  if (lane == 31) scratch[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    T w = lane < nwarps ? scratch[lane] : T(0);
    w = warp_inclusive_scan(w);
    scratch[lane] = w;
  }
  __syncthreads();
  T before = warp > 0 ? scratch[warp - 1] : T(0);
  *total = scratch[nwarps - 1];
  __syncthreads();
  return before + inc - v;
}

// Largest index b in [0, n) with a[b] <= x, for non-decreasing a (a[0] <= x).
template <typename T>
CPKV_DEV int upper_index(const T *a, int n, T x) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (a[mid] <= x) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
// Number of SMs of the current device (cached per device; thread-safe).
int device_sm_count();

// Raise `kernel`'s dynamic shared-memory limit to `bytes` on the current
// device, once per device and kernel (thread-safe).  CPKV_OK or CPKV_ERR_CUDA.
int ensure_dynamic_smem(const void *kernel, int bytes);

// One-dimensional grid for a persistent kernel of `threads`-thread CTAs with
// `smem` bytes of dynamic shared memory: the SM count times the CTAs that stay
// resident on one SM (occupancy calculator, cached per device, kernel and
// size), at most `cap_per_sm` CTAs per SM, at most `units` CTAs, at least 1.
int persistent_grid(const void *kernel, int threads, size_t smem, int cap_per_sm, int64_t units);

// Map the last launch error to CPKV_ERR_CUDA.
inline int launch_status() {
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? CPKV_OK : CPKV_ERR_CUDA;
}

// Launch a kernel that takes one parameter block by value, as a programmatic
// dependent of the previous kernel on `s` when `dependent` is set (see
// release_dependents / wait_prerequisite).  CPKV_OK or CPKV_ERR_CUDA.
template <typename Params>
int launch_kernel(void (*kernel)(Params), dim3 grid, dim3 block, size_t smem, bool dependent, cudaStream_t s,
                  const Params &prm) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = dependent ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kernel, prm) != cudaSuccess) {
    (void)cudaGetLastError();
    return CPKV_ERR_CUDA;
  }
  return launch_status();
}

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Most one-warp bulk-ring CTAs per SM for pages of a single `piece_bytes`
// piece: enough to keep about 56 KB of loads in flight per SM
// (`loads_in_flight` pieces per CTA), at least `floor_cap`, at most 32.
// Measured: 1152-byte pages (one 576xbf16 token) go from 218 to 53 us per
// traced-batch gather when the cap rises from 3 to 24; 8448-byte pages are
// best at 3.
inline int ring_cap_one_piece(int64_t piece_bytes, int loads_in_flight, int floor_cap) {
  const int64_t per_cta = (int64_t)loads_in_flight * (piece_bytes > 0 ? piece_bytes : 1);
  int64_t cap = (int64_t)(56 * 1024) / per_cta;
  if (cap < floor_cap) cap = floor_cap;
  return cap > 32 ? 32 : (int)cap;
}

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Whether an early (programmatic dependent) launch of a persistent grid of
// `grid` one-warp CTAs pays: only when it runs at most 4 CTAs per SM.  There
// its CTAs start in the room the previous kernel leaves and overlap that
// kernel's tail (traced pages, 3-4 per SM: fused 4.05 -> 3.81 ms per step;
// index-key pages, 3 per SM: fused 3.947 -> 3.700 ms).  With many small CTAs
// per SM (one-token pages, 24) the early CTAs crowd the previous kernel's
// tail and the step got slower (fused 4.27 -> 4.70 ms).  The grouped
// small-page kernels (8 KB groups, 6-8 CTAs per SM) do not ask: they launch
// early whenever the caller allows it, which measured faster for all three.
inline bool early_launch_pays(int grid) { return grid <= 4 * device_sm_count(); }

}  // namespace cpkv
