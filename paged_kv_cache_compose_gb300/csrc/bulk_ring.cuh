// A single-warp ring of bulk async copies (TMA, non-tensor form) through
// shared memory: global -> shared with mbarrier completion, shared -> global
// as bulk groups.  Shared by the page gather, the fill and the fused compose.
//
// kStages shared-memory stages of `piece_bytes` each; at most kLoads loads in
// flight, so kStages - kLoads stages hold stores that are still draining and
// loads overlap stores.  Lane 0 issues every copy; the other lanes only take
// part in the warp-uniform bookkeeping.  Loads carry an L2 evict_first policy
// (each byte is read once); stores too, unless the caller keeps them in L2
// for the next kernel.  Waits on the mbarriers are
// bounded by a time limit: on a timeout the ring raises
// CPKV_STATUS_TIMEOUT, stops issuing and still waits (bounded) for every load
// it issued before the CTA may exit.
//
// kDiscard: a push may mark its source as dead after the copy.  Once that
// load has landed in shared memory, the warp drops the source's L2 lines
// (`discard.global.L2`, the 128-byte lines that lie wholly inside the piece)
// so that dirty data nobody reads again is never written back to DRAM; the
// source bytes are undefined afterwards.
#pragma once

#include "common.cuh"

namespace cpkv {

constexpr uint64_t kRingWaitLimitNs = 2000000000ull;  // 2 s; a piece lands in microseconds

// Drop the L2 lines that lie wholly inside [src, src + bytes) without
// writing them back (warp-uniform call; the bytes become undefined).
// Invariant of every consuming caller: a discarded staging line reverts to
// whatever DRAM last held, so each staging byte that a later read sees (a
// staged row, a pad row, a lane-copied plane slice) must be rewritten before
// that read.  The fills write every row of a current page and zero every pad
// row after a request's last token; a fill that skipped any of them would
// leak stale DRAM bytes into the next dense buffer.
CPKV_DEV void warp_discard_l2(const uint8_t *src, uint32_t bytes) {
  const uintptr_t first = (reinterpret_cast<uintptr_t>(src) + 127) & ~static_cast<uintptr_t>(127);
  const uintptr_t end = (reinterpret_cast<uintptr_t>(src) + bytes) & ~static_cast<uintptr_t>(127);
  for (uintptr_t a = first + 128 * (uintptr_t)(threadIdx.x & 31); a < end; a += 32 * 128)
    asm volatile("discard.global.L2 [%0], 128;" ::"l"(a) : "memory");
}

template <int kStages, int kLoads, bool kDiscard = false>
struct BulkRing {
  static_assert(kLoads >= 1 && kLoads <= kStages && kStages <= 8, "ring shape");
  uint8_t *smem;          // kStages * piece_bytes of dynamic shared memory
  uint64_t *full;         // kStages mbarriers (shared)
  uint8_t **ring_dst;     // kStages destinations (shared)
  uint32_t *ring_bytes;   // kStages sizes (shared)
  int *ring_live;         // kStages flags: a load was issued into the stage (shared)
  const uint8_t **ring_src;  // kDiscard: kStages sources to drop from L2 once loaded, or nullptr (shared)
  int32_t *status;
  int32_t piece_bytes;
  int64_t head, tail;     // consumed / issued (warp-uniform)
  bool dead;              // lane 0: a bounded wait gave up
  uint64_t load_policy, store_policy;

  // keep_stores: stores get L2 evict_last (the next kernel reads them back)
  // instead of evict_first.
  CPKV_DEV void init(uint8_t *smem_, uint64_t *full_, uint8_t **dst_, uint32_t *bytes_, int *live_,
                     int32_t *status_, int32_t piece_bytes_, bool keep_stores = false,
                     const uint8_t **src_ = nullptr) {
    smem = smem_; full = full_; ring_dst = dst_; ring_bytes = bytes_; ring_live = live_; ring_src = src_;
    status = status_; piece_bytes = piece_bytes_;
    head = tail = 0;
    dead = false;
    load_policy = l2_policy_evict_first();
    store_policy = keep_stores ? l2_policy_evict_last() : load_policy;
    if ((threadIdx.x & 31) == 0) {
      for (int s = 0; s < kStages; ++s) mbar_init(&full[s], 1);
      fence_barrier_init();
    }
    __syncwarp();
  }

  // Wait for the oldest load and store it (warp-uniform call).
  CPKV_DEV void consume() {
    const int s = (int)(head % kStages);
    bool landed = false;
    if ((threadIdx.x & 31) == 0) {
      const uint32_t parity = (uint32_t)((head / kStages) & 1);
      if (ring_live[s]) {
        landed = mbar_wait_bounded(&full[s], parity, kRingWaitLimitNs);
        if (!landed && !dead) {
          dead = true;
          raise_status(status, CPKV_STATUS_TIMEOUT);
        }
      }
      if (landed && !dead) bulk_store_s2g_hint(ring_dst[s], smem + (size_t)s * piece_bytes, ring_bytes[s], store_policy);
      bulk_commit();
    }
    if (kDiscard) {  // the load has landed: its source may go
      const int drop = __shfl_sync(0xffffffffu, (threadIdx.x & 31) == 0 && landed && !dead ? 1 : 0, 0);
      if (drop && ring_src[s] != nullptr) warp_discard_l2(ring_src[s], ring_bytes[s]);
    }
    ++head;
  }

  // Copy `bytes` (a multiple of 16, <= piece_bytes) from src to dst (warp-uniform call).
  // discard_src (kDiscard rings): drop the source's L2 lines once loaded.
  CPKV_DEV void push(const void *src, void *dst, uint32_t bytes, bool discard_src = false) {
    if (tail - head == kLoads) consume();
    const int s = (int)(tail % kStages);
    if ((threadIdx.x & 31) == 0) {
      // the stage's previous store must have finished reading shared memory
      if (tail >= kStages) bulk_wait_read_dyn((int)(head - tail + kStages - 1));
      ring_live[s] = 0;
      if (kDiscard) ring_src[s] = discard_src ? static_cast<const uint8_t *>(src) : nullptr;
      if (!dead) {
        ring_dst[s] = static_cast<uint8_t *>(dst);
        ring_bytes[s] = bytes;
        ring_live[s] = 1;
        mbar_arrive_expect_tx(&full[s], bytes);
        bulk_load_g2s_hint(smem + (size_t)s * piece_bytes, src, bytes, &full[s], load_policy);
      }
    }
    ++tail;
    __syncwarp();
  }

  // Store everything in flight and wait until the stores are complete.
  CPKV_DEV void drain() {
    while (head < tail) consume();
    if ((threadIdx.x & 31) == 0) bulk_wait_all();
    __syncwarp();
  }
};

// Zero `bytes` (a multiple of 16) at dst with 16-byte stores across the warp.
CPKV_DEV void warp_zero(uint8_t *dst, uint32_t bytes) {
  const uint4 z = make_uint4(0, 0, 0, 0);
  for (uint32_t i = threadIdx.x & 31; i < bytes / 16; i += 32) st_stream16(dst + 16 * (size_t)i, z);
}

// The same with an L2 cache policy on the stores.
CPKV_DEV void warp_zero_hint(uint8_t *dst, uint32_t bytes, uint64_t pol) {
  const uint4 z = make_uint4(0, 0, 0, 0);
  for (uint32_t i = threadIdx.x & 31; i < bytes / 16; i += 32) st16_hint(dst + 16 * (size_t)i, z, pol);
}

}  // namespace cpkv
