// A single-warp ring of page groups for small pages (at most 4 KB): a stage
// holds G consecutive dense pages (G = 8 KB / page bytes, at most 32), lane j
// describing the group's page j.  Shared by the slot-dense gather
// (gather_groups_kernel) and the single-pass compose (compose_fused_groups).
//
// Each page of a group is a copy of `copy` bytes from `src` followed by zero
// bytes up to the page's end, or a zero page (src == nullptr).  Consecutive
// pages whose sources are contiguous within one table entry, every page but
// the last of them whole, form a run that is loaded into the stage with ONE
// bulk copy (page-run merging: a contiguous stretch of a pool, a staging or
// a writer's rows is one copy); zero bytes are written into the stage by the
// warp, followed by a proxy fence; the whole group is stored with ONE bulk
// copy, since dense pages d0 .. d0 + n - 1 are contiguous.  A stage therefore
// holds up to 8 KB, so 6 CTAs per SM keep enough bytes in flight where one
// 1152-byte page per stage needed 24, and the store side issues 8 KB copies.
// Runs never cross table entries, so a consumed staging run (kConsume: its L2
// lines are dropped once loaded) never covers other bytes.  Every mbarrier
// wait is bounded, as in bulk_ring.cuh.
#pragma once

#include "bulk_ring.cuh"

namespace cpkv {

// Ring shape, measured on one-token pages (78-layer traced lengths, ms per
// step for the fill + gather with stagings kept / the fused compose): 4
// stages, 2 loading, 6 CTAs per SM 4.50 / 4.03; 4 stages with 3 loading
// 4.51 / 4.05; 3 stages with 2 or 1 loading and 8 CTAs per SM 4.77 / 4.21
// and 5.07 / 4.04; 2 stages, 12 CTAs per SM 4.76 / 4.09.
constexpr int kGroupStages = 4;
constexpr int kGroupLoads = 2;         // stages with loads in flight per CTA
constexpr int kGroupBytes = 8 * 1024;  // stage size
constexpr int kMaxCtasPerSmGroups = 6;

// One page of a group, as lane j sees it.
struct GroupPage {
  const uint8_t *src;  // nullptr: zero page
  uint32_t copy;       // bytes copied from src (a multiple of 16, at most the page)
  int32_t entry;       // source table entry (runs never cross entries)
  bool staging;        // a staging page: its load waits for the previous kernel; consumed when kConsume
};

// Page runs of a group (warp-uniform call): page j continues page j - 1 when
// both are copies from one table entry, page j - 1 is whole and page j's
// source starts where it ends.  A run's first lane gets start, the run's
// length and its bytes (whole pages, then the last page's copy).
struct PageRun {
  bool start;
  int run;
  uint32_t bytes;
};

CPKV_DEV PageRun page_runs(bool copy, const uint8_t *src, uint32_t my_copy, int32_t entry, uint32_t pb) {
  const unsigned all = 0xffffffffu;
  const int lane = threadIdx.x & 31;
  const unsigned long long prev_src = __shfl_up_sync(all, reinterpret_cast<unsigned long long>(src), 1);
  const uint32_t prev_copy = __shfl_up_sync(all, copy ? my_copy : 0u, 1);
  const int32_t prev_entry = __shfl_up_sync(all, entry, 1);
  const bool cont = lane > 0 && copy && prev_copy == pb && prev_entry == entry &&
                    reinterpret_cast<unsigned long long>(src) == prev_src + pb;
  const unsigned cont_mask = __ballot_sync(all, cont);
  PageRun r;
  r.start = copy && !cont;
  // run length: this page plus the continuing pages right after it
  const unsigned after = lane < 31 ? cont_mask >> (lane + 1) : 0u;
  r.run = r.start ? __ffs(~after) : 1;  // trailing ones of `after`, plus one
  const uint32_t last_copy = __shfl_sync(all, copy ? my_copy : 0u, (lane + r.run - 1) & 31);
  r.bytes = r.start ? (uint32_t)(r.run - 1) * pb + last_copy : 0;
  return r;
}

template <bool kConsume>
struct GroupRing {
  uint8_t *smem;        // kGroupStages * stage_bytes (dynamic shared memory)
  uint64_t *full;       // kGroupStages mbarriers
  uint8_t **dst;        // kGroupStages dense destinations (shared)
  uint32_t *bytes;      // kGroupStages group sizes (shared)
  int *live;            // kGroupStages: the stage was armed (shared)
  const uint8_t *(*drop_src)[32];  // kConsume: staging runs to drop once loaded (shared)
  uint32_t (*drop_bytes)[32];
  int *drop_n;
  int32_t *status;
  uint32_t stage_bytes;
  uint64_t pol;
  int64_t head, tail;   // consumed / issued (warp-uniform)
  bool dead;            // a bounded wait gave up (warp-uniform)
  bool open;            // store_gate

  CPKV_DEV void init(uint8_t *smem_, uint64_t *full_, uint8_t **dst_, uint32_t *bytes_, int *live_,
                     const uint8_t *(*drop_src_)[32], uint32_t (*drop_bytes_)[32], int *drop_n_, int32_t *status_,
                     uint32_t stage_bytes_) {
    smem = smem_; full = full_; dst = dst_; bytes = bytes_; live = live_;
    drop_src = drop_src_; drop_bytes = drop_bytes_; drop_n = drop_n_; status = status_;
    stage_bytes = stage_bytes_;
    pol = l2_policy_evict_first();
    head = tail = 0;
    dead = false;
    open = false;
    if ((threadIdx.x & 31) == 0) {
      for (int s = 0; s < kGroupStages; ++s) mbar_init(&full[s], 1);
      fence_barrier_init();
    }
    __syncwarp();
  }

  // Wait for the oldest group and store it (warp-uniform call).
  CPKV_DEV void consume() {
    const int s = (int)(head % kGroupStages);
    store_gate(&open);
    int ok = 0, dead_now = dead ? 1 : 0;
    if ((threadIdx.x & 31) == 0) {
      bool landed = false;
      if (live[s]) {
        landed = mbar_wait_bounded(&full[s], (uint32_t)((head / kGroupStages) & 1), kRingWaitLimitNs);
        if (!landed && !dead_now) {
          dead_now = 1;
          raise_status(status, CPKV_STATUS_TIMEOUT);
        }
      }
      if (landed && !dead_now) bulk_store_s2g_hint(dst[s], smem + (size_t)s * stage_bytes, bytes[s], pol);
      bulk_commit();
      ok = landed && !dead_now;
    }
    ok = __shfl_sync(0xffffffffu, ok, 0);
    dead = __shfl_sync(0xffffffffu, dead_now, 0) != 0;
    if (kConsume && ok)
      for (int k = 0; k < drop_n[s]; ++k) warp_discard_l2(drop_src[s][k], drop_bytes[s][k]);
    ++head;
  }

  // Issue a group of n pages of pb bytes each, stored to `dense` (the group's
  // first dense page); lane j < n describes page j (lanes past n: any value,
  // ignored).  Warp-uniform call.
  CPKV_DEV void push_group(uint8_t *dense, int n, uint32_t pb, GroupPage pg) {
    const unsigned all = 0xffffffffu;
    const int lane = threadIdx.x & 31;
    if (tail - head == kGroupLoads) consume();
    const int s = (int)(tail % kGroupStages);
    uint8_t *stage = smem + (size_t)s * stage_bytes;
    const bool mine = lane < n;
    const bool copy = mine && pg.src != nullptr && pg.copy > 0;
    const uint32_t my_copy = copy ? pg.copy : 0;
    const PageRun pr = page_runs(copy, pg.src, my_copy, pg.entry, pb);
    const bool start = pr.start;
    const uint32_t run_bytes = pr.bytes;
    uint32_t total = my_copy;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) total += __shfl_xor_sync(all, total, o);
    const unsigned zero_mask = __ballot_sync(all, mine && my_copy < pb);
    const bool staging = copy && pg.staging;
    const unsigned drop_mask = __ballot_sync(all, kConsume && start && staging);
    // the stage's previous store must have finished reading shared memory
    if (lane == 0 && tail >= kGroupStages) bulk_wait_read_dyn((int)(head - tail + kGroupStages - 1));
    __syncwarp();
    if (zero_mask != 0) {
      const uint4 z = make_uint4(0, 0, 0, 0);
      for (unsigned m = zero_mask; m != 0; m &= m - 1) {
        const int j = __ffs(m) - 1;
        const uint32_t from = __shfl_sync(all, my_copy, j);
        uint4 *page = reinterpret_cast<uint4 *>(stage + (size_t)j * pb);
        for (uint32_t i = from / 16 + lane; i < pb / 16; i += 32) page[i] = z;
      }
      fence_proxy_async_smem();  // the zeros are read by the bulk store (async proxy)
    }
    if (__any_sync(all, staging)) store_gate(&open);  // staging rows only after the previous kernel
    if (lane == 0) {
      live[s] = 0;
      if (!dead) {
        dst[s] = dense;
        bytes[s] = (uint32_t)n * pb;
        live[s] = 1;
        mbar_arrive_expect_tx(&full[s], total);  // 0 bytes: the phase completes now
      }
      if (kConsume) drop_n[s] = dead ? 0 : __popc(drop_mask);
    }
    if (kConsume && (drop_mask >> lane) & 1u) {
      const int k = __popc(drop_mask & ((1u << lane) - 1u));
      drop_src[s][k] = pg.src;
      drop_bytes[s][k] = run_bytes;
    }
    __syncwarp();
    if (start && !dead) bulk_load_g2s_hint(stage + (size_t)lane * pb, pg.src, run_bytes, &full[s], pol);
    ++tail;
    __syncwarp();
  }

  // Store everything in flight and wait until the stores are complete.
  CPKV_DEV void drain() {
    store_gate(&open);
    while (head < tail) consume();
    if ((threadIdx.x & 31) == 0) bulk_wait_all();
    __syncwarp();
  }
};

}  // namespace cpkv
