// cpkv_compose_layer on row-layout pages of at most 4 KB (one-token pages):
// one layer of the staging compose ("staging-direct compose" message of
// commits d63fbd4) — the fill of the current pages into the writers'
// stagings, then the slot-dense gather over the 2*cp pointer table — in a
// single launch that moves groups of consecutive dense pages.  The outputs
// (stagings and dense buffer) are byte-identical to cpkv_fill_current
// followed by cpkv_compose_gather on the same plan arrays.
#include <stdint.h>

#include "group_ring.cuh"
#include "layer_params.cuh"

namespace cpkv {
namespace {

// The staging compose over G = 8 KB / page-bytes consecutive dense pages at a
// time (at least 1, at most 32), through the small-page gather's page runs
// (group_ring.cuh).  A group first loads its pool pages and its current
// pages' rows into a stage (runs merged: consecutive pool pages of one owner,
// consecutive rows of one writer) and zeroes its zero slots and pad rows
// there.  Once they have landed, the warp stores each current page, rows and
// zero pads, from the stage to its staging slot with 16-byte stores (the
// fill; L2 evict_last), fences its generic-proxy global writes against the
// async proxy, and bulk-loads the pages back from the stagings into the same
// places of the stage (the gather's current part; runs merged over
// consecutive slots of one writer).  The group's dense pages are stored with
// one bulk copy once that read-back has landed, which is waited for when the
// next group is consumed, so it overlaps that group's loads.  Every staging
// page is written and read back, and each dense page is written once.
//
// Measured on the traced lengths with one-token pages (78 layers, 1152-byte
// pages, round-robin writers, launched plainly; ms per step, stagings kept /
// consumed; the stage count S, groups loading L and groups reading back K):
//   8 KB groups, S 3, L 2, K 1, 8 CTAs per SM (the form here)  4.69 / 5.41
//     consumed lines dropped after the dense store is issued,
//     launched early (the form here)                           4.36 / 4.90
//     (dropped before the dense store, launched early           4.36 / 5.05)
//     with every bulk copy issued by lane 0 in a loop over runs 4.80 / 5.57
//     with the group loads also issued by their runs' lanes      4.85 / 5.26
//   (the rows below with lane 0 issuing every copy)
//   8 KB, S 2, L 1, K 1, 12 CTAs per SM                        5.04 / 4.95
//   8 KB, S 4, 6 CTAs per SM (L, K of 2 and 1, 2 and 2, 3 and 1) 5.67 / 6.73-6.78
//   the same with a full proxy fence (shared and global)       5.97 / 6.77
//   4, 5, 6 or 7 KB groups, S 3, 16, 12, 10 or 9 CTAs per SM   4.91, 4.82, 4.92, 5.06 (kept)
//   10, 12 or 16 KB groups, S 3                                4.96, 5.62, 5.94 (kept)
//   4 KB groups, S 4, 12 CTAs per SM                           5.03 / 5.62
//   4 KB groups, S 4, 8 CTAs per SM; 2 KB, 24                  6.90; 7.03 (kept)
//   read-back by the lanes (coherent loads of their own stores, no fence),
//   8 KB groups, S 4                                           8.20-8.52 / 8.89-9.35
//   two warps per CTA, a producer (descriptors, zeros, loads) and a
//   consumer (staging stores, read-backs, dense stores) handing stages over
//   through mbarriers, launched early: 8 KB groups, S 3, 8 CTAs per SM
//   4.71 / 6.76; S 4 with 8, 6 or 4 KB groups (6, 8, 12 CTAs per SM)
//   4.60-4.64 (kept), against 4.36 / 4.91 for this one-warp form
// against 4.49 / 4.74 ms for the row fill followed by the group gather
// (4.40 / 4.64 launched early).  A
// warp waits on its loads, its staging stores' fence and its read-backs in
// turn and spends about 940 instructions per 8 KB group (700 per 4 KB
// group, ncu), so the throughput follows the number of warps per SM and the
// bytes each handles.
constexpr int kLayerGroupBytes = 8 * 1024;  // stage size
constexpr int kMaxCtasPerSmLayerGroups = 8;
constexpr int kLayerGroupStages = 3;
constexpr int kLayerGroupLoads = 2;  // groups with loads in flight per CTA
constexpr int kLayerGroupBacks = 1;  // groups with read-backs in flight per CTA
static_assert(kLayerGroupLoads + kLayerGroupBacks <= kLayerGroupStages, "ring shape");

// Make this thread's generic-proxy global writes ordered with its later
// async-proxy accesses (bulk copies reading what it just stored).
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Drop from L2 the lines that lie wholly inside each lane's run [src, src +
// bytes) (lanes with start set), without writing them back: all runs' lines
// are spread over the warp's lanes, so a group of small pages takes one
// discard instruction per 32 lines instead of one per run.  Warp-uniform
// call; the bytes become undefined, as for warp_discard_l2 (bulk_ring.cuh).
// The group gather (group_ring.cuh) measured slower with it (5.46 against
// 4.74 ms per traced step on one-token pages) and drops run by run.
__device__ __forceinline__ void warp_discard_runs(bool start, const uint8_t *src, uint32_t bytes) {
  const unsigned all = 0xffffffffu;
  const int lane = threadIdx.x & 31;
  unsigned long long first = 0;
  uint32_t n = 0;
  if (start) {
    first = (reinterpret_cast<unsigned long long>(src) + 127) & ~127ull;
    const unsigned long long end = (reinterpret_cast<unsigned long long>(src) + bytes) & ~127ull;
    n = end > first ? (uint32_t)((end - first) / 128) : 0u;
  }
  const unsigned runs = __ballot_sync(all, n != 0);
  uint32_t total = n;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) total += __shfl_xor_sync(all, total, o);
  for (uint32_t base = 0; base < total; base += 32) {
    const uint32_t idx = base + lane;
    unsigned long long a = 0;
    uint32_t cum = 0;
    for (unsigned m = runs; m != 0; m &= m - 1) {  // the run holding line idx
      const int j = __ffs(m) - 1;
      const uint32_t nj = __shfl_sync(all, n, j);
      const unsigned long long fj = __shfl_sync(all, first, j);
      if (idx >= cum && idx < cum + nj) a = fj + 128ull * (idx - cum);
      cum += nj;
    }
    if (idx < total) asm volatile("discard.global.L2 [%0], 128;" ::"l"(a) : "memory");
  }
}

template <bool kConsume>
struct LayerGroupRing {
  static constexpr int S = kLayerGroupStages;
  uint8_t *smem;
  uint64_t *full;      // per stage: the group's loads (pool pages, rows)
  uint64_t *back;      // per stage: the group's read-back (completes once per group, 0 bytes without current pages)
  uint8_t **dense;     // per stage: the group's first dense page
  uint32_t *bytes;     // per stage: the group's dense bytes
  int *live;           // per stage: loads were issued (else nothing lands)
  unsigned *cur_mask;  // per stage: lanes holding current pages
  const uint8_t *(*stg)[32];  // per stage: each lane's staging page
  int32_t (*entry)[32];       // per stage: each lane's table entry
  int32_t *status;
  uint32_t stage_bytes, pb;
  uint64_t stream_pol, keep_pol;
  // groups [0, stored) stored to the dense buffer, [stored, head) read back
  // in flight, [head, tail) loading
  int64_t head, tail, stored;
  bool dead, open;

  CPKV_DEV bool wait_bar(uint64_t *bar, int64_t use) {
    bool ok = true;
    if ((threadIdx.x & 31) == 0 && !dead) {
      ok = mbar_wait_bounded(bar, (uint32_t)((use / S) & 1), kRingWaitLimitNs);
      if (!ok) raise_status(status, CPKV_STATUS_TIMEOUT);
    }
    const int bad = __shfl_sync(0xffffffffu, ok ? 0 : 1, 0);
    if (bad) dead = true;
    __syncwarp();
    return !dead;
  }

  // The oldest consumed group's read-back has landed: store it to the dense
  // buffer (exactly one bulk group per group, in group order), then drop its
  // staging lines (kConsume).
  CPKV_DEV void finish_oldest() {
    const int64_t g = stored;
    const int s = (int)(g % S);
    const bool ok = wait_bar(&back[s], g);
    if ((threadIdx.x & 31) == 0) {
      if (!dead) bulk_store_s2g_hint(dense[s], smem + (size_t)s * stage_bytes, bytes[s], stream_pol);
      bulk_commit();
    }
    __syncwarp();
    if (kConsume && ok && cur_mask[s] != 0u) {  // after the store has been issued
      const int lane = threadIdx.x & 31;
      const bool cur = (cur_mask[s] >> lane) & 1u;
      const PageRun pr = page_runs(cur, stg[s][lane], cur ? pb : 0u, entry[s][lane], pb);
      warp_discard_runs(pr.start, stg[s][lane], pr.bytes);
    }
    ++stored;
    __syncwarp();
  }

  // Consume the oldest loading group: stage its current pages out to their
  // staging slots and start their read-back.
  CPKV_DEV void consume() {
    const int lane = threadIdx.x & 31;
    store_gate(&open);
    while (head - stored >= kLayerGroupBacks) finish_oldest();
    const int64_t g = head++;
    const int s = (int)(g % S);
    if (live[s]) wait_bar(&full[s], g);  // lane 0 saw the loads land: every lane may read the stage
    const unsigned cm = cur_mask[s];
    if (dead) return;  // nothing more is issued; finish_oldest only commits
    if (cm == 0u) {
      if (lane == 0) mbar_arrive_expect_tx(&back[s], 0);
      __syncwarp();
      return;
    }
    uint8_t *stage = smem + (size_t)s * stage_bytes;
    // the fill: each current page, rows and pad zeros, to its staging slot
    for (unsigned m = cm; m != 0; m &= m - 1) {
      const int j = __ffs(m) - 1;
      uint8_t *to = const_cast<uint8_t *>(stg[s][j]);
      const uint4 *from = reinterpret_cast<const uint4 *>(stage + (size_t)j * pb);
      for (uint32_t i = lane; i < pb / 16; i += 32) st16_hint(to + 16 * (size_t)i, from[i], keep_pol);
    }
    fence_proxy_async_global();  // the stores above before the bulk loads below (another proxy)
    __syncwarp();
    // the gather's current part: the same pages back from the stagings
    const bool cur = (cm >> lane) & 1u;
    const PageRun pr = page_runs(cur, stg[s][lane], cur ? pb : 0u, entry[s][lane], pb);
    if (lane == 0) mbar_arrive_expect_tx(&back[s], (uint32_t)__popc(cm) * pb);
    __syncwarp();
    // each run's first lane issues its read-back (the group loads below go
    // through lane 0, which measured faster there)
    if (pr.start) bulk_load_g2s_hint(stage + (size_t)lane * pb, stg[s][lane], pr.bytes, &back[s], stream_pol);
    __syncwarp();
  }

  // kind: 0 no page (lanes past n), 1 zero page, 2 pool page, 3 current page.
  CPKV_DEV void push(uint8_t *dense_first, int n, int kind, const uint8_t *src, uint32_t copy, int32_t ent,
                     uint8_t *stg_page) {
    const unsigned all = 0xffffffffu;
    const int lane = threadIdx.x & 31;
    if (tail - head == kLayerGroupLoads) consume();
    const int64_t t = tail;
    const int s = (int)(t % S);
    // the stage's previous group (t - S) has been stored (ring shape: stored
    // >= head - backs >= t - loads + 1 - backs); its store must have read
    // shared memory
    while (stored < t - S + 1) finish_oldest();
    if (lane == 0 && t >= S) bulk_wait_read_dyn((int)(stored - (t - S) - 1));
    __syncwarp();
    uint8_t *stage = smem + (size_t)s * stage_bytes;
    const bool cpy = kind >= 2;
    const uint32_t my_copy = cpy ? copy : 0;
    const PageRun pr = page_runs(cpy, src, my_copy, ent, pb);
    uint32_t total = my_copy;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) total += __shfl_xor_sync(all, total, o);
    const unsigned zero_mask = __ballot_sync(all, kind == 1 || (kind == 3 && my_copy < pb));
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
    const unsigned cm = __ballot_sync(all, kind == 3);
    stg[s][lane] = kind == 3 ? stg_page : nullptr;
    entry[s][lane] = ent;
    if (lane == 0) {
      dense[s] = dense_first;
      bytes[s] = (uint32_t)n * pb;
      cur_mask[s] = cm;
      live[s] = 0;
      if (!dead) {
        live[s] = 1;
        mbar_arrive_expect_tx(&full[s], total);  // 0 bytes: the phase completes now
      }
    }
    __syncwarp();
    for (unsigned m = __ballot_sync(all, pr.start); m != 0; m &= m - 1) {
      const int j = __ffs(m) - 1;
      const unsigned long long from = __shfl_sync(all, reinterpret_cast<unsigned long long>(src), j);
      const uint32_t b = __shfl_sync(all, pr.bytes, j);
      if (lane == 0 && !dead)
        bulk_load_g2s_hint(stage + (size_t)j * pb, reinterpret_cast<const uint8_t *>(from), b, &full[s], stream_pol);
    }
    ++tail;
    __syncwarp();
  }

  CPKV_DEV void drain() {
    store_gate(&open);
    while (head < tail) consume();
    while (stored < head) finish_oldest();
    if ((threadIdx.x & 31) == 0) bulk_wait_all();
    __syncwarp();
  }
};

template <int MAXB, bool CONSUME>
__global__ void __launch_bounds__(32) compose_layer_groups_kernel(const __grid_constant__ LayerParams<MAXB, 1> p) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t full[kLayerGroupStages];
  __shared__ __align__(8) uint64_t back[kLayerGroupStages];
  __shared__ uint8_t *st_dense[kLayerGroupStages];
  __shared__ uint32_t st_bytes[kLayerGroupStages];
  __shared__ int st_live[kLayerGroupStages];
  __shared__ unsigned st_cur[kLayerGroupStages];
  __shared__ const uint8_t *st_stg[kLayerGroupStages][32];
  __shared__ int32_t st_entry[kLayerGroupStages][32];
  __shared__ int32_t cur_page_start[MAXB + 1];
  __shared__ int64_t token_start[MAXB + 1];
  const int lane = threadIdx.x;
  release_dependents();
  {  // request-level exclusive scans, 32 requests per step
    int32_t carry_pages = 0;
    int64_t carry_tok = 0;
    for (int base = 0; base < p.B; base += 32) {
      const int b = base + lane;
      const int32_t n = b < p.B ? p.cur_lens[b] : 0;
      const int32_t np = (n + p.ps - 1) / p.ps;
      const int32_t inc_p = warp_inclusive_scan<int32_t>(np);
      const int64_t inc_t = warp_inclusive_scan<int64_t>((int64_t)n);
      if (b < p.B) {
        cur_page_start[b] = carry_pages + inc_p - np;
        token_start[b] = carry_tok + inc_t - n;
      }
      carry_pages += __shfl_sync(0xffffffffu, inc_p, 31);
      carry_tok += __shfl_sync(0xffffffffu, inc_t, 31);
    }
    if (lane == 0) {
      cur_page_start[p.B] = carry_pages;
      token_start[p.B] = carry_tok;
    }
    __syncwarp();
  }
  const uint32_t pb = (uint32_t)p.page_bytes;
  const int64_t R = p.page_bytes / p.ps;
  const int G = p.pieces;  // pages per group (LayerParams.pieces holds G here)
  LayerGroupRing<CONSUME> ring;
  ring.smem = smem;
  ring.full = full;
  ring.back = back;
  ring.dense = st_dense;
  ring.bytes = st_bytes;
  ring.live = st_live;
  ring.cur_mask = st_cur;
  ring.stg = st_stg;
  ring.entry = st_entry;
  ring.status = p.status;
  ring.stage_bytes = (uint32_t)G * pb;
  ring.pb = pb;
  ring.stream_pol = l2_policy_evict_first();
  ring.keep_pol = l2_policy_evict_last();
  ring.head = ring.tail = ring.stored = 0;
  ring.dead = false;
  ring.open = false;
  if (lane == 0) {
    for (int s = 0; s < kLayerGroupStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&back[s], 1);
    }
    fence_barrier_init();
  }
  __syncwarp();

  const int64_t step = gridDim.x;
  auto load_desc = [&](int64_t v, int32_t &o, int32_t &s) {
    o = -1;
    s = 0;
    if (v < p.units && lane < min64(G, p.dense_cap - v * G)) {
      o = p.owner[v * G + lane];
      s = p.src[v * G + lane];
    }
  };
  auto row0_of = [&](int32_t o, int32_t s) -> int32_t {
    if (o < p.cp || o >= 2 * p.cp || s < 1 || s > p.C || p.B == 0) return -1;
    const int b = upper_index<int32_t>(cur_page_start, p.B, s - 1);
    return p.token_writer_row[token_start[b] + (int64_t)(s - 1 - cur_page_start[b]) * p.ps];
  };
  // descriptors two groups ahead, first rows of current pages one group ahead
  int64_t u = blockIdx.x;
  int32_t o0, s0, o1, s1;
  load_desc(u, o0, s0);
  load_desc(u + step, o1, s1);
  int32_t r0 = row0_of(o0, s0);
  for (; u < p.units; u += step) {
    const int64_t d0 = u * G;
    const int n = (int)min64(G, p.dense_cap - d0);
    int32_t o2, s2;
    load_desc(u + 2 * step, o2, s2);
    const int32_t r1 = row0_of(o1, s1);
    int kind = 0;
    const uint8_t *src = nullptr;
    uint32_t copy = 0;
    uint8_t *stg = nullptr;
    if (lane < n) {
      kind = 1;
      if (o0 >= 0 && o0 < p.cp && s0 >= 0 && s0 < p.cap_pages[o0]) {
        kind = 2;
        src = p.table[o0] + (int64_t)s0 * p.page_bytes;
        copy = pb;
      } else if (o0 >= p.cp && o0 < 2 * p.cp) {
        int64_t nr = 0;
        const int32_t bad = current_rows(p, cur_page_start, true, o0, s0, r0, &nr);
        if (bad) {
          raise_status(p.status, bad);
        } else {
          kind = 3;
          src = p.cur_rows[0][o0 - p.cp] + (int64_t)r0 * R;
          copy = (uint32_t)(nr * R);
          stg = const_cast<uint8_t *>(p.table[o0]) + (int64_t)s0 * p.page_bytes;
        }
      } else if (o0 != -1) {
        raise_status(p.status, CPKV_STATUS_DESC_OOB);
      }
    }
    ring.push(p.dense + d0 * p.page_bytes, n, kind, src, copy, o0, stg);
    o0 = o1; s0 = s1; r0 = r1;
    o1 = o2; s1 = s2;
  }
  ring.drain();
}

}  // namespace

template <int MAXB>
int launch_layer_groups(LayerParams<MAXB, 1> prm, bool consume, bool early, cudaStream_t s) {
  // Launched early whenever asked: at 8 CTAs per SM that measured faster
  // (4.69 -> 4.36 ms per one-token step), where early_launch_pays would refuse.
  const int64_t per = kLayerGroupBytes / prm.page_bytes;
  const int64_t G = per < 1 ? 1 : (per < 32 ? per : 32);
  const int64_t gunits = ceil_div(prm.dense_cap, G);
  const size_t gsmem = (size_t)kLayerGroupStages * (size_t)(G * prm.page_bytes);
  prm.units = gunits;
  prm.pieces = (int32_t)G;
  prm.piece_bytes = (int32_t)prm.page_bytes;
  void (*kernel)(LayerParams<MAXB, 1>) =
      consume ? compose_layer_groups_kernel<MAXB, true> : compose_layer_groups_kernel<MAXB, false>;
  const void *fn = reinterpret_cast<const void *>(kernel);
  if (ensure_dynamic_smem(fn, (int)gsmem) != CPKV_OK) return CPKV_ERR_CUDA;
  const int grid = persistent_grid(fn, 32, gsmem, kMaxCtasPerSmLayerGroups, gunits);
  return launch_kernel(kernel, dim3(grid), dim3(32), gsmem, early, s, prm);
}

template int launch_layer_groups<64>(LayerParams<64, 1>, bool, bool, cudaStream_t);
template int launch_layer_groups<CPKV_MAX_BATCH>(LayerParams<CPKV_MAX_BATCH, 1>, bool, bool, cudaStream_t);

}  // namespace cpkv
