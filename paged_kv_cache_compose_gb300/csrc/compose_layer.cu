// cpkv_compose_layer: one layer of the staging compose ("staging-direct
// compose" message of commits d63fbd4) — the fill of the current pages into
// the writers' stagings followed by the slot-dense gather over the 2*cp
// pointer table — in a single launch.
//
// Every CTA walks its units (pieces of dense pages, u = blockIdx.x + i*grid)
// once; one warp drives a ring of bulk copies (for planar pages a second warp
// does the plain stores: zero slots, pad slices, lane-copied planes):
//   - a pool page or zero slot goes to the dense buffer (the prefix part of
//     the gather);
//   - a current page's rows, copied from its writer's current-row buffer, go
//     to staging slot src of writer owner - cp (the fill), and zero pad rows
//     go to both the staging slot and the dense page;
//   - a few bulk groups later, once `cp.async.bulk.wait_group` shows that the
//     staging store has completed, the same rows are copied back from the
//     staging slot into the dense page (the current part of the gather).
// A CTA reads back only staging pieces it wrote itself, so no CTA waits on
// another, and the fill's reads share DRAM time with the prefix pages'
// streams instead of running alone.  Every staging row is written and read
// back; the pad rows, zero in both places, are written to the dense page
// directly instead of being read back.  Staging stores carry an L2
// evict_last policy (their read-back follows within microseconds), all other
// copies evict_first.  With consume_staging the staged lines are dropped from
// L2 once read back, so they are never written back to DRAM.
//
// Pages may be planar (cpkv_compose_layer_planes): plane q of a page holds
// the ps tokens' plane_bytes[q]-byte slices, the planes one after the other.
// A plane whose slices are 16-byte multiples starting 16-byte aligned in the
// page is staged and read back as above; the slices of any other plane (the
// 4-byte scales of the NSA indexer keys) are copied by the warp's lanes,
// 4 bytes at a time, into both the staging slot and the dense page.  The row
// layout is the one-plane case.
//
// Row-layout pages of at most 4 KB take a grouped form instead
// (compose_layer_groups_kernel, below).  An earlier grouped form that staged
// each current page with its own 1152-byte bulk store and read it back once
// the bulk group had completed measured 7.64-7.71 ms per traced step on
// one-token pages, against 6.96-7.03 ms for the per-page form above; the
// grouped form below stages with the lanes' 16-byte stores and a proxy fence.
//
// The staging layout and the current pages' rows follow the plan of
// cpkv_plan_build: current page i (src = i + 1) holds its n_i tokens, whose
// rows are consecutive in their writer's buffer starting at
// token_writer_row of the page's first token.  The outputs (stagings and
// dense buffer) are byte-identical to cpkv_fill_current followed by
// cpkv_compose_gather on those plan arrays (cpkv_fill_current_planes for
// planar pages).
#include <stdint.h>

#include "group_ring.cuh"

namespace cpkv {
namespace {

constexpr int kStages = 4;
constexpr int kLoadsInFlight = 2;
constexpr int kMaxCtasPerSm = 3;
constexpr int kMaxPieceBytes = 24 * 1024;
constexpr int kReadbackQueue = 8;  // staging pieces waiting for their read-back, per CTA
constexpr int kReadbackLag = 4;    // bulk groups committed after a staging store before its read-back
constexpr int kMaxPlanes = 4;
constexpr int kWordsPerLane = 8;   // 4-byte words a lane keeps in flight when lanes copy a plane slice

// Wait until at most n (0..7; more counts as 7) of this thread's most recent
// bulk groups are still pending, and every older one has completed: its
// writes are done, not only its shared-memory reads.
__device__ __forceinline__ void bulk_wait_complete_dyn(int64_t n) {
  switch (n <= 0 ? 0 : (n >= 7 ? 7 : (int)n)) {
    case 0: asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); break;
    case 1: asm volatile("cp.async.bulk.wait_group 1;" ::: "memory"); break;
    case 2: asm volatile("cp.async.bulk.wait_group 2;" ::: "memory"); break;
    case 3: asm volatile("cp.async.bulk.wait_group 3;" ::: "memory"); break;
    case 4: asm volatile("cp.async.bulk.wait_group 4;" ::: "memory"); break;
    case 5: asm volatile("cp.async.bulk.wait_group 5;" ::: "memory"); break;
    case 6: asm volatile("cp.async.bulk.wait_group 6;" ::: "memory"); break;
    default: asm volatile("cp.async.bulk.wait_group 7;" ::: "memory"); break;
  }
}

// Every thread passes store_gate (common.cuh) before its first global store.
// It waits only when the launch is a programmatic dependent (at most 4 CTAs
// per SM, as for the fused compose: the CTAs may start in the slots the
// previous launch's tail frees and issue loads first).

struct Readback {
  const uint8_t *src;  // staging piece
  uint8_t *dst;        // dense piece
  uint32_t bytes;
  int64_t q;           // ring index of the copy that stored the staging piece
};

// NP: plane slots (1 for the row layout, which keeps the launch's parameter
// block small).
template <int MAXB, int NP>
struct LayerParams {
  const uint8_t *table[2 * CPKV_MAX_CP];  // pools, then stagings
  int64_t cap_pages[2 * CPKV_MAX_CP];
  const uint8_t *cur_rows[NP][CPKV_MAX_CP];  // plane q of writer w's current rows
  int64_t cur_cap[CPKV_MAX_CP];              // rows of writer w (every plane)
  int64_t plane_off[NP];                     // byte offset of plane q in a page
  int32_t plane_bytes[NP];
  int32_t plane_bulk[NP];                    // plane q is staged with bulk copies
  const int32_t *owner, *src, *token_writer_row;
  uint8_t *dense;
  int32_t *status;
  int64_t dense_cap, page_bytes, units, C;
  int32_t cp, ps, B, pieces, piece_bytes, n_planes;
  int32_t cur_lens[MAXB];
};

__device__ __forceinline__ uint32_t ld_stream4(const void *p) {
  uint32_t v;
  asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

__device__ __forceinline__ void st4(void *p, uint32_t v) {
  asm volatile("st.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void st4_hint(void *p, uint32_t v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.u32 [%0], %1, %2;" ::"l"(p), "r"(v), "l"(pol) : "memory");
}

// Copy `bytes` (a multiple of 4) from src to dst, and to stg (L2 policy
// `pol`) when STAGE, with the warp's lanes, kWordsPerLane loads in flight per
// lane.
template <bool STAGE>
__device__ __forceinline__ void warp_copy_words(const uint8_t *src, uint8_t *stg, uint8_t *dst, uint32_t bytes,
                                                uint64_t pol) {
  const uint32_t words = bytes / 4, lane = threadIdx.x & 31;
  for (uint32_t base = 0; base < words; base += 32 * kWordsPerLane) {
    uint32_t v[kWordsPerLane];
#pragma unroll
    for (int k = 0; k < kWordsPerLane; ++k) {
      const uint32_t i = base + k * 32 + lane;
      if (i < words) v[k] = ld_stream4(src + 4 * (size_t)i);
    }
#pragma unroll
    for (int k = 0; k < kWordsPerLane; ++k) {
      const uint32_t i = base + k * 32 + lane;
      if (i < words) {
        if (STAGE) st4_hint(stg + 4 * (size_t)i, v[k], pol);
        st4(dst + 4 * (size_t)i, v[k]);
      }
    }
  }
}

// Zero `bytes` (a multiple of 4) at dst with the warp's lanes: 16-byte stores
// when dst and bytes allow, else 4-byte stores; with an L2 policy when `hint`.
__device__ __forceinline__ void warp_zero_span(uint8_t *dst, uint32_t bytes, bool hint, uint64_t pol) {
  if (((reinterpret_cast<uintptr_t>(dst) | bytes) & 15u) == 0) {
    if (hint) warp_zero_hint(dst, bytes, pol);
    else warp_zero(dst, bytes);
    return;
  }
  for (uint32_t i = threadIdx.x & 31; i < bytes / 4; i += 32) {
    if (hint) st4_hint(dst + 4 * (size_t)i, 0u, pol);
    else st4(dst + 4 * (size_t)i, 0u);
  }
}

// Where a current page's rows come from: n rows starting at row0 of its
// writer's buffer.  Returns 0, or the status bit to raise when the descriptor
// (CPKV_STATUS_DESC_OOB: also a staging slot past the staging's capacity when
// `staged`) or the rows (CPKV_STATUS_ROW_OOB) are out of range; such a page is
// zero-filled in the dense buffer and its staging slot is left untouched.
template <typename Params>
__device__ __forceinline__ int32_t current_rows(const Params &p, const int32_t *cur_page_start, bool staged,
                                                int32_t o, int32_t s, int32_t row0, int64_t *n) {
  const int32_t w = o - p.cp, i = s - 1;
  if (i < 0 || i >= p.C || p.B == 0 || (staged && s >= p.cap_pages[o])) return CPKV_STATUS_DESC_OOB;
  const int b = upper_index<int32_t>(cur_page_start, p.B, i);
  const int32_t kp = i - cur_page_start[b];
  *n = min64(p.ps, (int64_t)p.cur_lens[b] - (int64_t)kp * p.ps);
  if (*n < 1) return CPKV_STATUS_DESC_OOB;
  return row0 >= 0 && row0 + *n <= p.cur_cap[w] ? 0 : CPKV_STATUS_ROW_OOB;
}

// The bulk ring with a per-piece choice of L2 policy for the store, and a
// queue of staging read-backs.  Every consume() commits exactly one bulk
// group, so the store of the copy with ring index q is group q, and group q
// has completed once wait_group(head - q - 1) returns.  kConsume: a
// read-back's staging lines are dropped from L2 once it has landed.
template <bool kConsume>
struct LayerRing : BulkRing<kStages, kLoadsInFlight, kConsume> {
  using Base = BulkRing<kStages, kLoadsInFlight, kConsume>;
  using Base::consume;
  using Base::head;
  using Base::push;
  using Base::store_policy;
  using Base::tail;
  uint32_t keep_mask;  // bit s: the piece in stage s is stored with keep_policy (warp-uniform)
  uint64_t keep_policy, stream_policy;
  Readback *rq;        // kReadbackQueue entries (shared; lane 0 writes, the warp reads)
  int64_t rq_head, rq_tail;
  bool stores_open;    // the previous launch has completed (store_gate)

  CPKV_DEV void consume_one() {
    store_gate(&stores_open);
    store_policy = ((keep_mask >> (int)(head % kStages)) & 1u) ? keep_policy : stream_policy;
    consume();
  }
  CPKV_DEV void push_with(const void *src, void *dst, uint32_t bytes, bool keep_in_l2, bool discard_src = false) {
    if (tail - head == kLoadsInFlight) consume_one();  // push() then finds a free load slot
    const uint32_t bit = 1u << (int)(tail % kStages);
    keep_mask = keep_in_l2 ? (keep_mask | bit) : (keep_mask & ~bit);
    push(src, dst, bytes, discard_src);
  }
  // Issue the oldest read-back once its staging store has completed.
  CPKV_DEV void readback_front() {
    const Readback r = rq[rq_head % kReadbackQueue];
    while (head <= r.q) consume_one();  // the staging store has been issued
    if ((threadIdx.x & 31) == 0) bulk_wait_complete_dyn(head - r.q - 1);
    __syncwarp();
    ++rq_head;
    push_with(r.src, r.dst, r.bytes, false, kConsume);
  }
  // Issue the read-backs whose stores are kReadbackLag groups old (all of
  // them when `all`).
  CPKV_DEV void service(bool all) {
    while (rq_head < rq_tail) {
      const int64_t q = rq[rq_head % kReadbackQueue].q;
      if (!all && rq_tail - rq_head < kReadbackQueue && head - q - 1 < kReadbackLag) break;
      readback_front();
    }
  }
  // Store `bytes` of rows into a staging piece now; copy them back from there
  // into the dense piece later.
  CPKV_DEV void stage(const uint8_t *rows, uint8_t *stg, uint8_t *dst, uint32_t bytes) {
    if (rq_tail - rq_head == kReadbackQueue) readback_front();
    const int64_t q = tail;
    push_with(rows, stg, bytes, true);
    if ((threadIdx.x & 31) == 0) rq[rq_tail % kReadbackQueue] = Readback{stg, dst, bytes, q};
    __syncwarp();
    ++rq_tail;
  }
  CPKV_DEV void drain_all() {
    service(true);
    while (head < tail) consume_one();
    if ((threadIdx.x & 31) == 0) bulk_wait_all();
    __syncwarp();
  }
};

// PLANAR false: one plane, staged with bulk copies (the row layout).
// STAGED false: the single-GPU compose without stagings (owner cp + w names
// writer w's current page src - 1, read straight from its rows).
// CONSUME (with STAGED): the stagings are consumed (their read-back lines are
// dropped from L2).
template <int MAXB, bool PLANAR, bool STAGED, bool CONSUME>
__global__ void __launch_bounds__(64, 1)
    compose_layer_kernel(const __grid_constant__ LayerParams<MAXB, PLANAR ? kMaxPlanes : 1> p) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t full[kStages];
  __shared__ uint8_t *ring_dst[kStages];
  __shared__ uint32_t ring_bytes[kStages];
  __shared__ int ring_live[kStages];
  __shared__ int32_t cur_page_start[MAXB + 1];
  __shared__ int64_t token_start[MAXB + 1];
  __shared__ Readback readbacks[kReadbackQueue];
  __shared__ const uint8_t *ring_src[kStages];
  const int lane = threadIdx.x & 31;
  const bool copy_warp = threadIdx.x < 32;
  // Planar pages: warp 0 issues every bulk copy, warp 1 does every plain
  // store (zero slots, pad slices, lane-copied plane slices), so that a load
  // it waits on never holds up the ring; the two warps write disjoint bytes.
  // Row layout (one warp): the same warp does both.
  const bool copy_role = copy_warp, store_role = PLANAR ? !copy_warp : true;
  const uint64_t keep = l2_policy_evict_last();  // staging stores
  release_dependents();
  bool stores_open = false;  // plain stores of this warp wait for the previous launch once

  if (copy_warp) {  // request-level exclusive scans, 32 requests per step
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
  }
  __syncthreads();

  LayerRing<CONSUME> ring;
  if (copy_warp) {
    ring.init(smem, full, ring_dst, ring_bytes, ring_live, p.status, p.piece_bytes, false, ring_src);
    ring.keep_mask = 0;
    ring.keep_policy = keep;
    ring.stream_policy = ring.load_policy;
    ring.rq = readbacks;
    ring.rq_head = ring.rq_tail = 0;
    ring.stores_open = false;
  }
  const int64_t step = gridDim.x;
  for (int64_t base = blockIdx.x; base < p.units; base += 32 * step) {
    const int64_t mine = base + lane * step;
    int32_t my_o = -1, my_s = 0, my_row0 = -1;
    if (mine < p.units) {
      my_o = p.owner[mine / p.pieces];
      my_s = p.src[mine / p.pieces];
    }
    if (my_o >= p.cp && my_o < 2 * p.cp && my_s >= 1 && my_s <= p.C && p.B > 0) {
      const int b = upper_index<int32_t>(cur_page_start, p.B, my_s - 1);
      my_row0 = p.token_writer_row[token_start[b] + (int64_t)(my_s - 1 - cur_page_start[b]) * p.ps];
    }
    for (int j = 0; j < 32; ++j) {
      const int64_t u = base + j * step;
      if (u >= p.units) break;  // uniform across the warp
      const int32_t o = __shfl_sync(0xffffffffu, my_o, j);
      const int32_t s = __shfl_sync(0xffffffffu, my_s, j);
      const int32_t row0 = __shfl_sync(0xffffffffu, my_row0, j);
      const int64_t d = u / p.pieces;
      const int32_t k = (int32_t)(u - d * p.pieces);
      const int64_t off = (int64_t)k * p.piece_bytes;
      const uint32_t bytes = (uint32_t)min64(p.piece_bytes, p.page_bytes - off);
      uint8_t *dst = p.dense + d * p.page_bytes + off;
      if (!(o >= p.cp && o < 2 * p.cp)) {  // pool pages, zero slots, invalid descriptors
        if (o >= 0 && o < p.cp && s >= 0 && s < p.cap_pages[o]) {
          if (copy_role) ring.push_with(p.table[o] + (int64_t)s * p.page_bytes + off, dst, bytes, false);
        } else if (store_role) {
          if (o != -1 && lane == 0 && k == 0) raise_status(p.status, CPKV_STATUS_DESC_OOB);
          store_gate(&stores_open);
          warp_zero(dst, bytes);
        }
      } else {
        int64_t n = 0;
        const int32_t bad = current_rows(p, cur_page_start, STAGED, o, s, row0, &n);
        if (bad) {
          if (store_role) {
            if (lane == 0 && k == 0) raise_status(p.status, bad);
            store_gate(&stores_open);
            warp_zero(dst, bytes);
          }
        } else {
          // per plane: the rows' slices inside this piece, then the pad slices
          uint8_t *stg_page = STAGED ? const_cast<uint8_t *>(p.table[o]) + (int64_t)s * p.page_bytes : nullptr;
          uint8_t *dense_page = p.dense + d * p.page_bytes;
          const int64_t end = off + bytes;
          const int n_planes = PLANAR ? p.n_planes : 1;
          for (int q = 0; q < n_planes; ++q) {
            const int64_t P = PLANAR ? p.plane_off[q] : 0, w = p.plane_bytes[q];
            const bool bulk = PLANAR ? p.plane_bulk[q] != 0 : true;
            const int64_t rows_end = P + n * w, plane_end = P + (int64_t)p.ps * w;
            const int64_t lo = off > P ? off : P, hi = min64(end, rows_end);
            if (lo < hi && (bulk ? copy_role : store_role)) {
              const uint8_t *from = p.cur_rows[q][o - p.cp] + (int64_t)row0 * w + (lo - P);
              if (bulk && STAGED) ring.stage(from, stg_page + lo, dense_page + lo, (uint32_t)(hi - lo));
              else if (bulk) ring.push_with(from, dense_page + lo, (uint32_t)(hi - lo), false);
              else {
                store_gate(&stores_open);
                warp_copy_words<STAGED>(from, stg_page + lo, dense_page + lo, (uint32_t)(hi - lo), keep);
              }
            }
            const int64_t zlo = off > rows_end ? off : rows_end, zhi = min64(end, plane_end);
            if (zlo < zhi && store_role) {
              store_gate(&stores_open);
              if (STAGED) warp_zero_span(stg_page + zlo, (uint32_t)(zhi - zlo), true, keep);
              warp_zero_span(dense_page + zlo, (uint32_t)(zhi - zlo), false, 0);
            }
          }
        }
      }
      if (copy_warp) ring.service(false);
    }
  }
  if (copy_warp) ring.drain_all();
}

// ---------------------------------------------------------------------------
// Small pages (row layout, at most 4 KB): groups of consecutive dense pages
// ---------------------------------------------------------------------------
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
// against 4.49 / 4.74 ms for the row fill followed by the group gather
// (launched early: 4.35 / 5.05 here, 4.40 / 4.64 for fill + gather).  A
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

  // The oldest consumed group's read-back has landed: drop its staging lines
  // (kConsume) and store it to the dense buffer (exactly one bulk group per
  // group, in group order).
  CPKV_DEV void finish_oldest() {
    const int64_t g = stored;
    const int s = (int)(g % S);
    const bool ok = wait_bar(&back[s], g);
    if (kConsume && ok && cur_mask[s] != 0u) {
      const int lane = threadIdx.x & 31;
      const bool cur = (cur_mask[s] >> lane) & 1u;
      const PageRun pr = page_runs(cur, stg[s][lane], cur ? pb : 0u, entry[s][lane], pb);
      warp_discard_runs(pr.start, stg[s][lane], pr.bytes);
    }
    if ((threadIdx.x & 31) == 0) {
      if (!dead) bulk_store_s2g_hint(dense[s], smem + (size_t)s * stage_bytes, bytes[s], stream_pol);
      bulk_commit();
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
}  // namespace cpkv

namespace {

// Launch one instantiation of the kernel on a persistent grid sized by the
// occupancy calculator; as a programmatic dependent of the previous kernel
// when `early` and the grid runs at most 4 CTAs per SM (early_launch_pays:
// index-key pages 4.345 -> 4.089 ms per step, traced 4.25 -> 3.91 ms).
template <typename Params>
int launch_layer(void (*kernel)(Params), int threads, int64_t units, size_t smem, int cap_per_sm, bool early,
                 cudaStream_t s, const Params &prm) {
  using namespace cpkv;
  const void *fn = reinterpret_cast<const void *>(kernel);
  if (ensure_dynamic_smem(fn, kStages * kMaxPieceBytes) != CPKV_OK) return CPKV_ERR_CUDA;
  const int grid = persistent_grid(fn, threads, smem, cap_per_sm, units);
  return launch_kernel(kernel, dim3(grid), dim3(threads), smem, early && early_launch_pays(grid), s, prm);
}

// staged: h_src_table / h_src_cap_pages hold 2*cp entries (pools, then
// stagings); else cp entries (pools only) and no staging is written.
int compose_layer_impl(bool staged, bool consume_staging, bool early, int B, int page_size, int cp_size, int n_planes,
                       const int32_t *h_plane_bytes, const int32_t *h_cur_lens, const void *const *h_cur_planes,
                       const int64_t *h_cur_rows_cap, const void *const *h_src_table, const int64_t *h_src_cap_pages,
                       const int32_t *d_owner, const int32_t *d_src, const int32_t *d_token_writer_row,
                       int64_t dense_cap_pages, void *d_dense, int32_t *d_status, cudaStream_t s) {
  using namespace cpkv;
  if (B < 0 || page_size <= 0 || cp_size < 1 || cp_size > CPKV_MAX_CP) return CPKV_ERR_ARG;
  if (n_planes < 1 || n_planes > kMaxPlanes || h_plane_bytes == nullptr || dense_cap_pages < 0) return CPKV_ERR_ARG;
  int64_t row_bytes = 0;
  for (int q = 0; q < n_planes; ++q) {
    if (h_plane_bytes[q] <= 0 || h_plane_bytes[q] % 4 != 0) return CPKV_ERR_ARG;
    row_bytes += h_plane_bytes[q];
  }
  if (((int64_t)page_size * row_bytes) % 16 != 0) return CPKV_ERR_ARG;
  if (B > CPKV_MAX_BATCH) return CPKV_ERR_LIMIT;
  if (h_cur_planes == nullptr || h_cur_rows_cap == nullptr || h_src_table == nullptr || h_src_cap_pages == nullptr ||
      d_status == nullptr)
    return CPKV_ERR_ARG;
  if (B > 0 && h_cur_lens == nullptr) return CPKV_ERR_ARG;
  int64_t T = 0, C = 0;
  for (int b = 0; b < B; ++b) {
    if (h_cur_lens[b] < 0) return CPKV_ERR_ARG;
    T += h_cur_lens[b];
    C += ceil_div(h_cur_lens[b], page_size);
  }
  if (T > INT32_MAX - 1 || C > INT32_MAX - 2) return CPKV_ERR_LIMIT;
  const int n_table = staged ? 2 * cp_size : cp_size;
  for (int k = 0; k < n_table; ++k) {
    if (h_src_cap_pages[k] < 0) return CPKV_ERR_ARG;
    if (h_src_cap_pages[k] > 0 && (h_src_table[k] == nullptr || !aligned16(h_src_table[k]))) return CPKV_ERR_ARG;
  }
  for (int w = 0; w < cp_size; ++w) {
    if (staged && C > 0 && h_src_cap_pages[cp_size + w] < C + 1) return CPKV_ERR_CAPACITY;  // staging slots 1..C
    if (h_cur_rows_cap[w] < 0) return CPKV_ERR_ARG;
    for (int q = 0; q < n_planes; ++q) {
      const void *rows = h_cur_planes[q * cp_size + w];
      if (h_cur_rows_cap[w] > 0 && (rows == nullptr || !aligned16(rows))) return CPKV_ERR_ARG;
    }
  }
  if (dense_cap_pages == 0) return CPKV_OK;
  if (d_owner == nullptr || d_src == nullptr || d_dense == nullptr || !aligned16(d_dense)) return CPKV_ERR_ARG;
  if (T > 0 && d_token_writer_row == nullptr) return CPKV_ERR_ARG;
  const int64_t page_bytes = (int64_t)page_size * row_bytes;
  const int64_t pieces = ceil_div(page_bytes, kMaxPieceBytes);
  const int64_t piece_bytes = ceil_div(ceil_div(page_bytes, pieces), 16) * 16;
  if (pieces > INT32_MAX || dense_cap_pages > INT64_MAX / pieces) return CPKV_ERR_LIMIT;
  const int64_t units = dense_cap_pages * pieces;
  const size_t smem = (size_t)kStages * piece_bytes;
  const int cap_per_sm = pieces > 1 ? kMaxCtasPerSm : ring_cap_one_piece(piece_bytes, kLoadsInFlight, kMaxCtasPerSm);

#define CPKV_FILL_LAYER(prm)                                                                           \
  for (int k = 0; k < 2 * CPKV_MAX_CP; ++k) {                                                          \
    prm.table[k] = k < n_table ? static_cast<const uint8_t *>(h_src_table[k]) : nullptr;               \
    prm.cap_pages[k] = k < n_table ? h_src_cap_pages[k] : 0;                                           \
  }                                                                                                    \
  for (int q = 0; q < (int)(sizeof(prm.plane_bytes) / sizeof(int32_t)); ++q)                           \
    for (int w = 0; w < CPKV_MAX_CP; ++w)                                                              \
      prm.cur_rows[q][w] =                                                                             \
          q < n_planes && w < cp_size ? static_cast<const uint8_t *>(h_cur_planes[q * cp_size + w]) : nullptr; \
  for (int w = 0; w < CPKV_MAX_CP; ++w) prm.cur_cap[w] = w < cp_size ? h_cur_rows_cap[w] : 0;         \
  {                                                                                                    \
    int64_t at = 0;                                                                                    \
    for (int q = 0; q < (int)(sizeof(prm.plane_bytes) / sizeof(int32_t)); ++q) {                     \
      const int32_t wq = q < n_planes ? h_plane_bytes[q] : 0;                                          \
      prm.plane_off[q] = at;                                                                           \
      prm.plane_bytes[q] = wq;                                                                         \
      prm.plane_bulk[q] = (wq % 16 == 0 && at % 16 == 0) ? 1 : 0;                                      \
      at += (int64_t)page_size * wq;                                                                   \
    }                                                                                                  \
  }                                                                                                    \
  prm.owner = d_owner; prm.src = d_src; prm.token_writer_row = d_token_writer_row;                     \
  prm.dense = static_cast<uint8_t *>(d_dense); prm.status = d_status; prm.dense_cap = dense_cap_pages;   \
  prm.page_bytes = page_bytes; prm.units = units; prm.C = C; prm.cp = cp_size; prm.ps = page_size;     \
  prm.B = B; prm.pieces = (int32_t)pieces; prm.piece_bytes = (int32_t)piece_bytes; prm.n_planes = n_planes; \
  for (int b = 0; b < B; ++b) prm.cur_lens[b] = h_cur_lens[b];

  // Row layout without stagings is cpkv_compose_fused (fused.cu); the
  // callers route it there.
  const bool planar = !(n_planes == 1 && h_plane_bytes[0] % 16 == 0);
  if (!planar && !staged) return CPKV_ERR_ARG;
  if (!planar && pieces == 1 && page_bytes * 2 <= kGroupBytes) {
    // small pages: groups of consecutive dense pages, staged and read back by
    // the warp; launched early whenever asked (8 CTAs per SM: 4.69 -> 4.36 ms
    // per one-token step, where early_launch_pays would refuse)
    const int64_t G = kLayerGroupBytes / page_bytes < 1 ? 1 : (kLayerGroupBytes / page_bytes < 32 ? kLayerGroupBytes / page_bytes : 32);
    const int64_t gunits = ceil_div(dense_cap_pages, G);
    const size_t gsmem = (size_t)kLayerGroupStages * (size_t)(G * page_bytes);
#define CPKV_LAYER_GROUPS(MB, CO)                                                                   \
  {                                                                                                 \
    const void *kernel = reinterpret_cast<const void *>(compose_layer_groups_kernel<MB, CO>);       \
    if (ensure_dynamic_smem(kernel, gsmem) != CPKV_OK) return CPKV_ERR_CUDA;                          \
    const int grid = persistent_grid(kernel, 32, gsmem, kMaxCtasPerSmLayerGroups, gunits);          \
    LayerParams<MB, 1> prm;                                                                         \
    CPKV_FILL_LAYER(prm)                                                                            \
    prm.units = gunits; prm.pieces = (int32_t)G; prm.piece_bytes = (int32_t)page_bytes;             \
    return launch_kernel(compose_layer_groups_kernel<MB, CO>, dim3(grid), dim3(32), gsmem, early, s, \
                         prm);                                                                      \
  }
    if (B <= 64 && consume_staging) CPKV_LAYER_GROUPS(64, true)
    if (B <= 64) CPKV_LAYER_GROUPS(64, false)
    if (consume_staging) CPKV_LAYER_GROUPS(CPKV_MAX_BATCH, true)
    CPKV_LAYER_GROUPS(CPKV_MAX_BATCH, false)
#undef CPKV_LAYER_GROUPS
  }
  // one instantiation per (batch template, planar, staged, consumed)
#define CPKV_LAUNCH_LAYER(MAXB, NP, PL, ST, CO, THREADS)                                   \
  {                                                                                        \
    LayerParams<MAXB, NP> prm;                                                             \
    CPKV_FILL_LAYER(prm)                                                                   \
    return launch_layer(compose_layer_kernel<MAXB, PL, ST, CO>, THREADS, units, smem, cap_per_sm,             \
                        early, s,                                                 \
                        prm);                                                                   \
  }
  if (B <= 64) {
    if (planar && !staged) CPKV_LAUNCH_LAYER(64, kMaxPlanes, true, false, false, 64)
    if (planar && consume_staging) CPKV_LAUNCH_LAYER(64, kMaxPlanes, true, true, true, 64)
    if (planar) CPKV_LAUNCH_LAYER(64, kMaxPlanes, true, true, false, 64)
    if (consume_staging) CPKV_LAUNCH_LAYER(64, 1, false, true, true, 32)
    CPKV_LAUNCH_LAYER(64, 1, false, true, false, 32)
  }
  if (planar && !staged) CPKV_LAUNCH_LAYER(CPKV_MAX_BATCH, kMaxPlanes, true, false, false, 64)
  if (planar && consume_staging) CPKV_LAUNCH_LAYER(CPKV_MAX_BATCH, kMaxPlanes, true, true, true, 64)
  if (planar) CPKV_LAUNCH_LAYER(CPKV_MAX_BATCH, kMaxPlanes, true, true, false, 64)
  if (consume_staging) CPKV_LAUNCH_LAYER(CPKV_MAX_BATCH, 1, false, true, true, 32)
  CPKV_LAUNCH_LAYER(CPKV_MAX_BATCH, 1, false, true, false, 32)
#undef CPKV_LAUNCH_LAYER
#undef CPKV_FILL_LAYER
}

}  // namespace

extern "C" int cpkv_compose_layer(int B, int page_size, int cp_size, int64_t row_bytes, const int32_t *h_cur_lens,
                                  const void *const *h_cur_rows, const int64_t *h_cur_rows_cap,
                                  const void *const *h_src_table, const int64_t *h_src_cap_pages,
                                  const int32_t *d_owner, const int32_t *d_src, const int32_t *d_token_writer_row,
                                  int64_t dense_cap_pages, void *d_dense, int flags, int32_t *d_status,
                                  cpkv_stream_t stream) {
  if (row_bytes <= 0 || row_bytes % 16 != 0 || row_bytes > INT32_MAX) return CPKV_ERR_ARG;
  if ((flags & ~(CPKV_FLAG_CONSUME_STAGING | CPKV_FLAG_EARLY_INPUTS)) != 0) return CPKV_ERR_ARG;
  const int32_t plane = (int32_t)row_bytes;
  const bool consume = (flags & CPKV_FLAG_CONSUME_STAGING) != 0, early = (flags & CPKV_FLAG_EARLY_INPUTS) != 0;
  return compose_layer_impl(true, consume, early, B, page_size, cp_size, 1, &plane, h_cur_lens, h_cur_rows,
                            h_cur_rows_cap, h_src_table, h_src_cap_pages, d_owner, d_src, d_token_writer_row,
                            dense_cap_pages, d_dense, d_status, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int cpkv_compose_layer_planes(int B, int page_size, int cp_size, int n_planes,
                                         const int32_t *h_plane_bytes, const int32_t *h_cur_lens,
                                         const void *const *h_cur_planes, const int64_t *h_cur_rows_cap,
                                         const void *const *h_src_table, const int64_t *h_src_cap_pages,
                                         const int32_t *d_owner, const int32_t *d_src,
                                         const int32_t *d_token_writer_row, int64_t dense_cap_pages, void *d_dense,
                                         int flags, int32_t *d_status, cpkv_stream_t stream) {
  if ((flags & ~(CPKV_FLAG_CONSUME_STAGING | CPKV_FLAG_EARLY_INPUTS)) != 0) return CPKV_ERR_ARG;
  const bool consume = (flags & CPKV_FLAG_CONSUME_STAGING) != 0, early = (flags & CPKV_FLAG_EARLY_INPUTS) != 0;
  return compose_layer_impl(true, consume, early, B, page_size, cp_size, n_planes, h_plane_bytes, h_cur_lens,
                            h_cur_planes, h_cur_rows_cap, h_src_table, h_src_cap_pages, d_owner, d_src,
                            d_token_writer_row,
                            dense_cap_pages, d_dense, d_status, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int cpkv_compose_fused_planes(int B, int page_size, int cp_size, int n_planes,
                                         const int32_t *h_plane_bytes, const int32_t *h_cur_lens,
                                         const void *const *h_pools, const int64_t *h_pool_cap_pages,
                                         const void *const *h_cur_planes, const int64_t *h_cur_rows_cap,
                                         const int32_t *d_owner, const int32_t *d_src,
                                         const int32_t *d_token_writer_row, int64_t dense_cap_pages, void *d_dense,
                                         int flags, int32_t *d_status, cpkv_stream_t stream) {
  if ((flags & ~CPKV_FLAG_EARLY_INPUTS) != 0) return CPKV_ERR_ARG;
  if (n_planes == 1 && h_plane_bytes != nullptr && h_plane_bytes[0] > 0 && h_plane_bytes[0] % 16 == 0)
    return cpkv_compose_fused(B, page_size, cp_size, h_plane_bytes[0], h_cur_lens, h_pools, h_pool_cap_pages,
                              h_cur_planes, h_cur_rows_cap, d_owner, d_src, d_token_writer_row, dense_cap_pages,
                              d_dense, flags, d_status, stream);
  return compose_layer_impl(false, false, (flags & CPKV_FLAG_EARLY_INPUTS) != 0, B, page_size, cp_size, n_planes,
                            h_plane_bytes, h_cur_lens, h_cur_planes, h_cur_rows_cap, h_pools, h_pool_cap_pages,
                            d_owner, d_src, d_token_writer_row, dense_cap_pages, d_dense, d_status,
                            reinterpret_cast<cudaStream_t>(stream));
}
