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
// (compose_layer_groups_kernel in compose_layer_groups.cu).  An earlier
// grouped form that staged each current page with its own 1152-byte bulk
// store and read it back once the bulk group had completed measured
// 7.64-7.71 ms per traced step on one-token pages, against 6.96-7.03 ms for
// the per-piece form here; the grouped form stages with the lanes' 16-byte
// stores and a proxy fence.
//
// The staging layout and the current pages' rows follow the plan of
// cpkv_plan_build: current page i (src = i + 1) holds its n_i tokens, whose
// rows are consecutive in their writer's buffer starting at
// token_writer_row of the page's first token.  The outputs (stagings and
// dense buffer) are byte-identical to cpkv_fill_current followed by
// cpkv_compose_gather on those plan arrays (cpkv_fill_current_planes for
// planar pages).
#include <stdint.h>

#include "bulk_ring.cuh"
#include "layer_params.cuh"

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
  if (!planar && pieces == 1 && page_bytes <= kLayerGroupMaxPageBytes) {
    // small pages: groups of consecutive dense pages, staged and read back by
    // the warp (compose_layer_groups.cu)
#define CPKV_LAYER_GROUPS(MB)                                                                       \
  {                                                                                                 \
    LayerParams<MB, 1> prm;                                                                         \
    CPKV_FILL_LAYER(prm)                                                                            \
    return launch_layer_groups<MB>(prm, consume_staging, early, s);                                 \
  }
    if (B <= 64) CPKV_LAYER_GROUPS(64)
    CPKV_LAYER_GROUPS(CPKV_MAX_BATCH)
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
