// cpkv_compose_gather: the slot-dense page gather ("staging-direct compose"
// message of commits d63fbd4: ONE gather covers prefix pages through pool
// pointers and all current pages through staging pointers, via a
// concatenated 2*cp pointer table; "compose_v2" message: owner -1 zero-fills).
//
// Every dense page is ps*R contiguous bytes copied from one contiguous
// source page, so the kernel moves pages with bulk async copies (TMA,
// non-tensor form): global -> shared with mbarrier completion, then
// shared -> global tracked by bulk groups.  Each page is cut into `pieces`
// equal 16-byte-multiple units (<= 16 KB); units are dealt round-robin to a
// persistent grid of one-warp CTAs: up to 4 per SM for pages of several
// pieces, and for pages of one piece enough to keep about 56 KB of loads in
// flight per SM (3 for 8448-byte pages, 24 for 1152-byte ones; see
// ring_cap_one_piece).  Each CTA runs a BulkRing of
// 4 shared-memory stages with at most 2 loads outstanding, so the other
// stages hold stores still draining: loads and stores overlap instead of a
// stage waiting for its own store.  Every copy carries an L2 evict_first
// policy: pool pages, staging pages and dense pages are each touched once per
// layer, and streaming them must not evict the staging the fill has just
// written for this gather.  Zero units (owner -1 or an invalid descriptor)
// are written with plain 16-byte stores by the whole warp.  Every mbarrier
// wait is bounded (see bulk_ring.cuh).  With CPKV_GATHER_CONSUME_STAGING the
// stagings are consumed: once a staging piece has landed in shared memory
// its L2 lines are dropped, so the fill's dirty staging lines are never
// written back to DRAM.
//
// With CPKV_GATHER_EARLY_INPUTS and a grid of at most 4 CTAs per SM
// (early_launch_pays: pages of several pieces, index-key pages) the gather is
// launched as a programmatic dependent of the previous kernel (its fill: the
// page-run fills release it at their start, the row fills as their blocks
// finish).  Its CTAs start beside or after the fill, load descriptors and
// pool pieces at once, and each waits for the fill (store_gate) before its
// first staging load and before its first store.  Measured per 78-layer step: traced 4.284 -> 4.200 ms;
// fp8 unchanged (19.77 ms); index keys 4.143 -> 4.128 ms; one-token pages,
// where the per-page ring ran 24 small CTAs per SM, 5.195 -> 5.555 ms, so
// such grids launch plainly.  The group gather of pages of at most 4 KB (6
// CTAs per SM) launches early: 4.49 -> 4.41 ms per one-token step.
// The gather itself releases its dependents at its start (the next layer's
// fill, launched with CPKV_FLAG_EARLY_INPUTS, may start while it runs).
#include <stdint.h>

#include "group_ring.cuh"

namespace cpkv {
namespace {

constexpr int kStages = 4;
constexpr int kLoadsInFlight = 2;
constexpr int kMaxPieceBytes = 16 * 1024;
// One-warp CTAs per SM, as many as shared memory allows up to: 4 when pages
// are cut into several pieces, 3 for pages of one piece (more CTAs measured
// slower there).
constexpr int kMaxCtasPerSmPieces = 4;
constexpr int kMaxCtasPerSmOnePiece = 3;

struct GatherParams {
  const uint8_t *table[2 * CPKV_MAX_CP];
  int64_t cap_pages[2 * CPKV_MAX_CP];
  const int32_t *owner, *src;
  uint8_t *dense;
  int32_t *status;
  int64_t dense_cap, page_bytes, units;  // units: pieces, or page groups (gather_groups_kernel)
  int32_t n_table, n_pool, pieces, piece_bytes, kinds;
  int32_t group;                          // pages per group (gather_groups_kernel)
};

struct Unit {
  const uint8_t *src;  // nullptr: zero-fill
  uint8_t *dst;
  uint32_t bytes;
};

// Kind of a descriptor: pool page, staging page, or zero slot (owner -1 and
// invalid descriptors, which are zero-filled).
__device__ __forceinline__ int slot_kind(const GatherParams &p, int32_t o) {
  if (o >= 0 && o < p.n_pool) return CPKV_GATHER_POOL;
  if (o >= p.n_pool && o < p.n_table) return CPKV_GATHER_STAGING;
  return CPKV_GATHER_ZERO;
}

// Unit u of this launch, given its page's descriptor (o, s).
__device__ __forceinline__ Unit resolve_unit(const GatherParams &p, int64_t u, int32_t o, int32_t s, bool report,
                                             bool *skip) {
  const int64_t d = u / p.pieces;
  const int32_t k = (int32_t)(u - d * p.pieces);
  const int64_t off = (int64_t)k * p.piece_bytes;
  Unit x;
  x.bytes = (uint32_t)min64(p.piece_bytes, p.page_bytes - off);
  x.dst = p.dense + d * p.page_bytes + off;
  x.src = nullptr;
  *skip = (slot_kind(p, o) & p.kinds) == 0;
  if (*skip || o == -1) return x;
  if (o < -1 || o >= p.n_table || s < 0 || s >= p.cap_pages[o]) {
    if (report && k == 0) raise_status(p.status, CPKV_STATUS_DESC_OOB);
    return x;
  }
  x.src = p.table[o] + (int64_t)s * p.page_bytes + off;
  return x;
}

// kConsume: the staging pages are consumed; once a staging piece has been
// loaded its L2 lines are dropped without write-back.
template <bool kConsume>
__global__ void __launch_bounds__(32) gather_pages_kernel(const __grid_constant__ GatherParams p) {
  // A fill launched after this gather with CPKV_FLAG_EARLY_INPUTS may start
  // its loads now; its stores wait for this kernel to complete.
  release_dependents();
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t full[kStages];
  __shared__ uint8_t *ring_dst[kStages];
  __shared__ uint32_t ring_bytes[kStages];
  __shared__ int ring_live[kStages];
  __shared__ const uint8_t *ring_src[kStages];
  BulkRing<kStages, kLoadsInFlight, kConsume> ring;
  ring.init(smem, full, ring_dst, ring_bytes, ring_live, p.status, p.piece_bytes, false, ring_src);
  // The CTA's units are u = blockIdx.x + i * gridDim.x.  Their descriptors
  // are loaded 32 at a time (one per lane) and handed out with shuffles, so
  // no copy waits on a descriptor load of its own.
  const int lane = threadIdx.x;
  const int64_t step = gridDim.x;
  bool open = false;  // store_gate: warp-uniform here
  for (int64_t base = blockIdx.x; base < p.units; base += 32 * step) {
    const int64_t mine = base + lane * step;
    int32_t my_o = -1, my_s = 0;
    if (mine < p.units) {
      my_o = p.owner[mine / p.pieces];
      my_s = p.src[mine / p.pieces];
    }
    for (int j = 0; j < 32; ++j) {
      const int64_t u = base + j * step;
      if (u >= p.units) break;  // uniform across the warp
      const int32_t o = __shfl_sync(0xffffffffu, my_o, j);
      const int32_t sr = __shfl_sync(0xffffffffu, my_s, j);
      bool skip;
      const Unit x = resolve_unit(p, u, o, sr, lane == 0, &skip);
      if (skip) continue;
      // staging loads and stores (a zero unit, or a push that stores the
      // oldest stage) wait for the previous kernel when launched early
      if (x.src == nullptr || o >= p.n_pool || ring.tail - ring.head == kLoadsInFlight) store_gate(&open);
      if (x.src == nullptr) warp_zero(x.dst, x.bytes);
      else ring.push(x.src, x.dst, x.bytes, kConsume && o >= p.n_pool);
    }
  }
  store_gate(&open);
  ring.drain();
}

// ---------------------------------------------------------------------------
// Small pages: groups of consecutive dense pages, with page-run merging
// ---------------------------------------------------------------------------
// Pages of at most 4 KB are moved a group at a time through the group ring
// (group_ring.cuh, shared with the fused compose on small pages): a unit is
// G consecutive dense pages (G = 8 KB / page bytes, at most 32), and lane j
// resolves the group's page j.  Consecutive pages whose sources are
// consecutive pages of one table entry form a run, loaded into the stage with
// ONE bulk copy (page-
// run merging: a contiguous stretch of a pool or a staging is one copy); zero
// pages (owner -1, invalid descriptors) are zero-filled in shared memory by
// the warp; the whole group is stored with ONE bulk copy, since dense pages
// d0 .. d0 + n - 1 are contiguous.  A stage therefore holds up to 8 KB, so
// 6 CTAs per SM keep enough bytes in flight where one 1152-byte page per
// stage needed 24, and the store side issues 8 KB copies.  With fewer, leaner
// CTAs the next layer's early fill fits beside the gather.  Measured per
// 78-layer step on one-token pages: 5.312 -> 4.863 ms (gather alone 53.2 ->
// 52.2 us); 16 KB groups at 3-4 CTAs per SM were slower (5.07-5.45 ms), as
// were 3 groups in flight (5.38 ms).  Runs never
// cross table entries or mix pools with stagings, so a consumed staging run
// never covers pool bytes.  Used only when every slot kind is written (a
// skipped slot must keep its bytes).
template <bool kConsume>
__global__ void __launch_bounds__(32) gather_groups_kernel(const __grid_constant__ GatherParams p) {
  release_dependents();  // as in gather_pages_kernel
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t full[kGroupStages];
  __shared__ uint8_t *st_dst[kGroupStages];
  __shared__ uint32_t st_bytes[kGroupStages];
  __shared__ int st_live[kGroupStages];
  __shared__ const uint8_t *st_drop_src[kGroupStages][32];
  __shared__ uint32_t st_drop_bytes[kGroupStages][32];
  __shared__ int st_drop_n[kGroupStages];
  const int lane = threadIdx.x;
  const uint32_t pb = (uint32_t)p.page_bytes;
  GroupRing<kConsume> ring;
  ring.init(smem, full, st_dst, st_bytes, st_live, st_drop_src, st_drop_bytes, st_drop_n, p.status,
            (uint32_t)(p.group * p.page_bytes));
  // Group u covers dense pages [u * G, min(u * G + G, dense_cap)).  The next
  // group's descriptors are loaded before the current group is issued.
  const int G = p.group;
  const int64_t step = gridDim.x;
  int32_t o = -1, sr = 0;
  int64_t u = blockIdx.x;
  if (u < p.units && lane < min64(G, p.dense_cap - u * G)) {
    o = p.owner[u * G + lane];
    sr = p.src[u * G + lane];
  }
  for (; u < p.units; u += step) {
    const int64_t d0 = u * G;
    const int n = (int)min64(G, p.dense_cap - d0);
    const int64_t v = u + step;
    int32_t o_next = -1, s_next = 0;
    if (v < p.units && lane < min64(G, p.dense_cap - v * G)) {
      o_next = p.owner[v * G + lane];
      s_next = p.src[v * G + lane];
    }
    // my page: a whole-page copy from its table entry, or zeros (owner -1,
    // invalid descriptors)
    GroupPage pg{nullptr, 0, -1, false};
    if (lane < n && o != -1) {
      if (o < -1 || o >= p.n_table || sr < 0 || sr >= p.cap_pages[o]) {
        raise_status(p.status, CPKV_STATUS_DESC_OOB);
      } else {
        pg.src = p.table[o] + (int64_t)sr * p.page_bytes;
        pg.copy = pb;
        pg.entry = o;
        pg.staging = o >= p.n_pool;
      }
    }
    ring.push_group(p.dense + d0 * p.page_bytes, n, pb, pg);
    o = o_next;
    sr = s_next;
  }
  ring.drain();
}

}  // namespace
}  // namespace cpkv

extern "C" int cpkv_compose_gather_kinds(int page_size, int cp_size, int64_t row_bytes,
                                         const void *const *h_src_table, const int64_t *h_src_cap_pages,
                                         const int32_t *d_owner, const int32_t *d_src, int64_t dense_cap_pages,
                                         int kinds, void *d_dense, int32_t *d_status, cpkv_stream_t stream) {
  using namespace cpkv;
  if (kinds < 0 || kinds > (CPKV_GATHER_ALL | CPKV_GATHER_CONSUME_STAGING | CPKV_GATHER_EARLY_INPUTS))
    return CPKV_ERR_ARG;
  const bool consume = (kinds & CPKV_GATHER_CONSUME_STAGING) != 0;
  const bool early = (kinds & CPKV_GATHER_EARLY_INPUTS) != 0;
  kinds &= CPKV_GATHER_ALL;
  if (page_size <= 0 || cp_size < 1 || cp_size > CPKV_MAX_CP) return CPKV_ERR_ARG;
  if (row_bytes <= 0 || ((int64_t)page_size * row_bytes) % 16 != 0 || dense_cap_pages < 0) return CPKV_ERR_ARG;
  if (h_src_table == nullptr || h_src_cap_pages == nullptr || d_status == nullptr) return CPKV_ERR_ARG;
  if (dense_cap_pages == 0) return CPKV_OK;
  if (d_owner == nullptr || d_src == nullptr || d_dense == nullptr || !aligned16(d_dense)) return CPKV_ERR_ARG;
  const int n_table = 2 * cp_size;
  for (int k = 0; k < n_table; ++k) {
    if (h_src_cap_pages[k] < 0) return CPKV_ERR_ARG;
    if (h_src_cap_pages[k] > 0 && (h_src_table[k] == nullptr || !aligned16(h_src_table[k]))) return CPKV_ERR_ARG;
  }
  const int64_t page_bytes = (int64_t)page_size * row_bytes;
  const int64_t pieces = ceil_div(page_bytes, kMaxPieceBytes);
  const int64_t piece_bytes = ceil_div(ceil_div(page_bytes, pieces), 16) * 16;
  if (pieces > INT32_MAX || dense_cap_pages > INT64_MAX / pieces) return CPKV_ERR_LIMIT;

  GatherParams prm;
  for (int k = 0; k < 2 * CPKV_MAX_CP; ++k) {
    prm.table[k] = k < n_table ? static_cast<const uint8_t *>(h_src_table[k]) : nullptr;
    prm.cap_pages[k] = k < n_table ? h_src_cap_pages[k] : 0;
  }
  prm.owner = d_owner;
  prm.src = d_src;
  prm.dense = static_cast<uint8_t *>(d_dense);
  prm.status = d_status;
  prm.dense_cap = dense_cap_pages;
  prm.page_bytes = page_bytes;
  prm.units = dense_cap_pages * pieces;
  prm.n_table = n_table;
  prm.n_pool = cp_size;
  prm.kinds = kinds;
  prm.pieces = (int32_t)pieces;
  prm.piece_bytes = (int32_t)piece_bytes;
  prm.group = 1;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

  if (pieces == 1 && kinds == CPKV_GATHER_ALL && page_bytes * 2 <= kGroupBytes) {
    // small pages, every slot written: groups of pages, runs merged
    const int64_t G = kGroupBytes / page_bytes < 32 ? kGroupBytes / page_bytes : 32;
    prm.group = (int32_t)G;
    prm.units = ceil_div(dense_cap_pages, G);
    const size_t gsmem = (size_t)kGroupStages * (size_t)(G * page_bytes);
    const void *gkernel = consume ? reinterpret_cast<const void *>(gather_groups_kernel<true>)
                                  : reinterpret_cast<const void *>(gather_groups_kernel<false>);
    if (ensure_dynamic_smem(gkernel, kGroupStages * kGroupBytes) != CPKV_OK) return CPKV_ERR_CUDA;
    const int ggrid = persistent_grid(gkernel, 32, gsmem, kMaxCtasPerSmGroups, prm.units);
    const bool gdep = early;  // 6 CTAs per SM of 8 KB groups: early pays (4.49 -> 4.41 ms per one-token step)
    if (consume) return launch_kernel(gather_groups_kernel<true>, dim3(ggrid), dim3(32), gsmem, gdep, s, prm);
    return launch_kernel(gather_groups_kernel<false>, dim3(ggrid), dim3(32), gsmem, gdep, s, prm);
  }

  const size_t smem = (size_t)kStages * piece_bytes;
  const void *kernel = consume ? reinterpret_cast<const void *>(gather_pages_kernel<true>)
                               : reinterpret_cast<const void *>(gather_pages_kernel<false>);
  if (ensure_dynamic_smem(kernel, kStages * kMaxPieceBytes) != CPKV_OK) return CPKV_ERR_CUDA;
  const int grid =
      persistent_grid(kernel, 32, smem,
                      pieces > 1 ? kMaxCtasPerSmPieces
                                 : ring_cap_one_piece(piece_bytes, kLoadsInFlight, kMaxCtasPerSmOnePiece),
                      prm.units);
  const bool dependent = early && early_launch_pays(grid);
  if (consume) return launch_kernel(gather_pages_kernel<true>, dim3(grid), dim3(32), smem, dependent, s, prm);
  return launch_kernel(gather_pages_kernel<false>, dim3(grid), dim3(32), smem, dependent, s, prm);
}

extern "C" int cpkv_compose_gather(int page_size, int cp_size, int64_t row_bytes,
                                   const void *const *h_src_table, const int64_t *h_src_cap_pages,
                                   const int32_t *d_owner, const int32_t *d_src, int64_t dense_cap_pages,
                                   void *d_dense, int32_t *d_status, cpkv_stream_t stream) {
  return cpkv_compose_gather_kinds(page_size, cp_size, row_bytes, h_src_table, h_src_cap_pages, d_owner, d_src,
                                   dense_cap_pages, CPKV_GATHER_ALL, d_dense, d_status, stream);
}
