// cpkv_compose_fused: the single-GPU compose in one pass per layer.
//
// The staging exchange of the pages ("staging-direct compose" message of
// commits d63fbd4) exists because current pages are computed on other GPUs:
// each rank fills its own current pages into its staging, and every rank
// gathers all of them back.  When every writer region lives on this GPU the
// round trip through staging is not needed: a current page's rows are already
// contiguous in its writer's current-row buffer (tokens of one page are
// consecutive in batch order and have one writer), so the dense page can be
// copied straight from there, followed by zero pad rows.  The pages' own
// measurements point the same way: the staging-direct design measured 62.8 ms
// per batch against a 60.8 ms ideal, the gap being structure, not copies.
//
// One launch per layer moves every dense page exactly once:
//   owner -1           -> zeros
//   owner r < cp       -> page src of pool slab r (modulo-owner prefix page)
//   owner cp + w       -> current page i = src - 1 of writer w: its n_i rows
//                         from cur_rows[w] starting at token_writer_row of the
//                         page's first token, then ps - n_i zero rows
// The descriptors are the ones cpkv_plan_build writes for the gather.  The
// output is byte-identical to cpkv_fill_current followed by
// cpkv_compose_gather.  Same bulk-copy ring as the gather (bulk_ring.cuh),
// with up to 3 one-warp CTAs per SM for pages of several pieces and the
// gather's in-flight rule for pages of one piece.
#include <stdint.h>

#include "group_ring.cuh"

namespace cpkv {
namespace {

constexpr int kStages = 4;
constexpr int kLoadsInFlight = 2;
constexpr int kMaxCtasPerSm = 3;  // one-warp CTAs per SM, at most; fewer when their rings do not fit
// With CPKV_FLAG_EARLY_INPUTS and a grid of at most 4 CTAs per SM
// (early_launch_pays), the kernel is
// launched as a programmatic dependent of the previous kernel on the stream:
// its CTAs may start in SM slots that the previous launch's tail frees, read
// their inputs at once, and wait for that launch (store_gate) only before
// their first global store.  Measured per 78-layer step: traced
// 4.045 -> 3.807 ms, fp8 17.99 -> 17.64 ms; waiting before the first load
// instead kept only 4.045 -> 3.993 ms.  Index-key pages (one 8448-byte
// piece, 3 CTAs per SM): 3.947 -> 3.700 ms.  One-token pages run 24 small
// CTAs per SM, where the next launch's CTAs would sit beside the current
// ones from the start (4.27 -> 4.70 ms), so that grid launches plainly.
// In a plain launch the waits return at once.
constexpr int kMaxPieceBytes = 24 * 1024;

template <int MAXB>
struct FusedParams {
  const uint8_t *pool[CPKV_MAX_CP];
  int64_t pool_cap[CPKV_MAX_CP];
  const uint8_t *cur_rows[CPKV_MAX_CP];
  int64_t cur_cap[CPKV_MAX_CP];
  const int32_t *owner, *src, *token_writer_row;
  uint8_t *dense;
  int32_t *status;
  int64_t dense_cap, page_bytes, units, R, C;
  int32_t cp, ps, B, pieces, piece_bytes;
  int32_t cur_lens[MAXB];
};

template <int MAXB>
__global__ void __launch_bounds__(32) compose_fused_kernel(const __grid_constant__ FusedParams<MAXB> p) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t full[kStages];
  __shared__ uint8_t *ring_dst[kStages];
  __shared__ uint32_t ring_bytes[kStages];
  __shared__ int ring_live[kStages];
  __shared__ int32_t cur_page_start[MAXB + 1];  // first batch current page of request b
  __shared__ int64_t token_start[MAXB + 1];     // first batch token of request b
  const int lane = threadIdx.x;
  release_dependents();
  bool stores_open = false;  // store_gate: warp-uniform here

  // request-level exclusive scans, 32 requests per step
  {
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

  BulkRing<kStages, kLoadsInFlight> ring;
  ring.init(smem, full, ring_dst, ring_bytes, ring_live, p.status, p.piece_bytes);
  // units u = blockIdx.x + i * gridDim.x; descriptors loaded 32 at a time
  const int64_t step = gridDim.x;
  for (int64_t base = blockIdx.x; base < p.units; base += 32 * step) {
   const int64_t mine = base + lane * step;
   int32_t my_o = -1, my_s = 0;
   if (mine < p.units) {
     my_o = p.owner[mine / p.pieces];
     my_s = p.src[mine / p.pieces];
   }
   // for a current page, also its first token's row in the writer's buffer
   int32_t my_row0 = -1;
   if (my_o >= p.cp && my_o < 2 * p.cp && my_s >= 1 && my_s <= p.C && p.B > 0) {
     const int b = upper_index<int32_t>(cur_page_start, p.B, my_s - 1);
     const int64_t tok0 = token_start[b] + (int64_t)(my_s - 1 - cur_page_start[b]) * p.ps;
     my_row0 = p.token_writer_row[tok0];
   }
   for (int jj = 0; jj < 32; ++jj) {
    const int64_t u = base + jj * step;
    if (u >= p.units) break;  // uniform across the warp
    const int64_t d = u / p.pieces;
    const int32_t k = (int32_t)(u - d * p.pieces);
    const int64_t off = (int64_t)k * p.piece_bytes;
    const uint32_t bytes = (uint32_t)min64(p.piece_bytes, p.page_bytes - off);
    uint8_t *dst = p.dense + d * p.page_bytes + off;
    const int32_t o = __shfl_sync(0xffffffffu, my_o, jj);
    const int32_t s = __shfl_sync(0xffffffffu, my_s, jj);
    const int32_t row0 = __shfl_sync(0xffffffffu, my_row0, jj);
    if (o >= 0 && o < p.cp && s >= 0 && s < p.pool_cap[o]) {
      if (ring.tail - ring.head == kLoadsInFlight) store_gate(&stores_open);  // this push stores
      ring.push(p.pool[o] + (int64_t)s * p.page_bytes + off, dst, bytes);
      continue;
    }
    int64_t copy = 0;  // bytes of this piece that come from current rows
    const uint8_t *from = nullptr;
    bool bad = o != -1 && !(o >= p.cp && o < 2 * p.cp);
    if (!bad && o >= p.cp) {
      const int32_t w = o - p.cp;
      const int32_t i = s - 1;  // batch current page index
      if (i < 0 || i >= p.C || p.B == 0) {
        bad = true;
      } else {
        const int b = upper_index<int32_t>(cur_page_start, p.B, i);
        const int32_t kp = i - cur_page_start[b];
        const int64_t n = min64(p.ps, (int64_t)p.cur_lens[b] - (int64_t)kp * p.ps);
        if (n < 1 || row0 < 0 || row0 + n > p.cur_cap[w]) {
          bad = true;
        } else {
          const int64_t rows_bytes = n * p.R;
          copy = off < rows_bytes ? min64(bytes, rows_bytes - off) : 0;
          from = p.cur_rows[w] + (int64_t)row0 * p.R + off;
        }
      }
    }
    if (bad) {
      if (lane == 0 && k == 0) raise_status(p.status, CPKV_STATUS_DESC_OOB);
      copy = 0;
    }
    if (copy > 0) {
      if (ring.tail - ring.head == kLoadsInFlight) store_gate(&stores_open);  // this push stores
      ring.push(from, dst, (uint32_t)copy);
    }
    if (copy < bytes) {
      store_gate(&stores_open);
      warp_zero(dst + copy, bytes - (uint32_t)copy);
    }
   }
  }
  store_gate(&stores_open);
  ring.drain();
}

// ---------------------------------------------------------------------------
// Small pages (at most 4 KB, one piece): groups of consecutive dense pages
// through the group ring (group_ring.cuh), as the small-page gather does.
// Lane j describes the group's page j: a pool page (a whole-page copy), a
// current page (its n rows from the writer's buffer, then zero pad rows), or
// zeros.  Runs merge consecutive pool pages of one owner and consecutive
// current pages of one writer whose rows follow each other.  A current
// page's first row (token_writer_row of its first token) depends on its
// descriptor, so descriptors are loaded two groups ahead and first rows one
// group ahead.  Measured per 78-layer step on one-token pages (1152 bytes):
// 4.27 -> 4.055 ms against one page per ring slot at 24 CTAs per SM; the
// kernel alone 0.85 -> 0.893 of the copy peak.  The grid runs 6 CTAs per SM
// and launches early whenever asked, unlike the one-page-per-slot ring at 24
// CTAs per SM that early_launch_pays keeps plain: 4.05 -> 3.72 ms per step.
template <int MAXB>
__device__ __forceinline__ int32_t group_row0(const FusedParams<MAXB> &p, const int32_t *cur_page_start,
                                              const int64_t *token_start, int32_t o, int32_t s) {
  if (o < p.cp || o >= 2 * p.cp || s < 1 || s > p.C || p.B == 0) return -1;
  const int b = upper_index<int32_t>(cur_page_start, p.B, s - 1);
  return p.token_writer_row[token_start[b] + (int64_t)(s - 1 - cur_page_start[b]) * p.ps];
}

template <int MAXB>
__global__ void __launch_bounds__(32) compose_fused_groups_kernel(const __grid_constant__ FusedParams<MAXB> p) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t full[kGroupStages];
  __shared__ uint8_t *st_dst[kGroupStages];
  __shared__ uint32_t st_bytes[kGroupStages];
  __shared__ int st_live[kGroupStages];
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
  GroupRing<false> ring;
  ring.init(smem, full, st_dst, st_bytes, st_live, nullptr, nullptr, nullptr, p.status,
            (uint32_t)(p.pieces * p.page_bytes));
  const int G = p.pieces;  // pages per group (FusedParams.pieces holds G here)
  const int64_t step = gridDim.x;
  auto load_desc = [&](int64_t v, int32_t &o, int32_t &s) {
    o = -1;
    s = 0;
    if (v < p.units && lane < min64(G, p.dense_cap - v * G)) {
      o = p.owner[v * G + lane];
      s = p.src[v * G + lane];
    }
  };
  int64_t u = blockIdx.x;
  int32_t o0, s0, o1, s1;
  load_desc(u, o0, s0);
  load_desc(u + step, o1, s1);
  int32_t r0 = group_row0(p, cur_page_start, token_start, o0, s0);
  for (; u < p.units; u += step) {
    const int64_t d0 = u * G;
    const int n = (int)min64(G, p.dense_cap - d0);
    int32_t o2, s2;
    load_desc(u + 2 * step, o2, s2);
    const int32_t r1 = group_row0(p, cur_page_start, token_start, o1, s1);
    GroupPage pg{nullptr, 0, -1, false};
    if (lane < n && o0 != -1) {
      if (o0 >= 0 && o0 < p.cp && s0 >= 0 && s0 < p.pool_cap[o0]) {
        pg.src = p.pool[o0] + (int64_t)s0 * p.page_bytes;
        pg.copy = pb;
        pg.entry = o0;
      } else {
        bool bad = !(o0 >= p.cp && o0 < 2 * p.cp) || s0 < 1 || s0 > p.C || p.B == 0;
        if (!bad) {
          const int32_t w = o0 - p.cp, i = s0 - 1;
          const int b = upper_index<int32_t>(cur_page_start, p.B, i);
          const int64_t nr = min64(p.ps, (int64_t)p.cur_lens[b] - (int64_t)(i - cur_page_start[b]) * p.ps);
          if (nr < 1 || r0 < 0 || r0 + nr > p.cur_cap[w]) {
            bad = true;
          } else {
            pg.src = p.cur_rows[w] + (int64_t)r0 * p.R;
            pg.copy = (uint32_t)(nr * p.R);
            pg.entry = o0;
          }
        }
        if (bad) raise_status(p.status, CPKV_STATUS_DESC_OOB);
      }
    }
    ring.push_group(p.dense + d0 * p.page_bytes, n, pb, pg);
    o0 = o1; s0 = s1; r0 = r1;
    o1 = o2; s1 = s2;
  }
  ring.drain();
}

// Launch, as a programmatic dependent of the previous kernel when `dependent`.
template <typename Params>
int launch_fused(void (*kernel)(Params), int grid, size_t smem, bool dependent, cudaStream_t s,
                 const Params &prm) {
  return launch_kernel(kernel, dim3(grid), dim3(32), smem, dependent, s, prm);
}

}  // namespace
}  // namespace cpkv

extern "C" int cpkv_compose_fused(int B, int page_size, int cp_size, int64_t row_bytes, const int32_t *h_cur_lens,
                                  const void *const *h_pools, const int64_t *h_pool_cap_pages,
                                  const void *const *h_cur_rows, const int64_t *h_cur_rows_cap,
                                  const int32_t *d_owner, const int32_t *d_src, const int32_t *d_token_writer_row,
                                  int64_t dense_cap_pages, void *d_dense, int flags, int32_t *d_status,
                                  cpkv_stream_t stream) {
  using namespace cpkv;
  if ((flags & ~CPKV_FLAG_EARLY_INPUTS) != 0) return CPKV_ERR_ARG;
  const bool early = (flags & CPKV_FLAG_EARLY_INPUTS) != 0;
  if (B < 0 || page_size <= 0 || cp_size < 1 || cp_size > CPKV_MAX_CP) return CPKV_ERR_ARG;
  if (row_bytes <= 0 || row_bytes % 16 != 0 || dense_cap_pages < 0) return CPKV_ERR_ARG;
  if (B > CPKV_MAX_BATCH) return CPKV_ERR_LIMIT;
  if (h_pools == nullptr || h_pool_cap_pages == nullptr || h_cur_rows == nullptr || h_cur_rows_cap == nullptr ||
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
  if (dense_cap_pages == 0) return CPKV_OK;
  if (d_owner == nullptr || d_src == nullptr || d_dense == nullptr || !aligned16(d_dense)) return CPKV_ERR_ARG;
  if (T > 0 && d_token_writer_row == nullptr) return CPKV_ERR_ARG;
  for (int k = 0; k < cp_size; ++k) {
    if (h_pool_cap_pages[k] < 0 || h_cur_rows_cap[k] < 0) return CPKV_ERR_ARG;
    if (h_pool_cap_pages[k] > 0 && (h_pools[k] == nullptr || !aligned16(h_pools[k]))) return CPKV_ERR_ARG;
    if (h_cur_rows_cap[k] > 0 && (h_cur_rows[k] == nullptr || !aligned16(h_cur_rows[k]))) return CPKV_ERR_ARG;
  }
  const int64_t page_bytes = (int64_t)page_size * row_bytes;
  const int64_t pieces = ceil_div(page_bytes, kMaxPieceBytes);
  const int64_t piece_bytes = ceil_div(ceil_div(page_bytes, pieces), 16) * 16;
  if (pieces > INT32_MAX || dense_cap_pages > INT64_MAX / pieces) return CPKV_ERR_LIMIT;
  const int64_t units = dense_cap_pages * pieces;
  const size_t smem = (size_t)kStages * piece_bytes;
  const int cap_per_sm = pieces > 1 ? kMaxCtasPerSm : ring_cap_one_piece(piece_bytes, kLoadsInFlight, kMaxCtasPerSm);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

#define CPKV_FILL_FUSED(prm)                                                                        \
  for (int k = 0; k < CPKV_MAX_CP; ++k) {                                                           \
    prm.pool[k] = k < cp_size ? static_cast<const uint8_t *>(h_pools[k]) : nullptr;                 \
    prm.pool_cap[k] = k < cp_size ? h_pool_cap_pages[k] : 0;                                        \
    prm.cur_rows[k] = k < cp_size ? static_cast<const uint8_t *>(h_cur_rows[k]) : nullptr;          \
    prm.cur_cap[k] = k < cp_size ? h_cur_rows_cap[k] : 0;                                           \
  }                                                                                                 \
  prm.owner = d_owner; prm.src = d_src; prm.token_writer_row = d_token_writer_row;                  \
  prm.dense = static_cast<uint8_t *>(d_dense); prm.status = d_status; prm.dense_cap = dense_cap_pages; \
  prm.page_bytes = page_bytes; prm.units = units; prm.R = row_bytes; prm.C = C; prm.cp = cp_size;  \
  prm.ps = page_size; prm.B = B; prm.pieces = (int32_t)pieces; prm.piece_bytes = (int32_t)piece_bytes; \
  for (int b = 0; b < B; ++b) prm.cur_lens[b] = h_cur_lens[b];

  if (pieces == 1 && page_bytes * 2 <= kGroupBytes) {
    // small pages: groups of consecutive dense pages, runs merged
    const int64_t G = kGroupBytes / page_bytes < 32 ? kGroupBytes / page_bytes : 32;
    const int64_t gunits = ceil_div(dense_cap_pages, G);
    const size_t gsmem = (size_t)kGroupStages * (size_t)(G * page_bytes);
#define CPKV_FUSED_GROUPS(MB)                                                                       \
  {                                                                                                 \
    const void *kernel = reinterpret_cast<const void *>(compose_fused_groups_kernel<MB>);           \
    if (ensure_dynamic_smem(kernel, kGroupStages * kGroupBytes) != CPKV_OK) return CPKV_ERR_CUDA;   \
    const int grid = persistent_grid(kernel, 32, gsmem, kMaxCtasPerSmGroups, gunits);               \
    FusedParams<MB> prm;                                                                            \
    CPKV_FILL_FUSED(prm)                                                                            \
    prm.units = gunits; prm.pieces = (int32_t)G; prm.piece_bytes = (int32_t)page_bytes;             \
    return launch_fused(compose_fused_groups_kernel<MB>, grid, gsmem, early, s, prm); \
  }
    if (B <= 64) CPKV_FUSED_GROUPS(64)
    CPKV_FUSED_GROUPS(CPKV_MAX_BATCH)
#undef CPKV_FUSED_GROUPS
  }

  if (B <= 64) {
    const void *kernel = reinterpret_cast<const void *>(compose_fused_kernel<64>);
    if (ensure_dynamic_smem(kernel, kStages * kMaxPieceBytes) != CPKV_OK) return CPKV_ERR_CUDA;
    const int grid = persistent_grid(kernel, 32, smem, cap_per_sm, units);
    FusedParams<64> prm;
    CPKV_FILL_FUSED(prm)
    return launch_fused(compose_fused_kernel<64>, grid, smem, early && early_launch_pays(grid), s, prm);
  }
  const void *kernel = reinterpret_cast<const void *>(compose_fused_kernel<CPKV_MAX_BATCH>);
  if (ensure_dynamic_smem(kernel, kStages * kMaxPieceBytes) != CPKV_OK) return CPKV_ERR_CUDA;
  const int grid = persistent_grid(kernel, 32, smem, cap_per_sm, units);
  FusedParams<CPKV_MAX_BATCH> prm;
  CPKV_FILL_FUSED(prm)
#undef CPKV_FILL_FUSED
  return launch_fused(compose_fused_kernel<CPKV_MAX_BATCH>, grid, smem, early && early_launch_pays(grid), s, prm);
}
