// cpkv_plan_build: the per-batch compose plan on the device.
//
// Two launches on the caller's stream, the second a programmatic dependent
// of the first (it starts early and waits for the first only before it
// touches what the first writes):
//   1. plan_init   — blocks [0, nInit): page_inverse[:] = -1,
//                    staging_page_inverse[:] = 0 (P entries each, the only
//                    P-sized work); blocks [nInit, nInit + NB): per token
//                    block j, the rows of each writer in its K current pages
//                    (workspace[j][w]).
//   2. plan_main   — blocks [0, nA): one thread per dense slot: descriptors
//                    (owner, src) and the inverse scatters, plus the spans
//                    (block 0); blocks [nA, nA + NB): K current pages per
//                    block: per-writer row bases and the per-token arrays.
// The per-writer row base of a current page (the row of its first token in
// its writer's current-row buffer) is an exclusive sum over earlier pages of
// the same writer.  It is taken in two levels: across token blocks from the
// workspace (a block adds the totals of the blocks before it, cp values
// each), inside a block by warp matching and a scan over its warps.  So the
// work is linear in the number of current pages; K grows as the page size
// shrinks (about 2048 tokens per block, 32 to 1024 pages), which keeps
// blocks few and full on one-token pages.  Measured per build, 10 builds back
// to back in a CUDA graph: traced batch 6.36 us, fp8 batch 8.0 us, traced
// lengths on one-token pages 8.2 us.  Each block counting the pages before it
// itself (no workspace, no wait for plan_init) measured slower: 6.77, 9.5 and
// 8.2 us.  The first form, each 32-page block rescanning all earlier pages,
// took 78 us per build on one-token pages.
// (Token blocks that hold only part of a warp's pages, and warps without a
// short page, skip the per-lane row sums: a full page holds ps rows.)
// Host lengths travel as kernel parameters (__grid_constant__), so nothing
// is copied host-to-device and nothing syncs.  Every block that needs them
// rebuilds the request-level exclusive scans in shared memory (B <= 1024).
//
// Method: "staging-direct compose" message of commits d63fbd4 (spans,
// descriptors, staging-remapped inverse, mixed_locs / staging rows built once
// per batch); "prefetch staging" message of commits 0d87bc5 (slot i + 1,
// row 0 reserved); modulo-owner prefix placement ("owner_check" message).
#include <stdint.h>

#include "common.cuh"

namespace cpkv {
namespace {

constexpr int kPlanThreads = 1024;
constexpr int kTokensPerBlock = 2048;    // tokens a token block writes, about
constexpr int kMaxPagesPerBlock = 1024;  // one current page per thread

template <int MAXB>
struct PlanParams {
  int B, ps, cp, nA, nInit, K, NB;  // K current pages per token block, NB token blocks
  bool vec;                         // the inverses are 16-byte aligned
  int64_t P, dense_cap, D, C, T;
  const int32_t *prefix_pages, *cur_pages, *writer;
  int32_t *prefix_spans, *cur_spans, *owner, *src, *page_inverse, *staging_page_inverse;
  int64_t *mixed_locs, *staging_rows;
  int32_t *token_writer_row, *status;
  int32_t *block_rows;  // workspace [NB][cp]: rows of writer w in token block j's pages
  int32_t prefix_lens[MAXB];
  int32_t cur_lens[MAXB];
};

// Request-level exclusive scans, one request per thread (B <= 1024).
template <int MAXB>
struct RequestScan {
  int32_t dense_start[MAXB + 1];        // first dense slot of request b
  int32_t cur_page_start[MAXB + 1];     // first batch current page index
  int32_t prefix_page_start[MAXB + 1];  // CSR offset into prefix_pages
  int64_t token_start[MAXB + 1];        // first batch token
  int64_t scratch64[33];
};

template <int MAXB>
__device__ void build_request_scan(const PlanParams<MAXB> &p, RequestScan<MAXB> &rs) {
  if (p.B <= 32) {  // one warp: shuffle scans and a single barrier
    if (threadIdx.x < 32) {
      const int b = threadIdx.x;
      int64_t npp = 0, ncp = 0, cur = 0;
      if (b < p.B) {
        npp = p.prefix_lens[b] / p.ps;
        cur = p.cur_lens[b];
        ncp = (cur + p.ps - 1) / p.ps;
      }
      const int64_t ds = warp_inclusive_scan<int64_t>(npp + ncp);
      const int64_t cs = warp_inclusive_scan<int64_t>(ncp);
      const int64_t pp = warp_inclusive_scan<int64_t>(npp);
      const int64_t ts = warp_inclusive_scan<int64_t>(cur);
      if (b < p.B) {
        rs.dense_start[b] = (int32_t)(ds - npp - ncp);
        rs.cur_page_start[b] = (int32_t)(cs - ncp);
        rs.prefix_page_start[b] = (int32_t)(pp - npp);
        rs.token_start[b] = ts - cur;
      }
      if (b == 31) {  // lanes past B add nothing, so lane 31 holds the totals
        rs.dense_start[p.B] = (int32_t)ds;
        rs.cur_page_start[p.B] = (int32_t)cs;
        rs.prefix_page_start[p.B] = (int32_t)pp;
        rs.token_start[p.B] = ts;
      }
    }
    __syncthreads();
    return;
  }
  const int b = threadIdx.x;
  const int ps = p.ps;
  int64_t npp = 0, ncp = 0, cur = 0;
  if (b < p.B) {
    npp = p.prefix_lens[b] / ps;
    cur = p.cur_lens[b];
    ncp = (cur + ps - 1) / ps;
  }
  int64_t tot;
  const int64_t ds = block_exclusive_scan<int64_t>(npp + ncp, rs.scratch64, &tot);
  if (b < p.B) rs.dense_start[b] = (int32_t)ds;
  if (b == 0) rs.dense_start[p.B] = (int32_t)tot;
  const int64_t cs = block_exclusive_scan<int64_t>(ncp, rs.scratch64, &tot);
  if (b < p.B) rs.cur_page_start[b] = (int32_t)cs;
  if (b == 0) rs.cur_page_start[p.B] = (int32_t)tot;
  const int64_t pp = block_exclusive_scan<int64_t>(npp, rs.scratch64, &tot);
  if (b < p.B) rs.prefix_page_start[b] = (int32_t)pp;
  if (b == 0) rs.prefix_page_start[p.B] = (int32_t)tot;
  const int64_t ts = block_exclusive_scan<int64_t>(cur, rs.scratch64, &tot);
  if (b < p.B) rs.token_start[b] = ts;
  if (b == 0) rs.token_start[p.B] = tot;
  __syncthreads();
}

template <int MAXB>
__device__ bool slot_is_prefix(const PlanParams<MAXB> &p, const RequestScan<MAXB> &rs, int32_t slot) {
  if (slot < 0 || slot >= p.D || p.B == 0) return false;
  const int b = upper_index<int32_t>(rs.dense_start, p.B, slot);
  return slot - rs.dense_start[b] < p.prefix_lens[b] / p.ps;
}

// One thread per dense slot: descriptors and inverse scatters.
template <int MAXB>
__device__ void plan_dense_slots(const PlanParams<MAXB> &p, const RequestScan<MAXB> &rs) {
  const int64_t d = (int64_t)blockIdx.x * kPlanThreads + threadIdx.x;
  if (blockIdx.x == 0 && threadIdx.x < p.B) {
    const int b = threadIdx.x;
    const int32_t npp = p.prefix_lens[b] / p.ps;
    p.prefix_spans[2 * b] = rs.dense_start[b];
    p.prefix_spans[2 * b + 1] = npp;
    p.cur_spans[2 * b] = rs.dense_start[b] + npp;
    p.cur_spans[2 * b + 1] = rs.cur_page_start[b + 1] - rs.cur_page_start[b];
  }
  if (d >= p.dense_cap) return;
  int32_t owner = -1, src = 0;
  if (d < p.D) {
    const int b = upper_index<int32_t>(rs.dense_start, p.B, (int32_t)d);
    const int32_t k = (int32_t)d - rs.dense_start[b];
    const int32_t npp = p.prefix_lens[b] / p.ps;
    const unsigned int slot = (unsigned int)d;
    // the page tables are loaded before waiting for plan_init
    const bool is_prefix = k < npp;
    const int32_t i = is_prefix ? 0 : rs.cur_page_start[b] + (k - npp);
    const int32_t lp = is_prefix ? p.prefix_pages[rs.prefix_page_start[b] + k] : p.cur_pages[i];
    const int32_t w = is_prefix ? 0 : p.writer[i];
    wait_prerequisite();
    if (is_prefix) {
      if (lp < 1 || lp >= p.P) {
        raise_status(p.status, CPKV_STATUS_PAGE_OOB);
      } else {
        owner = lp % p.cp;
        src = lp / p.cp;
        const unsigned int old = atomicMin(reinterpret_cast<unsigned int *>(p.page_inverse) + lp, slot);
        // a collision with a current page's slot breaks single-writer
        if (old != 0xffffffffu && !slot_is_prefix(p, rs, (int32_t)old))
          raise_status(p.status, CPKV_STATUS_CURRENT_IN_PREFIX);
      }
    } else {
      if (lp < 1 || lp >= p.P) {
        raise_status(p.status, CPKV_STATUS_PAGE_OOB);
      } else if (w < 0 || w >= p.cp) {
        raise_status(p.status, CPKV_STATUS_WRITER_OOB);
      } else {
        owner = p.cp + w;
        src = i + 1;
        if (atomicExch(p.staging_page_inverse + lp, i + 1) != 0)
          raise_status(p.status, CPKV_STATUS_DUP_CURRENT_PAGE);
        const unsigned int old = atomicMin(reinterpret_cast<unsigned int *>(p.page_inverse) + lp, slot);
        if (old != 0xffffffffu && slot_is_prefix(p, rs, (int32_t)old))
          raise_status(p.status, CPKV_STATUS_CURRENT_IN_PREFIX);
      }
    }
  }
  p.owner[d] = owner;
  p.src[d] = src;
}

// Current page i of the batch: its rows n (ps, or fewer on a request's last
// page), its first token, its dense slot, and its writer (-1 when out of
// range).
template <int MAXB>
struct CurPage {
  int32_t n, w, slot;
  int64_t tok0;
};

template <int MAXB>
__device__ CurPage<MAXB> current_page(const PlanParams<MAXB> &p, const RequestScan<MAXB> &rs, int64_t i) {
  CurPage<MAXB> c;
  const int b = upper_index<int32_t>(rs.cur_page_start, p.B, (int32_t)i);
  const int32_t kp = (int32_t)i - rs.cur_page_start[b];  // page index inside the request
  c.n = min(p.ps, p.cur_lens[b] - kp * p.ps);
  c.tok0 = rs.token_start[b] + (int64_t)kp * p.ps;
  c.slot = rs.dense_start[b] + p.prefix_lens[b] / p.ps + kp;
  c.w = p.writer[i];
  if (c.w < 0 || c.w >= p.cp) c.w = -1;
  return c;
}

// Rows of the lanes below this one whose writer is the same (`peers`, from
// __match_any_sync), and the group's total (warp-uniform call).  A lane
// whose page is full holds ps rows, so a warp without short pages (only a
// request's last page can be short) counts lanes; otherwise the rows are
// summed over the lanes by shuffles.
__device__ __forceinline__ void same_writer_rows(unsigned int peers, int32_t n, bool valid, int ps, int32_t *before,
                                                 int32_t *total) {
  const int lane = threadIdx.x & 31;
  const unsigned int below = (1u << lane) - 1u;
  if (__ballot_sync(0xffffffffu, valid && n != ps) == 0u) {
    *before = ps * __popc(peers & below);
    *total = ps * __popc(peers);
    return;
  }
  int32_t b = 0, t = 0;
#pragma unroll
  for (int l = 0; l < 32; ++l) {
    const int32_t nl = __shfl_sync(0xffffffffu, n, l);
    if ((peers >> l) & 1u) {
      t += nl;
      if (l < lane) b += nl;
    }
  }
  *before = b;
  *total = t;
}

// Add the rows of each writer in current pages [first, last) to rows[w]
// (shared, block-wide call: one page per thread per round, lanes of one
// writer summed in the warp, one shared atomic per writer and warp).
// Every page counts ps rows (one coalesced load of the writers per round,
// lanes of one writer counted by the warp); then each request whose last
// page is short and in the range takes back the rows that page lacks.
template <int MAXB>
__device__ void add_writer_rows(const PlanParams<MAXB> &p, const RequestScan<MAXB> &rs, int64_t first,
                                int64_t last, int32_t *rows) {
  for (int64_t base = first; base < last; base += kPlanThreads) {  // uniform trip count: full warps in match
    const int64_t i = base + threadIdx.x;
    int32_t w = -1;
    if (i < last) {
      w = p.writer[i];
      if (w < 0 || w >= p.cp) w = -1;
    }
    const unsigned int peers = __match_any_sync(0xffffffffu, w);
    if (w >= 0 && (int)(threadIdx.x & 31) == __ffs(peers) - 1) atomicAdd(&rows[w], p.ps * __popc(peers));
  }
  for (int b = threadIdx.x; b < p.B; b += kPlanThreads) {
    const int32_t rem = p.cur_lens[b] % p.ps;
    const int64_t lastp = rs.cur_page_start[b + 1] - 1;
    if (rem != 0 && lastp >= first && lastp < last) {
      const int32_t w = p.writer[lastp];
      if (w >= 0 && w < p.cp) atomicAdd(&rows[w], rem - p.ps);
    }
  }
}

// Token block j of plan_init (batches of more than kDirectMaxPages current
// pages): rows of each writer in current pages [j K, (j + 1) K), to the
// workspace.
template <int MAXB>
__device__ void plan_block_rows(const PlanParams<MAXB> &p, int j) {
  __shared__ RequestScan<MAXB> rs;
  __shared__ int32_t rows[CPKV_MAX_CP];
  if (threadIdx.x < CPKV_MAX_CP) rows[threadIdx.x] = 0;
  build_request_scan(p, rs);  // ends with __syncthreads()
  add_writer_rows(p, rs, (int64_t)j * p.K, min64((int64_t)(j + 1) * p.K, p.C), rows);
  __syncthreads();
  if ((int)threadIdx.x < p.cp) p.block_rows[(int64_t)j * p.cp + threadIdx.x] = rows[threadIdx.x];
}

template <int MAXB>
__global__ void __launch_bounds__(kPlanThreads) plan_init(const __grid_constant__ PlanParams<MAXB> p) {
  // plan_main may start now: it waits for this grid only before its first
  // access to the inverses or the workspace.
  release_dependents();
  if ((int)blockIdx.x >= p.nInit) {
    plan_block_rows(p, blockIdx.x - p.nInit);
    return;
  }
  const int64_t tid = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  const int64_t stride = (int64_t)p.nInit * blockDim.x;
  int32_t *pi = p.page_inverse, *spi = p.staging_page_inverse;
  int64_t done = 0;
  if (p.vec) {
    const int64_t n4 = p.P >> 2;
    int4 *pi4 = reinterpret_cast<int4 *>(pi);
    int4 *spi4 = reinterpret_cast<int4 *>(spi);
    for (int64_t i = tid; i < n4; i += stride) {
      pi4[i] = make_int4(-1, -1, -1, -1);
      spi4[i] = make_int4(0, 0, 0, 0);
    }
    done = n4 << 2;
  }
  for (int64_t i = done + tid; i < p.P; i += stride) {
    pi[i] = -1;
    spi[i] = 0;
  }
}

// Token block j of plan_main: per-writer row bases of current pages
// [i0, i0 + K), i0 = j K, then their tokens' mixed_locs / staging_rows /
// token_writer_row.
template <int MAXB>
__device__ void plan_current_tokens(const PlanParams<MAXB> &p, const RequestScan<MAXB> &rs, int j) {
  __shared__ int32_t base_rows[CPKV_MAX_CP];          // rows of writer w before i0
  __shared__ int32_t warp_rows[kPlanThreads / 32][CPKV_MAX_CP];  // per warp, then scanned over warps
  __shared__ int32_t page_tok0[kMaxPagesPerBlock];
  __shared__ int32_t page_slot[kMaxPagesPerBlock];
  __shared__ int32_t page_rows[kMaxPagesPerBlock];
  __shared__ int32_t page_row_base[kMaxPagesPerBlock];

  const int ps = p.ps, cp = p.cp;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  constexpr int kWarps = kPlanThreads / 32;
  const int64_t i0 = (int64_t)j * p.K;  // this block's first current page
  const int npages = (int)min64(p.K, p.C - i0);
  if (threadIdx.x < CPKV_MAX_CP) base_rows[threadIdx.x] = 0;
  for (int k = threadIdx.x; k < kWarps * CPKV_MAX_CP; k += kPlanThreads) (&warp_rows[0][0])[k] = 0;
  __syncthreads();

  // this block's pages, one per thread; the rows of same-writer pages below
  // it in the warp, and each writer's total per warp
  const int t = threadIdx.x;
  int32_t w = -1, n = 0;
  if (t < npages) {
    const CurPage<MAXB> c = current_page(p, rs, i0 + t);
    w = c.w;
    n = c.n;
    page_tok0[t] = (int32_t)c.tok0;
    page_slot[t] = c.slot;
    page_rows[t] = c.n;
  }
  int32_t before = 0;
  if (warp * 32 < npages) {  // warps that hold pages
    const unsigned int peers = __match_any_sync(0xffffffffu, w);
    int32_t total;
    same_writer_rows(peers, n, w >= 0, ps, &before, &total);
    if (w >= 0 && lane == __ffs(peers) - 1) warp_rows[warp][w] = total;
  }
  __syncthreads();

  // the token locations that need no row base, while plan_init still runs
  for (int u = threadIdx.x; u < npages * ps; u += kPlanThreads) {
    const int jj = u / ps, off = u - jj * ps;
    if (off >= page_rows[jj]) continue;
    const int64_t tok = (int64_t)page_tok0[jj] + off;
    p.mixed_locs[tok] = (int64_t)page_slot[jj] * ps + off;
    p.staging_rows[tok] = (i0 + jj + 1) * ps + off;
  }

  // rows of each writer in the pages before this block: the totals of the
  // token blocks before this one, from the workspace (plan_init)
  wait_prerequisite();
  for (int64_t k = threadIdx.x; k < (int64_t)j * cp; k += kPlanThreads) {
    const int32_t v = p.block_rows[k];
    if (v != 0) atomicAdd(&base_rows[(int)(k % cp)], v);
  }
  __syncthreads();
  // exclusive scan of each writer's rows over the warps that hold pages
  if (threadIdx.x < cp) {
    const int used = (npages + 31) / 32;
    int32_t run = base_rows[threadIdx.x];
    for (int k = 0; k < used; ++k) {
      const int32_t v = warp_rows[k][threadIdx.x];
      warp_rows[k][threadIdx.x] = run;
      run += v;
    }
  }
  __syncthreads();
  if (t < npages) page_row_base[t] = w < 0 ? -1 : warp_rows[warp][w] + before;
  __syncthreads();

  for (int u = threadIdx.x; u < npages * ps; u += kPlanThreads) {
    const int jj = u / ps, off = u - jj * ps;
    if (off >= page_rows[jj]) continue;
    p.token_writer_row[(int64_t)page_tok0[jj] + off] = page_row_base[jj] < 0 ? -1 : page_row_base[jj] + off;
  }
}

template <int MAXB>
__global__ void __launch_bounds__(kPlanThreads) plan_main(const __grid_constant__ PlanParams<MAXB> p) {
  __shared__ RequestScan<MAXB> rs;
  build_request_scan(p, rs);
  if ((int)blockIdx.x < p.nA) {
    plan_dense_slots(p, rs);
  } else {
    plan_current_tokens(p, rs, blockIdx.x - p.nA);
  }
}

// Current pages per token block for page size ps: about kTokensPerBlock
// tokens, a multiple of 32 between 32 and kMaxPagesPerBlock.
inline int pages_per_token_block(int ps) {
  int64_t k = kTokensPerBlock / ps;
  k = (k + 31) / 32 * 32;
  if (k < 32) k = 32;
  if (k > kMaxPagesPerBlock) k = kMaxPagesPerBlock;
  return (int)k;
}

inline int64_t workspace_bytes_for(int64_t C, int ps, int cp) {
  return ceil_div(C, pages_per_token_block(ps)) * cp * (int64_t)sizeof(int32_t);
}

// plan_init is launched plainly; plan_main is its programmatic dependent:
// its request scans, page-table loads, descriptors and page walks overlap the
// init, and only the inverse scatters and the reads of the workspace wait for
// it (wait_prerequisite).
template <int MAXB>
int launch_plan(const PlanParams<MAXB> &prm, cudaStream_t s) {
  {
    const int rc = launch_kernel(plan_init<MAXB>, dim3(prm.nInit + prm.NB), dim3(kPlanThreads), 0, false, s, prm);
    if (rc != CPKV_OK) return rc;
  }
  const int grid = prm.nA + prm.NB;
  if (grid == 0) return CPKV_OK;
  return launch_kernel(plan_main<MAXB>, dim3(grid), dim3(kPlanThreads), 0, true, s, prm);
}

template <int MAXB>
void fill_common(PlanParams<MAXB> &prm, int B, const int32_t *pl, const int32_t *cl) {
  for (int b = 0; b < B; ++b) {
    prm.prefix_lens[b] = pl[b];
    prm.cur_lens[b] = cl[b];
  }
}

}  // namespace
}  // namespace cpkv

extern "C" int cpkv_plan_workspace_bytes(int B, int page_size, int cp_size, const int32_t *h_cur_lens,
                                         int64_t *h_bytes) {
  using namespace cpkv;
  if (B < 0 || page_size <= 0 || cp_size < 1 || cp_size > CPKV_MAX_CP || h_bytes == nullptr) return CPKV_ERR_ARG;
  if (B > CPKV_MAX_BATCH) return CPKV_ERR_LIMIT;
  if (B > 0 && h_cur_lens == nullptr) return CPKV_ERR_ARG;
  int64_t C = 0;
  for (int b = 0; b < B; ++b) {
    if (h_cur_lens[b] < 0) return CPKV_ERR_ARG;
    C += ceil_div(h_cur_lens[b], page_size);
  }
  if (C > INT32_MAX - 2) return CPKV_ERR_LIMIT;
  *h_bytes = workspace_bytes_for(C, page_size, cp_size);
  return CPKV_OK;
}

extern "C" int cpkv_plan_build(int B, int page_size, int cp_size, int64_t num_pool_pages,
                               const int32_t *h_prefix_lens, const int32_t *h_cur_lens,
                               const int32_t *d_prefix_pages, const int32_t *d_cur_pages,
                               const int32_t *d_writer, int64_t dense_cap_pages, int32_t *d_prefix_spans,
                               int32_t *d_cur_spans, int32_t *d_owner, int32_t *d_src,
                               int32_t *d_page_inverse, int32_t *d_staging_page_inverse,
                               int64_t *d_mixed_locs, int64_t *d_staging_rows, int32_t *d_token_writer_row,
                               void *d_workspace, int64_t workspace_bytes, int32_t *d_status,
                               cpkv_stream_t stream) {
  using namespace cpkv;
  if (cp_size < 1 || cp_size > CPKV_MAX_CP || num_pool_pages < 1 || dense_cap_pages < 0) return CPKV_ERR_ARG;
  if (B > CPKV_MAX_BATCH) return CPKV_ERR_LIMIT;
  if (num_pool_pages > INT32_MAX || dense_cap_pages > INT32_MAX - 1) return CPKV_ERR_LIMIT;
  cpkv_sizes sz;
  int rc = cpkv_plan_sizes(B, page_size, h_prefix_lens, h_cur_lens, &sz);
  if (rc != CPKV_OK) return rc;
  if (dense_cap_pages < sz.D) return CPKV_ERR_CAPACITY;
  if (d_page_inverse == nullptr || d_staging_page_inverse == nullptr || d_status == nullptr)
    return CPKV_ERR_ARG;
  if (B > 0 && (d_prefix_spans == nullptr || d_cur_spans == nullptr)) return CPKV_ERR_ARG;
  if (dense_cap_pages > 0 && (d_owner == nullptr || d_src == nullptr)) return CPKV_ERR_ARG;
  if (sz.D - sz.C > 0 && d_prefix_pages == nullptr) return CPKV_ERR_ARG;
  if (sz.C > 0 && (d_cur_pages == nullptr || d_writer == nullptr)) return CPKV_ERR_ARG;
  if (sz.T > 0 && (d_mixed_locs == nullptr || d_staging_rows == nullptr || d_token_writer_row == nullptr))
    return CPKV_ERR_ARG;
  const int K = pages_per_token_block(page_size);
  const int64_t NB = ceil_div(sz.C, K);
  const int64_t need = workspace_bytes_for(sz.C, page_size, cp_size);
  if (workspace_bytes < 0) return CPKV_ERR_ARG;
  if (need > 0 && (d_workspace == nullptr || (reinterpret_cast<uintptr_t>(d_workspace) & 3u) != 0))
    return CPKV_ERR_ARG;
  if (workspace_bytes < need) return CPKV_ERR_CAPACITY;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

  const bool vec = aligned16(d_page_inverse) && aligned16(d_staging_page_inverse);
  const int64_t init_work = vec ? (num_pool_pages >> 2) + 3 : num_pool_pages;
  const int64_t init_blocks = ceil_div(init_work, kPlanThreads);
  const int nInit = (int)(init_blocks < 2 * device_sm_count() ? (init_blocks > 0 ? init_blocks : 1)
                                                              : 2 * device_sm_count());
  int nA = (int)ceil_div(dense_cap_pages, kPlanThreads);
  if (nA == 0 && B > 0) nA = 1;  // block 0 writes the spans

#define CPKV_FILL_PLAN(prm)                                                                        \
  prm.B = B; prm.ps = page_size; prm.cp = cp_size; prm.nA = nA; prm.nInit = nInit; prm.K = K;     \
  prm.NB = (int)NB; prm.vec = vec; prm.P = num_pool_pages;                                         \
  prm.dense_cap = dense_cap_pages; prm.D = sz.D; prm.C = sz.C; prm.T = sz.T;                       \
  prm.prefix_pages = d_prefix_pages; prm.cur_pages = d_cur_pages; prm.writer = d_writer;           \
  prm.prefix_spans = d_prefix_spans; prm.cur_spans = d_cur_spans; prm.owner = d_owner;             \
  prm.src = d_src; prm.page_inverse = d_page_inverse; prm.staging_page_inverse = d_staging_page_inverse; \
  prm.mixed_locs = d_mixed_locs; prm.staging_rows = d_staging_rows;                                \
  prm.token_writer_row = d_token_writer_row; prm.status = d_status;                                \
  prm.block_rows = static_cast<int32_t *>(d_workspace);                                            \
  fill_common(prm, B, h_prefix_lens, h_cur_lens);

  if (B <= 64) {
    PlanParams<64> prm;
    CPKV_FILL_PLAN(prm)
    return launch_plan(prm, s);
  }
  PlanParams<CPKV_MAX_BATCH> prm;
  CPKV_FILL_PLAN(prm)
#undef CPKV_FILL_PLAN
  return launch_plan(prm, s);
}
