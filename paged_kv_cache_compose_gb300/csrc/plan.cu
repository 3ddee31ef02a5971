// cpkv_plan_build: the per-batch compose plan on the device.
//
// Two launches on the caller's stream, the second a programmatic dependent
// of the first (it starts early and waits only before the inverse scatters):
//   1. plan_init_inverses  — page_inverse[:] = -1, staging_page_inverse[:] = 0
//                            (P entries each; the only P-sized work).
//   2. plan_main           — blocks [0, nA): one thread per dense slot:
//                            descriptors (owner, src) and the inverse
//                            scatters, plus the spans (block 0);
//                            blocks [nA, nA + nB): 32 current pages per block:
//                            per-writer row bases and the per-token arrays.
// Host lengths travel as kernel parameters (__grid_constant__), so nothing
// is copied host-to-device and nothing syncs.  Every block rebuilds the
// request-level exclusive scans in shared memory (B <= 1024, one block scan).
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
constexpr int kPagesPerBlock = 32;  // current pages handled by one token block (one warp lane each)

template <int MAXB>
struct PlanParams {
  int B, ps, cp, nA;
  int64_t P, dense_cap, D, C, T;
  const int32_t *prefix_pages, *cur_pages, *writer;
  int32_t *prefix_spans, *cur_spans, *owner, *src, *page_inverse, *staging_page_inverse;
  int64_t *mixed_locs, *staging_rows;
  int32_t *token_writer_row, *status;
  int32_t prefix_lens[MAXB];
  int32_t cur_lens[MAXB];
};

__global__ void plan_init_inverses(int32_t *__restrict__ pi, int32_t *__restrict__ spi, int64_t P,
                                   bool vec) {
  // plan_main may start now: it waits for this grid only before its first
  // access to the inverses.
  release_dependents();
  const int64_t tid = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  if (vec) {
    const int64_t n4 = P >> 2;
    int4 *pi4 = reinterpret_cast<int4 *>(pi);
    int4 *spi4 = reinterpret_cast<int4 *>(spi);
    for (int64_t i = tid; i < n4; i += stride) {
      pi4[i] = make_int4(-1, -1, -1, -1);
      spi4[i] = make_int4(0, 0, 0, 0);
    }
    for (int64_t i = (n4 << 2) + tid; i < P; i += stride) {
      pi[i] = -1;
      spi[i] = 0;
    }
  } else {
    for (int64_t i = tid; i < P; i += stride) {
      pi[i] = -1;
      spi[i] = 0;
    }
  }
}

// Request-level exclusive scans, one request per thread (B <= 1024).
struct RequestScan {
  int32_t dense_start[CPKV_MAX_BATCH + 1];   // first dense slot of request b
  int32_t cur_page_start[CPKV_MAX_BATCH + 1];  // first batch current page index
  int32_t prefix_page_start[CPKV_MAX_BATCH + 1];  // CSR offset into prefix_pages
  int64_t token_start[CPKV_MAX_BATCH + 1];   // first batch token
  int64_t scratch64[33];
};

template <int MAXB>
__device__ void build_request_scan(const PlanParams<MAXB> &p, RequestScan &rs) {
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
__device__ bool slot_is_prefix(const PlanParams<MAXB> &p, const RequestScan &rs, int32_t slot) {
  if (slot < 0 || slot >= p.D || p.B == 0) return false;
  const int b = upper_index<int32_t>(rs.dense_start, p.B, slot);
  return slot - rs.dense_start[b] < p.prefix_lens[b] / p.ps;
}

// One thread per dense slot: descriptors and inverse scatters.
template <int MAXB>
__device__ void plan_dense_slots(const PlanParams<MAXB> &p, const RequestScan &rs) {
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
    // the page tables are loaded before waiting for plan_init_inverses
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

// 32 current pages per block: per-writer token row bases, then per-token
// mixed_locs / staging_rows / token_writer_row.
template <int MAXB>
__device__ void plan_current_tokens(const PlanParams<MAXB> &p, const RequestScan &rs, int blk) {
  __shared__ int32_t full_pages[CPKV_MAX_CP];  // pages of writer w before this block
  __shared__ int64_t short_rows[CPKV_MAX_CP];  // missing rows of w's partial pages before this block
  __shared__ int64_t page_tok0[kPagesPerBlock];
  __shared__ int32_t page_slot[kPagesPerBlock];
  __shared__ int32_t page_rows[kPagesPerBlock];
  __shared__ int32_t page_row_base[kPagesPerBlock];

  const int ps = p.ps, cp = p.cp;
  const int64_t i0 = (int64_t)blk * kPagesPerBlock;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (threadIdx.x < CPKV_MAX_CP) {
    full_pages[threadIdx.x] = 0;
    short_rows[threadIdx.x] = 0;
  }
  __syncthreads();

  // pages of each writer before i0 (warp-aggregated shared atomics)
  for (int64_t base = 0; base < i0; base += kPlanThreads) {  // uniform trip count: full warps in match
    const int64_t i = base + threadIdx.x;
    int32_t w = -1;
    if (i < i0) {
      w = p.writer[i];
      if (w < 0 || w >= cp) w = -1;
    }
    const unsigned int peers = __match_any_sync(0xffffffffu, w);
    if (w >= 0 && lane == __ffs(peers) - 1) atomicAdd(&full_pages[w], __popc(peers));
  }
  // each request's last page, if partial and before i0, holds fewer rows
  for (int b = threadIdx.x; b < p.B; b += kPlanThreads) {
    const int32_t rem = p.cur_lens[b] % ps;
    const int32_t last = rs.cur_page_start[b + 1] - 1;
    if (rem != 0 && last < i0) {
      const int32_t w = p.writer[last];
      if (w >= 0 && w < cp) atomicAdd(reinterpret_cast<unsigned long long *>(&short_rows[w]),
                                      (unsigned long long)(ps - rem));
    }
  }
  __syncthreads();

  if (warp == 0) {
    const int64_t i = i0 + lane;
    int32_t w = -1, n = 0;
    if (i < p.C) {
      const int b = upper_index<int32_t>(rs.cur_page_start, p.B, (int32_t)i);
      const int32_t kp = (int32_t)i - rs.cur_page_start[b];  // page index inside the request
      n = min(ps, p.cur_lens[b] - kp * ps);
      w = p.writer[i];
      page_tok0[lane] = rs.token_start[b] + (int64_t)kp * ps;
      page_slot[lane] = rs.dense_start[b] + p.prefix_lens[b] / ps + kp;
      page_rows[lane] = n;
      if (w < 0 || w >= cp) w = -1;
    }
    // rows of same-writer pages earlier in this block
    int32_t before = 0;
#pragma unroll
    for (int l = 0; l < 32; ++l) {
      const int32_t wl = __shfl_sync(0xffffffffu, w, l);
      const int32_t nl = __shfl_sync(0xffffffffu, n, l);
      if (l < lane && wl == w) before += nl;
    }
    if (i < p.C) {
      page_row_base[lane] =
          w < 0 ? -1 : (int32_t)((int64_t)full_pages[w] * ps - short_rows[w] + before);
    }
  }
  __syncthreads();

  const int npages = (int)min64(kPagesPerBlock, p.C - i0);
  for (int u = threadIdx.x; u < npages * ps; u += kPlanThreads) {
    const int j = u / ps, off = u - j * ps;
    if (off >= page_rows[j]) continue;
    const int64_t t = page_tok0[j] + off;
    p.mixed_locs[t] = (int64_t)page_slot[j] * ps + off;
    p.staging_rows[t] = (i0 + j + 1) * ps + off;
    p.token_writer_row[t] = page_row_base[j] < 0 ? -1 : page_row_base[j] + off;
  }
}

template <int MAXB>
__global__ void __launch_bounds__(kPlanThreads) plan_main(const __grid_constant__ PlanParams<MAXB> p) {
  __shared__ RequestScan rs;
  build_request_scan(p, rs);
  if ((int)blockIdx.x < p.nA) {
    plan_dense_slots(p, rs);
  } else {
    plan_current_tokens(p, rs, blockIdx.x - p.nA);
  }
}

// plan_main is a programmatic dependent of plan_init_inverses: its request
// scans, page-table loads, descriptors and token arrays overlap the init;
// only the inverse scatters wait for it (wait_prerequisite).
template <int MAXB>
int launch_plan(const PlanParams<MAXB> &prm, int nB, cudaStream_t s) {
  const int grid = prm.nA + nB;
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

extern "C" int cpkv_plan_build(int B, int page_size, int cp_size, int64_t num_pool_pages,
                               const int32_t *h_prefix_lens, const int32_t *h_cur_lens,
                               const int32_t *d_prefix_pages, const int32_t *d_cur_pages,
                               const int32_t *d_writer, int64_t dense_cap_pages, int32_t *d_prefix_spans,
                               int32_t *d_cur_spans, int32_t *d_owner, int32_t *d_src,
                               int32_t *d_page_inverse, int32_t *d_staging_page_inverse,
                               int64_t *d_mixed_locs, int64_t *d_staging_rows, int32_t *d_token_writer_row,
                               int32_t *d_status, cpkv_stream_t stream) {
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
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

  {
    const bool vec = aligned16(d_page_inverse) && aligned16(d_staging_page_inverse);
    const int64_t work = vec ? (num_pool_pages >> 2) + 3 : num_pool_pages;
    const int64_t blocks = ceil_div(work, 256);
    const int grid = (int)(blocks < 4 * device_sm_count() ? (blocks > 0 ? blocks : 1) : 4 * device_sm_count());
    plan_init_inverses<<<grid, 256, 0, s>>>(d_page_inverse, d_staging_page_inverse, num_pool_pages, vec);
    rc = launch_status();
    if (rc != CPKV_OK) return rc;
  }

  int nA = (int)ceil_div(dense_cap_pages, kPlanThreads);
  if (nA == 0 && B > 0) nA = 1;  // block 0 writes the spans
  const int nB = (int)ceil_div(sz.C, kPagesPerBlock);

#define CPKV_FILL_PLAN(prm)                                                                        \
  prm.B = B; prm.ps = page_size; prm.cp = cp_size; prm.nA = nA; prm.P = num_pool_pages;           \
  prm.dense_cap = dense_cap_pages; prm.D = sz.D; prm.C = sz.C; prm.T = sz.T;                       \
  prm.prefix_pages = d_prefix_pages; prm.cur_pages = d_cur_pages; prm.writer = d_writer;           \
  prm.prefix_spans = d_prefix_spans; prm.cur_spans = d_cur_spans; prm.owner = d_owner;             \
  prm.src = d_src; prm.page_inverse = d_page_inverse; prm.staging_page_inverse = d_staging_page_inverse; \
  prm.mixed_locs = d_mixed_locs; prm.staging_rows = d_staging_rows;                                \
  prm.token_writer_row = d_token_writer_row; prm.status = d_status;                                \
  fill_common(prm, B, h_prefix_lens, h_cur_lens);

  if (B <= 64) {
    PlanParams<64> prm;
    CPKV_FILL_PLAN(prm)
    return launch_plan(prm, nB, s);
  }
  PlanParams<CPKV_MAX_BATCH> prm;
  CPKV_FILL_PLAN(prm)
#undef CPKV_FILL_PLAN
  return launch_plan(prm, nB, s);
}
