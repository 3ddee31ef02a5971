// cpkv_fill_current: the per-layer fill of current rows into the writers'
// stagings ("staging-direct compose" message of commits d63fbd4: the fill is
// a single index copy of layer-invariant row indices; "fp8 -> uint8"
// message of commits 0d87bc5: rows are opaque bytes).
//
// One launch.  Blocks [0, nRow) copy rows: one warp per token row, each lane
// moving 16-byte vectors, RIF rows in flight per warp (all loads issued
// before the stores); the grid is one resident wave.  RIF follows the row
// width so that a warp keeps about 2-3 KB in flight: 2 rows of up to 96
// vectors (the 1152-byte MLA row), 4 rows of up to 64 vectors (the 656-byte
// fp8 NSA row).  Blocks [nRow, nRow + B) zero the pad rows after each
// request's last token, up to the end of its staging page.  Current rows are
// read once (L2 evict_first); staging rows are written with evict_last
// because the gather that follows reads them back.
//
// With CPKV_FLAG_EARLY_INPUTS the fill is launched as a programmatic
// dependent of the previous kernel on the stream (the previous layer's
// gather, which releases its dependents at its start).  The fill's blocks
// then take the SM room the gather's one-warp CTAs leave free, resolve their
// indices and load their first rows while the gather runs, and each thread
// waits for the gather (store_gate) before its first store: the staging the
// fill overwrites is what that gather reads.  Measured per 78-layer traced
// step: 4.451 -> 4.290 ms; one-token pages 5.457 -> 5.192 ms; fp8 unchanged
// (19.99 ms).  In a plain launch the gate returns at once.  The row fill
// releases its dependents as each block finishes, the page-run fill below at
// its start, for a gather launched with CPKV_GATHER_EARLY_INPUTS.
//
// (A variant that moves whole pages with bulk copies when a page's indices
// form a run was slower here: each page first needs a round trip of index
// loads, and a layer has only a few pages per CTA to overlap them with.)
//
// With CPKV_FILL_PAGE_RUNS the caller promises the plan's page runs, and
// fill_pages_kernel below moves each current page as one run instead.
#include <stdint.h>

#include "common.cuh"

namespace cpkv {
namespace {

constexpr int kFillThreads = 256;
constexpr int kWarpsPerBlock = kFillThreads / 32;
constexpr int kBlocksPerSm = 4;    // one resident wave (<= 64 registers x 256 threads x 4 = 64K)

template <int MAXB>
struct FillParams {
  const uint8_t *cur_rows[CPKV_MAX_CP];
  int64_t cur_cap[CPKV_MAX_CP];
  uint8_t *staging[CPKV_MAX_CP];
  const int64_t *staging_rows;
  const int32_t *token_writer_row, *writer;
  int32_t *status;
  int64_t T, C, staging_cap_rows, R;
  int ps, cp, B, nRow, vpr;  // vpr = R / 16
  int64_t units;             // page mode: chunks of current pages (C * upp)
  int32_t upp;               // page mode: chunks per page
  int32_t cur_lens[MAXB];
};

struct RowJob {
  const uint8_t *src;
  uint8_t *dst;
};

// Resolve token t to (source row, staging row); nullptr src when skipped.
template <int MAXB>
__device__ RowJob resolve_row(const FillParams<MAXB> &p, int64_t t) {
  RowJob j{nullptr, nullptr};
  const int64_t sr = p.staging_rows[t];
  const int64_t slot = sr / p.ps;
  if (sr < p.ps || sr >= p.staging_cap_rows || slot > p.C) {
    raise_status(p.status, CPKV_STATUS_ROW_OOB);
    return j;
  }
  const int32_t w = p.writer[slot - 1];
  if (w < 0 || w >= p.cp) {
    raise_status(p.status, CPKV_STATUS_WRITER_OOB);
    return j;
  }
  const int32_t r = p.token_writer_row[t];
  if (r < 0 || r >= p.cur_cap[w]) {
    raise_status(p.status, CPKV_STATUS_ROW_OOB);
    return j;
  }
  j.src = p.cur_rows[w] + (int64_t)r * p.R;
  j.dst = p.staging[w] + sr * p.R;
  return j;
}

// Warp w handles rows w*RIF + i*stride + [0, RIF) in iteration i (stride =
// RIF * warps).  The indices of 32/RIF iterations are resolved at once, one
// row per lane (their dependent index loads overlap), and each iteration
// takes its rows' pointers by shuffle.  RIF rows are copied per iteration,
// each lane moving VPL 16-byte vectors per row (vpr <= 32 * VPL), all loads
// issued before the stores.
template <int MAXB, int RIF, int VPL>
__device__ void copy_rows_unrolled(const FillParams<MAXB> &p, uint64_t read_once, uint64_t keep) {
  static_assert(32 % RIF == 0, "RIF divides the warp");
  constexpr int kIters = 32 / RIF;  // iterations resolved per batch
  const int lane = threadIdx.x & 31;
  const int64_t warp_id = (int64_t)blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
  const int64_t stride = (int64_t)p.nRow * kWarpsPerBlock * RIF;
  const int vpr = p.vpr;
  bool stores_open = false;
  for (int64_t tb = warp_id * RIF; tb < p.T; tb += kIters * stride) {
    const int64_t tl = tb + (int64_t)(lane / RIF) * stride + (lane % RIF);
    const RowJob mine = tl < p.T ? resolve_row(p, tl) : RowJob{nullptr, nullptr};
    for (int it = 0; it < kIters; ++it) {
      const int64_t t0 = tb + (int64_t)it * stride;
      if (t0 >= p.T) break;  // uniform across the warp
      RowJob job[RIF];
      uint4 v[RIF][VPL];
#pragma unroll
      for (int r = 0; r < RIF; ++r) {
        const int from = it * RIF + r;
        job[r].src = reinterpret_cast<const uint8_t *>(
            __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(mine.src), from));
        job[r].dst = reinterpret_cast<uint8_t *>(
            __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(mine.dst), from));
      }
#pragma unroll
      for (int r = 0; r < RIF; ++r) {
#pragma unroll
        for (int k = 0; k < VPL; ++k) {
          const int c = lane + 32 * k;
          if (job[r].src != nullptr && c < vpr) v[r][k] = ld_stream16_hint(job[r].src + 16 * (int64_t)c, read_once);
        }
      }
      store_gate(&stores_open);
#pragma unroll
      for (int r = 0; r < RIF; ++r) {
#pragma unroll
        for (int k = 0; k < VPL; ++k) {
          const int c = lane + 32 * k;
          if (job[r].src != nullptr && c < vpr) st16_hint(job[r].dst + 16 * (int64_t)c, v[r][k], keep);
        }
      }
    }
  }
}

// Rows wider than 128 vectors (2 KB): one row per warp, a plain loop.
template <int MAXB>
__device__ void copy_rows_wide(const FillParams<MAXB> &p, uint64_t read_once, uint64_t keep) {
  const int lane = threadIdx.x & 31;
  const int64_t warp_id = (int64_t)blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
  const int64_t nwarps = (int64_t)p.nRow * kWarpsPerBlock;
  bool stores_open = false;
  for (int64_t t = warp_id; t < p.T; t += nwarps) {
    const RowJob job = resolve_row(p, t);
    if (job.src == nullptr) continue;
    store_gate(&stores_open);
    for (int c = lane; c < p.vpr; c += 32)
      st16_hint(job.dst + 16 * (int64_t)c, ld_stream16_hint(job.src + 16 * (int64_t)c, read_once), keep);
  }
}

// Zero the rows after request b's last token up to the end of its staging page.
template <int MAXB>
__device__ void zero_pad_rows(const FillParams<MAXB> &p, int b) {
  __shared__ int64_t last_tok;
  if (b >= p.B) return;
  const int32_t rem = p.cur_lens[b] % p.ps;
  if (rem == 0) return;
  if (threadIdx.x == 0) {
    int64_t s = 0;
    for (int k = 0; k <= b; ++k) s += p.cur_lens[k];
    last_tok = s - 1;
  }
  __syncthreads();
  const int64_t sr = p.staging_rows[last_tok];
  const int64_t slot = sr / p.ps;
  if (sr < p.ps || sr >= p.staging_cap_rows || slot > p.C) {
    if (threadIdx.x == 0) raise_status(p.status, CPKV_STATUS_ROW_OOB);
    return;
  }
  const int32_t w = p.writer[slot - 1];
  if (w < 0 || w >= p.cp) {
    if (threadIdx.x == 0) raise_status(p.status, CPKV_STATUS_WRITER_OOB);
    return;
  }
  wait_prerequisite();
  const int64_t first = sr + 1, end = (slot + 1) * p.ps;  // [first, end) rows to zero
  uint8_t *base = p.staging[w] + first * p.R;
  const int64_t nvec = (end - first) * p.vpr;
  const uint4 z = make_uint4(0, 0, 0, 0);
  const uint64_t keep = l2_policy_evict_last();
  for (int64_t i = threadIdx.x; i < nvec; i += kFillThreads) st16_hint(base + 16 * i, z, keep);
}

// ---------------------------------------------------------------------------
// Page mode (CPKV_FILL_PAGE_RUNS): the plan of cpkv_plan_build stages current
// page i's n_i tokens at rows (i + 1) ps .. (i + 1) ps + n_i - 1 of its
// writer's staging and reads them from n_i consecutive rows of the writer's
// buffer, from token_writer_row of the page's first token.  So a page is one
// contiguous run on both sides, and the fill moves it in chunks of
// 4 KB (32 lanes x 8 16-byte vectors): a unit is one chunk of
// one page (the last chunks of a short page are partly or wholly pad, zeroed
// in the same pass).  A warp resolves the pages of 32 units at once, one
// unit per lane: the page's writer and first source row are two independent
// loads (no per-row index chain), plus the first staging row and the last
// source row, which must fit the run (a page that does not is skipped and
// raises ROW_OOB).  Each unit then issues all its loads before its stores, so
// a warp keeps 4 KB in flight.  Units u = warp + k * warps: consecutive
// warps stream consecutive chunks.
// Measured (same box, two runs each): traced 78-layer step 4.183 ms against
// 4.202 with the row fill, fp8 19.70-19.80 against 19.90.  Alone the kernel
// is no faster than the row fill (15.5 against 14.3 us): both are bound by
// the rounds of load latency of a 51 MB copy, not by index loads.  Shapes
// tried: 2 KB chunks with 8 blocks of 256 or 4 of 512 threads per SM (32
// registers, spills) 4.63-4.68 ms; 8 blocks of 128 threads 4.226 ms; the
// pages through the gather's bulk-copy ring (one-warp CTAs, 16 KB pieces)
// 4.175 ms traced but 20.10 ms fp8.
constexpr int kPageChunkVecs = 256;  // 4 KB chunks
constexpr int kPageVpl = kPageChunkVecs / 32;
constexpr int kPageThreads = 256;
constexpr int kPageWarps = kPageThreads / 32;
constexpr int kPageBlocksPerSm = 4;  // one resident wave
// The page fill's grid: 3 blocks per SM when that leaves each warp at most
// this many chunks, else 4.  Launched early beside a gather that holds 3-4
// one-warp CTAs per SM, only 3 fill blocks fit there at once; with 3 per SM
// all of them start (and release the next gather) while the previous gather
// runs.  Measured per 78-layer step (same box, two runs each): traced (12 654
// chunks, 3.5 per warp at 3 per SM) 4.10 -> 3.99-4.00 ms; fp8 (22 715
// chunks) unchanged at 19.86 ms with 4 per SM, where 3 per SM measured 20.96-
// 23.04 ms and 2 per SM 19.63 ms (three runs, against 19.70-19.71 at 4 per
// SM: too small a gain to extend the rule from two workloads); the traced
// step at 2 per SM 4.14 ms.
constexpr int64_t kPageUnitsPerWarp3 = 4;

struct PageUnit {
  const uint8_t *src;  // nullptr: skip
  uint8_t *dst;
  int32_t copy, total;  // bytes copied from src, bytes written (the rest zero)
};

template <int MAXB>
__device__ PageUnit resolve_page_unit(const FillParams<MAXB> &p, const int32_t *cur_page_start,
                                      const int64_t *token_start, int64_t u) {
  PageUnit x{nullptr, nullptr, 0, 0};
  if (u >= p.units) return x;
  const int64_t i = u / p.upp;
  const int32_t c = (int32_t)(u - i * p.upp);
  const int b = upper_index<int32_t>(cur_page_start, p.B, (int32_t)i);
  const int32_t kp = (int32_t)i - cur_page_start[b];
  const int32_t n = min(p.ps, p.cur_lens[b] - kp * p.ps);
  const int64_t tok0 = token_start[b] + (int64_t)kp * p.ps;
  // independent loads: writer, first and last source rows, first staging row
  const int32_t w = p.writer[i];
  const int32_t r0 = p.token_writer_row[tok0];
  const int32_t r1 = p.token_writer_row[tok0 + n - 1];
  const int64_t s0 = p.staging_rows[tok0];
  if (w < 0 || w >= p.cp) {
    if (c == 0) raise_status(p.status, CPKV_STATUS_WRITER_OOB);
    return x;
  }
  if (r0 < 0 || r1 != r0 + n - 1 || (int64_t)r0 + n > p.cur_cap[w] || s0 != (i + 1) * p.ps) {
    if (c == 0) raise_status(p.status, CPKV_STATUS_ROW_OOB);
    return x;
  }
  const int64_t page_bytes = (int64_t)p.ps * p.R;
  const int64_t off = (int64_t)c * (kPageChunkVecs * 16);
  x.total = (int32_t)min64(kPageChunkVecs * 16, page_bytes - off);
  const int64_t rows_bytes = (int64_t)n * p.R;
  x.copy = (int32_t)(off < rows_bytes ? min64(x.total, rows_bytes - off) : 0);
  x.src = p.cur_rows[w] + (int64_t)r0 * p.R + off;
  x.dst = p.staging[w] + (i + 1) * page_bytes + off;
  return x;
}

template <int MAXB>
__global__ void __launch_bounds__(kPageThreads, kPageBlocksPerSm) fill_pages_kernel(const __grid_constant__ FillParams<MAXB> p) {
  __shared__ int32_t cur_page_start[MAXB + 1];
  __shared__ int64_t token_start[MAXB + 1];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (warp == 0) {  // request-level exclusive scans, 32 requests per step
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
  // the gather of these stagings (CPKV_GATHER_EARLY_INPUTS) may launch now:
  // its CTAs load pool pages beside this fill and wait for it to complete
  // before any staging load or store.  Releasing it here rather than as the
  // blocks finish measured faster with the page runs (traced 78-layer step
  // 4.18 -> 4.09 ms, fp8 19.79 -> 19.82 ms; same box, two runs each).  The
  // row fill below keeps releasing at its end: at its start the traced step
  // with row fills went 4.19 -> 4.10 ms, but one-token pages, whose group
  // gather runs 6 CTAs per SM beside it, 4.40 -> 4.98 ms.
  release_dependents();
  const uint64_t read_once = l2_policy_evict_first();
  const uint64_t keep = l2_policy_evict_last();
  const int64_t nw = (int64_t)gridDim.x * kPageWarps;
  const int64_t gw = (int64_t)blockIdx.x * kPageWarps + warp;
  bool stores_open = false;
  for (int64_t base = gw; base < p.units; base += 32 * nw) {
    const PageUnit mine = resolve_page_unit(p, cur_page_start, token_start, base + lane * nw);
    for (int j = 0; j < 32; ++j) {
      if (base + j * nw >= p.units) break;  // uniform across the warp
      const uint8_t *src = reinterpret_cast<const uint8_t *>(
          __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(mine.src), j));
      uint8_t *dst = reinterpret_cast<uint8_t *>(
          __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(mine.dst), j));
      const int32_t copy = __shfl_sync(0xffffffffu, mine.copy, j);
      const int32_t total = __shfl_sync(0xffffffffu, mine.total, j);
      if (src == nullptr) continue;  // uniform
      uint4 v[kPageVpl];
#pragma unroll
      for (int k = 0; k < kPageVpl; ++k) {
        const int32_t off = 16 * (lane + 32 * k);
        v[k] = off < copy ? ld_stream16_hint(src + off, read_once) : make_uint4(0, 0, 0, 0);
      }
      store_gate(&stores_open);
#pragma unroll
      for (int k = 0; k < kPageVpl; ++k) {
        const int32_t off = 16 * (lane + 32 * k);
        if (off < total) st16_hint(dst + off, v[k], keep);
      }
    }
  }
  // an early-launched fill finishes only after the kernel before it, even if
  // it stored nothing (chains of early launches stay ordered)
  if (threadIdx.x == 0) store_gate(&stores_open);
}

// RIF = 0 selects the wide-row loop.
template <int MAXB, int RIF, int VPL>
__global__ void __launch_bounds__(kFillThreads, kBlocksPerSm) fill_current_kernel(const __grid_constant__ FillParams<MAXB> p) {
  if ((int)blockIdx.x < p.nRow) {
    const uint64_t read_once = l2_policy_evict_first();
    const uint64_t keep = l2_policy_evict_last();
    if constexpr (RIF == 0) copy_rows_wide(p, read_once, keep);
    else copy_rows_unrolled<MAXB, RIF, VPL>(p, read_once, keep);
  } else {
    zero_pad_rows(p, blockIdx.x - p.nRow);
  }
  // the gather of these stagings (CPKV_GATHER_EARLY_INPUTS) may launch once
  // every block is here; it waits for this kernel before reading a staging
  release_dependents();
}

template <int MAXB>
int launch_fill(const FillParams<MAXB> &prm, int grid, bool early, cudaStream_t s) {
  void (*kernel)(FillParams<MAXB>);
  if (prm.vpr <= 32) kernel = fill_current_kernel<MAXB, 4, 1>;
  else if (prm.vpr <= 64) kernel = fill_current_kernel<MAXB, 4, 2>;
  else if (prm.vpr <= 96) kernel = fill_current_kernel<MAXB, 2, 3>;
  else if (prm.vpr <= 128) kernel = fill_current_kernel<MAXB, 2, 4>;
  else kernel = fill_current_kernel<MAXB, 0, 0>;
  return launch_kernel(kernel, dim3(grid), dim3(kFillThreads), 0, early, s, prm);
}

}  // namespace
}  // namespace cpkv

extern "C" int cpkv_fill_current(int B, int page_size, int cp_size, int64_t row_bytes,
                                 const int32_t *h_cur_lens, const void *const *h_cur_rows,
                                 const int64_t *h_cur_rows_cap, void *const *h_staging,
                                 int64_t staging_cap_pages, const int64_t *d_staging_rows,
                                 const int32_t *d_token_writer_row, const int32_t *d_writer,
                                 int64_t num_cur_pages, int flags, int32_t *d_status, cpkv_stream_t stream) {
  using namespace cpkv;
  if (B < 0 || page_size <= 0 || cp_size < 1 || cp_size > CPKV_MAX_CP) return CPKV_ERR_ARG;
  if ((flags & ~(CPKV_FLAG_EARLY_INPUTS | CPKV_FILL_PAGE_RUNS)) != 0) return CPKV_ERR_ARG;
  const bool early = (flags & CPKV_FLAG_EARLY_INPUTS) != 0;
  if (row_bytes <= 0 || row_bytes % 16 != 0) return CPKV_ERR_ARG;
  if (B > CPKV_MAX_BATCH) return CPKV_ERR_LIMIT;
  if (h_cur_rows == nullptr || h_cur_rows_cap == nullptr || h_staging == nullptr || d_status == nullptr)
    return CPKV_ERR_ARG;
  if (B > 0 && h_cur_lens == nullptr) return CPKV_ERR_ARG;
  int64_t T = 0, C = 0;
  for (int b = 0; b < B; ++b) {
    if (h_cur_lens[b] < 0) return CPKV_ERR_ARG;
    T += h_cur_lens[b];
    C += ceil_div(h_cur_lens[b], page_size);
  }
  if (num_cur_pages != C) return CPKV_ERR_ARG;
  if (staging_cap_pages < C + 1) return CPKV_ERR_CAPACITY;
  if (T > 0 && (d_staging_rows == nullptr || d_token_writer_row == nullptr || d_writer == nullptr))
    return CPKV_ERR_ARG;
  for (int w = 0; w < cp_size; ++w) {
    if (h_staging[w] == nullptr || !aligned16(h_staging[w])) return CPKV_ERR_ARG;
    if (h_cur_rows_cap[w] < 0) return CPKV_ERR_ARG;
    if (h_cur_rows_cap[w] > 0 && (h_cur_rows[w] == nullptr || !aligned16(h_cur_rows[w]))) return CPKV_ERR_ARG;
  }
  if (T == 0 && C == 0) return CPKV_OK;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

#define CPKV_FILL_FILL(prm)                                                                  \
  for (int w = 0; w < CPKV_MAX_CP; ++w) {                                                    \
    prm.cur_rows[w] = w < cp_size ? static_cast<const uint8_t *>(h_cur_rows[w]) : nullptr;   \
    prm.cur_cap[w] = w < cp_size ? h_cur_rows_cap[w] : 0;                                    \
    prm.staging[w] = w < cp_size ? static_cast<uint8_t *>(h_staging[w]) : nullptr;           \
  }                                                                                          \
  prm.staging_rows = d_staging_rows; prm.token_writer_row = d_token_writer_row;              \
  prm.writer = d_writer; prm.status = d_status; prm.T = T; prm.C = C;                        \
  prm.staging_cap_rows = staging_cap_pages * page_size; prm.R = row_bytes;                   \
  prm.ps = page_size; prm.cp = cp_size; prm.B = B; prm.nRow = nRow;                          \
  prm.vpr = (int)(row_bytes / 16); prm.units = C * upp; prm.upp = (int32_t)upp;              \
  for (int b = 0; b < B; ++b) prm.cur_lens[b] = h_cur_lens[b];

  // page mode for pages of at least one chunk (smaller pages are rows: the
  // row kernel moves the same bytes)
  const int64_t page_bytes = (int64_t)page_size * row_bytes;
  const bool pages = (flags & CPKV_FILL_PAGE_RUNS) != 0 && page_bytes >= kPageChunkVecs * 16;
  const int64_t upp = ceil_div(page_bytes, kPageChunkVecs * 16);
  const int64_t row_warps = pages ? ceil_div(C * upp, 2) : ceil_div(T, 2);
  const int64_t row_blocks_needed = ceil_div(row_warps, pages ? kPageWarps : kWarpsPerBlock);
  const int64_t sms = device_sm_count();
  const int page_blocks = C * upp <= sms * 3 * kPageWarps * kPageUnitsPerWarp3 ? 3 : kPageBlocksPerSm;
  const int64_t row_blocks_cap = sms * (pages ? page_blocks : kBlocksPerSm);
  const int nRow = (int)(row_blocks_needed < row_blocks_cap ? row_blocks_needed : row_blocks_cap);

  if (B <= 64) {
    FillParams<64> prm;
    CPKV_FILL_FILL(prm)
    if (pages) return launch_kernel(fill_pages_kernel<64>, dim3(nRow), dim3(kPageThreads), 0, early, s, prm);
    return launch_fill(prm, nRow + B, early, s);
  }
  FillParams<CPKV_MAX_BATCH> prm;
  CPKV_FILL_FILL(prm)
#undef CPKV_FILL_FILL
  if (pages)
    return launch_kernel(fill_pages_kernel<CPKV_MAX_BATCH>, dim3(nRow), dim3(kPageThreads), 0, early, s, prm);
  return launch_fill(prm, nRow + B, early, s);
}
