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
// (19.99 ms).  In a plain launch the gate returns at once.  The fill itself
// releases its dependents as each block finishes, for a gather launched with
// CPKV_GATHER_EARLY_INPUTS.
//
// (A variant that moves whole pages with bulk copies when a page's indices
// form a run was slower here: each page first needs a round trip of index
// loads, and a layer has only a few pages per CTA to overlap them with.)
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
  if ((flags & ~CPKV_FLAG_EARLY_INPUTS) != 0) return CPKV_ERR_ARG;
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

  const int64_t row_warps = ceil_div(T, 2);
  const int64_t row_blocks_needed = ceil_div(row_warps, kWarpsPerBlock);
  const int64_t row_blocks_cap = (int64_t)device_sm_count() * kBlocksPerSm;
  const int nRow = (int)(row_blocks_needed < row_blocks_cap ? row_blocks_needed : row_blocks_cap);

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
  prm.vpr = (int)(row_bytes / 16);                                                           \
  for (int b = 0; b < B; ++b) prm.cur_lens[b] = h_cur_lens[b];

  if (B <= 64) {
    FillParams<64> prm;
    CPKV_FILL_FILL(prm)
    return launch_fill(prm, nRow + B, early, s);
  }
  FillParams<CPKV_MAX_BATCH> prm;
  CPKV_FILL_FILL(prm)
#undef CPKV_FILL_FILL
  return launch_fill(prm, nRow + B, early, s);
}
