// cpkv_fill_current: the per-layer fill of current rows into the writers'
// stagings ("staging-direct compose" message of commits d63fbd4: the fill is
// a single index copy of layer-invariant row indices; "fp8 -> uint8"
// message of commits 0d87bc5: rows are opaque bytes).
//
// The work is cut by current page: the tokens of page i are consecutive in
// batch order, so with the plan's row indices they form one run of
// consecutive source rows (in their writer's current-row buffer) and one run
// of consecutive staging rows starting on a page boundary.  For each page the
// warp first checks that the page's indices really form such a run; if so it
// moves the page with the bulk-copy ring (bulk_ring.cuh) in pieces of at most
// 24 KB, and zeroes the pad rows after a request's last token up to the end
// of its staging page.  Any page whose indices do not form a run is copied row
// by row, exactly as an index copy (16-byte vectors), with its pad rows zeroed
// after the request's last token.  Either way the result is the index copy
// the contract describes.
//
// Current rows are read once (L2 evict_first); staging rows are stored with
// evict_last because the gather that follows reads them back from L2.
#include <stdint.h>

#include "bulk_ring.cuh"

namespace cpkv {
namespace {

constexpr int kStages = 4;
constexpr int kLoadsInFlight = 2;
constexpr int kCtasPerSm = 2;
constexpr int kMaxPieceBytes = 24 * 1024;

template <int MAXB>
struct FillParams {
  const uint8_t *cur_rows[CPKV_MAX_CP];
  int64_t cur_cap[CPKV_MAX_CP];
  uint8_t *staging[CPKV_MAX_CP];
  const int64_t *staging_rows;
  const int32_t *token_writer_row, *writer;
  int32_t *status;
  int64_t C, staging_cap_rows, R, page_bytes, units;
  int32_t ps, cp, B, pieces, piece_bytes;
  int32_t cur_lens[MAXB];
};

// Copy one token row (index-copy semantics), validating every index.
template <int MAXB>
__device__ void copy_row(const FillParams<MAXB> &p, int64_t t, uint64_t read_once, uint64_t keep) {
  const int lane = threadIdx.x & 31;
  const int64_t sr = p.staging_rows[t];
  const int64_t slot = sr / p.ps;
  if (sr < p.ps || sr >= p.staging_cap_rows || slot > p.C) {
    if (lane == 0) raise_status(p.status, CPKV_STATUS_ROW_OOB);
    return;
  }
  const int32_t w = p.writer[slot - 1];
  if (w < 0 || w >= p.cp) {
    if (lane == 0) raise_status(p.status, CPKV_STATUS_WRITER_OOB);
    return;
  }
  const int32_t r = p.token_writer_row[t];
  if (r < 0 || r >= p.cur_cap[w]) {
    if (lane == 0) raise_status(p.status, CPKV_STATUS_ROW_OOB);
    return;
  }
  const uint8_t *src = p.cur_rows[w] + (int64_t)r * p.R;
  uint8_t *dst = p.staging[w] + sr * p.R;
  for (int64_t c = lane; c < p.R / 16; c += 32)
    st16_hint(dst + 16 * c, ld_stream16_hint(src + 16 * c, read_once), keep);
}

// Zero the rows after staging row `sr_last` up to the end of its page.
template <int MAXB>
__device__ void zero_after(const FillParams<MAXB> &p, int64_t sr_last, uint64_t keep) {
  const int64_t slot = sr_last / p.ps;
  if (sr_last < p.ps || sr_last >= p.staging_cap_rows || slot > p.C) {
    if ((threadIdx.x & 31) == 0) raise_status(p.status, CPKV_STATUS_ROW_OOB);
    return;
  }
  const int32_t w = p.writer[slot - 1];
  if (w < 0 || w >= p.cp) {
    if ((threadIdx.x & 31) == 0) raise_status(p.status, CPKV_STATUS_WRITER_OOB);
    return;
  }
  const int64_t first = sr_last + 1, end = (slot + 1) * p.ps;
  if (first < end) warp_zero_hint(p.staging[w] + first * p.R, (uint32_t)((end - first) * p.R), keep);
}

template <int MAXB>
__global__ void __launch_bounds__(32) fill_pages_kernel(const __grid_constant__ FillParams<MAXB> p) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t full[kStages];
  __shared__ uint8_t *ring_dst[kStages];
  __shared__ uint32_t ring_bytes[kStages];
  __shared__ int ring_live[kStages];
  __shared__ int32_t cur_page_start[MAXB + 1];  // first batch current page of request b
  __shared__ int64_t token_start[MAXB + 1];     // first batch token of request b
  const int lane = threadIdx.x;
  const uint64_t read_once = l2_policy_evict_first();
  const uint64_t keep = l2_policy_evict_last();

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

  BulkRing<kStages, kLoadsInFlight> ring;
  ring.init(smem, full, ring_dst, ring_bytes, ring_live, p.status, p.piece_bytes, /*keep_stores=*/true);
  for (int64_t u = blockIdx.x; u < p.units; u += gridDim.x) {
    const int64_t i = u / p.pieces;  // batch current page
    const int32_t k = (int32_t)(u - i * p.pieces);
    const int b = upper_index<int32_t>(cur_page_start, p.B, (int32_t)i);
    const int32_t kp = (int32_t)i - cur_page_start[b];
    const int64_t tok0 = token_start[b] + (int64_t)kp * p.ps;
    const int64_t n = min64(p.ps, (int64_t)p.cur_lens[b] - (int64_t)kp * p.ps);  // rows of this page
    const bool last_of_request = (int64_t)kp * p.ps + n == p.cur_lens[b];

    // does the page form one run: page-aligned staging rows, consecutive source rows?
    const int64_t sr0 = p.staging_rows[tok0];
    const int32_t r0 = p.token_writer_row[tok0];
    const int64_t slot = sr0 / p.ps;
    bool run = sr0 % p.ps == 0 && sr0 >= p.ps && slot <= p.C && sr0 + p.ps <= p.staging_cap_rows;
    int32_t w = -1;
    if (run) {
      w = p.writer[slot - 1];
      run = w >= 0 && w < p.cp && r0 >= 0 && (int64_t)r0 + n <= p.cur_cap[w];
    }
    bool mine = true;
    for (int64_t j = lane; j < n; j += 32)
      mine &= p.staging_rows[tok0 + j] == sr0 + j && p.token_writer_row[tok0 + j] == r0 + j;
    run = __all_sync(0xffffffffu, mine) && run;

    if (run) {
      const int64_t off = (int64_t)k * p.piece_bytes;
      const uint32_t bytes = (uint32_t)min64(p.piece_bytes, p.page_bytes - off);
      uint8_t *dst = p.staging[w] + sr0 * p.R + off;
      const int64_t rows_bytes = n * p.R;
      const int64_t copy = off < rows_bytes ? min64(bytes, rows_bytes - off) : 0;
      if (copy > 0) ring.push(p.cur_rows[w] + (int64_t)r0 * p.R + off, dst, (uint32_t)copy);
      // rows past n exist only on a request's last (partial) page: zero them
      if (copy < bytes && last_of_request) warp_zero_hint(dst + copy, bytes - (uint32_t)copy, keep);
    } else if (k == 0) {
      for (int64_t j = 0; j < n; ++j) copy_row(p, tok0 + j, read_once, keep);
      __syncwarp();  // the row copies are ordered before the pad zeroing
      if (last_of_request && p.cur_lens[b] % p.ps != 0) zero_after(p, p.staging_rows[tok0 + n - 1], keep);
    }
  }
  ring.drain();
}

template <int MAXB>
int launch_fill(const FillParams<MAXB> &prm, int grid, size_t smem, cudaStream_t s, int slot) {
  static int configured[256][2] = {{0}};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 256 && !configured[dev][slot]) {
    if (cudaFuncSetAttribute(fill_pages_kernel<MAXB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kStages * kMaxPieceBytes) != cudaSuccess)
      return CPKV_ERR_CUDA;
    configured[dev][slot] = 1;
  }
  fill_pages_kernel<MAXB><<<grid, 32, smem, s>>>(prm);
  return launch_status();
}

}  // namespace
}  // namespace cpkv

extern "C" int cpkv_fill_current(int B, int page_size, int cp_size, int64_t row_bytes,
                                 const int32_t *h_cur_lens, const void *const *h_cur_rows,
                                 const int64_t *h_cur_rows_cap, void *const *h_staging,
                                 int64_t staging_cap_pages, const int64_t *d_staging_rows,
                                 const int32_t *d_token_writer_row, const int32_t *d_writer,
                                 int64_t num_cur_pages, int32_t *d_status, cpkv_stream_t stream) {
  using namespace cpkv;
  if (B < 0 || page_size <= 0 || cp_size < 1 || cp_size > CPKV_MAX_CP) return CPKV_ERR_ARG;
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
  if (T > INT32_MAX - 1 || C > INT32_MAX - 2) return CPKV_ERR_LIMIT;
  if (staging_cap_pages < C + 1) return CPKV_ERR_CAPACITY;
  if (T > 0 && (d_staging_rows == nullptr || d_token_writer_row == nullptr || d_writer == nullptr))
    return CPKV_ERR_ARG;
  for (int w = 0; w < cp_size; ++w) {
    if (h_staging[w] == nullptr || !aligned16(h_staging[w])) return CPKV_ERR_ARG;
    if (h_cur_rows_cap[w] < 0) return CPKV_ERR_ARG;
    if (h_cur_rows_cap[w] > 0 && (h_cur_rows[w] == nullptr || !aligned16(h_cur_rows[w]))) return CPKV_ERR_ARG;
  }
  if (C == 0) return CPKV_OK;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

  const int64_t page_bytes = (int64_t)page_size * row_bytes;
  const int64_t pieces = ceil_div(page_bytes, kMaxPieceBytes);
  const int64_t piece_bytes = ceil_div(ceil_div(page_bytes, pieces), 16) * 16;
  if (pieces > INT32_MAX || C > INT64_MAX / pieces) return CPKV_ERR_LIMIT;
  const int64_t units = C * pieces;
  const int64_t cap = (int64_t)device_sm_count() * kCtasPerSm;
  const int grid = (int)(units < cap ? units : cap);
  const size_t smem = (size_t)kStages * piece_bytes;

#define CPKV_FILL_FILL(prm)                                                                  \
  for (int w = 0; w < CPKV_MAX_CP; ++w) {                                                    \
    prm.cur_rows[w] = w < cp_size ? static_cast<const uint8_t *>(h_cur_rows[w]) : nullptr;   \
    prm.cur_cap[w] = w < cp_size ? h_cur_rows_cap[w] : 0;                                    \
    prm.staging[w] = w < cp_size ? static_cast<uint8_t *>(h_staging[w]) : nullptr;           \
  }                                                                                          \
  prm.staging_rows = d_staging_rows; prm.token_writer_row = d_token_writer_row;              \
  prm.writer = d_writer; prm.status = d_status; prm.C = C;                                   \
  prm.staging_cap_rows = staging_cap_pages * page_size; prm.R = row_bytes;                   \
  prm.page_bytes = page_bytes; prm.units = units; prm.ps = page_size; prm.cp = cp_size;      \
  prm.B = B; prm.pieces = (int32_t)pieces; prm.piece_bytes = (int32_t)piece_bytes;          \
  for (int b = 0; b < B; ++b) prm.cur_lens[b] = h_cur_lens[b];

  if (B <= 64) {
    FillParams<64> prm;
    CPKV_FILL_FILL(prm)
    return launch_fill(prm, grid, smem, s, 0);
  }
  FillParams<CPKV_MAX_BATCH> prm;
  CPKV_FILL_FILL(prm)
#undef CPKV_FILL_FILL
  return launch_fill(prm, grid, smem, s, 1);
}
