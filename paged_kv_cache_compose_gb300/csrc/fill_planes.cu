// cpkv_fill_current_planes: the per-layer fill for planar pages — the
// "index" kind of the pages, whose fill kernel is its own and is only pointed
// at the staging page inverse ("prefetch staging" message of commits
// 0d87bc5).  A planar page of ps tokens stores its planes one after the
// other; plane p holds the ps tokens' w_p-byte slices in token order (the NSA
// indexer keys: a 128-byte fp8 key plane, then a 4-byte fp32 scale plane).
// A token row therefore is not contiguous in the page, which is why an index
// copy of whole rows cannot fill it.
//
// For every token t (an index copy over planes, any row indices):
//   sr = staging_rows[t], slot = sr / ps, off = sr % ps, w = writer[slot - 1]
//   plane p of staging[w] page slot, token off  <-  cur_planes[p][w] row
//   token_writer_row[t]
// and for every request whose current length is not a multiple of ps, the
// slices after its last token up to the end of that page are zero in every
// plane.
//
// Blocks [0, nTile) take tiles of 128 tokens: the tile's indices are resolved
// once into shared memory, then each plane is copied as a flat loop over
// (token, unit) with consecutive threads on consecutive units, so a warp
// reads and writes contiguous bytes (a unit is 16 bytes when the plane allows
// it, else 4).  Blocks [nTile, nTile + B) zero the pad slices.
//
// With CPKV_FLAG_EARLY_INPUTS the fill is launched as a programmatic
// dependent of the previous kernel on the stream (the previous layer's
// gather) and each thread waits for it (store_gate) before its first store,
// as in cpkv_fill_current.
#include <stdint.h>

#include "common.cuh"

namespace cpkv {
namespace {

constexpr int kThreads = 128;  // also the tokens per tile
constexpr int kMaxPlanes = 4;
constexpr int kUnroll = 4;     // units per thread in flight

template <int MAXB>
struct PlaneParams {
  const uint8_t *planes[kMaxPlanes][CPKV_MAX_CP];  // writer w's rows of plane p
  int64_t cur_cap[CPKV_MAX_CP];
  uint8_t *staging[CPKV_MAX_CP];
  const int64_t *staging_rows;
  const int32_t *token_writer_row, *writer;
  int32_t *status;
  int64_t T, C, staging_cap_rows, page_bytes;
  int32_t plane_bytes[kMaxPlanes], plane_start[kMaxPlanes], plane_unit[kMaxPlanes];
  int32_t chunk_start[kMaxPlanes + 1];  // page mode: first chunk of plane p within a page (last: chunks per page)
  int64_t units;                        // page mode: C * chunks per page
  int32_t n_planes, ps, cp, B, nTile;
  int32_t cur_lens[MAXB];
};

template <int MAXB>
__device__ void copy_tile(const PlaneParams<MAXB> &p, int64_t t0, bool *stores_open) {
  __shared__ uint8_t *dst_page[kThreads];  // staging page base of each token (nullptr: skip)
  __shared__ int32_t dst_off[kThreads];    // token slot inside the page
  __shared__ int32_t src_row[kThreads];
  __shared__ int32_t src_w[kThreads];
  const int j = threadIdx.x;
  const int64_t t = t0 + j;
  uint8_t *page = nullptr;
  int32_t off = 0, row = 0, w = 0;
  if (t < p.T) {
    const int64_t sr = p.staging_rows[t];
    const int64_t slot = sr / p.ps;
    if (sr < p.ps || sr >= p.staging_cap_rows || slot > p.C) {
      raise_status(p.status, CPKV_STATUS_ROW_OOB);
    } else {
      w = p.writer[slot - 1];
      row = p.token_writer_row[t];
      if (w < 0 || w >= p.cp) raise_status(p.status, CPKV_STATUS_WRITER_OOB);
      else if (row < 0 || row >= p.cur_cap[w]) raise_status(p.status, CPKV_STATUS_ROW_OOB);
      else {
        page = p.staging[w] + slot * p.page_bytes;
        off = (int32_t)(sr - slot * p.ps);
      }
    }
  }
  dst_page[j] = page;
  dst_off[j] = off;
  src_row[j] = row;
  src_w[j] = w;
  __syncthreads();
  const int ntok = (int)min64(kThreads, p.T - t0);
  // rows are read once (evict_first); the staging is read back by the gather
  // right after this kernel (evict_last)
  const uint64_t stream_pol = l2_policy_evict_first(), keep_pol = l2_policy_evict_last();
  for (int pl = 0; pl < p.n_planes; ++pl) {
    const int32_t wp = p.plane_bytes[pl], unit = p.plane_unit[pl], start = p.plane_start[pl];
    const int32_t upt = wp / unit;  // units per token
    const int total = ntok * upt;
    // kUnroll units per thread in flight: all loads, then all stores
    for (int base = 0; base < total; base += kThreads * kUnroll) {
      uint4 v[kUnroll];
      uint8_t *dst[kUnroll];
#pragma unroll
      for (int r = 0; r < kUnroll; ++r) {
        const int i = base + j + r * kThreads;
        dst[r] = nullptr;
        if (i < total) {
          const int k = i / upt, u = i - k * upt;
          uint8_t *dp = dst_page[k];
          if (dp != nullptr) {
            dst[r] = dp + start + (int64_t)dst_off[k] * wp + (int64_t)u * unit;
            const uint8_t *s = p.planes[pl][src_w[k]] + (int64_t)src_row[k] * wp + (int64_t)u * unit;
            if (unit == 16) v[r] = ld_stream16_hint(s, stream_pol);
            else v[r].x = __ldg(reinterpret_cast<const uint32_t *>(s));
          }
        }
      }
      store_gate(stores_open);
#pragma unroll
      for (int r = 0; r < kUnroll; ++r) {
        if (dst[r] == nullptr) continue;
        if (unit == 16) st16_hint(dst[r], v[r], keep_pol);
        else *reinterpret_cast<uint32_t *>(dst[r]) = v[r].x;
      }
    }
  }
}

// Zero the slices after request b's last token up to the end of its page.
template <int MAXB>
__device__ void zero_pad(const PlaneParams<MAXB> &p, int b) {
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
  uint8_t *page = p.staging[w] + slot * p.page_bytes;
  const int64_t first = sr - slot * p.ps + 1;  // first pad token slot
  for (int pl = 0; pl < p.n_planes; ++pl) {
    uint32_t *z = reinterpret_cast<uint32_t *>(page + p.plane_start[pl] + first * p.plane_bytes[pl]);
    const int64_t words = (p.ps - first) * p.plane_bytes[pl] / 4;
    for (int64_t i = threadIdx.x; i < words; i += kThreads) z[i] = 0u;
  }
}

// ---------------------------------------------------------------------------
// Page mode (CPKV_FILL_PAGE_RUNS): with the plan of cpkv_plan_build, current
// page i's n_i tokens are consecutive rows of each plane of their writer,
// from token_writer_row of the page's first token, and their slices are
// consecutive in each plane of staging slot i + 1.  So each plane of a page
// is one contiguous run on both sides: a unit is one chunk of at most 4 KB of
// one plane of one page, moved with 16-byte vectors when its source,
// destination and sizes allow it, else with 4-byte words, the pad slices of a
// short page zeroed in the same pass.  A warp resolves the pages of 32 units
// at once with independent loads (writer, first and last source row, first
// staging row; a page that does not fit the run is skipped and raises
// ROW_OOB), as in the row page fill.  The index keys: two 4 KB key chunks and
// one 256-byte scale chunk per page.
constexpr int kPageThreads = 256;
constexpr int kPageWarps = kPageThreads / 32;
constexpr int kPageBlocksPerSm = 4;
constexpr int kChunkBytes = 4096;
constexpr int kChunkVpl = kChunkBytes / 16 / 32;  // 16-byte vectors per lane and chunk
constexpr int kWordVpl = 8;                       // 4-byte words per lane and pass

struct PlaneUnit {
  const uint8_t *src;  // nullptr: skip
  uint8_t *dst;
  int32_t copy, total;
};

template <int MAXB>
__device__ PlaneUnit resolve_plane_unit(const PlaneParams<MAXB> &p, const int32_t *cur_page_start,
                                        const int64_t *token_start, int64_t u) {
  PlaneUnit x{nullptr, nullptr, 0, 0};
  if (u >= p.units) return x;
  const int32_t upp = p.chunk_start[p.n_planes];
  const int64_t i = u / upp;
  const int32_t c = (int32_t)(u - i * upp);
  int q = 0;
  while (q + 1 < p.n_planes && p.chunk_start[q + 1] <= c) ++q;
  const int32_t k = c - p.chunk_start[q];
  const int b = upper_index<int32_t>(cur_page_start, p.B, (int32_t)i);
  const int32_t kp = (int32_t)i - cur_page_start[b];
  const int32_t n = min(p.ps, p.cur_lens[b] - kp * p.ps);
  const int64_t tok0 = token_start[b] + (int64_t)kp * p.ps;
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
  const int32_t wp = p.plane_bytes[q];
  const int64_t seg = (int64_t)p.ps * wp, off = (int64_t)k * kChunkBytes;
  x.total = (int32_t)min64(kChunkBytes, seg - off);
  const int64_t rows_bytes = (int64_t)n * wp;
  x.copy = (int32_t)(off < rows_bytes ? min64(x.total, rows_bytes - off) : 0);
  x.src = p.planes[q][w] + (int64_t)r0 * wp + off;
  x.dst = p.staging[w] + (i + 1) * p.page_bytes + p.plane_start[q] + off;
  return x;
}

template <int MAXB>
__global__ void __launch_bounds__(kPageThreads, kPageBlocksPerSm)
    fill_planes_pages_kernel(const __grid_constant__ PlaneParams<MAXB> p) {
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
  // the gather may launch now, as in cpkv_fill_current's page runs (index-key
  // 78-layer step 4.06 -> 4.00 ms against releasing as the blocks finish)
  release_dependents();
  const uint64_t read_once = l2_policy_evict_first(), keep = l2_policy_evict_last();
  const int64_t nw = (int64_t)gridDim.x * kPageWarps;
  const int64_t gw = (int64_t)blockIdx.x * kPageWarps + warp;
  bool stores_open = false;
  for (int64_t base = gw; base < p.units; base += 32 * nw) {
    const PlaneUnit mine = resolve_plane_unit(p, cur_page_start, token_start, base + lane * nw);
    for (int j = 0; j < 32; ++j) {
      if (base + j * nw >= p.units) break;  // uniform across the warp
      const uint8_t *src = reinterpret_cast<const uint8_t *>(
          __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(mine.src), j));
      uint8_t *dst = reinterpret_cast<uint8_t *>(
          __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(mine.dst), j));
      const int32_t copy = __shfl_sync(0xffffffffu, mine.copy, j);
      const int32_t total = __shfl_sync(0xffffffffu, mine.total, j);
      if (src == nullptr) continue;  // uniform
      if (((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst) | (uint32_t)copy |
            (uint32_t)total) & 15u) == 0) {
        uint4 v[kChunkVpl];
#pragma unroll
        for (int r = 0; r < kChunkVpl; ++r) {
          const int32_t off = 16 * (lane + 32 * r);
          v[r] = off < copy ? ld_stream16_hint(src + off, read_once) : make_uint4(0, 0, 0, 0);
        }
        store_gate(&stores_open);
#pragma unroll
        for (int r = 0; r < kChunkVpl; ++r) {
          const int32_t off = 16 * (lane + 32 * r);
          if (off < total) st16_hint(dst + off, v[r], keep);
        }
      } else {  // 4-byte slices at an offset that is not a 16-byte multiple
        for (int32_t w0 = 0; w0 < total / 4; w0 += 32 * kWordVpl) {
          uint32_t v[kWordVpl];
#pragma unroll
          for (int r = 0; r < kWordVpl; ++r) {
            const int32_t i = w0 + lane + 32 * r;
            v[r] = 4 * i < copy ? __ldg(reinterpret_cast<const uint32_t *>(src) + i) : 0u;
          }
          store_gate(&stores_open);
#pragma unroll
          for (int r = 0; r < kWordVpl; ++r) {
            const int32_t i = w0 + lane + 32 * r;
            if (4 * i < total) reinterpret_cast<uint32_t *>(dst)[i] = v[r];
          }
        }
      }
    }
  }
  // an early-launched fill finishes only after the kernel before it
  if (threadIdx.x == 0) store_gate(&stores_open);
}

template <int MAXB>
__global__ void __launch_bounds__(kThreads) fill_planes_kernel(const __grid_constant__ PlaneParams<MAXB> p) {
  if ((int)blockIdx.x < p.nTile) {
    bool stores_open = false;
    for (int64_t t0 = (int64_t)blockIdx.x * kThreads; t0 < p.T; t0 += (int64_t)p.nTile * kThreads) {
      copy_tile(p, t0, &stores_open);
      __syncthreads();  // the tile's shared indices are reused by the next tile
    }
  } else {
    zero_pad(p, blockIdx.x - p.nTile);
  }
  release_dependents();  // as in cpkv_fill_current
}

}  // namespace
}  // namespace cpkv

extern "C" int cpkv_fill_current_planes(int B, int page_size, int cp_size, int n_planes, const int32_t *h_plane_bytes,
                                        const int32_t *h_cur_lens, const void *const *h_cur_planes,
                                        const int64_t *h_cur_rows_cap, void *const *h_staging,
                                        int64_t staging_cap_pages, const int64_t *d_staging_rows,
                                        const int32_t *d_token_writer_row, const int32_t *d_writer,
                                        int64_t num_cur_pages, int flags, int32_t *d_status,
                                        cpkv_stream_t stream) {
  using namespace cpkv;
  if (B < 0 || page_size <= 0 || cp_size < 1 || cp_size > CPKV_MAX_CP) return CPKV_ERR_ARG;
  if ((flags & ~(CPKV_FLAG_EARLY_INPUTS | CPKV_FILL_PAGE_RUNS)) != 0) return CPKV_ERR_ARG;
  const bool early = (flags & CPKV_FLAG_EARLY_INPUTS) != 0;
  const bool pages = (flags & CPKV_FILL_PAGE_RUNS) != 0;
  if (n_planes < 1 || n_planes > kMaxPlanes || h_plane_bytes == nullptr) return CPKV_ERR_ARG;
  if (B > CPKV_MAX_BATCH) return CPKV_ERR_LIMIT;
  if (h_cur_planes == nullptr || h_cur_rows_cap == nullptr || h_staging == nullptr || d_status == nullptr)
    return CPKV_ERR_ARG;
  if (B > 0 && h_cur_lens == nullptr) return CPKV_ERR_ARG;
  int64_t row_bytes = 0;
  for (int p = 0; p < n_planes; ++p) {
    if (h_plane_bytes[p] <= 0 || h_plane_bytes[p] % 4 != 0) return CPKV_ERR_ARG;
    row_bytes += h_plane_bytes[p];
  }
  const int64_t page_bytes = (int64_t)page_size * row_bytes;
  if (page_bytes % 16 != 0 || page_bytes > INT32_MAX) return CPKV_ERR_ARG;
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
    for (int p = 0; p < n_planes; ++p) {
      const void *ptr = h_cur_planes[p * cp_size + w];
      if (h_cur_rows_cap[w] > 0 && (ptr == nullptr || !aligned16(ptr))) return CPKV_ERR_ARG;
    }
  }
  if (T == 0) return CPKV_OK;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int64_t tiles = ceil_div(T, kThreads);
  const int64_t cap = (int64_t)device_sm_count() * 16;
  const int nTile = (int)(tiles < cap ? tiles : cap);

#define CPKV_FILL_PLANES(prm)                                                                          \
  for (int p = 0; p < kMaxPlanes; ++p)                                                                 \
    for (int w = 0; w < CPKV_MAX_CP; ++w)                                                              \
      prm.planes[p][w] = (p < n_planes && w < cp_size)                                                 \
                             ? static_cast<const uint8_t *>(h_cur_planes[p * cp_size + w]) : nullptr;  \
  for (int w = 0; w < CPKV_MAX_CP; ++w) {                                                              \
    prm.cur_cap[w] = w < cp_size ? h_cur_rows_cap[w] : 0;                                              \
    prm.staging[w] = w < cp_size ? static_cast<uint8_t *>(h_staging[w]) : nullptr;                     \
  }                                                                                                    \
  {                                                                                                    \
    int32_t start = 0;                                                                                 \
    for (int p = 0; p < kMaxPlanes; ++p) {                                                             \
      const int32_t wp = p < n_planes ? h_plane_bytes[p] : 0;                                          \
      prm.plane_bytes[p] = wp;                                                                         \
      prm.plane_start[p] = start;                                                                      \
      prm.plane_unit[p] = (wp % 16 == 0 && start % 16 == 0) ? 16 : 4;                                 \
      start += page_size * wp;                                                                         \
    }                                                                                                  \
  }                                                                                                    \
  prm.staging_rows = d_staging_rows; prm.token_writer_row = d_token_writer_row; prm.writer = d_writer; \
  prm.status = d_status; prm.T = T; prm.C = C; prm.staging_cap_rows = staging_cap_pages * page_size;  \
  prm.page_bytes = page_bytes; prm.n_planes = n_planes; prm.ps = page_size; prm.cp = cp_size;         \
  prm.B = B; prm.nTile = nTile;                                                                        \
  {                                                                                                    \
    int32_t cs = 0;                                                                                    \
    for (int p = 0; p <= kMaxPlanes; ++p) {                                                            \
      prm.chunk_start[p] = cs;                                                                         \
      if (p < n_planes) cs += (int32_t)ceil_div((int64_t)page_size * h_plane_bytes[p], kChunkBytes);   \
    }                                                                                                  \
    prm.chunk_start[n_planes] = cs;                                                                    \
    prm.units = C * cs;                                                                                \
  }                                                                                                    \
  for (int b = 0; b < B; ++b) prm.cur_lens[b] = h_cur_lens[b];

  // page mode: one resident wave of 4 blocks per SM, about 2 units per warp
  int64_t upp = 0;
  for (int p = 0; p < n_planes; ++p) upp += ceil_div((int64_t)page_size * h_plane_bytes[p], kChunkBytes);
  const int64_t pblocks = ceil_div(ceil_div(C * upp, 2), kPageWarps);
  const int64_t pcap = (int64_t)device_sm_count() * kPageBlocksPerSm;
  const int nPage = (int)(pblocks < pcap ? (pblocks > 0 ? pblocks : 1) : pcap);

  if (B <= 64) {
    PlaneParams<64> prm;
    CPKV_FILL_PLANES(prm)
    if (pages) return launch_kernel(fill_planes_pages_kernel<64>, dim3(nPage), dim3(kPageThreads), 0, early, s, prm);
    return launch_kernel(fill_planes_kernel<64>, dim3(nTile + B), dim3(kThreads), 0, early, s, prm);
  }
  PlaneParams<CPKV_MAX_BATCH> prm;
  CPKV_FILL_PLANES(prm)
#undef CPKV_FILL_PLANES
  if (pages)
    return launch_kernel(fill_planes_pages_kernel<CPKV_MAX_BATCH>, dim3(nPage), dim3(kPageThreads), 0, early, s, prm);
  return launch_kernel(fill_planes_kernel<CPKV_MAX_BATCH>, dim3(nTile + B), dim3(kThreads), 0, early, s, prm);
}
