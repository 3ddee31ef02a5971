// cpkv_ragged_plan_build: the NSA indexer's per-batch ragged index plan of
// one CP rank ("CPU-gap fixes" message of commits d63fbd4: a per-batch plan
// replaces the per-layer rebuild of the O(total q) topk offset list and the
// int32 segment / kv_lens / q_starts / q_lens / k_bases / q_bases /
// current_bases descriptors; all inputs are batch metadata keyed on cp_index).
//
// One launch of G CTAs of 1024 threads.  Every CTA rebuilds the request-level
// scans (chunk ids, k bases) in shared memory, then walks cp_index in tiles of
// 1024 owned chunks with two block scans per tile (segment starts, token
// counts) and carries across tiles.  CTA 0 writes the segment arrays.  The
// rank's q tokens are cut into G equal ranges; CTA g writes the topk offsets
// of range g with coalesced stores (a token finds its chunk by binary search
// over the tile's token offsets in shared memory).
#include <stdint.h>

#include "common.cuh"

namespace cpkv {
namespace {

constexpr int kRaggedThreads = 1024;

template <int MAXB>
struct RaggedParams {
  int B, chunk, k_align;
  int64_t n;
  const int32_t *cp_index;
  int32_t *topk;
  int64_t topk_cap;
  int32_t *seg_req, *kv_lens, *q_starts, *q_lens, *k_bases, *q_bases, *current_bases;
  int64_t seg_cap;
  int64_t *counts;
  int32_t *status;
  int64_t q_span;  // q tokens per CTA for the topk offsets
  int32_t prefix_lens[MAXB];
  int32_t q_lens_in[MAXB];
};

template <int MAXB>
__global__ void __launch_bounds__(kRaggedThreads) ragged_plan_kernel(const __grid_constant__ RaggedParams<MAXB> p) {
  __shared__ int32_t chunk_first[CPKV_MAX_BATCH + 1];  // first chunk id of request b
  __shared__ int64_t kbase[CPKV_MAX_BATCH + 1];        // k base of request b
  __shared__ int64_t scratch[33];
  __shared__ int64_t tile_qpos[kRaggedThreads];
  __shared__ int32_t tile_kb[kRaggedThreads];
  __shared__ int64_t tile_q0, tile_q1;

  const int tid = threadIdx.x;
  const int B = p.B, chunk = p.chunk;
  {
    int64_t nch = 0, kv_al = 0;
    if (tid < B) {
      nch = (p.q_lens_in[tid] + chunk - 1) / chunk;
      const int64_t kv = (int64_t)p.prefix_lens[tid] + p.q_lens_in[tid];
      kv_al = (kv + p.k_align - 1) / p.k_align * p.k_align;
    }
    int64_t tot;
    const int64_t cf = block_exclusive_scan<int64_t>(nch, scratch, &tot);
    if (tid < B) chunk_first[tid] = (int32_t)cf;
    if (tid == 0) chunk_first[B] = (int32_t)tot;
    const int64_t kb = block_exclusive_scan<int64_t>(kv_al, scratch, &tot);
    if (tid < B) kbase[tid] = kb;
    if (tid == 0) kbase[B] = tot;
    __syncthreads();
  }
  const int64_t total_chunks = chunk_first[B];

  int64_t seg_carry = 0, q_carry = 0;
  const int64_t ntiles = (p.n + kRaggedThreads - 1) / kRaggedThreads;
  for (int64_t tile = 0; tile < ntiles; ++tile) {
    const int64_t k = tile * kRaggedThreads + tid;
    bool ok = false, start = false, end = false;
    int b = 0;
    int64_t off = 0, len = 0;
    if (k < p.n) {
      const int64_t id = p.cp_index[k];
      const int64_t prev = k > 0 ? (int64_t)p.cp_index[k - 1] : -1;
      ok = id >= 0 && id < total_chunks && (k == 0 || id > prev) && B > 0;
      if (!ok) {
        raise_status(p.status, CPKV_STATUS_CHUNK_OOB);
      } else {
        b = upper_index<int32_t>(chunk_first, B, (int32_t)id);
        off = (id - chunk_first[b]) * chunk;
        len = min64(chunk, p.q_lens_in[b] - off);
        const int64_t next = k + 1 < p.n ? (int64_t)p.cp_index[k + 1] : -1;
        start = k == 0 || id != prev + 1 || id == chunk_first[b];
        end = k + 1 == p.n || next != id + 1 || id + 1 == chunk_first[b + 1];
      }
    }
    int64_t nstart, ntok;
    const int64_t seg_before = block_exclusive_scan<int64_t>(start ? 1 : 0, scratch, &nstart);
    const int64_t qpos = q_carry + block_exclusive_scan<int64_t>(len, scratch, &ntok);
    const int64_t s = seg_carry + seg_before + (start ? 1 : 0) - 1;  // this chunk's segment

    if (blockIdx.x == 0) {
      if (ok && start) {
        if (s < p.seg_cap) {
          p.seg_req[s] = b;
          p.q_starts[s] = (int32_t)off;
          p.k_bases[s] = (int32_t)kbase[b];
          p.current_bases[s] = (int32_t)(kbase[b] + p.prefix_lens[b]);
          p.q_bases[s] = (int32_t)qpos;
        } else {
          raise_status(p.status, CPKV_STATUS_OUT_CAPACITY);
        }
      }
      __syncthreads();  // segment starts of this tile are visible to the block
      if (ok && end && s >= 0 && s < p.seg_cap) {
        const int64_t seg_end = off + len;  // token offset after the segment, inside request b
        p.q_lens[s] = (int32_t)(seg_end - p.q_starts[s]);
        p.kv_lens[s] = (int32_t)(p.prefix_lens[b] + seg_end);
      }
    }

    // this CTA's slice of the tile's q tokens
    const int64_t lo_q = (int64_t)blockIdx.x * p.q_span, hi_q = lo_q + p.q_span;
    if (q_carry < hi_q && q_carry + ntok > lo_q) {
      tile_qpos[tid] = qpos;
      tile_kb[tid] = (int32_t)kbase[b];
      if (tid == 0) {
        tile_q0 = q_carry > lo_q ? q_carry : lo_q;
        tile_q1 = q_carry + ntok < hi_q ? q_carry + ntok : hi_q;
      }
      __syncthreads();
      const int nk = (int)min64(kRaggedThreads, p.n - tile * kRaggedThreads);
      for (int64_t q = tile_q0 + tid; q < tile_q1; q += kRaggedThreads) {
        // chunk of token q: last chunk in the tile whose qpos <= q
        int lo = 0, hi = nk - 1;
        while (lo < hi) {
          const int mid = (lo + hi + 1) >> 1;
          if (tile_qpos[mid] <= q) lo = mid;
          else hi = mid - 1;
        }
        if (q < p.topk_cap) p.topk[q] = tile_kb[lo];
        else raise_status(p.status, CPKV_STATUS_OUT_CAPACITY);
      }
      __syncthreads();
    }
    seg_carry += nstart;
    q_carry += ntok;
  }
  if (blockIdx.x == 0 && tid == 0 && p.counts != nullptr) {
    p.counts[0] = seg_carry;
    p.counts[1] = q_carry;
  }
}

}  // namespace
}  // namespace cpkv

extern "C" int cpkv_ragged_plan_build(int B, int chunk, int k_align, int topk, const int32_t *h_prefix_lens,
                                      const int32_t *h_q_lens, const int32_t *d_cp_index, int64_t n_owned,
                                      int32_t *d_topk_offsets, int64_t topk_cap, int32_t *d_seg_req,
                                      int32_t *d_kv_lens, int32_t *d_q_starts, int32_t *d_q_lens,
                                      int32_t *d_k_bases, int32_t *d_q_bases, int32_t *d_current_bases,
                                      int64_t seg_cap, int64_t *d_counts, int32_t *d_status,
                                      cpkv_stream_t stream) {
  using namespace cpkv;
  // topk is the consumer's index width: no plan array depends on it, but a
  // plan for a non-positive width is a caller error
  if (B < 0 || chunk <= 0 || k_align <= 0 || topk <= 0 || n_owned < 0 || topk_cap < 0 || seg_cap < 0)
    return CPKV_ERR_ARG;
  if (B > CPKV_MAX_BATCH) return CPKV_ERR_LIMIT;
  if (d_status == nullptr || d_counts == nullptr) return CPKV_ERR_ARG;
  if (B > 0 && (h_prefix_lens == nullptr || h_q_lens == nullptr)) return CPKV_ERR_ARG;
  if (n_owned > 0 && d_cp_index == nullptr) return CPKV_ERR_ARG;
  if (seg_cap > 0 && (d_seg_req == nullptr || d_kv_lens == nullptr || d_q_starts == nullptr ||
                      d_q_lens == nullptr || d_k_bases == nullptr || d_q_bases == nullptr ||
                      d_current_bases == nullptr))
    return CPKV_ERR_ARG;
  if (topk_cap > 0 && d_topk_offsets == nullptr) return CPKV_ERR_ARG;
  int64_t total_chunks = 0, total_kv = 0;
  for (int b = 0; b < B; ++b) {
    if (h_prefix_lens[b] < 0 || h_q_lens[b] < 0) return CPKV_ERR_ARG;
    total_chunks += ceil_div(h_q_lens[b], chunk);
    total_kv += ceil_div((int64_t)h_prefix_lens[b] + h_q_lens[b], k_align) * k_align;
  }
  if (total_chunks > INT32_MAX || total_kv > INT32_MAX) return CPKV_ERR_LIMIT;
  if (n_owned > INT32_MAX) return CPKV_ERR_LIMIT;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // one CTA per kTokensPerCta q tokens (upper bound n_owned * chunk), at most one per SM
  constexpr int64_t kTokensPerCta = 2048;
  const int64_t q_max = n_owned * chunk;
  const int64_t sms = device_sm_count();
  int64_t g = ceil_div(q_max, kTokensPerCta);
  g = g < 1 ? 1 : (g < sms ? g : sms);
  const int grid = (int)g;
  const int64_t q_span = q_max > 0 ? ceil_div(q_max, g) : 1;

#define CPKV_FILL_RAGGED(prm)                                                                   \
  prm.B = B; prm.chunk = chunk; prm.k_align = k_align; prm.n = n_owned; prm.cp_index = d_cp_index; \
  prm.topk = d_topk_offsets; prm.topk_cap = topk_cap; prm.seg_req = d_seg_req; prm.kv_lens = d_kv_lens; \
  prm.q_starts = d_q_starts; prm.q_lens = d_q_lens; prm.k_bases = d_k_bases; prm.q_bases = d_q_bases; \
  prm.current_bases = d_current_bases; prm.seg_cap = seg_cap; prm.counts = d_counts;            \
  prm.status = d_status; prm.q_span = q_span;                                                   \
  for (int b = 0; b < B; ++b) { prm.prefix_lens[b] = h_prefix_lens[b]; prm.q_lens_in[b] = h_q_lens[b]; }

  if (B <= 64) {
    RaggedParams<64> prm;
    CPKV_FILL_RAGGED(prm)
    ragged_plan_kernel<64><<<grid, kRaggedThreads, 0, s>>>(prm);
    return launch_status();
  }
  RaggedParams<CPKV_MAX_BATCH> prm;
  CPKV_FILL_RAGGED(prm)
#undef CPKV_FILL_RAGGED
  ragged_plan_kernel<CPKV_MAX_BATCH><<<grid, kRaggedThreads, 0, s>>>(prm);
  return launch_status();
}
