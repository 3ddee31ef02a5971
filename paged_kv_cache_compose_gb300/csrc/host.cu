// Host-only entry points of the cpkv library: batch sizing, writer token
// counts, ragged-plan sizing, error strings, device queries.  No GPU work.
#include <stdint.h>

#include "common.cuh"

namespace cpkv {

int device_sm_count() {
  static int cache[256] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 256) return 148;
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cache[dev] = n;
  }
  return cache[dev];
}

}  // namespace cpkv

extern "C" int cpkv_plan_sizes(int B, int page_size, const int32_t *h_prefix_lens,
                               const int32_t *h_cur_lens, cpkv_sizes *out) {
  if (B < 0 || page_size <= 0 || out == nullptr) return CPKV_ERR_ARG;
  if (B > 0 && (h_prefix_lens == nullptr || h_cur_lens == nullptr)) return CPKV_ERR_ARG;
  int64_t T = 0, C = 0, D = 0;
  for (int b = 0; b < B; ++b) {
    const int64_t pl = h_prefix_lens[b], cl = h_cur_lens[b];
    if (pl < 0 || cl < 0) return CPKV_ERR_ARG;
    if (pl % page_size != 0) return CPKV_ERR_UNALIGNED_PREFIX;
    const int64_t npp = pl / page_size, ncp = cpkv::ceil_div(cl, page_size);
    T += cl;
    C += ncp;
    D += npp + ncp;
  }
  // Every index array is int32 and staging slots reach C + 1.
  if (T > INT32_MAX - 1 || D > INT32_MAX - 1 || C > INT32_MAX - 2) return CPKV_ERR_LIMIT;
  out->T = T;
  out->C = C;
  out->D = D;
  return CPKV_OK;
}

extern "C" int cpkv_writer_token_counts(int B, int page_size, int cp_size, const int32_t *h_cur_lens,
                                        const int32_t *h_writer, int64_t C,
                                        int64_t *h_tokens_per_writer) {
  if (B < 0 || page_size <= 0 || cp_size < 1 || cp_size > CPKV_MAX_CP || h_tokens_per_writer == nullptr)
    return CPKV_ERR_ARG;
  if (B > 0 && h_cur_lens == nullptr) return CPKV_ERR_ARG;
  if (C > 0 && h_writer == nullptr) return CPKV_ERR_ARG;
  for (int w = 0; w < cp_size; ++w) h_tokens_per_writer[w] = 0;
  int64_t i = 0;
  for (int b = 0; b < B; ++b) {
    if (h_cur_lens[b] < 0) return CPKV_ERR_ARG;
    for (int64_t k = 0; k < h_cur_lens[b]; k += page_size) {
      if (i >= C) return CPKV_ERR_ARG;
      const int32_t w = h_writer[i];
      if (w < 0 || w >= cp_size) return CPKV_ERR_ARG;
      const int64_t n = h_cur_lens[b] - k < page_size ? h_cur_lens[b] - k : page_size;
      h_tokens_per_writer[w] += n;
      ++i;
    }
  }
  return i == C ? CPKV_OK : CPKV_ERR_ARG;
}

extern "C" int cpkv_ragged_plan_sizes(int B, int chunk, const int32_t *h_q_lens, const int32_t *h_cp_index,
                                      int64_t n_owned, int64_t *h_S, int64_t *h_Q) {
  if (B < 0 || chunk <= 0 || n_owned < 0 || h_S == nullptr || h_Q == nullptr) return CPKV_ERR_ARG;
  if ((B > 0 && h_q_lens == nullptr) || (n_owned > 0 && h_cp_index == nullptr)) return CPKV_ERR_ARG;
  // chunk ids of request b are [first[b], first[b+1])
  int64_t total = 0;
  for (int b = 0; b < B; ++b) {
    if (h_q_lens[b] < 0) return CPKV_ERR_ARG;
    total += cpkv::ceil_div(h_q_lens[b], chunk);
  }
  int64_t S = 0, Q = 0, prev = -1, req = 0, first = 0;
  for (int64_t k = 0; k < n_owned; ++k) {
    const int64_t id = h_cp_index[k];
    if (id < 0 || id >= total || id <= prev) return CPKV_ERR_ARG;
    while (first + cpkv::ceil_div(h_q_lens[req], chunk) <= id) {
      first += cpkv::ceil_div(h_q_lens[req], chunk);
      ++req;
    }
    const int64_t off = (id - first) * chunk;
    const int64_t len = h_q_lens[req] - off < chunk ? h_q_lens[req] - off : chunk;
    if (!(k > 0 && id == prev + 1 && id != first)) ++S;
    Q += len;
    prev = id;
  }
  *h_S = S;
  *h_Q = Q;
  return CPKV_OK;
}

extern "C" const char *cpkv_error_string(int code) {
  switch (code) {
    case CPKV_OK: return "CPKV_OK";
    case CPKV_ERR_ARG: return "CPKV_ERR_ARG: invalid argument";
    case CPKV_ERR_UNALIGNED_PREFIX: return "CPKV_ERR_UNALIGNED_PREFIX: prefix length not a multiple of page_size";
    case CPKV_ERR_CAPACITY: return "CPKV_ERR_CAPACITY: capacity too small";
    case CPKV_ERR_LIMIT: return "CPKV_ERR_LIMIT: size beyond this build's limits";
    case CPKV_ERR_CUDA: return "CPKV_ERR_CUDA: kernel launch failed";
    default: return "unknown cpkv error";
  }
}

extern "C" int cpkv_version(void) { return CPKV_VERSION; }
