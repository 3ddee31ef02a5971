// Host-only entry points of the cpkv library: batch sizing, writer token
// counts, ragged-plan sizing, error strings, device queries.  No GPU work.
#include <stdint.h>

#include <mutex>
#include <vector>

#include "common.cuh"

namespace cpkv {
namespace {

std::mutex g_query_mu;  // guards the device-query caches below

struct KernelQuery {
  int dev;
  const void *kernel;
  size_t smem;
  int threads;
  int value;
};
std::vector<KernelQuery> g_smem_limits;  // value: the limit set
std::vector<KernelQuery> g_resident;     // value: resident CTAs per SM
int g_sm_count[256] = {0};

int current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    (void)cudaGetLastError();
    return -1;
  }
  return dev;
}

}  // namespace

int device_sm_count() {
  const int dev = current_device();
  if (dev < 0 || dev >= 256) return 1;
  std::lock_guard<std::mutex> lock(g_query_mu);
  if (g_sm_count[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
      (void)cudaGetLastError();
      return 1;
    }
    g_sm_count[dev] = n;
  }
  return g_sm_count[dev];
}

int ensure_dynamic_smem(const void *kernel, int bytes) {
  const int dev = current_device();
  if (dev < 0) return CPKV_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_query_mu);
  for (const KernelQuery &q : g_smem_limits)
    if (q.dev == dev && q.kernel == kernel && q.value >= bytes) return CPKV_OK;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess) {
    (void)cudaGetLastError();
    return CPKV_ERR_CUDA;
  }
  g_smem_limits.push_back(KernelQuery{dev, kernel, 0, 0, bytes});
  return CPKV_OK;
}

int persistent_grid(const void *kernel, int threads, size_t smem, int cap_per_sm, int64_t units) {
  const int sms = device_sm_count();
  const int dev = current_device();
  int per_sm = 0;
  {
    std::lock_guard<std::mutex> lock(g_query_mu);
    for (const KernelQuery &q : g_resident)
      if (q.dev == dev && q.kernel == kernel && q.smem == smem && q.threads == threads) per_sm = q.value;
    if (per_sm == 0) {
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem) != cudaSuccess ||
          per_sm < 1) {
        (void)cudaGetLastError();
        per_sm = 1;
      }
      g_resident.push_back(KernelQuery{dev, kernel, smem, threads, per_sm});
    }
  }
  if (per_sm > cap_per_sm) per_sm = cap_per_sm;
  const int64_t grid = (int64_t)sms * per_sm;
  return (int)(units < grid ? (units > 0 ? units : 1) : grid);
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
