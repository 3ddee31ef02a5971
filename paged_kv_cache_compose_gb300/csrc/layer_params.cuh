// The parameter block of the one-launch layer compose, shared by the
// per-piece kernel (compose_layer.cu) and the grouped kernel for small pages
// (compose_layer_groups.cu), and the rule that resolves a current page's
// rows.
#pragma once

#include <stdint.h>

#include "common.cuh"

namespace cpkv {

// NP: plane slots (1 for the row layout, which keeps the launch's parameter
// block small).
template <int MAXB, int NP>
struct LayerParams {
  const uint8_t *table[2 * CPKV_MAX_CP];  // pools, then stagings
  int64_t cap_pages[2 * CPKV_MAX_CP];
  const uint8_t *cur_rows[NP][CPKV_MAX_CP];  // plane q of writer w's current rows
  int64_t cur_cap[CPKV_MAX_CP];              // rows of writer w (every plane)
  int64_t plane_off[NP];                     // byte offset of plane q in a page
  int32_t plane_bytes[NP];
  int32_t plane_bulk[NP];                    // plane q is staged with bulk copies
  const int32_t *owner, *src, *token_writer_row;
  uint8_t *dense;
  int32_t *status;
  int64_t dense_cap, page_bytes, units, C;
  int32_t cp, ps, B, pieces, piece_bytes, n_planes;
  int32_t cur_lens[MAXB];
};

// Where a current page's rows come from: n rows starting at row0 of its
// writer's buffer.  Returns 0, or the status bit to raise when the descriptor
// (CPKV_STATUS_DESC_OOB: also a staging slot past the staging's capacity when
// `staged`) or the rows (CPKV_STATUS_ROW_OOB) are out of range; such a page is
// zero-filled in the dense buffer and its staging slot is left untouched.
template <typename Params>
__device__ __forceinline__ int32_t current_rows(const Params &p, const int32_t *cur_page_start, bool staged,
                                                int32_t o, int32_t s, int32_t row0, int64_t *n) {
  const int32_t w = o - p.cp, i = s - 1;
  if (i < 0 || i >= p.C || p.B == 0 || (staged && s >= p.cap_pages[o])) return CPKV_STATUS_DESC_OOB;
  const int b = upper_index<int32_t>(cur_page_start, p.B, i);
  const int32_t kp = i - cur_page_start[b];
  *n = min64(p.ps, (int64_t)p.cur_lens[b] - (int64_t)kp * p.ps);
  if (*n < 1) return CPKV_STATUS_DESC_OOB;
  return row0 >= 0 && row0 + *n <= p.cur_cap[w] ? 0 : CPKV_STATUS_ROW_OOB;
}

// Row-layout pages of at most this many bytes go through the grouped kernel.
constexpr int64_t kLayerGroupMaxPageBytes = 4096;

// Launch compose_layer_groups_kernel for row pages of at most
// kLayerGroupMaxPageBytes (prm as for the per-piece kernel; units, pieces and
// piece_bytes are set here).  CPKV_OK or CPKV_ERR_CUDA.
template <int MAXB>
int launch_layer_groups(LayerParams<MAXB, 1> prm, bool consume, bool early, cudaStream_t s);

}  // namespace cpkv
