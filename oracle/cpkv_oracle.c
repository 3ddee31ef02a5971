/*
 * CPU oracle of the paged-KV compose of a context-parallel prefill.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously correct
 * statement of what the compose computes.  It is used by the tests, by the
 * smoke check and by the benchmark's CPU-baseline leg, never by the product
 * path.  It shares no code, header or constant with the CUDA library.
 *
 * Sources (commit-log pages of an SGLang fork; no code is printed there):
 *   [A] commits d63fbd4 (test/manual), "staging-direct compose" message:
 *       current rows are written into a slot-ordered staging through a
 *       staging-remapped page inverse; ONE slot-dense gather over one
 *       pointer table of 2*cp sources fills every dense page slot; the
 *       descriptor of a current page names its writer's staging (owner
 *       cp + writer) and its slot there (src);
 *       mixed_locs / staging row indices are computed once per batch and the
 *       per-layer fill is a single index copy into the zeroed staging.
 *   [B] same page, "touched-pages staging" message: the staging keeps only the
 *       current pages of one batch, in the order of the merged spans; a
 *       page's slot is its batch current index, the same on every rank.
 *   [D] same page, "symm counting barrier" message: under the page-aligned
 *       in-seq split every current page has exactly one writer rank.
 *   [E] same page, "compose_v2" message: a descriptor owner of -1 zero-fills
 *       its slot (it replaces the dense zero-fill).
 *   [P] commits 0d87bc5 (python), "prefetch staging" message: staging row 0
 *       is reserved, the slot of current page i is i + 1; page id 0 is the
 *       dummy page.
 *   [M] commits 0d87bc5 (python), "owner_check" / "span_owner" messages: the
 *       owner of a logical page is a modulo function of its id.
 *   [S] commits 0d87bc5 (python), "bs=1 spans" message: per-request prefix
 *       and current slot spans are the canonical description of the dense
 *       regions (an empty prefix list means no prefix).
 *   [C] commits d63fbd4, "CPU-gap fixes" message: the ragged index plan holds
 *       a per-q-token topk offset list and int32 segment / kv_lens /
 *       q_starts / q_lens / k_bases / q_bases / current_bases arrays, built
 *       from batch metadata keyed on cp_index.
 *
 * Readings where the pages are silent (all are listed with the design notes):
 *   - logical page lp lives on owner lp % cp at local page lp / cp [M];
 *   - dense layout: request-major, prefix pages then current pages, rows
 *     after the last current token up to the page boundary are zero;
 *   - page_inverse keeps the smallest dense slot of a page that appears in
 *     several prefixes (a shared radix prefix);
 *   - ragged plan: q tokens are cut into `chunk`-token chunks numbered
 *     request-major; a segment is a maximal run of owned chunks of one
 *     request with consecutive ids.
 *
 * Everything is integer indexing and byte copies: results are exact.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_OK 0
#define ORC_BAD_ARG (-1)
#define ORC_UNALIGNED_PREFIX (-2)
#define ORC_CAPACITY (-3)

/* data-dependent violations (same meaning as in the CUDA library's status
 * word, re-stated here so the two share no header) */
#define ORC_PAGE_OOB 1
#define ORC_WRITER_OOB 2
#define ORC_DUP_CURRENT_PAGE 4
#define ORC_CURRENT_IN_PREFIX 8
#define ORC_DESC_OOB 16
#define ORC_ROW_OOB 32
#define ORC_CHUNK_OOB 64

static int64_t ceil_div64(int64_t a, int64_t b) { return (a + b - 1) / b; }

/* Total tokens T, current pages C and dense pages D of a batch. */
int oracle_sizes(int B, int ps, const int32_t *prefix_lens, const int32_t *cur_lens,
                 int64_t *T, int64_t *C, int64_t *D) {
  if (B < 0 || ps <= 0) return ORC_BAD_ARG;
  int64_t t = 0, c = 0, d = 0;
  for (int b = 0; b < B; ++b) {
    if (prefix_lens[b] < 0 || cur_lens[b] < 0) return ORC_BAD_ARG;
    if (prefix_lens[b] % ps != 0) return ORC_UNALIGNED_PREFIX;
    int64_t npp = prefix_lens[b] / ps;
    int64_t ncp = ceil_div64(cur_lens[b], ps);
    t += cur_lens[b];
    c += ncp;
    d += npp + ncp;
  }
  *T = t; *C = c; *D = d;
  return ORC_OK;
}

/*
 * Compose plan [A][B][P][S][M]: spans, gather descriptors, the page inverse,
 * the staging-remapped page inverse and the per-token locations, written as
 * one walk over requests in batch order.
 *
 *   prefix_spans[b] = (dense start, prefix pages)
 *   cur_spans[b]    = (dense start + prefix pages, current pages)
 *   prefix slot:      owner = lp % cp,        src = lp / cp
 *   current page i:   owner = cp + writer[i], src = i + 1
 *   slots >= D:       owner = -1,             src = 0
 *   page_inverse[lp]          = dense slot of lp (smallest), else -1
 *   staging_page_inverse[lp]  = i + 1 for current page i, else 0
 *   mixed_locs[t]   = dense slot of t's page * ps + offset in page
 *   staging_rows[t] = (i + 1) * ps + offset in page
 *   token_writer_row[t] = number of earlier tokens (batch order) whose page
 *                         has the same writer
 */
int oracle_compose_plan(int B, int ps, int cp, int64_t P, const int32_t *prefix_lens,
                        const int32_t *cur_lens, const int32_t *prefix_pages,
                        const int32_t *cur_pages, const int32_t *writer, int64_t dense_cap,
                        int32_t *prefix_spans, int32_t *cur_spans, int32_t *owner,
                        int32_t *src, int32_t *page_inverse, int32_t *staging_page_inverse,
                        int64_t *mixed_locs, int64_t *staging_rows, int32_t *token_writer_row,
                        int32_t *status) {
  if (cp < 1 || cp > 64 || P < 1) return ORC_BAD_ARG;
  int64_t T, C, D;
  int rc = oracle_sizes(B, ps, prefix_lens, cur_lens, &T, &C, &D);
  if (rc) return rc;
  if (dense_cap < D) return ORC_CAPACITY;

  for (int64_t lp = 0; lp < P; ++lp) {
    page_inverse[lp] = -1;
    staging_page_inverse[lp] = 0;
  }
  int64_t *writer_count = (int64_t *)calloc((size_t)cp, sizeof(int64_t));
  int32_t st = 0;

  int64_t dense = 0;    /* next dense slot */
  int64_t pfx_cur = 0;  /* cursor into prefix_pages */
  int64_t cur_page = 0; /* batch current page index i */
  int64_t tok = 0;      /* batch token index t */
  for (int b = 0; b < B; ++b) {
    int64_t npp = prefix_lens[b] / ps;
    int64_t ncp = ceil_div64(cur_lens[b], ps);
    prefix_spans[2 * b] = (int32_t)dense;
    prefix_spans[2 * b + 1] = (int32_t)npp;
    cur_spans[2 * b] = (int32_t)(dense + npp);
    cur_spans[2 * b + 1] = (int32_t)ncp;

    for (int64_t k = 0; k < npp; ++k) {
      int64_t d = dense + k;
      int32_t lp = prefix_pages[pfx_cur + k];
      if (lp < 1 || lp >= P) {
        st |= ORC_PAGE_OOB;
        owner[d] = -1;
        src[d] = 0;
        continue;
      }
      owner[d] = lp % cp;
      src[d] = lp / cp;
      if (page_inverse[lp] == -1) page_inverse[lp] = (int32_t)d;
    }
    for (int64_t k = 0; k < ncp; ++k) {
      int64_t d = dense + npp + k;
      int64_t i = cur_page + k;
      int32_t lp = cur_pages[i];
      int32_t w = writer[i];
      if (lp < 1 || lp >= P) { st |= ORC_PAGE_OOB; owner[d] = -1; src[d] = 0; continue; }
      if (w < 0 || w >= cp) { st |= ORC_WRITER_OOB; owner[d] = -1; src[d] = 0; continue; }
      owner[d] = cp + w;
      src[d] = (int32_t)(i + 1);
      if (staging_page_inverse[lp] != 0) st |= ORC_DUP_CURRENT_PAGE;
      staging_page_inverse[lp] = (int32_t)(i + 1);
      if (page_inverse[lp] == -1) page_inverse[lp] = (int32_t)d;
    }
    for (int64_t k = 0; k < cur_lens[b]; ++k) {
      int64_t t = tok + k;
      int64_t i = cur_page + k / ps;
      int64_t off = k % ps;
      mixed_locs[t] = (dense + npp + k / ps) * ps + off;
      staging_rows[t] = (i + 1) * ps + off;
      int32_t w = writer[i];
      if (w >= 0 && w < cp) token_writer_row[t] = (int32_t)(writer_count[w]++);
      else token_writer_row[t] = -1;
    }
    dense += npp + ncp;
    pfx_cur += npp;
    cur_page += ncp;
    tok += cur_lens[b];
  }
  for (int64_t d = D; d < dense_cap; ++d) { owner[d] = -1; src[d] = 0; }

  /* a current page must not also be a prefix page (single writer [D]) */
  pfx_cur = 0;
  for (int b = 0; b < B; ++b) {
    int64_t npp = prefix_lens[b] / ps;
    for (int64_t k = 0; k < npp; ++k) {
      int32_t lp = prefix_pages[pfx_cur + k];
      if (lp >= 1 && lp < P && staging_page_inverse[lp] != 0) st |= ORC_CURRENT_IN_PREFIX;
    }
    pfx_cur += npp;
  }
  free(writer_count);
  *status |= st;
  return ORC_OK;
}

/*
 * The plain definition of the composed dense KV [A][S]: for every request in
 * batch order, its prefix rows read from the pool through its logical page
 * table, then its current rows, then zero rows up to the next page boundary;
 * dense pages past the batch (up to dense_cap) are zero.  No descriptor,
 * inverse or staging is involved.
 *
 * pool_slabs[r] is owner r's slab [slab_pages][ps][R]; cur_rows is [T][R] in
 * batch order; dense_out is [dense_cap * ps][R].
 */
int oracle_compose_dense(int B, int ps, int cp, int64_t R, int64_t slab_pages,
                         const int32_t *prefix_lens, const int32_t *cur_lens,
                         const int32_t *prefix_pages, const uint8_t *const *pool_slabs,
                         const uint8_t *cur_rows, int64_t dense_cap, uint8_t *dense_out) {
  int64_t T, C, D;
  int rc = oracle_sizes(B, ps, prefix_lens, cur_lens, &T, &C, &D);
  if (rc) return rc;
  if (dense_cap < D) return ORC_CAPACITY;
  int64_t row = 0;     /* dense row being written */
  int64_t pfx_cur = 0; /* cursor into prefix_pages */
  int64_t tok = 0;     /* batch token index */
  for (int b = 0; b < B; ++b) {
    for (int64_t k = 0; k < prefix_lens[b]; ++k) {
      int64_t lp = prefix_pages[pfx_cur + k / ps];
      int64_t off = k % ps;
      int64_t owner = lp % cp, local = lp / cp;
      if (lp < 1 || local >= slab_pages) return ORC_BAD_ARG;
      memcpy(dense_out + row * R, pool_slabs[owner] + (local * ps + off) * R, (size_t)R);
      ++row;
    }
    for (int64_t k = 0; k < cur_lens[b]; ++k) {
      memcpy(dense_out + row * R, cur_rows + (tok + k) * R, (size_t)R);
      ++row;
    }
    while (row % ps != 0) {
      memset(dense_out + row * R, 0, (size_t)R);
      ++row;
    }
    pfx_cur += prefix_lens[b] / ps;
    tok += cur_lens[b];
  }
  for (; row < dense_cap * ps; ++row) memset(dense_out + row * R, 0, (size_t)R);
  return ORC_OK;
}

/*
 * The staging content defined by [A][B][P]: in writer w's staging, page
 * i + 1 holds the rows of current page i when writer[i] == w, followed by zero
 * rows.  Pages of other writers and page 0 are not defined; this routine
 * leaves them untouched.  staging[w] is [staging_cap_pages * ps][R].
 */
int oracle_staging(int B, int ps, int cp, int64_t R, const int32_t *cur_lens,
                   const int32_t *writer, const uint8_t *cur_rows, uint8_t *const *staging,
                   int64_t staging_cap_pages) {
  int64_t i = 0, tok = 0;
  for (int b = 0; b < B; ++b) {
    for (int64_t k0 = 0; k0 < cur_lens[b]; k0 += ps) {
      int64_t n = cur_lens[b] - k0 < ps ? cur_lens[b] - k0 : ps;
      int32_t w = writer[i];
      if (w < 0 || w >= cp || i + 1 >= staging_cap_pages) return ORC_BAD_ARG;
      uint8_t *page = staging[w] + (i + 1) * ps * R;
      for (int64_t r = 0; r < ps; ++r) {
        if (r < n) memcpy(page + r * R, cur_rows + (tok + k0 + r) * R, (size_t)R);
        else memset(page + r * R, 0, (size_t)R);
      }
      ++i;
    }
    tok += cur_lens[b];
  }
  return ORC_OK;
}

/*
 * The fill as the index copy of [A], for any row indices: for every token t,
 * with w = writer[staging_rows[t] / ps - 1],
 *     staging[w] row staging_rows[t] <- cur_rows[w] row token_writer_row[t]
 * in token order, then for every request whose current length is not a
 * multiple of ps, the rows after its last token's staging row up to the end
 * of that staging page are set to zero.  A row index outside its buffer or a
 * writer outside [0, cp) skips that token and raises ORC_ROW_OOB /
 * ORC_WRITER_OOB.  cur_rows[w] is [cur_cap[w]][R]; staging[w] is
 * [staging_cap_pages * ps][R].
 */
int oracle_fill_index_copy(int B, int ps, int cp, int64_t R, const int32_t *cur_lens,
                           const int64_t *staging_rows, const int32_t *token_writer_row,
                           const int32_t *writer, int64_t C, const uint8_t *const *cur_rows,
                           const int64_t *cur_cap, uint8_t *const *staging, int64_t staging_cap_pages,
                           int32_t *status) {
  int64_t T = 0;
  for (int b = 0; b < B; ++b) T += cur_lens[b];
  for (int64_t t = 0; t < T; ++t) {
    int64_t sr = staging_rows[t];
    int64_t slot = sr / ps;
    if (sr < ps || sr >= staging_cap_pages * ps || slot > C) { *status |= ORC_ROW_OOB; continue; }
    int32_t w = writer[slot - 1];
    if (w < 0 || w >= cp) { *status |= ORC_WRITER_OOB; continue; }
    int32_t r = token_writer_row[t];
    if (r < 0 || r >= cur_cap[w]) { *status |= ORC_ROW_OOB; continue; }
    memcpy(staging[w] + sr * R, cur_rows[w] + (int64_t)r * R, (size_t)R);
  }
  int64_t last = -1;
  for (int b = 0; b < B; ++b) {
    last += cur_lens[b];
    if (cur_lens[b] % ps == 0) continue;
    int64_t sr = staging_rows[last];
    int64_t slot = sr / ps;
    if (sr < ps || sr >= staging_cap_pages * ps || slot > C) { *status |= ORC_ROW_OOB; continue; }
    int32_t w = writer[slot - 1];
    if (w < 0 || w >= cp) { *status |= ORC_WRITER_OOB; continue; }
    for (int64_t row = sr + 1; row < (slot + 1) * ps; ++row) memset(staging[w] + row * R, 0, (size_t)R);
  }
  return ORC_OK;
}

/*
 * Planar pages (the index kind of [P]: its own fill kernel, pointed at the
 * staging page inverse).  Reading taken here: a page of ps tokens stores
 * n_planes planes one after the other; plane p holds the ps tokens' w_p-byte
 * slices in token order, so token `off` of the page has its plane-p slice at
 * byte  ps * (w_0 + ... + w_{p-1}) + off * w_p  of the page, and a page is
 * ps * (w_0 + ... + w_{n-1}) bytes.  One plane of width R is the row layout.
 *
 * The fill as an index copy over planes: for every token t, with
 * sr = staging_rows[t], slot = sr / ps, off = sr % ps and
 * w = writer[slot - 1], plane p of staging[w] page `slot` row `off` <-
 * cur_planes[p * cp + w] row token_writer_row[t] (w_p bytes); then for every
 * request whose current length is not a multiple of ps, the slices of the
 * rows after its last token up to the end of that page are zero in every
 * plane.  Violations skip the token and raise ORC_ROW_OOB / ORC_WRITER_OOB.
 */
int oracle_fill_planes(int B, int ps, int cp, int n_planes, const int32_t *plane_bytes,
                       const int32_t *cur_lens, const int64_t *staging_rows,
                       const int32_t *token_writer_row, const int32_t *writer, int64_t C,
                       const uint8_t *const *cur_planes, const int64_t *cur_cap,
                       uint8_t *const *staging, int64_t staging_cap_pages, int32_t *status) {
  int64_t page_bytes = 0;
  for (int p = 0; p < n_planes; ++p) page_bytes += (int64_t)ps * plane_bytes[p];
  int64_t T = 0;
  for (int b = 0; b < B; ++b) T += cur_lens[b];
  for (int64_t t = 0; t < T; ++t) {
    int64_t sr = staging_rows[t];
    int64_t slot = sr / ps, off = sr % ps;
    if (sr < ps || sr >= staging_cap_pages * ps || slot > C) { *status |= ORC_ROW_OOB; continue; }
    int32_t w = writer[slot - 1];
    if (w < 0 || w >= cp) { *status |= ORC_WRITER_OOB; continue; }
    int32_t r = token_writer_row[t];
    if (r < 0 || r >= cur_cap[w]) { *status |= ORC_ROW_OOB; continue; }
    int64_t plane_start = 0;
    for (int p = 0; p < n_planes; ++p) {
      int64_t wp = plane_bytes[p];
      memcpy(staging[w] + slot * page_bytes + plane_start + off * wp, cur_planes[p * cp + w] + r * wp,
             (size_t)wp);
      plane_start += ps * wp;
    }
  }
  int64_t last = -1;
  for (int b = 0; b < B; ++b) {
    last += cur_lens[b];
    if (cur_lens[b] % ps == 0) continue;
    int64_t sr = staging_rows[last];
    int64_t slot = sr / ps;
    if (sr < ps || sr >= staging_cap_pages * ps || slot > C) { *status |= ORC_ROW_OOB; continue; }
    int32_t w = writer[slot - 1];
    if (w < 0 || w >= cp) { *status |= ORC_WRITER_OOB; continue; }
    int64_t plane_start = 0;
    for (int p = 0; p < n_planes; ++p) {
      int64_t wp = plane_bytes[p];
      for (int64_t off = sr % ps + 1; off < ps; ++off)
        memset(staging[w] + slot * page_bytes + plane_start + off * wp, 0, (size_t)wp);
      plane_start += ps * wp;
    }
  }
  return ORC_OK;
}

/*
 * The plain definition of the composed dense KV for planar pages: request by
 * request, its prefix tokens' slices copied from their pool pages, then its
 * current tokens' slices from the batch-ordered current planes
 * (cur_planes[p] is [T][w_p]), then zero slices up to the page boundary;
 * pages past the batch are zero.  Pool slab r is [slab_pages][page_bytes].
 */
int oracle_compose_dense_planes(int B, int ps, int cp, int n_planes, const int32_t *plane_bytes,
                                int64_t slab_pages, const int32_t *prefix_lens, const int32_t *cur_lens,
                                const int32_t *prefix_pages, const uint8_t *const *pool_slabs,
                                const uint8_t *const *cur_planes, int64_t dense_cap, uint8_t *dense_out) {
  int64_t T, C, D;
  int rc = oracle_sizes(B, ps, prefix_lens, cur_lens, &T, &C, &D);
  if (rc) return rc;
  if (dense_cap < D) return ORC_CAPACITY;
  int64_t page_bytes = 0;
  for (int p = 0; p < n_planes; ++p) page_bytes += (int64_t)ps * plane_bytes[p];
  int64_t row = 0, pfx_cur = 0, tok = 0;  /* row = dense token position */
  for (int b = 0; b < B; ++b) {
    int64_t n_tok = prefix_lens[b] + cur_lens[b];
    int64_t padded = ((n_tok + ps - 1) / ps) * ps;
    for (int64_t k = 0; k < padded; ++k) {
      int64_t page = (row + k) / ps, off = (row + k) % ps;
      int64_t plane_start = 0;
      for (int p = 0; p < n_planes; ++p) {
        int64_t wp = plane_bytes[p];
        uint8_t *dst = dense_out + page * page_bytes + plane_start + off * wp;
        if (k < prefix_lens[b]) {
          int64_t lp = prefix_pages[pfx_cur + k / ps];
          int64_t owner = lp % cp, local = lp / cp;
          if (lp < 1 || local >= slab_pages) return ORC_BAD_ARG;
          memcpy(dst, pool_slabs[owner] + local * page_bytes + plane_start + (k % ps) * wp, (size_t)wp);
        } else if (k < n_tok) {
          memcpy(dst, cur_planes[p] + (tok + k - prefix_lens[b]) * wp, (size_t)wp);
        } else {
          memset(dst, 0, (size_t)wp);
        }
        plane_start += ps * wp;
      }
    }
    row += padded;
    pfx_cur += prefix_lens[b] / ps;
    tok += cur_lens[b];
  }
  if (row < dense_cap * ps) memset(dense_out + (row / ps) * page_bytes, 0, (size_t)((dense_cap - row / ps) * page_bytes));
  return ORC_OK;
}

/*
 * Slot-dense page gather [A][E], descriptor by descriptor: dense page d is a
 * copy of page src[d] of table[owner[d]], or zeros when owner[d] == -1.  A
 * descriptor outside the table or the source's capacity is a violation: the
 * slot is zero-filled and ORC_DESC_OOB is raised.
 */
int oracle_gather(int ps, int n_table, int64_t R, const uint8_t *const *table,
                  const int64_t *cap_pages, const int32_t *owner, const int32_t *src,
                  int64_t dense_cap, uint8_t *dense_out, int32_t *status) {
  int64_t page_bytes = ps * R;
  for (int64_t d = 0; d < dense_cap; ++d) {
    uint8_t *dst = dense_out + d * page_bytes;
    int32_t o = owner[d];
    if (o == -1) { memset(dst, 0, (size_t)page_bytes); continue; }
    if (o < -1 || o >= n_table || src[d] < 0 || src[d] >= cap_pages[o]) {
      *status |= ORC_DESC_OOB;
      memset(dst, 0, (size_t)page_bytes);
      continue;
    }
    memcpy(dst, table[o] + (int64_t)src[d] * page_bytes, (size_t)page_bytes);
  }
  return ORC_OK;
}

/*
 * Ragged index plan [C].  Request b's q tokens are cut into ceil(q_b/chunk)
 * chunks; chunk ids run request-major over the batch.  cp_index lists the
 * chunk ids this rank owns, ascending.  Walking cp_index in order, a chunk
 * opens a new segment unless it is the next chunk (id + 1) of the same
 * request as the previous owned chunk.  Per segment s of request b:
 *   seg_req[s]       = b
 *   q_starts[s]      = token offset of the segment inside request b's q
 *   q_lens[s]        = tokens in the segment
 *   kv_lens[s]       = prefix_b + q_starts[s] + q_lens[s]
 *   k_bases[s]       = sum over b' < b of align_up(prefix_b' + q_b', k_align)
 *   current_bases[s] = k_bases[s] + prefix_b
 *   q_bases[s]       = tokens of this rank in earlier segments
 * and topk_offsets[j] = k_bases of the segment holding this rank's j-th q
 * token.  Returns S and Q_r through out_S / out_Qr.
 */
int oracle_ragged_plan(int B, int chunk, int k_align, const int32_t *prefix_lens,
                       const int32_t *q_lens, const int32_t *cp_index, int64_t n_owned,
                       int32_t *topk_offsets, int32_t *seg_req, int32_t *kv_lens,
                       int32_t *q_starts, int32_t *q_lens_out, int32_t *k_bases,
                       int32_t *q_bases, int32_t *current_bases, int64_t *out_S,
                       int64_t *out_Qr, int32_t *status) {
  if (B < 0 || chunk <= 0 || k_align <= 0) return ORC_BAD_ARG;
  int64_t *chunk_start = (int64_t *)malloc(sizeof(int64_t) * (size_t)(B + 1));
  int64_t *kbase = (int64_t *)malloc(sizeof(int64_t) * (size_t)(B + 1));
  chunk_start[0] = 0;
  kbase[0] = 0;
  for (int b = 0; b < B; ++b) {
    chunk_start[b + 1] = chunk_start[b] + ceil_div64(q_lens[b], chunk);
    int64_t kv = (int64_t)prefix_lens[b] + q_lens[b];
    kbase[b + 1] = kbase[b] + ceil_div64(kv, k_align) * k_align;
  }
  int64_t total_chunks = chunk_start[B];
  int64_t S = 0, Q = 0;
  int64_t prev_id = -2;
  int prev_req = -1;
  for (int64_t k = 0; k < n_owned; ++k) {
    int64_t id = cp_index[k];
    if (id < 0 || id >= total_chunks || id <= prev_id) { *status |= ORC_CHUNK_OOB; break; }
    int b = 0;
    while (chunk_start[b + 1] <= id) ++b; /* request holding chunk id */
    int64_t off = (id - chunk_start[b]) * chunk;
    int64_t len = q_lens[b] - off < chunk ? q_lens[b] - off : chunk;
    if (!(b == prev_req && id == prev_id + 1)) {
      seg_req[S] = b;
      q_starts[S] = (int32_t)off;
      q_lens_out[S] = 0;
      k_bases[S] = (int32_t)kbase[b];
      current_bases[S] = (int32_t)(kbase[b] + prefix_lens[b]);
      q_bases[S] = (int32_t)Q;
      ++S;
    }
    q_lens_out[S - 1] += (int32_t)len;
    kv_lens[S - 1] = prefix_lens[b] + q_starts[S - 1] + q_lens_out[S - 1];
    for (int64_t j = 0; j < len; ++j) topk_offsets[Q + j] = (int32_t)kbase[b];
    Q += len;
    prev_id = id;
    prev_req = b;
  }
  *out_S = S;
  *out_Qr = Q;
  free(chunk_start);
  free(kbase);
  return ORC_OK;
}
