/*
 * cpkv — paged-KV compose of a context-parallel LLM prefill, for one GB300.
 *
 * Plain C ABI.  Every pointer argument is either a HOST pointer (prefix h_)
 * or a DEVICE pointer (prefix d_) of the current CUDA device.  The caller
 * owns all memory; the library allocates nothing, never synchronises the
 * stream and never traps.  All GPU work is enqueued on `stream` and is
 * asynchronous.  Lengths that size outputs are read from host arrays, so no
 * call needs a device-to-host copy.
 *
 * Error handling (two channels):
 *   - the return value: CPKV_OK, or a negative CPKV_ERR_* code for bad
 *     arguments detected on the host before anything is launched (nothing is
 *     written then), or CPKV_ERR_CUDA when a launch fails;
 *   - `d_status`: a caller-owned int32 in device memory.  Kernels OR
 *     CPKV_STATUS_* bits into it when they meet data that violates the
 *     contract (a page id out of range, a duplicate current page, ...).  The
 *     offending element is skipped or zero-filled as each call documents; all
 *     other outputs are still produced.  The library never clears it: zero it
 *     before a batch and read it whenever the caller synchronises anyway.
 *
 * Source of the method (commit-log pages of an SGLang fork):
 *   "staging-direct compose" message of commits d63fbd4 (test/manual):
 *     current rows are written straight into a slot-ordered staging through
 *     a per-batch staging-remapped page inverse; one slot-dense page gather
 *     over a concatenated 2*cp source-pointer table fills every dense page;
 *     mixed_locs / staging rows are layer-invariant and computed once per
 *     batch; the per-layer fill is a single index copy.
 *   "touched-pages staging" message (same page): a page's staging slot is
 *     its index among the batch's current pages; staging is sized by current pages only.
 *   "prefetch staging" message of commits 0d87bc5 (python): staging row 0 is
 *     reserved, current page i sits at slot i + 1; page id 0 is the dummy.
 *   "compose_v2" message (commits d63fbd4): an owner of -1 zero-fills.
 *   "CPU-gap fixes" message (commits d63fbd4): the per-batch ragged index
 *     plan of the NSA indexer.
 *
 * Notation: B requests, ps = page_size, cp = cp_size, R = row bytes,
 * npp_b = prefix_len_b / ps, ncp_b = ceil(cur_len_b / ps), T = sum cur_len,
 * C = sum ncp, D = sum (npp + ncp).  Logical page lp of the pool lives on
 * owner lp % cp at local page lp / cp (modulo-owner placement); page 0 is the
 * dummy page and is never a valid page id.
 */
#ifndef CPKV_H_
#define CPKV_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define CPKV_VERSION 1
#define CPKV_MAX_CP 64       /* largest cp_size (2*cp source pointers)      */
#define CPKV_MAX_BATCH 1024  /* largest B (host lengths travel as kernel parameters) */

/* A cudaStream_t, passed as an opaque handle (0 = the legacy default stream). */
typedef void *cpkv_stream_t;

/* Return codes. */
#define CPKV_OK 0
#define CPKV_ERR_ARG (-1)              /* null/misaligned pointer, bad size or count   */
#define CPKV_ERR_UNALIGNED_PREFIX (-2) /* a prefix length is not a multiple of ps      */
#define CPKV_ERR_CAPACITY (-3)         /* an output or staging capacity is too small   */
#define CPKV_ERR_LIMIT (-4)            /* B, cp or a size exceeds what this build takes */
#define CPKV_ERR_CUDA (-5)             /* a kernel launch failed                        */

/* Device status bits (ORed into *d_status). */
#define CPKV_STATUS_PAGE_OOB 1            /* page id outside [1, num_pool_pages)         */
#define CPKV_STATUS_WRITER_OOB 2          /* writer rank outside [0, cp)                 */
#define CPKV_STATUS_DUP_CURRENT_PAGE 4    /* a current page id appears twice             */
#define CPKV_STATUS_CURRENT_IN_PREFIX 8   /* a current page id is also a prefix page     */
#define CPKV_STATUS_DESC_OOB 16           /* gather descriptor outside table/capacity    */
#define CPKV_STATUS_ROW_OOB 32            /* fill row index outside its buffer           */
#define CPKV_STATUS_CHUNK_OOB 64          /* cp_index not ascending or out of range      */
#define CPKV_STATUS_OUT_CAPACITY 128      /* a device-sized output exceeded its capacity */
#define CPKV_STATUS_TIMEOUT 256           /* a bounded wait gave up (should never occur) */

/* Sizes of a batch, derived from host lengths. */
typedef struct {
  int64_t T; /* current tokens */
  int64_t C; /* current pages  */
  int64_t D; /* dense pages (prefix + current) */
} cpkv_sizes;

/*
 * cpkv_plan_sizes — T, C and D of a batch (host only, no GPU work).
 * h_prefix_lens, h_cur_lens: host int32 [B], non-negative; prefix lengths
 * must be multiples of page_size (the chunked-prefill message of commits
 * 0d87bc5 keeps unaligned prefixes out of multi-request batches because the
 * page-aligned CP split rejects them).
 * Returns CPKV_ERR_UNALIGNED_PREFIX for an unaligned prefix, CPKV_ERR_ARG for
 * B < 0, page_size <= 0, a negative length or a null pointer (B > 0),
 * CPKV_ERR_LIMIT when T, C or D would not fit int32 indices.
 */
int cpkv_plan_sizes(int B, int page_size, const int32_t *h_prefix_lens, const int32_t *h_cur_lens,
                    cpkv_sizes *out);

/*
 * cpkv_writer_token_counts — tokens each writer rank computes (host only).
 * h_writer: host int32 [C], writer rank of each current page in batch order.
 * h_tokens_per_writer: host int64 [cp_size], written.  Sizes the per-writer
 * current-row buffers passed to cpkv_fill_current.  A writer outside [0, cp)
 * returns CPKV_ERR_ARG.
 */
int cpkv_writer_token_counts(int B, int page_size, int cp_size, const int32_t *h_cur_lens,
                             const int32_t *h_writer, int64_t C, int64_t *h_tokens_per_writer);

/*
 * cpkv_plan_build — the per-batch compose plan, built on the device.
 * ("staging-direct compose": spans, descriptors, the page inverse, the
 * staging-remapped page inverse and mixed_locs / staging row indices are
 * layer-invariant and built once per batch.)
 *
 * Inputs:
 *   h_prefix_lens, h_cur_lens  host int32 [B] (B <= CPKV_MAX_BATCH)
 *   d_prefix_pages  device int32 [sum npp], CSR by request: the logical pages
 *                   of request b's prefix, in token order
 *   d_cur_pages     device int32 [C], CSR by request: the logical pages that
 *                   hold request b's current tokens
 *   d_writer        device int32 [C]: writer rank of each current page
 *   num_pool_pages  P: valid page ids are [1, P)
 *   dense_cap_pages capacity of the dense buffer in pages, >= D
 * Outputs (device, caller-allocated, fully written):
 *   d_prefix_spans  int32 [B][2]  (dense start, npp_b)
 *   d_cur_spans     int32 [B][2]  (dense start + npp_b, ncp_b)
 *   d_owner, d_src  int32 [dense_cap_pages] gather descriptors:
 *                     prefix slot of lp:  owner = lp % cp,   src = lp / cp
 *                     current page i:     owner = cp + w_i,  src = i + 1
 *                     slots >= D:         owner = -1,        src = 0
 *   d_page_inverse         int32 [P]: dense slot of lp (smallest if lp is in
 *                          several prefixes), -1 if lp is not in the batch
 *   d_staging_page_inverse int32 [P]: i + 1 if lp is current page i, else 0
 *   d_mixed_locs     int64 [T]: dense row of each current token
 *   d_staging_rows   int64 [T]: staging row (i + 1) * ps + offset
 *   d_token_writer_row int32 [T]: row of the token in its writer's
 *                    current-row buffer (batch order within each writer)
 * Workspace (device, caller-allocated, at least the bytes that
 * cpkv_plan_workspace_bytes gives, 4-byte aligned; may be NULL when that is
 * 0): the per-writer row totals of each block of current pages, written by
 * the call's first kernel and read by its second.  Its contents between
 * calls are irrelevant (every entry read is written first in the same call),
 * and two calls whose kernels overlap on the GPU must not share one.
 * Status bits: PAGE_OOB / WRITER_OOB (the slot gets owner -1), DUP_CURRENT_PAGE,
 * CURRENT_IN_PREFIX.
 * Errors: ARG (bad sizes, null or unaligned pointers), UNALIGNED_PREFIX,
 * CAPACITY (dense_cap_pages < D, workspace_bytes too small), LIMIT, CUDA.
 */
int cpkv_plan_build(int B, int page_size, int cp_size, int64_t num_pool_pages,
                    const int32_t *h_prefix_lens, const int32_t *h_cur_lens,
                    const int32_t *d_prefix_pages, const int32_t *d_cur_pages, const int32_t *d_writer,
                    int64_t dense_cap_pages, int32_t *d_prefix_spans, int32_t *d_cur_spans,
                    int32_t *d_owner, int32_t *d_src, int32_t *d_page_inverse,
                    int32_t *d_staging_page_inverse, int64_t *d_mixed_locs, int64_t *d_staging_rows,
                    int32_t *d_token_writer_row, void *d_workspace, int64_t workspace_bytes, int32_t *d_status,
                    cpkv_stream_t stream);

/*
 * cpkv_plan_workspace_bytes — device workspace that cpkv_plan_build needs for
 * a batch (host only): 4 * cp_size bytes per block of current pages, a block
 * being about 2048 current tokens (32 to 1024 pages; so a few KB for batches
 * of a few hundred thousand tokens).  0 when the batch has no current page.
 * Errors: ARG (B < 0, page_size <= 0, cp_size outside [1, CPKV_MAX_CP], a
 * negative length, a null pointer), LIMIT (B > CPKV_MAX_BATCH, too many
 * current pages for int32 indices).
 */
int cpkv_plan_workspace_bytes(int B, int page_size, int cp_size, const int32_t *h_cur_lens, int64_t *h_bytes);

/*
 * cpkv_plan_build_noalloc — cpkv_plan_build for callers that cannot allocate
 * device memory, not even the small workspace: a plugin inside a framework
 * whose caching allocator owns all device memory (a raw cudaMalloc would
 * bypass it, and cudaMalloc / cudaFree synchronise the device), or a server
 * that reserved nearly all of HBM for its KV cache pool up front.  The pages
 * have no counterpart of this call; it exists for such callers only.
 *
 * Same arguments, outputs, status bits and errors as cpkv_plan_build, minus
 * the workspace: the call uses a fixed 64 KiB array in device memory that the
 * library holds on every GPU it is loaded on until the process exits, and
 * allocates nothing.  The caller still passes every input and output.
 *   - Limit: batches whose cpkv_plan_workspace_bytes exceeds 65536 bytes
 *     (more than 16384 / cp_size blocks of current pages, e.g. about 4M
 *     current tokens at cp_size 8) return CPKV_ERR_LIMIT, nothing launched.
 *   - Set-up: the first call on a device, with that device current, looks up
 *     the array's device address (cudaGetSymbolAddress) and keeps it; make
 *     that first call before any stream capture on the device.  A failed
 *     look-up returns CPKV_ERR_CUDA.
 *   - Sharing: all calls on a device use the one array, which keeps the last
 *     call's contents (no entry needs clearing: a call reads only what it
 *     wrote).  Calls whose kernels overlap on the GPU race on it; order them
 *     on one stream or with events.
 */
int cpkv_plan_build_noalloc(int B, int page_size, int cp_size, int64_t num_pool_pages,
                            const int32_t *h_prefix_lens, const int32_t *h_cur_lens,
                            const int32_t *d_prefix_pages, const int32_t *d_cur_pages, const int32_t *d_writer,
                            int64_t dense_cap_pages, int32_t *d_prefix_spans, int32_t *d_cur_spans,
                            int32_t *d_owner, int32_t *d_src, int32_t *d_page_inverse,
                            int32_t *d_staging_page_inverse, int64_t *d_mixed_locs, int64_t *d_staging_rows,
                            int32_t *d_token_writer_row, int32_t *d_status, cpkv_stream_t stream);

/* Flags of cpkv_fill_current(_planes), cpkv_compose_layer(_planes) and
 * cpkv_compose_fused(_planes). */
/* The stagings are consumed, as with CPKV_GATHER_CONSUME_STAGING (layer
 * compose only): each staged piece's L2 lines are dropped once it has been
 * read back, and the staging bytes are undefined after the call. */
#define CPKV_FLAG_CONSUME_STAGING 1
/* Early inputs: the caller promises that nothing the call reads (the plan
 * arrays, the pools, the current rows) or raises bits in (the status word) is
 * written by the kernel launched just before it on the stream, and that
 * every other writer of those inputs had
 * finished before that kernel started or is joined to this call by an event
 * wait on the stream after that kernel (an event wait stays a full
 * dependency; in a CUDA graph it is a full edge).  The call is then launched
 * as a programmatic dependent of the previous kernel: its CTAs may start
 * while that kernel still runs (in SM slots it leaves free or its tail frees)
 * and read inputs at once, and each thread waits for that kernel to complete
 * (griddepcontrol.wait) before its first global store, so every write stays
 * ordered after it.  In a per-layer loop whose inputs were produced before
 * the loop this holds; directly after the kernel that writes the current
 * rows or the plan it does not.  The fused and layer composes take the early
 * launch when their grid runs at most 4 CTAs per SM (pages of several
 * pieces, 8448-byte index-key pages) and for row pages of at most 4 KB, which
 * go in groups of consecutive dense pages at 6 or 8 CTAs per SM; other grids
 * of more CTAs per SM launch plainly, where the early launch measured
 * slower.  Chains of early launches stay
 * ordered: every early-launched kernel of this library has at least one
 * thread pass that wait before it can finish, so it completes only after its
 * predecessor, and no store runs ahead of a kernel two launches back. */
#define CPKV_FLAG_EARLY_INPUTS 2
/* Page runs (cpkv_fill_current, cpkv_fill_current_planes): the caller promises that the index
 * arrays are those of cpkv_plan_build for this batch, so that current page i
 * (n_i tokens, batch order) is staged at rows (i + 1) * ps .. (i + 1) * ps +
 * n_i - 1 of its writer's staging and read from n_i consecutive rows of that
 * writer's buffer, starting at d_token_writer_row of the page's first token.
 * The fill then moves each page as one run in 4 KB chunks (one index lookup
 * per page instead of per row) and zeroes the pad rows of short pages in the
 * same pass; the stagings end up byte-identical.  Each page's first staging
 * row and its first and last source rows are checked against the run: a
 * page that does not fit raises ROW_OOB and is not written (other
 * violations inside the run are not detected).  Pages under 4 KB take the
 * row fill, which needs no promise.  For planar pages each plane of a page
 * is a run (n_i consecutive slices of the writer's plane rows into the page's
 * plane), moved in chunks of up to 4 KB with 16-byte vectors where source,
 * destination and sizes allow, else 4-byte words. */
#define CPKV_FILL_PAGE_RUNS 4

/*
 * cpkv_fill_current — per layer: write every current row into its writer's
 * staging.  In the "staging-direct compose" message this is one index copy
 * per layer with layer-invariant row indices; rows are opaque bytes, so fp8
 * needs nothing special ("fp8 -> uint8" message of commits 0d87bc5).
 *
 * For every token t with writer w = d_writer[d_staging_rows[t] / ps - 1]:
 *   staging[w] row d_staging_rows[t]  <-  cur_rows[w] row d_token_writer_row[t]
 * and for every request b whose current length is not a multiple of ps, the
 * rows after its last token up to the end of that staging page are zeroed.
 * No other staging row is written (page 0 and other writers' pages keep their
 * bytes).
 *
 *   h_cur_lens        host int32 [B]
 *   h_cur_rows        host array [cp] of device pointers: writer w's current
 *                     rows, [h_cur_rows_cap[w]][R] bytes, 16-byte aligned
 *   h_staging         host array [cp] of device pointers: writer w's staging,
 *                     [staging_cap_pages * ps][R] bytes, 16-byte aligned;
 *                     staging_cap_pages >= C + 1
 *   d_staging_rows, d_token_writer_row: from cpkv_plan_build; d_writer [C]
 *   row_bytes         R, a multiple of 16
 *   flags             CPKV_FLAG_EARLY_INPUTS, CPKV_FILL_PAGE_RUNS (or 0);
 *                     other bits return CPKV_ERR_ARG
 * Status bits: ROW_OOB / WRITER_OOB (that row is skipped).
 */
int cpkv_fill_current(int B, int page_size, int cp_size, int64_t row_bytes, const int32_t *h_cur_lens,
                      const void *const *h_cur_rows, const int64_t *h_cur_rows_cap,
                      void *const *h_staging, int64_t staging_cap_pages,
                      const int64_t *d_staging_rows, const int32_t *d_token_writer_row,
                      const int32_t *d_writer, int64_t num_cur_pages, int flags, int32_t *d_status,
                      cpkv_stream_t stream);

/*
 * cpkv_fill_current_planes — per layer: the fill for planar pages (the
 * NSA indexer's "index" kind, whose fill the pages keep separate from the
 * token-KV index copy and point at the staging page inverse; "prefetch
 * staging" message of commits 0d87bc5).  A planar page of ps tokens stores
 * n_planes planes one after the other; plane p holds the ps tokens'
 * h_plane_bytes[p]-byte slices in token order (reading: the indexer keys are
 * a 128-byte fp8 key plane followed by a 4-byte fp32 scale plane, a page of
 * 64 * 132 = 8448 bytes).  One plane of width R is the row layout.
 *
 * For every token t, with sr = d_staging_rows[t], slot = sr / ps,
 * off = sr % ps, w = d_writer[slot - 1]:
 *   plane p of staging[w] page slot, token off  <-  row d_token_writer_row[t]
 *   of h_cur_planes[p * cp + w]
 * then, for every request whose current length is not a multiple of ps, the
 * slices after its last token up to the end of that page are zeroed in every
 * plane.  Other staging bytes are not written.
 *   n_planes          1..4; h_plane_bytes[p] a positive multiple of 4 and
 *                     ps * sum(h_plane_bytes) a multiple of 16
 *   h_cur_planes      host array [n_planes * cp] of device pointers: writer
 *                     w's rows of plane p, [h_cur_rows_cap[w]][plane_bytes[p]],
 *                     16-byte aligned
 *   h_staging         host array [cp] of device pointers, each
 *                     [staging_cap_pages][ps * sum(plane_bytes)] bytes
 *   flags             CPKV_FLAG_EARLY_INPUTS, CPKV_FILL_PAGE_RUNS (or 0);
 *                     other bits return CPKV_ERR_ARG
 * The gather of planar pages is cpkv_compose_gather with
 * row_bytes = sum(plane_bytes) (pages are copied as opaque bytes).
 * Status bits: ROW_OOB / WRITER_OOB (that token is skipped).
 */
int cpkv_fill_current_planes(int B, int page_size, int cp_size, int n_planes, const int32_t *h_plane_bytes,
                             const int32_t *h_cur_lens, const void *const *h_cur_planes,
                             const int64_t *h_cur_rows_cap, void *const *h_staging, int64_t staging_cap_pages,
                             const int64_t *d_staging_rows, const int32_t *d_token_writer_row,
                             const int32_t *d_writer, int64_t num_cur_pages, int flags, int32_t *d_status,
                             cpkv_stream_t stream);

/*
 * cpkv_compose_gather — per layer: the slot-dense page gather.  ONE call
 * fills every dense page: prefix pages from the owners' pools, all current
 * pages from the writers' stagings.
 *
 *   h_src_table      host array [2*cp] of device pointers:
 *                    [pool_0 .. pool_{cp-1} | staging_0 .. staging_{cp-1}],
 *                    each a page array [h_src_cap_pages[k]][ps][R], 16-byte aligned
 *   d_owner, d_src   device int32 [dense_cap_pages] (from cpkv_plan_build)
 *   d_dense          device [dense_cap_pages * ps][R], 16-byte aligned
 *   row_bytes        R; pages are opaque ps*R bytes, which must be a
 *                    multiple of 16 (R itself need not be)
 * dense page d <- page d_src[d] of table[d_owner[d]] (ps*R contiguous bytes);
 * owner -1 -> zeros.  A descriptor outside the table or the source's capacity
 * raises DESC_OOB and its page is zero-filled.
 * The gather releases its programmatic dependents when it starts: a kernel
 * launched after it with CPKV_FLAG_EARLY_INPUTS (the next layer's fill) may
 * start while it runs and waits for it before storing.
 * Pages of at most 4 KB are moved a group of consecutive dense pages at a
 * time, and a run of consecutive source pages within one table entry is one
 * copy (page-run merging); the result is the same bytes.
 */
int cpkv_compose_gather(int page_size, int cp_size, int64_t row_bytes,
                        const void *const *h_src_table, const int64_t *h_src_cap_pages,
                        const int32_t *d_owner, const int32_t *d_src, int64_t dense_cap_pages,
                        void *d_dense, int32_t *d_status, cpkv_stream_t stream);

/* Slot kinds of a gather descriptor (for cpkv_compose_gather_kinds). */
#define CPKV_GATHER_POOL 1     /* owner in [0, cp): a prefix page from a pool            */
#define CPKV_GATHER_STAGING 2  /* owner in [cp, 2cp): a current page from a staging      */
#define CPKV_GATHER_ZERO 4     /* owner -1 (and any invalid descriptor): a zero page      */
#define CPKV_GATHER_ALL 7
/* Flag for cpkv_compose_gather_kinds: the staging pages this call reads are
 * consumed.  After a staging piece has been loaded, its L2 lines are dropped
 * without being written back to DRAM, so the staging bytes are undefined
 * after the call (the dense buffer is unaffected).  For stagings that are
 * refilled before they are read again, as in the per-layer loop.  Each
 * staging page may be named by at most one descriptor of the call (plans of
 * cpkv_plan_build name each staging slot once); a second read of a consumed
 * page would see undefined bytes. */
#define CPKV_GATHER_CONSUME_STAGING 8
/* Flag for cpkv_compose_gather_kinds: early inputs, as CPKV_FLAG_EARLY_INPUTS
 * but for the gather behind its fill.  The caller promises that the plan
 * arrays and the pools were complete before the previous kernel on the
 * stream started and that nothing still running writes them; that previous
 * kernel may write the stagings (the fill).  When its grid runs at most 4
 * CTAs per SM (pages of several pieces, index-key pages), and for pages of
 * at most 4 KB (moved in groups of consecutive dense pages), the gather is
 * then launched as a programmatic dependent of that kernel (the page-run
 * fills release it at their start, the row fills as their blocks finish):
 * its CTAs may start beside or after the fill and load descriptors and pool
 * pages at once, and
 * each waits for the previous kernel to complete (griddepcontrol.wait) before
 * its first staging load and before its first store.  Any other grid of
 * more CTAs per SM is launched plainly. */
#define CPKV_GATHER_EARLY_INPUTS 16

/*
 * cpkv_compose_gather_kinds — the gather restricted to some slot kinds;
 * slots of other kinds are left untouched.  This splits a layer's compose
 * the way the layer-ahead prefetcher of the pages does ("prefetch staging"
 * message of commits 0d87bc5): the prefix pages (and zero slots) of layer
 * l + 1 do not depend on layer l and can be gathered early, e.g. on a side
 * stream (kinds = CPKV_GATHER_POOL | CPKV_GATHER_ZERO); consuming the layer
 * is then the fill followed by the current pages only
 * (kinds = CPKV_GATHER_STAGING).  The two calls together write exactly what
 * one cpkv_compose_gather writes.  kinds may also carry
 * CPKV_GATHER_CONSUME_STAGING and CPKV_GATHER_EARLY_INPUTS; any other value
 * returns CPKV_ERR_ARG.  Other
 * arguments as cpkv_compose_gather.
 */
int cpkv_compose_gather_kinds(int page_size, int cp_size, int64_t row_bytes,
                              const void *const *h_src_table, const int64_t *h_src_cap_pages,
                              const int32_t *d_owner, const int32_t *d_src, int64_t dense_cap_pages, int kinds,
                              void *d_dense, int32_t *d_status, cpkv_stream_t stream);

/*
 * cpkv_compose_layer — per layer: cpkv_fill_current followed by
 * cpkv_compose_gather in one launch, for the plan of cpkv_plan_build.  Each
 * CTA copies its pool pages (and zeroes its zero slots) into the dense
 * buffer, stores the rows of its current pages into their staging slots,
 * and reads each staged piece back into the dense page once that store has
 * completed.  The stagings and the dense buffer end up byte-identical to the
 * two-call form; every staged row is written and read back (pad rows, zero
 * in both, are written to the dense page directly).  Pages of at most 4 KB
 * go in groups of consecutive dense pages: a group's current pages, pad
 * rows included, are stored to their staging slots and read back whole
 * before the group is stored to the dense buffer.
 *   h_cur_lens       host int32 [B]
 *   h_cur_rows       host array [cp] of device pointers, writer w's current
 *                    rows [h_cur_rows_cap[w]][R], 16-byte aligned
 *   h_src_table      host array [2*cp] of device pointers
 *                    [pool_0 .. pool_{cp-1} | staging_0 .. staging_{cp-1}],
 *                    page arrays of h_src_cap_pages[k] pages; each staging
 *                    needs at least C + 1 pages
 *   d_owner, d_src, d_token_writer_row: from cpkv_plan_build (current page
 *                    i = src - 1 holds n_i rows that are consecutive in its
 *                    writer's buffer from token_writer_row of its first token)
 *   d_dense          device [dense_cap_pages * ps][R], 16-byte aligned
 *   flags            CPKV_FLAG_CONSUME_STAGING, CPKV_FLAG_EARLY_INPUTS (or 0);
 *                    other bits return CPKV_ERR_ARG
 * A descriptor outside the table or its capacity raises DESC_OOB, current
 * rows outside the writer's buffer raise ROW_OOB; either dense page is
 * zero-filled and its staging slot is not written.  Errors: ARG for bad
 * sizes, null or unaligned pointers, CAPACITY for a staging under C + 1
 * pages, LIMIT for B > CPKV_MAX_BATCH, CUDA for a failed launch.
 */
int cpkv_compose_layer(int B, int page_size, int cp_size, int64_t row_bytes, const int32_t *h_cur_lens,
                       const void *const *h_cur_rows, const int64_t *h_cur_rows_cap,
                       const void *const *h_src_table, const int64_t *h_src_cap_pages, const int32_t *d_owner,
                       const int32_t *d_src, const int32_t *d_token_writer_row, int64_t dense_cap_pages,
                       void *d_dense, int flags, int32_t *d_status, cpkv_stream_t stream);

/*
 * cpkv_compose_layer_planes — cpkv_compose_layer for planar pages (the
 * layout of cpkv_fill_current_planes): per layer, cpkv_fill_current_planes
 * followed by cpkv_compose_gather with row_bytes = sum(plane_bytes), in one
 * launch, with the same stagings and dense buffer as those two calls.  A
 * plane whose slices are 16-byte multiples at a 16-byte-aligned offset in
 * the page is staged and read back with bulk copies; the slices of any other
 * plane are written by the lanes to the staging and the dense page alike.
 *   n_planes          1..4; h_plane_bytes[p] a positive multiple of 4 and
 *                     ps * sum(h_plane_bytes) a multiple of 16
 *   h_cur_planes      host array [n_planes * cp] of device pointers: writer
 *                     w's rows of plane p, [h_cur_rows_cap[w]][plane_bytes[p]],
 *                     16-byte aligned
 *   other arguments, status bits and errors: as cpkv_compose_layer.
 */
int cpkv_compose_layer_planes(int B, int page_size, int cp_size, int n_planes, const int32_t *h_plane_bytes,
                              const int32_t *h_cur_lens, const void *const *h_cur_planes,
                              const int64_t *h_cur_rows_cap, const void *const *h_src_table,
                              const int64_t *h_src_cap_pages, const int32_t *d_owner, const int32_t *d_src,
                              const int32_t *d_token_writer_row, int64_t dense_cap_pages, void *d_dense,
                              int flags, int32_t *d_status, cpkv_stream_t stream);

/*
 * cpkv_compose_fused — per layer: the single-GPU compose in one pass, without
 * the staging round trip.  The staging exchange ("staging-direct compose")
 * carries current pages between GPUs; when every writer region is on this
 * GPU a current page can be copied straight from its writer's current-row
 * buffer.  Output is byte-identical to cpkv_fill_current followed by
 * cpkv_compose_gather, with the same descriptors:
 *   owner -1      -> zeros
 *   owner r < cp  -> page src of h_pools[r]
 *   owner cp + w  -> current page i = src - 1: the n_i consecutive rows of
 *                    h_cur_rows[w] starting at d_token_writer_row of the page's
 *                    first token, then ps - n_i zero rows
 * A descriptor outside these ranges (or rows outside the buffer) raises
 * DESC_OOB and its page is zero-filled.
 *   h_cur_lens       host int32 [B]
 *   h_pools          host array [cp] of device pointers, page arrays
 *                    [h_pool_cap_pages[r]][ps][R], 16-byte aligned
 *   h_cur_rows       host array [cp] of device pointers, [h_cur_rows_cap[w]][R]
 *   d_owner, d_src, d_token_writer_row: from cpkv_plan_build
 *   d_dense          device [dense_cap_pages * ps][R], 16-byte aligned
 *   flags            CPKV_FLAG_EARLY_INPUTS or 0; other bits return
 *                    CPKV_ERR_ARG
 */
int cpkv_compose_fused(int B, int page_size, int cp_size, int64_t row_bytes, const int32_t *h_cur_lens,
                       const void *const *h_pools, const int64_t *h_pool_cap_pages,
                       const void *const *h_cur_rows, const int64_t *h_cur_rows_cap, const int32_t *d_owner,
                       const int32_t *d_src, const int32_t *d_token_writer_row, int64_t dense_cap_pages,
                       void *d_dense, int flags, int32_t *d_status, cpkv_stream_t stream);

/*
 * cpkv_compose_fused_planes — cpkv_compose_fused for planar pages (the layout
 * of cpkv_fill_current_planes): output byte-identical to
 * cpkv_fill_current_planes followed by cpkv_compose_gather, in one pass
 * without stagings.  Plane slices that are 16-byte multiples at a
 * 16-byte-aligned page offset move with bulk copies, other slices with the
 * lanes.  One plane of a 16-byte-multiple width is cpkv_compose_fused.
 *   n_planes, h_plane_bytes, h_cur_planes: as cpkv_compose_layer_planes
 *   h_pools, h_pool_cap_pages, flags: as cpkv_compose_fused
 * A descriptor outside the table raises DESC_OOB, rows outside a writer's
 * buffer ROW_OOB; either page is zero-filled.  Errors: as cpkv_compose_layer.
 */
int cpkv_compose_fused_planes(int B, int page_size, int cp_size, int n_planes, const int32_t *h_plane_bytes,
                              const int32_t *h_cur_lens, const void *const *h_pools,
                              const int64_t *h_pool_cap_pages, const void *const *h_cur_planes,
                              const int64_t *h_cur_rows_cap, const int32_t *d_owner, const int32_t *d_src,
                              const int32_t *d_token_writer_row, int64_t dense_cap_pages, void *d_dense,
                              int flags, int32_t *d_status, cpkv_stream_t stream);

/*
 * cpkv_selftest_ring_timeout — diagnostics: runs the bounded wait of the
 * kernels' bulk-copy ring on a load that never arrives.  One warp arms a
 * ring stage for 16 bytes that no copy delivers, then drains the ring; the
 * wait gives up after the ring's time limit (2 s), the kernel raises
 * CPKV_STATUS_TIMEOUT in *d_status, writes nothing to d_dst16 (16 bytes,
 * 16-byte aligned) and returns normally.  No fault, no hang: the failure
 * path every gather, fused and layer kernel takes on a stalled copy.
 */
int cpkv_selftest_ring_timeout(void *d_dst16, int32_t *d_status, cpkv_stream_t stream);

/*
 * cpkv_ragged_plan_sizes — exact segment count S and q-token count Q_r of a
 * rank's ragged plan, from a host copy of its cp_index (host only).
 */
int cpkv_ragged_plan_sizes(int B, int chunk, const int32_t *h_q_lens, const int32_t *h_cp_index,
                           int64_t n_owned, int64_t *h_S, int64_t *h_Q);

/*
 * cpkv_ragged_plan_build — per batch: the NSA indexer's ragged index plan of
 * one CP rank ("CPU-gap fixes" message: a topk offset list plus int32
 * segment / kv_lens / q_starts / q_lens / k_bases / q_bases / current_bases
 * descriptors, all from batch metadata keyed on cp_index).
 *
 * Request b's q tokens are cut into ceil(q_b / chunk) chunks; chunk ids run
 * request-major over the batch.  d_cp_index (device int32 [n_owned]) lists the
 * chunk ids this rank owns, strictly ascending.  A segment is a maximal run
 * of owned chunks of one request with consecutive ids.  Per segment s of
 * request b:
 *   seg_req = b; q_starts = token offset inside request b's q; q_lens;
 *   kv_lens = prefix_b + q_starts + q_lens;
 *   k_bases = sum_{b' < b} align_up(prefix_b' + q_b', k_align);
 *   current_bases = k_bases + prefix_b; q_bases = exclusive sum of q_lens.
 * d_topk_offsets[j] = k_bases of the segment holding this rank's j-th token:
 * the base that turns the j-th query's topk key indices, which count from the
 * start of its request's keys, into rows of the ragged key buffer.
 * topk is the indexer's keys per query (2048 in the ragged config).  It is
 * the width of the consumer's index matrix [Q_r][topk]; no plan array depends
 * on it, and topk <= 0 returns CPKV_ERR_ARG.
 * Capacities: seg_cap >= S, topk_cap >= Q_r (S <= n_owned and
 * Q_r <= n_owned * chunk always hold).  d_counts (device int64 [2]) receives
 * (S, Q_r).  Status bits: CHUNK_OOB (bad cp_index), OUT_CAPACITY.
 */
int cpkv_ragged_plan_build(int B, int chunk, int k_align, int topk, const int32_t *h_prefix_lens,
                           const int32_t *h_q_lens, const int32_t *d_cp_index, int64_t n_owned,
                           int32_t *d_topk_offsets, int64_t topk_cap, int32_t *d_seg_req,
                           int32_t *d_kv_lens, int32_t *d_q_starts, int32_t *d_q_lens,
                           int32_t *d_k_bases, int32_t *d_q_bases, int32_t *d_current_bases,
                           int64_t seg_cap, int64_t *d_counts, int32_t *d_status, cpkv_stream_t stream);

/* Human-readable name of a return code. */
const char *cpkv_error_string(int code);

/* CPKV_VERSION of the loaded library. */
int cpkv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* CPKV_H_ */
