"""Per-batch and per-layer drivers over the C ABI.

``ComposePlan`` owns the device copies of one batch's metadata and the plan
arrays, and builds the plan once per batch (``cpkv_plan_build``).
``ComposeLayers`` owns the writers' staging regions and the dense buffers
(two, alternated by layer parity: a dense buffer is reused two layers later)
and runs the per-layer fill + gather.  Allocation uses torch device memory;
every computation is a library kernel.
"""
from __future__ import annotations

import numpy as np
import torch

from . import cpkv


class ComposePlan:
    def __init__(self, prefix_lens, cur_lens, prefix_pages, cur_pages, writer, *, page_size: int, cp_size: int,
                 num_pool_pages: int, dense_cap_pages: int | None = None, device="cuda"):
        self.prefix_lens = np.ascontiguousarray(prefix_lens, dtype=np.int32)
        self.cur_lens = np.ascontiguousarray(cur_lens, dtype=np.int32)
        self.page_size, self.cp_size, self.num_pool_pages = page_size, cp_size, num_pool_pages
        self.T, self.C, self.D = cpkv.cpkv_plan_sizes(self.prefix_lens, self.cur_lens, page_size)
        self.dense_cap_pages = self.D if dense_cap_pages is None else int(dense_cap_pages)
        self.B = len(self.prefix_lens)
        self.device = torch.device(device)
        host_writer = np.ascontiguousarray(writer, dtype=np.int32)
        self.host_writer = host_writer
        self.d_prefix_pages = torch.as_tensor(np.ascontiguousarray(prefix_pages, dtype=np.int32)).to(self.device)
        self.d_cur_pages = torch.as_tensor(np.ascontiguousarray(cur_pages, dtype=np.int32)).to(self.device)
        self.d_writer = torch.as_tensor(host_writer).to(self.device)
        self.bufs = cpkv.plan_buffers(self.B, self.T, self.dense_cap_pages, num_pool_pages, self.device,
                                      workspace_bytes=cpkv.cpkv_plan_workspace_bytes(self.cur_lens, page_size,
                                                                                     cp_size))
        self.d_status = torch.zeros(1, dtype=torch.int32, device=self.device)

    @property
    def tokens_per_writer(self):
        """Rows each writer computes (sizes its current-row buffer)."""
        return cpkv.cpkv_writer_token_counts(self.cur_lens, self.host_writer, self.page_size, self.cp_size)

    def build(self, stream=None):
        cpkv.cpkv_plan_build(self.prefix_lens, self.cur_lens, self.d_prefix_pages, self.d_cur_pages, self.d_writer,
                             page_size=self.page_size, cp_size=self.cp_size, num_pool_pages=self.num_pool_pages,
                             dense_cap_pages=self.dense_cap_pages, out=self.bufs, d_status=self.d_status,
                             stream=stream)
        return self

    def __getitem__(self, k):
        return self.bufs[k]

    @property
    def staging_cap_pages(self) -> int:
        return self.C + 1


class ComposeLayers:
    """Staging regions (one per writer, C + 1 pages each, row 0 reserved) and
    ``num_dense`` dense buffers of ``dense_cap_pages`` pages."""

    def __init__(self, plan: ComposePlan, row_bytes: int, num_dense: int = 2):
        self.plan = plan
        self.row_bytes = row_bytes
        ps, cp = plan.page_size, plan.cp_size
        self.staging = [torch.empty((plan.staging_cap_pages * ps, row_bytes), dtype=torch.uint8, device=plan.device)
                        for _ in range(cp)]
        self.dense = [torch.empty((plan.dense_cap_pages * ps, row_bytes), dtype=torch.uint8, device=plan.device)
                      for _ in range(num_dense)]

    def fill(self, cur_rows_per_writer, stream=None, early_inputs=False, page_runs=True):
        """``early_inputs``: the rows and the plan were complete before the
        previous kernel on the stream started (cpkv.FLAG_EARLY_INPUTS).
        ``page_runs``: the plan's index arrays move each current page as one
        run (cpkv.FILL_PAGE_RUNS; they are this plan's own, so it holds)."""
        p = self.plan
        cpkv.cpkv_fill_current(p.cur_lens, cur_rows_per_writer, self.staging, page_size=p.page_size,
                               cp_size=p.cp_size, row_bytes=self.row_bytes, staging_cap_pages=p.staging_cap_pages,
                               d_staging_rows=p["staging_rows"], d_token_writer_row=p["token_writer_row"],
                               d_writer=p.d_writer, num_cur_pages=p.C, d_status=p.d_status,
                               early_inputs=early_inputs, page_runs=page_runs, stream=stream)

    def fill_planes(self, cur_planes_per_writer, plane_bytes, stream=None, early_inputs=False, page_runs=True):
        """Planar-page fill (``cur_planes_per_writer[p][w]``); the row width of
        these buffers must be ``sum(plane_bytes)``.  ``page_runs``: each plane
        of a current page moves as one run (cpkv.FILL_PAGE_RUNS)."""
        p = self.plan
        cpkv.cpkv_fill_current_planes(p.cur_lens, cur_planes_per_writer, self.staging, page_size=p.page_size,
                                      cp_size=p.cp_size, plane_bytes=plane_bytes,
                                      staging_cap_pages=p.staging_cap_pages, d_staging_rows=p["staging_rows"],
                                      d_token_writer_row=p["token_writer_row"], d_writer=p.d_writer,
                                      num_cur_pages=p.C, d_status=p.d_status, early_inputs=early_inputs,
                                      page_runs=page_runs, stream=stream)

    def gather(self, pools, dense, stream=None, consume_staging=False, early_inputs=False):
        """``pools``: the cp owner slabs [slab_pages, ps, R] of this layer.
        ``consume_staging``: the stagings are refilled before their next read,
        so their L2 lines are dropped after the gather reads them (their bytes
        are undefined afterwards).  ``early_inputs``: the plan and the pools
        were complete before the previous kernel on the stream (the fill)
        started (cpkv.GATHER_EARLY_INPUTS)."""
        if consume_staging or early_inputs:
            kinds = cpkv.GATHER_ALL | (cpkv.GATHER_CONSUME_STAGING if consume_staging else 0)
            self.gather_kinds(pools, dense, kinds | (cpkv.GATHER_EARLY_INPUTS if early_inputs else 0), stream)
            return
        p = self.plan
        table = list(pools) + list(self.staging)
        caps = [t.shape[0] for t in pools] + [p.staging_cap_pages] * p.cp_size
        cpkv.cpkv_compose_gather(table, caps, p["owner"], p["src"], dense, page_size=p.page_size,
                                 cp_size=p.cp_size, row_bytes=self.row_bytes, dense_cap_pages=p.dense_cap_pages,
                                 d_status=p.d_status, stream=stream)

    def gather_kinds(self, pools, dense, kinds, stream=None):
        """The gather restricted to slot kinds (cpkv.GATHER_*)."""
        p = self.plan
        table = list(pools) + list(self.staging)
        caps = [t.shape[0] if t is not None else 0 for t in pools] + [p.staging_cap_pages] * p.cp_size
        cpkv.cpkv_compose_gather_kinds(table, caps, p["owner"], p["src"], dense, page_size=p.page_size,
                                       cp_size=p.cp_size, row_bytes=self.row_bytes,
                                       dense_cap_pages=p.dense_cap_pages, kinds=kinds, d_status=p.d_status,
                                       stream=stream)

    def prefetch(self, pools, dense, stream=None):
        """Layer-ahead part of a compose: prefix pages and zero slots only."""
        self.gather_kinds(pools, dense, cpkv.GATHER_POOL | cpkv.GATHER_ZERO, stream)

    def consume(self, cur_rows_per_writer, dense, stream=None):
        """The rest of the layer once its current rows exist: fill, then the
        current pages only."""
        self.fill(cur_rows_per_writer, stream)
        self.gather_kinds([None] * self.plan.cp_size, dense, cpkv.GATHER_STAGING, stream)

    def compose_fused(self, pools, cur_rows_per_writer, dense, stream=None, plane_bytes=None, early_inputs=False):
        """One-pass single-GPU compose of a layer (no staging round trip); for
        planar pages, ``plane_bytes`` and ``cur_rows_per_writer[p][w]``.
        ``early_inputs``: the plan, pools and rows were complete before the
        previous kernel on the stream started (cpkv.FLAG_EARLY_INPUTS)."""
        p = self.plan
        if plane_bytes is not None:
            cpkv.cpkv_compose_fused_planes(p.cur_lens, pools, cur_rows_per_writer, p["owner"], p["src"],
                                           p["token_writer_row"], dense, page_size=p.page_size, cp_size=p.cp_size,
                                           plane_bytes=plane_bytes, dense_cap_pages=p.dense_cap_pages,
                                           d_status=p.d_status, early_inputs=early_inputs, stream=stream)
            return
        cpkv.cpkv_compose_fused(p.cur_lens, pools, cur_rows_per_writer, p["owner"], p["src"], p["token_writer_row"],
                                dense, page_size=p.page_size, cp_size=p.cp_size, row_bytes=self.row_bytes,
                                dense_cap_pages=p.dense_cap_pages, d_status=p.d_status, early_inputs=early_inputs,
                                stream=stream)

    def compose_one_launch(self, pools, cur_rows_per_writer, dense, stream=None, plane_bytes=None,
                           consume_staging=False, early_inputs=False):
        """Fill + gather of a layer in a single launch (cpkv_compose_layer; for
        planar pages, ``plane_bytes`` and ``cur_rows_per_writer[p][w]``,
        cpkv_compose_layer_planes)."""
        p = self.plan
        table = list(pools) + list(self.staging)
        caps = [t.shape[0] for t in pools] + [p.staging_cap_pages] * p.cp_size
        if plane_bytes is not None:
            cpkv.cpkv_compose_layer_planes(p.cur_lens, cur_rows_per_writer, table, caps, p["owner"], p["src"],
                                           p["token_writer_row"], dense, page_size=p.page_size, cp_size=p.cp_size,
                                           plane_bytes=plane_bytes, dense_cap_pages=p.dense_cap_pages,
                                           d_status=p.d_status, consume_staging=consume_staging,
                                           early_inputs=early_inputs, stream=stream)
            return
        cpkv.cpkv_compose_layer(p.cur_lens, cur_rows_per_writer, table, caps, p["owner"], p["src"],
                                p["token_writer_row"], dense, page_size=p.page_size, cp_size=p.cp_size,
                                row_bytes=self.row_bytes, dense_cap_pages=p.dense_cap_pages, d_status=p.d_status,
                                consume_staging=consume_staging, early_inputs=early_inputs, stream=stream)

    def compose_layer(self, layer: int, pools, cur_rows_per_writer, stream=None, consume_staging=False,
                      early_inputs=False, page_runs=True):
        """Fill + gather of one layer into the dense buffer of its parity.
        ``early_inputs``: both kernels launch early (the fill behind the
        previous kernel, the gather behind the fill); the caller promises that
        the plan, pools and rows were complete before the previous kernel on
        the stream started."""
        dense = self.dense[layer % len(self.dense)]
        self.fill(cur_rows_per_writer, stream, early_inputs=early_inputs, page_runs=page_runs)
        self.gather(pools, dense, stream, consume_staging=consume_staging, early_inputs=early_inputs)
        return dense
