#!/usr/bin/env python
"""Benchmark of the paged-KV compose on one GB300 (or N independent replicas).

One step = one pass of the whole hot path over one batch: the compose plan
(once per batch), the ragged index plan of CP rank 0 (once per batch) and, for
each of the 78 layers, the fill of current rows into the writers' stagings
followed by the slot-dense page gather into that layer's dense buffer.

Default workload: the traced prefill batch (bs=12, 44 600 current tokens,
page_size 64, cp 8 emulated writer regions, MLA 576 x bf16 rows) over 78
layers, each layer with its own pool slab of 4096 pages and its own current
rows.  ``--config fp8_nsa`` runs the fp8 NSA layout (bs=32, 131 072 tokens,
656-byte rows, one 2^20-page pool shared by the layers).

Prints one JSON line (rank 0).  ``--impl reference`` times the CPU oracle on
a bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads as wl  # noqa: E402

METRIC = "compose GB/s and % of HBM peak; ms per 78-layer compose at bs=12/44.6K tokens"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 7900.0  # GB300 HBM3e, nominal (reported beside the measured or fallback peak)


# ---------------------------------------------------------------------------
# accounting
# ---------------------------------------------------------------------------

def layer_bytes(prefix_lens, cur_lens, page_size, row_bytes, dense_cap_pages, planes=None):
    """Algorithmic bytes of one layer's fill + gather.

    fill:   read T rows, write T rows + the pad rows of each request's last page
    gather: read every described page (prefix and current, D pages), write
            every dense slot (dense_cap pages; slots past D are zero-filled)
    layer:  the one-launch form reads back only the staged slices: not the pad
            rows, nor the slices of planes whose width or page offset is not a
            16-byte multiple (those go to the staging and the dense page from
            the same registers)
    """
    pl = np.asarray(prefix_lens, np.int64)
    cl = np.asarray(cur_lens, np.int64)
    ps, R = page_size, row_bytes
    T = int(cl.sum())
    pad = int(((ps - cl % ps) % ps).sum())
    D = int((pl // ps).sum() + ((cl + ps - 1) // ps).sum())
    fill_read, fill_write = T * R, (T + pad) * R
    gather_read, gather_write = D * ps * R, dense_cap_pages * ps * R
    unstaged, at = 0, 0
    for w in (planes or (R,)):
        if w % 16 or at % 16:
            unstaged += w
        at += ps * w
    return {
        "fill_read": fill_read, "fill_write": fill_write, "gather_read": gather_read,
        "gather_write": gather_write, "fill": fill_read + fill_write, "gather": gather_read + gather_write,
        "total": fill_read + fill_write + gather_read + gather_write,
        "single_pass_ideal": T * R + int((pl // ps).sum()) * ps * R + D * ps * R, "T": T, "D": D, "pad_rows": pad,
        # one-launch staging compose: the pad rows are written to the dense page, not read back
        "layer": fill_read + fill_write + gather_read - pad * R - T * unstaged + gather_write,
        # one-pass compose: current rows and prefix pages read once, every dense slot written once
        "fused": T * R + int((pl // ps).sum()) * ps * R + dense_cap_pages * ps * R,
        # bytes that must cross DRAM in any form of the compose: the current
        # rows read once, the prefix pages read once, every dense slot written
        # once (the staging round trip can stay on chip, and does in the step)
        "dram_min": T * R + int((pl // ps).sum()) * ps * R + dense_cap_pages * ps * R,
        "prefix_read": int((pl // ps).sum()) * ps * R, "staging_read": int(((cl + ps - 1) // ps).sum()) * ps * R,
    }


def kernel_dram_bytes(lb, kernel, consume_staging):
    """DRAM bytes per launch of a kernel timed alone (a graph of the step's
    launches of that kernel only, replayed back to back):
      fill    reads the current rows from DRAM; its staging writes land in
              L2, where the next replay rewrites the same lines
      gather  reads the prefix pages and writes every dense slot through
              DRAM; its staging reads come from L2 unless the gather consumes
              the stagings (then the previous replay dropped them and they
              come from DRAM)
      fused, layer  the single-pass bytes (a layer kernel's staging round
              trip stays in L2)"""
    if kernel == "fill":
        return lb["fill_read"]
    if kernel == "gather":
        return lb["prefix_read"] + lb["gather_write"] + (lb["staging_read"] if consume_staging else 0)
    return lb["dram_min"]


def kernel_source_sha(files) -> str:
    """Hash of the code of the kernel sources (comments and blank space
    removed, so that an edited comment keeps a capture valid)."""
    import hashlib
    import re

    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "paged_kv_cache_compose_gb300", "csrc", f), encoding="utf-8") as fh:
            text = fh.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def kernel_traffic(kernel: str, config: str):
    """DRAM bytes per launch of ``kernel`` from the committed ncu capture, or
    None when there is none for this workload or the kernel's sources changed
    since it was taken."""
    path = os.path.join(ROOT, "profiles", f"traffic_{kernel}_{config}.json")
    if not os.path.exists(path):
        return None
    try:
        with open(path) as f:
            d = json.load(f)
        if d.get("source_sha") != kernel_source_sha(d["sources"]):
            return None
    except Exception:
        return None
    return d.get("dram_bytes_per_launch")


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            with open(path) as f:
                d = json.load(f)
            for k in ("hbm_gbs", "hbm_GBs", "hbm_copy_gbs"):
                if k in d:
                    return float(d[k]), "measured", d
        except Exception:
            pass
    return FALLBACK_HBM_GBS, "fallback", {}


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except FileNotFoundError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# the workload on the GPU
# ---------------------------------------------------------------------------

class ComposeWorkload:
    """Device state of one benchmark replica: batch metadata, plan, pools,
    per-layer current rows, stagings, dense double buffer, ragged plan."""

    def __init__(self, config: str = "traced_78", device="cuda", num_layers: int | None = None,
                 variant: str = "staging", pool_pages: int | None = None, consume_staging: bool | None = None,
                 num_dense: int = 2, early: bool = True, fill_mode: str = "pages"):
        import torch

        from paged_kv_cache_compose_gb300 import cpkv
        from paged_kv_cache_compose_gb300.runtime import ComposeLayers, ComposePlan

        self.torch, self.cpkv = torch, cpkv
        self.config = config
        if pool_pages is not None and config not in ("fp8_nsa", "index_k"):
            raise ValueError("--pool-pages applies to the shared-pool workloads only")
        self.batch = b = (wl.CONFIGS[config]() if pool_pages is None
                          else wl.CONFIGS[config](num_pool_pages=pool_pages))
        self.num_layers = b.num_layers if num_layers is None else min(num_layers, b.num_layers)
        self.device = torch.device(device)
        self.plan = ComposePlan(b.prefix_lens, b.cur_lens, b.prefix_pages, b.cur_pages, b.writer,
                                page_size=b.page_size, cp_size=b.cp_size, num_pool_pages=b.num_pool_pages,
                                device=self.device)
        # dense buffers reused round-robin by layer (2: double buffering; one
        # per layer keeps every layer's output for a full parity check)
        self.layers = ComposeLayers(self.plan, b.row_bytes, num_dense=num_dense)
        self.early = bool(early)
        # the fill moves each current page as one run (its plan is cpkv_plan_build's), or row by row
        if fill_mode not in ("pages", "rows"):
            raise ValueError(fill_mode)
        self.fill_mode = fill_mode
        # pools: one per layer (own slab) unless the config shares one pool over its layers
        self.shared_pool = config in ("fp8_nsa", "index_k")
        n_pools = 1 if self.shared_pool else self.num_layers
        self.pools = [wl.device_pool(b, layer, self.device) for layer in range(n_pools)]
        # all layers' current rows in one allocation (so the end-to-end leg can
        # upload them with one copy): per layer, writer-major rows, or for planar
        # pages plane-major then writer-major, each block 16-byte aligned
        counts = [int(x) for x in self.plan.tokens_per_writer]
        planes = b.planes or (b.row_bytes,)
        blocks = [(p, w, -(-counts[w] * wp // 16) * 16) for p, wp in enumerate(planes) for w in range(b.cp_size)]
        per_layer = sum(n for _, _, n in blocks)
        self.rows_all = torch.empty((self.num_layers, per_layer), dtype=torch.uint8, device=self.device)
        self.rows = []
        for layer in range(self.num_layers):
            g = wl.device_current_rows(b, layer, self.device)
            parts = wl.device_split_rows_by_writer(b, g)
            views = [[None] * b.cp_size for _ in planes]
            off, col = 0, [0]
            for wp in planes:
                col.append(col[-1] + wp)
            for p, w, n in blocks:
                wp = planes[p]
                dst = self.rows_all[layer, off:off + counts[w] * wp].view(counts[w], wp)
                dst.copy_(parts[w][:, col[p]:col[p + 1]])
                views[p][w] = dst
                off += n
            self.rows.append(views if b.planes else views[0])
            del g
        # ragged index plan of CP rank 0 over the batch's q tokens
        self.rb = wl.ragged_from_compose(b)
        self.cp_index = self.rb.cp_index(0)
        S, Q = cpkv.cpkv_ragged_plan_sizes(self.rb.q_lens, self.cp_index, self.rb.chunk)
        self.ragged_out = cpkv.ragged_buffers(max(S, 1), max(Q, 1), self.device)
        self.d_cp_index = torch.from_numpy(self.cp_index).to(self.device)
        self.ragged_counts = torch.zeros(2, dtype=torch.int64, device=self.device)
        self.bytes = layer_bytes(b.prefix_lens, b.cur_lens, b.page_size, b.row_bytes, self.plan.dense_cap_pages,
                                 b.planes)
        self.graph = None
        self.variant = variant
        # the gather consumes the stagings (drops their L2 lines after reading
        # them): by default for row-major pages above 4 KB, where it measured
        # faster (traced -6%, fp8 -1%); the planar index-key pages measured
        # 1.5% slower, and one-token 1152-byte pages 5% (fill + group gather,
        # 4.64 against 4.40 ms) and 13% (one launch, 4.90 against 4.36 ms)
        if consume_staging is None:
            consume_staging = (variant in ("staging", "layer") and not b.planes
                               and b.page_size * b.row_bytes > 4096)
        self.consume_staging = bool(consume_staging) and variant in ("staging", "layer")
        if variant == "staging":
            self.launches_per_step = 3 + 2 * self.num_layers  # plan (2) + ragged (1) + (fill + gather) per layer
            self.layer_bytes = self.bytes["total"]
            self.kernels = {"fill": self.bytes["fill"], "gather": self.bytes["gather"]}
        elif variant == "fused":
            self.launches_per_step = 3 + self.num_layers  # plan (2) + ragged (1) + one fused compose per layer
            self.layer_bytes = self.bytes["fused"]
            self.kernels = {"fused": self.bytes["fused"]}
        elif variant == "layer":
            self.launches_per_step = 3 + self.num_layers  # plan (2) + ragged (1) + one fill+gather launch per layer
            self.layer_bytes = self.bytes["layer"]
            self.kernels = {"layer": self.bytes["layer"]}
        elif variant == "prefetch":
            # layer-ahead: prefix pages of layer l+1 gathered on a side stream while layer l is consumed
            self.launches_per_step = 3 + 3 * self.num_layers  # plan + ragged + (prefetch, fill, current gather)
            self.layer_bytes = self.bytes["total"]
            self.kernels = {"fill": self.bytes["fill"], "gather": self.bytes["gather"]}
            self.side = torch.cuda.Stream(device=self.device)
            self.prefetched = [torch.cuda.Event() for _ in range(self.num_layers)]
            self.consumed = [torch.cuda.Event() for _ in range(self.num_layers)]
            self.plan_ready = torch.cuda.Event()
        else:
            raise ValueError(variant)

    def pools_of(self, layer):
        return self.pools[0 if self.shared_pool else layer]

    def dense_of(self, layer):
        return self.layers.dense[layer % len(self.layers.dense)]

    def step(self, stream=None):
        """Enqueue one step on the current stream."""
        self.plan.build(stream)
        self.cpkv.cpkv_ragged_plan_build(self.rb.prefix_lens, self.rb.q_lens, self.d_cp_index, len(self.cp_index),
                                         chunk=self.rb.chunk, k_align=self.rb.k_align, topk=self.rb.topk, out=self.ragged_out,
                                         d_counts=self.ragged_counts, d_status=self.plan.d_status, stream=stream)
        if self.variant == "prefetch":
            return self._prefetch_layers()
        for layer in range(self.num_layers):
            self.run_kernel("all", layer, stream)

    def _prefetch_layers(self):
        """Layer l's prefix pages are gathered on the side stream one layer
        ahead; the main stream consumes layer l (fill + current pages) once
        its prefix is in.  The side stream reuses a dense buffer only after
        the layer that used it two layers earlier has been consumed."""
        torch = self.torch
        main = torch.cuda.current_stream()
        self.plan_ready.record(main)
        side = self.side
        side.wait_event(self.plan_ready)

        def prefetch(layer):
            with torch.cuda.stream(side):
                if layer >= 2:
                    side.wait_event(self.consumed[layer - 2])
                self.layers.prefetch(self.pools_of(layer), self.dense_of(layer))
                self.prefetched[layer].record(side)

        prefetch(0)
        for layer in range(self.num_layers):
            if layer + 1 < self.num_layers:
                prefetch(layer + 1)
            main.wait_event(self.prefetched[layer])
            self.layers.consume(self.rows[layer], self.dense_of(layer))
            self.consumed[layer].record(main)
        main.wait_stream(side)

    def run_kernel(self, kind, layer, stream=None):
        """Launch one layer's work: ``all`` of it, or one kernel of it."""
        dense = self.dense_of(layer)
        # Every input of a layer's compose (plan, pools, rows) is complete before
        # the step's layer loop starts (or, end to end, is joined to the layer
        # by an event wait on its upload), and no kernel of the loop writes
        # one, so the step launches its kernels early behind the previous one
        # (cpkv.FLAG_EARLY_INPUTS, cpkv.GATHER_EARLY_INPUTS).  The graphs that
        # time one kind of kernel alone launch plainly, so that their launches
        # never overlap and each one's duration is measured whole.
        early = kind == "all" and self.early
        if self.variant == "fused":
            self.layers.compose_fused(self.pools_of(layer), self.rows[layer], dense, stream,
                                      plane_bytes=list(self.batch.planes) if self.batch.planes else None,
                                      early_inputs=early)
            return
        if self.variant == "layer":
            self.layers.compose_one_launch(self.pools_of(layer), self.rows[layer], dense, stream,
                                           plane_bytes=list(self.batch.planes) if self.batch.planes else None,
                                           consume_staging=self.consume_staging, early_inputs=early)
            return
        if kind in ("all", "fill"):
            if self.batch.planes:
                self.layers.fill_planes(self.rows[layer], list(self.batch.planes), stream, early_inputs=early,
                                        page_runs=self.fill_mode == "pages")
            else:
                self.layers.fill(self.rows[layer], stream, early_inputs=early, page_runs=self.fill_mode == "pages")
        if kind in ("all", "gather"):
            self.layers.gather(self.pools_of(layer), dense, stream, consume_staging=self.consume_staging,
                               early_inputs=early)

    def kernel_graphs(self):
        """One more CUDA graph per kernel of the step (fills alone and gathers
        alone; the fused or layer kernel alone): the step's launches of that
        kernel, same inputs and launch shapes, launched plainly so that no two
        launches overlap, to time each kernel's launches."""
        torch = self.torch
        graphs = {}
        for kind in self.kernels:
            def body(kind=kind):
                for layer in range(self.num_layers):
                    self.run_kernel(kind, layer)
            s = torch.cuda.Stream()
            s.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(s):
                body()
            torch.cuda.current_stream().wait_stream(s)
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                body()
            graphs[kind] = g
        torch.cuda.synchronize()
        return graphs

    def capture(self):
        """Capture one step as a CUDA graph (after a warm-up run)."""
        torch = self.torch
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            self.step()
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            self.step()
        torch.cuda.synchronize()

    def run(self):
        if self.graph is not None:
            self.graph.replay()
        else:
            self.step()

    def status(self) -> int:
        return int(self.plan.d_status.item())


def _dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def aggregate(values_ms, units, ws):
    """Max time over ranks and total units over ranks (torch.distributed when ws > 1)."""
    if ws == 1:
        return float(values_ms), float(units)
    import torch
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(values_ms)], dtype=torch.float64, device=dev)
    u = torch.tensor([float(units)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


# ---------------------------------------------------------------------------
# CPU oracle timing (cpu_baseline leg and --impl reference)
# ---------------------------------------------------------------------------

def compact_pool(batch, slabs):
    """Relabel the batch's prefix pages onto a compact pool holding only the
    pages it references, keeping each page's owner (new id = cp * (j + 1) + owner,
    j = rank of the page among the owner's referenced pages).  The compose reads
    exactly the same bytes, so oracle results and work are unchanged; the host
    only has to hold the referenced pages.  ``slabs``: the cp owner slabs
    (torch CUDA tensors or numpy arrays) [slab_pages, ps, R]."""
    import dataclasses

    cp = batch.cp_size
    lp = np.asarray(batch.prefix_pages, np.int64)
    new_ids = np.empty_like(lp)
    host = []
    width = 1
    for o in range(cp):
        idx = np.nonzero(lp % cp == o)[0]
        uniq, inv = np.unique(lp[idx] // cp, return_inverse=True)
        new_ids[idx] = cp * (inv + 1) + o
        s = slabs[o]
        if hasattr(s, "index_select"):
            import torch

            pages = s.index_select(0, torch.from_numpy(uniq).to(s.device)).cpu().numpy()
        else:
            pages = s[uniq]
        host.append(pages)
        width = max(width, len(uniq) + 1)
    ps, R = batch.page_size, batch.row_bytes
    out = []
    for pages in host:
        slab = np.zeros((width, ps, R), np.uint8)
        slab[1:1 + len(pages)] = pages
        out.append(slab)
    # current pages are never read from the pool: give them fresh ids past the compact range
    cur_ids = cp * (width + 1 + np.arange(batch.C, dtype=np.int64))
    nb = dataclasses.replace(batch, prefix_pages=new_ids.astype(np.int32), cur_pages=cur_ids.astype(np.int32),
                             num_pool_pages=int(cp * (width + 2 + batch.C)))
    return nb, out


class HostPages:
    """One owner's pool slab on the host, generated page by page on demand
    (seeded by batch, layer and owner): indexing it with page ids yields
    [len(ids), ps, R] rows, so a compacted sample of a large pool never
    materialises the pages it does not reference."""

    def __init__(self, batch, layer: int, owner: int):
        self.batch, self.layer, self.owner = batch, layer, owner

    def __getitem__(self, ids):
        b = self.batch
        ids = np.asarray(ids, np.int64)
        out = np.empty((len(ids), b.page_size, b.row_bytes), np.uint8)
        for k, i in enumerate(ids.tolist()):
            rng = np.random.default_rng([b.seed, 7, self.layer, self.owner, i])
            out[k] = wl.random_rows(rng, b.page_size, b.row_bytes, b.row_kind)
        return out


def oracle_sample(work_or_batch, n_layers: int, shared_pool: bool = False):
    """Host inputs for ``n_layers`` layers of the workload: copied from the
    device replica when there is one, else generated on the host (only the
    referenced pages; ``shared_pool``: one pool for all layers); pools are
    compacted to the pages the batch references."""
    b = work_or_batch.batch if hasattr(work_or_batch, "batch") else work_or_batch
    pools, rows = [], []
    nb = b
    for layer in range(n_layers):
        if hasattr(work_or_batch, "pools_of"):
            w = work_or_batch
            nb, slabs = compact_pool(b, w.pools_of(layer))
            rows.append([r.cpu().numpy() for r in w.rows[layer]])
        else:
            if pools and shared_pool:
                slabs = pools[0]
            else:
                nb, slabs = compact_pool(b, [HostPages(b, layer, o) for o in range(b.cp_size)])
            rows.append(wl.split_rows_by_writer(b, wl.host_current_rows(b, layer)))
        pools.append(slabs)
    return nb, pools, rows


def oracle_step(b, pools, rows_per_writer, lib=None):
    """One bounded oracle step: plan once, then per sampled layer the staging
    (fill) and the descriptor gather.  Returns the algorithmic bytes moved."""
    import oracle

    plan = oracle.compose_plan(b.prefix_lens, b.cur_lens, b.prefix_pages, b.cur_pages, b.writer,
                               page_size=b.page_size, cp_size=b.cp_size, num_pool_pages=b.num_pool_pages, lib=lib)
    rb = wl.ragged_from_compose(b)
    oracle.ragged_plan(rb.prefix_lens, rb.q_lens, rb.cp_index(0), chunk=rb.chunk, k_align=rb.k_align, lib=lib)
    ps, R, cp = b.page_size, b.row_bytes, b.cp_size
    stg = [np.zeros(((plan["C"] + 1) * ps, R), np.uint8) for _ in range(cp)]
    tw = wl.token_writer(b)
    moved = 0
    lb = layer_bytes(b.prefix_lens, b.cur_lens, ps, R, plan["D"])
    for layer in range(len(pools)):
        # the oracle's staging takes batch-ordered rows: interleave the writers' rows back
        g = np.empty((b.T, R), np.uint8)
        for w in range(cp):
            g[tw == w] = rows_per_writer[layer][w]
        oracle.staging(b.cur_lens, b.writer, g, stg, page_size=ps, cp_size=cp, lib=lib)
        table = [s.reshape(-1) for s in pools[layer]] + [s.reshape(-1) for s in stg]
        caps = [s.shape[0] for s in pools[layer]] + [plan["C"] + 1] * cp
        oracle.gather(table, caps, plan["owner"], plan["src"], page_size=ps, row_bytes=R, dense_cap=plan["D"], lib=lib)
        moved += lb["total"]
    return moved


def host_cpu() -> dict:
    """The host the oracle runs on: logical CPUs and the CPU model."""
    import platform

    model = None
    try:
        fields = {}
        with open("/proc/cpuinfo") as f:
            for line in f:
                k, _, v = line.partition(":")
                fields.setdefault(k.strip(), v.strip())
        model = fields.get("model name") or (
            f"implementer {fields['CPU implementer']} part {fields['CPU part']}" if "CPU part" in fields else None)
    except OSError:
        pass
    return {"nproc": os.cpu_count(), "machine": platform.machine(), "model": model}


def time_oracle(b, pools, rows, min_seconds=10.0, max_seconds=30.0):
    """Run oracle steps until at least ``min_seconds`` of work; GB/s of the work."""
    import oracle

    lib = oracle.load()
    t0 = time.perf_counter()
    moved, steps = 0, 0
    while True:
        moved += oracle_step(b, pools, rows, lib)
        steps += 1
        el = time.perf_counter() - t0
        if el >= min_seconds or el >= max_seconds:
            break
    return moved / el / 1e9, el, steps


def _all_cores_worker(config, n_layers, shared_pool, seconds, barrier, out):
    """One process of the all-cores oracle baseline: host inputs generated
    from the workload's seeds, one untimed step, then oracle steps from the
    common start (a barrier) for ``seconds``.  Puts (bytes, t0, t1, steps),
    or an error string."""
    try:
        import oracle

        b, pools, rows = oracle_sample(wl.CONFIGS[config](), n_layers, shared_pool=shared_pool)
        lib = oracle.load()
        oracle_step(b, pools, rows, lib)
        barrier.wait(timeout=600)
        t0 = time.time()
        moved, steps = 0, 0
        while True:
            moved += oracle_step(b, pools, rows, lib)
            steps += 1
            t1 = time.time()
            if t1 - t0 >= seconds:
                break
        out.put((moved, t0, t1, steps))
    except Exception as e:  # reported by the parent, which then gives no number
        barrier.abort()
        out.put(f"{type(e).__name__}: {e}")


def time_oracle_all_cores(config, n_layers, shared_pool=False, seconds=10.0, workers=None):
    """The labelled all-cores variant of the CPU baseline: one single-threaded
    oracle process per host core, each running the same bounded sample on its
    own host-generated copy of the inputs, started together.  Returns
    (GB/s over the common wall-clock window, processes, seconds, steps), or
    None with the reason when a worker failed."""
    import multiprocessing as mp
    import queue

    ctx = mp.get_context("spawn")  # never fork a process that holds a CUDA context
    n = workers or os.cpu_count() or 1
    barrier, out = ctx.Barrier(n), ctx.Queue()
    procs = [ctx.Process(target=_all_cores_worker, args=(config, n_layers, shared_pool, seconds, barrier, out))
             for _ in range(n)]
    for p in procs:
        p.start()
    res, err = [], None
    try:
        for _ in range(n):
            r = out.get(timeout=900)
            if isinstance(r, str):
                err = err or r
            else:
                res.append(r)
    except queue.Empty:
        err = err or "a worker did not report within 900 s"
    for p in procs:
        p.join(timeout=60)
        if p.is_alive():
            p.terminate()
    if err is not None or len(res) != n:
        return None, err or "missing worker results"
    moved = sum(r[0] for r in res)
    t0, t1 = min(r[1] for r in res), max(r[2] for r in res)
    return (moved / (t1 - t0) / 1e9, n, t1 - t0, sum(r[3] for r in res)), None


# ---------------------------------------------------------------------------
# main
# ---------------------------------------------------------------------------

def warm_and_capture(work, warmup: int, graph: bool = True):
    """``warmup`` untimed steps (also the first use of every kernel), then the
    capture of one step as a CUDA graph and two more replays."""
    torch = work.torch
    for _ in range(warmup):
        work.run()
    torch.cuda.synchronize()
    if graph:
        work.capture()
        for _ in range(2):
            work.run()
        torch.cuda.synchronize()


def timed_steps(work, steps: int, flush=None):
    """Exactly ``steps`` steps timed with CUDA events on the launching stream:
    one pair around all of them and one pair around each.  ``flush``: a buffer
    larger than L2, written between steps outside the per-step events (the
    time is then the sum of the steps).  Returns (ms in all, sorted per-step ms)."""
    torch = work.torch
    per_step = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for s0, s1 in per_step:
        if flush is not None:
            flush.fill_(1)
        s0.record()
        work.run()
        s1.record()
    e1.record()
    torch.cuda.synchronize()
    step_ms = sorted(s0.elapsed_time(s1) for s0, s1 in per_step)
    return (sum(step_ms) if flush is not None else e0.elapsed_time(e1)), step_ms


def time_kernels(work, steps: int):
    """Average launch duration (ms) of each kernel of the step: CUDA events
    around replays of a graph that holds the step's launches of that kernel
    alone."""
    torch = work.torch
    kern = {}
    for kind, g in work.kernel_graphs().items():
        g.replay()
        torch.cuda.synchronize()
        k0, k1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = max(3, steps // 4)
        k0.record()
        for _ in range(reps):
            g.replay()
        k1.record()
        torch.cuda.synchronize()
        kern[kind] = k0.elapsed_time(k1) / (reps * work.num_layers)
    return kern


def kernel_rooflines(work, kern, hbm_peak):
    """Per kernel: algorithmic bytes per launch over its average launch time,
    the bytes of it that cross DRAM (kernel_dram_bytes) over the same time,
    and the DRAM bytes ncu measured per launch (kernel_traffic; None without
    a capture of the current sources)."""
    out = {}
    for k, ms in kern.items():
        alg = work.kernels[k]
        dram = kernel_dram_bytes(work.bytes, k, work.consume_staging)
        out[k] = {"avg_launch_ms": round(ms, 5), "algorithmic_bytes_per_launch": alg,
                  "achieved": round(alg / (ms / 1e3) / 1e9, 1), "frac": round(alg / (ms / 1e3) / 1e9 / hbm_peak, 4),
                  "dram_bytes_per_launch": dram, "dram_achieved": round(dram / (ms / 1e3) / 1e9, 1),
                  "dram_frac": round(dram / (ms / 1e3) / 1e9 / hbm_peak, 4),
                  "traffic": kernel_traffic(k, work.config)}
    return out


def step_fractions(work, ms_step, hbm_peak, ws=1):
    """The step's byte rates: algorithmic bytes (every byte each kernel reads
    and writes, the staging round trip included) and the bytes that must cross
    DRAM (current rows and prefix pages read once, every dense slot written
    once), each over the measured peak."""
    alg = work.layer_bytes * work.num_layers / (ms_step / 1e3) / 1e9
    dram = work.bytes["dram_min"] * work.num_layers / (ms_step / 1e3) / 1e9
    return {
        "dram_gbs": round(dram * ws, 1),
        "pct_of_hbm_peak_dram": round(100 * dram / hbm_peak, 2),
        "pct_algorithmic_over_peak": round(100 * alg / hbm_peak, 2),
        "pct_of_nominal_hbm_dram": round(100 * dram / NOMINAL_HBM_GBS, 2),
    }


def _free(torch):
    """Return the device memory of dropped objects to the driver."""
    import gc

    gc.collect()
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def extra_configs(a, device, hbm_peak):
    """The scope table's other measured rows, in the same run as the headline:
    the fp8 NSA compose over 78 layers (the headline's variant, timed the same
    way over fewer steps, with its kernels timed alone), the traced lengths on
    one-token pages (the headline's variant and one launch per layer), the
    ragged index plan of the ragged config (every CP rank) and the compose
    plan of the traced, fp8 and one-token-page batches."""
    import torch

    out = {}
    steps = max(5, min(a.steps, 20))

    def measure(config, variant, workload):
        t0 = time.perf_counter()
        work = ComposeWorkload(config, device=device, variant=variant, fill_mode=a.fill_mode,
                               early=a.launch == "early")
        setup_s = time.perf_counter() - t0
        warm_and_capture(work, 3)
        st0 = work.status()
        ms_total, step_ms = timed_steps(work, steps)
        ms_step = ms_total / steps
        kern = time_kernels(work, steps)
        b = work.batch
        res = {
            "workload": workload,
            "variant": work.variant, "consume_staging": work.consume_staging, "steps": steps,
            "ms_per_78_layer_compose": round(ms_step * 78 / work.num_layers, 4),
            "ms_per_step_stats": {"median": round(step_ms[len(step_ms) // 2], 4), "min": round(step_ms[0], 4),
                                  "max": round(step_ms[-1], 4)},
            "value": round(work.layer_bytes * work.num_layers / (ms_step / 1e3) / 1e9, 2), "unit": "GB/s",
            **step_fractions(work, ms_step, hbm_peak),
            "bytes_per_layer": work.layer_bytes, "dram_bytes_per_layer": work.bytes["dram_min"],
            "B": b.B, "T": b.T, "C": work.plan.C, "D": work.plan.D,
            "kernels": kernel_rooflines(work, kern, hbm_peak),
            "setup_s": round(setup_s, 1),
            "status_word": work.status() | st0,
        }
        del work
        _free(torch)
        return res

    out["fp8_nsa"] = measure(
        "fp8_nsa", a.variant,
        "fp8 NSA compose, 78 layers: bs=32, 131072 current tokens (lognormal split), prefix U[0,64K] "
        "page-floored, page_size=64, cp=8, 656-byte rows, one 2^20-page pool shared by the layers")
    # the traced lengths on one-token pages, through the kernels that move
    # groups of consecutive dense pages: the headline's variant and the
    # one-launch form
    ps1 = ("traced lengths on one-token pages, 78 layers: page_size=1, 88832 prefix + 44600 current pages "
           "of 1152 bytes per layer, a 2^18-page pool slab per layer")
    out["traced_78_ps1"] = measure("traced_78_ps1", a.variant, ps1)
    if a.variant != "layer":
        out["traced_78_ps1_layer"] = measure("traced_78_ps1", "layer", ps1)
    reps = max(20, a.steps)
    out["ragged_plan"] = ragged_plan_latency(reps, splits=("interleaved",))["interleaved"]
    out["compose_plan"] = compose_plan_latency(reps, ("traced", "fp8_nsa", "traced_78_ps1"))
    return out


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default="traced_78",
                    choices=["traced_78", "traced", "traced_78_ps1", "fp8_nsa", "index_k", "plans"],
                    help="plans: latency of the per-batch plan builders (ragged plan config, all CP ranks and "
                         "splits; compose plan of the traced, fp8 and one-token-page batches)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--variant", default="staging", choices=["staging", "fused", "prefetch", "layer"],
                    help="staging: fill + slot-dense gather per layer (the pages' method); "
                         "fused: one-pass single-GPU compose without the staging round trip; "
                         "prefetch: staging method with each layer's prefix pages gathered one layer ahead "
                         "on a side stream")
    ap.add_argument("--no-graph", action="store_true", help="launch layer by layer instead of replaying a CUDA graph")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra-configs", action="store_true",
                    help="skip the fp8 NSA, one-token-page, ragged-plan and compose-plan measurements that the "
                         "default (traced_78) run adds to its line")
    ap.add_argument("--cpu-layers", type=int, default=2, help="layers in the oracle's bounded sample")
    ap.add_argument("--no-cpu-all-cores", action="store_true",
                    help="skip the all-cores variant of the CPU baseline (one oracle process per core)")
    ap.add_argument("--layers", type=int, default=None,
                    help="run only the first N layers (small cases for profiling; the headline uses all 78)")
    ap.add_argument("--consume-staging", choices=["auto", "on", "off"], default="auto",
                    help="staging variant: the gather drops each staging piece's L2 lines after reading it "
                         "(the stagings are refilled before their next read); auto = on for row-major pages")
    ap.add_argument("--launch", choices=["early", "plain"], default="early",
                    help="early: each kernel of the layer loop launches as a programmatic dependent of the previous "
                         "one (all inputs exist before the loop); plain: ordinary launches")
    ap.add_argument("--fill-mode", choices=["pages", "rows"], default="pages",
                    help="staging variant: the fill moves each current page as one run (the plan's pages are "
                         "runs) or copies row by row through the index arrays")
    ap.add_argument("--pool-pages", type=int, default=None,
                    help="pool size of the shared-pool workloads (fp8_nsa, index_k): small device footprints for "
                         "profiling; every launch still moves the same pages")
    a = ap.parse_args(argv)
    a.warmup = max(a.warmup, 3)

    ws, rank, local = _dist_env()
    if a.impl == "reference":
        return run_reference(a, ws, rank)
    if a.config == "plans":
        return run_plans(a)

    import torch

    if ws > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    device = torch.device("cuda", local if ws > 1 else torch.cuda.current_device())
    torch.cuda.set_device(device)

    from paged_kv_cache_compose_gb300 import build as cpkv_build

    cpkv_build.build()
    work = ComposeWorkload(a.config, device=device, num_layers=a.layers, variant=a.variant, pool_pages=a.pool_pages,
                           consume_staging={"auto": None, "on": True, "off": False}[a.consume_staging],
                           fill_mode=a.fill_mode, early=a.launch == "early")
    hbm_peak, peak_src, _ = read_peaks()

    warm_and_capture(work, a.warmup, graph=not a.no_graph)
    st0 = work.status()

    # timed region
    clocks = ClockSampler(device.index)
    clocks.start()
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    # A one-layer workload re-reads the same pages every step, so L2 is
    # flushed between its steps by a write larger than L2, outside the
    # per-step events, and its time is the sum of the steps; the 78-layer
    # workloads read 27+ GB of distinct inputs per step and run back to back.
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=device) if work.num_layers == 1 else None
    ms_total, step_ms = timed_steps(work, a.steps, flush)
    if ws > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    ms_max, units_all = aggregate(ms_total, work.layer_bytes * work.num_layers * a.steps, ws)
    ms_step = ms_max / a.steps
    value_gbs = units_all / (ms_max / 1e3) / 1e9

    kern = time_kernels(work, a.steps)
    kernel_timing = ("alone: a CUDA graph of the step's launches of that kernel only, replayed, launched plainly "
                     "(in the step they launch early behind the previous kernel; here launches never overlap)")
    if work.consume_staging and work.variant == "staging":
        kernel_timing += (" (the gather consumes the stagings, so when replayed alone it reads them from DRAM: "
                          "all its algorithmic bytes cross DRAM; inside the step they are read from L2)")
    kroof = kernel_rooflines(work, kern, hbm_peak)
    top = {"fused": "fused", "layer": "layer"}.get(work.variant, "gather")
    status = work.status()

    traffic = kroof[top]["traffic"]

    # end to end through the public API with host buffers
    e2e = None
    if not a.no_e2e:
        e2e = run_e2e(work, a, ws)

    cpu = None
    if not a.no_cpu_baseline and rank == 0 and ws == 1:
        b, pools, rows = oracle_sample(work, min(a.cpu_layers, work.num_layers))
        gbs, secs, steps = time_oracle(b, pools, rows)
        cpu = {"value": round(gbs, 3), "unit": "GB/s", "cores": 1, "kind": "oracle",
               "sample": f"plan + ragged plan + {len(pools)} of {work.num_layers} layers (staging + gather) of "
                         f"the same batch and inputs, repeated {steps}x over {secs:.1f}s, single-threaded C",
               "host": host_cpu()}
    cpu_all = None
    if not a.no_cpu_baseline and not a.no_cpu_all_cores and rank == 0 and ws == 1:
        n_layers = min(a.cpu_layers, work.num_layers)
        got, why = time_oracle_all_cores(a.config, n_layers, shared_pool=work.shared_pool)
        if got is None:
            cpu_all = {"value": None, "unavailable": why}
        else:
            gbs_all, procs, secs, steps = got
            cpu_all = {"value": round(gbs_all, 3), "unit": "GB/s", "cores": procs, "kind": "oracle",
                       "sample": f"{procs} single-threaded oracle processes (one per host core) started together, "
                                 f"each running plan + ragged plan + {n_layers} of {work.num_layers} layers "
                                 f"(staging + gather) on its own host-generated inputs of the same batch; "
                                 f"{steps} steps in {secs:.1f}s in all"}

    b = work.batch
    workload_desc = (
        "traced prefill compose, 78 layers: bs=12, 44600 current tokens (lognormal split), prefix U[0,16K] "
        "page-floored, page_size=64, cp=8 writer regions on one GPU, MLA 576xbf16 rows, 4096-page pool slab per "
        "layer" if a.config == "traced_78" else
        "traced prefill compose, 1 layer: the same batch over its 200000-page randomly permuted pool"
        if a.config == "traced" else
        "traced prefill compose with one-token pages, 78 layers: the same lengths, page_size=1 (88832 prefix + "
        "44600 current pages of 1152 bytes per layer), 2^18-page pool slab per layer" if a.config == "traced_78_ps1"
        else
        "fp8 NSA compose, 78 layers: bs=32, 131072 current tokens, prefix U[0,64K], page_size=64, cp=8, 656-byte "
        "rows, one 2^20-page pool shared by the layers" if a.config == "fp8_nsa" else
        "NSA indexer-key compose, 78 layers: the fp8 NSA batch with planar pages of 64 x (128-byte fp8 key + "
        "4-byte scale) = 8448 bytes, one 2^20-page pool shared by the layers")
    config = {
        "workload": workload_desc,
        "B": b.B, "T": b.T, "C": work.plan.C, "D": work.plan.D, "layers": work.num_layers,
        "page_size": b.page_size, "cp_size": b.cp_size, "row_bytes": b.row_bytes,
        "variant": work.variant,
        "consume_staging": work.consume_staging,
        "fill_mode": work.fill_mode if work.variant in ("staging", "prefetch") else None,
        "launch": "early" if work.early else "plain",
        "bytes_per_layer": work.layer_bytes,
        "dram_bytes_per_layer": work.bytes["dram_min"],
        "l2": ("L2 flushed between steps (a 512 MB write outside the per-step events)" if work.num_layers == 1
               else "inputs larger than L2: every layer reads its own pool slab and rows (%.1f GB per step)" % (
                   (sum(s.numel() for p in work.pools for s in p) + work.rows_all.numel()) / 1e9)),
        "cuda_graph": not a.no_graph,
        "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU",
    }
    small = b.page_size * b.row_bytes <= 4096  # pages moved a group of consecutive dense pages at a time
    kernel_name = {
        "gather": ("gather_groups_kernel" if small else "gather_pages_kernel") + " (cpkv_compose_gather_kinds)",
        "fused": ("compose_layer_kernel (cpkv_compose_fused_planes)" if b.planes
                  else ("compose_fused_groups_kernel" if small else "compose_fused_kernel") + " (cpkv_compose_fused)"),
        "layer": ("compose_layer_kernel (cpkv_compose_layer_planes)" if b.planes
                  else ("compose_layer_groups_kernel" if small else "compose_layer_kernel") + " (cpkv_compose_layer)")}[top]
    roofline = {
        "bound": "hbm",
        "kernel": kernel_name,
        "achieved": kroof[top]["achieved"],
        "peak": hbm_peak,
        "peak_source": peak_src,
        "unit": "GB/s",
        "frac": kroof[top]["frac"],
        "traffic": traffic,
        "algorithmic_bytes_per_launch": work.kernels[top],
        "avg_launch_ms": kroof[top]["avg_launch_ms"],
        "dram_bytes_per_launch": kroof[top]["dram_bytes_per_launch"],
        "dram_frac": kroof[top]["dram_frac"],
        "timing": kernel_timing,
        **{k: v for k, v in kroof.items() if k != top},
    }

    fr = step_fractions(work, ms_step, hbm_peak, ws)
    launches = work.launches_per_step * a.steps
    extra = None
    if not a.no_extra_configs and a.config == "traced_78" and a.layers is None and ws == 1:
        # the headline's device memory goes before the fp8 workload (52 GB) is made
        del work
        _free(torch)
        extra = extra_configs(a, device, hbm_peak)
        for k in ("fp8_nsa", "traced_78_ps1", "traced_78_ps1_layer"):
            status |= extra.get(k, {}).get("status_word", 0)

    line = {
        "metric": METRIC,
        "value": round(value_gbs, 2),
        "unit": "GB/s",
        "n_gpus": ws,
        "steps": a.steps,
        "warmup": a.warmup,
        "ms_per_step": round(ms_step, 4),
        "ms_per_step_stats": {"median": round(step_ms[len(step_ms) // 2], 4), "min": round(step_ms[0], 4),
                              "max": round(step_ms[-1], 4), "steps_timed": len(step_ms)},
        "ms_per_78_layer_compose": round(ms_step * 78 / config["layers"], 4),
        **fr,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "u8",
        "data": "synthetic",
        "config": config,
        "roofline": roofline,
        "configs": extra,
        "cpu_baseline": cpu,
        "cpu_baseline_all_cores": cpu_all,
        "e2e": e2e,
        "gpu_launches": launches,
        "clocks": clk,
        "status_word": status | st0,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()
    return 0 if (status | st0) == 0 else 3


def build_e2e(work):
    """The end-to-end step through the public API with host buffers, as one
    CUDA graph.  Every replay uploads the batch metadata and all layers'
    current rows from pinned host memory (a copy of the workload's rows taken
    now), runs the step, and reads back the status word, the ragged counts
    and the last layer's composed dense buffer (the step's result) into
    pinned host memory.  The uploads run on a copy stream, one layer at a
    time, and layer l's compose waits (an event wait) only for layer l's
    rows, so the copies overlap the compose of earlier layers.  Returns
    (one, h2d, d2h, h_dense): one() replays the graph, synchronises and raises
    on a non-zero status word; h_dense holds the last layer's dense bytes."""
    torch = work.torch
    b = work.batch
    h_meta = [torch.from_numpy(np.ascontiguousarray(x, np.int32)).pin_memory()
              for x in (b.prefix_pages, b.cur_pages, b.writer)]
    d_meta = [work.plan.d_prefix_pages, work.plan.d_cur_pages, work.plan.d_writer]
    h_rows = work.rows_all.cpu().pin_memory()
    h_out = torch.empty(1, dtype=torch.int32).pin_memory()
    h_cnt = torch.empty(2, dtype=torch.int64).pin_memory()
    last = work.dense_of(work.num_layers - 1)
    h_dense = torch.empty(last.shape, dtype=last.dtype).pin_memory()
    h2d = sum(x.numel() * x.element_size() for x in h_meta) + h_rows.numel()
    d2h = h_out.numel() * 4 + h_cnt.numel() * 8 + h_dense.numel()
    copy = torch.cuda.Stream()
    landed = [torch.cuda.Event() for _ in range(work.num_layers)]

    def body():
        cur = torch.cuda.current_stream()
        for h, d in zip(h_meta, d_meta):
            if h.numel():
                d.copy_(h, non_blocking=True)
        copy.wait_stream(cur)
        with torch.cuda.stream(copy):
            for layer in range(work.num_layers):
                work.rows_all[layer].copy_(h_rows[layer], non_blocking=True)
                landed[layer].record(copy)
        work.plan.build()
        work.cpkv.cpkv_ragged_plan_build(work.rb.prefix_lens, work.rb.q_lens, work.d_cp_index, len(work.cp_index),
                                         chunk=work.rb.chunk, k_align=work.rb.k_align, topk=work.rb.topk, out=work.ragged_out,
                                         d_counts=work.ragged_counts, d_status=work.plan.d_status)
        for layer in range(work.num_layers):
            cur.wait_event(landed[layer])
            work.run_kernel("all", layer)
        cur.wait_stream(copy)
        h_dense.copy_(last, non_blocking=True)
        h_out.copy_(work.plan.d_status, non_blocking=True)
        h_cnt.copy_(work.ragged_counts, non_blocking=True)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        body()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        body()

    def one():
        g.replay()
        torch.cuda.current_stream().synchronize()
        if int(h_out[0]) != 0:
            raise RuntimeError(f"status word {int(h_out[0])}")

    return one, h2d, d2h, h_dense


def run_e2e(work, a, ws):
    """Same metric through the public API with host buffers (build_e2e);
    the host synchronises on the result every step.  The value is the bytes
    of all timed steps over their total time; the median step is reported
    beside it."""
    one, h2d, d2h, _ = build_e2e(work)
    for _ in range(2):
        one()
    steps = max(10, a.steps // 2)
    if ws > 1:
        work.torch.distributed.barrier()
    per = []
    t0 = time.perf_counter()
    for _ in range(steps):
        s0 = time.perf_counter()
        one()
        per.append(time.perf_counter() - s0)
    el = time.perf_counter() - t0
    ms_max, units_all = aggregate(el * 1e3, work.layer_bytes * work.num_layers * steps, ws)
    return {"value": round(units_all / (ms_max / 1e3) / 1e9, 2), "unit": "GB/s", "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "ms_per_step": round(ms_max / steps, 3), "steps": steps,
            "ms_per_step_median": round(1e3 * statistics.median(per), 3),
            "ms_per_step_min": round(1e3 * min(per), 3), "ms_per_step_max": round(1e3 * max(per), 3),
            "h2d_overlapped": True,
            "result": "the last layer's dense KV buffer, the status word and the ragged counts copied to pinned "
                      "host memory every step (the other layers' dense buffers stay on the device for attention)"}


def _graph_us(torch, fn, reps, per, inner=1):
    """µs per unit of ``fn`` (``per`` units per call), from CUDA events around
    ``reps`` replays of a graph that holds ``inner`` calls back to back.  With
    inner = 1 every replay also pays the graph launch from the host; with
    more, consecutive calls follow each other on the device."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(inner):
            fn()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) * 1e3 / (reps * per * inner)


def ragged_plan_latency(reps: int, splits=("interleaved", "contiguous", "zigzag")):
    """µs per ragged index plan build of the ragged config (B=64, 131 072 q
    tokens, cp=8, topk=2048): one CUDA graph per measured set, replayed
    (``us_per_rank``: a graph holding one rank's build, so each replay also
    pays its launch from the host; ``us_all_ranks``: all 8 ranks in one graph;
    ``us_per_build_back_to_back``: 10 x all ranks in one graph, per build)."""
    import torch

    from paged_kv_cache_compose_gb300 import cpkv

    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    base = wl.ragged_batch()
    out = {}
    for split in splits:
        rb = wl.RaggedBatch(base.name, base.seed, base.cp_size, base.chunk, base.k_align, base.prefix_lens,
                            base.q_lens, split=split)
        jobs = []
        for r in range(rb.cp_size):
            ci = rb.cp_index(r)
            S, Q = cpkv.cpkv_ragged_plan_sizes(rb.q_lens, ci, rb.chunk)
            jobs.append((torch.from_numpy(ci).cuda(), len(ci), cpkv.ragged_buffers(max(S, 1), max(Q, 1)),
                         torch.zeros(2, dtype=torch.int64, device="cuda")))

        def build(js):
            for d_ci, n, buf, cnt in js:
                cpkv.cpkv_ragged_plan_build(rb.prefix_lens, rb.q_lens, d_ci, n, chunk=rb.chunk, k_align=rb.k_align,
                                            topk=rb.topk, out=buf, d_counts=cnt, d_status=status)
        per_rank = [_graph_us(torch, lambda j=j: build([j]), reps, 1) for j in jobs]
        all_ranks = _graph_us(torch, lambda: build(jobs), reps, 1)
        back_to_back = _graph_us(torch, lambda: build(jobs), reps, len(jobs), inner=10)
        out[split] = {"us_per_rank": [round(x, 2) for x in per_rank], "us_all_ranks": round(all_ranks, 2),
                      "us_per_build_back_to_back": round(back_to_back, 2),
                      "B": rb.B, "q_tokens": int(rb.q_lens.sum()), "cp": rb.cp_size, "topk": rb.topk,
                      "status_word": int(status.item())}
    return out


COMPOSE_PLAN_BATCHES = {"traced": wl.traced_batch, "traced_78_slab": wl.traced_78_layer_batch,
                        "fp8_nsa": wl.fp8_nsa_batch, "traced_78_ps1": wl.traced_78_token_pages_batch}


def compose_plan_latency(reps: int, names=tuple(COMPOSE_PLAN_BATCHES)):
    """µs per compose plan build (cpkv_plan_build: inverses over the whole
    pool, descriptors, per-token arrays): ``us`` from a graph holding one
    build (each replay also pays its launch from the host), ``us_back_to_back``
    from a graph holding 10 builds in a row."""
    import torch

    from paged_kv_cache_compose_gb300.runtime import ComposePlan

    out = {}
    for name in names:
        b = COMPOSE_PLAN_BATCHES[name]()
        plan = ComposePlan(b.prefix_lens, b.cur_lens, b.prefix_pages, b.cur_pages, b.writer, page_size=b.page_size,
                           cp_size=b.cp_size, num_pool_pages=b.num_pool_pages)
        out[name] = {"us": round(_graph_us(torch, lambda: plan.build(), reps, 1), 2),
                     "us_back_to_back": round(_graph_us(torch, lambda: plan.build(), reps, 1, inner=10), 2),
                     "B": b.B, "T": b.T,
                     "C": plan.C, "D": plan.D, "page_size": b.page_size, "num_pool_pages": b.num_pool_pages,
                     "status_word": int(plan.d_status.item())}
    return out


def run_plans(a):
    """Latency of the plan builders, one CUDA graph per measured set, launched
    back to back (µs per build includes the launch inside the graph)."""
    from paged_kv_cache_compose_gb300 import build as cpkv_build

    cpkv_build.build()
    reps = max(20, a.steps)
    out = {"metric": "plan build latency", "unit": "us per build", "n_gpus": 1, "steps": reps, "data": "synthetic",
           "higher_is_better": False, "ragged": ragged_plan_latency(reps), "compose_plan": compose_plan_latency(reps)}
    out["status_word"] = 0
    for v in list(out["ragged"].values()) + list(out["compose_plan"].values()):
        out["status_word"] |= v["status_word"]
    print(json.dumps(out), flush=True)
    return 0 if out["status_word"] == 0 else 3


def run_reference(a, ws, rank):
    """The CPU oracle as the reference arm: each step is a bounded sample
    (plan, ragged plan and ``--cpu-layers`` layers of staging + gather)."""
    if rank != 0:
        return 0
    import oracle

    oracle.build()
    batch = wl.CONFIGS[a.config]()
    n = min(a.cpu_layers, batch.num_layers)
    b, pools, rows = oracle_sample(batch, n, shared_pool=a.config in ("fp8_nsa", "index_k"))
    lib = oracle.load()
    for _ in range(a.warmup):
        oracle_step(b, pools, rows, lib)
    t0 = time.perf_counter()
    moved = 0
    for _ in range(a.steps):
        moved += oracle_step(b, pools, rows, lib)
    el = time.perf_counter() - t0
    gbs = moved / el / 1e9
    ms_step = el * 1e3 / a.steps
    sample = (f"plan + ragged plan + {n} of {batch.num_layers} layers (staging + gather) per step, "
              f"host-generated inputs of the same batch, single-threaded C oracle")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 3), "unit": "GB/s", "n_gpus": ws,
        "steps": a.steps, "warmup": a.warmup, "ms_per_step": round(ms_step, 3),
        "ms_per_78_layer_compose": round(ms_step * 78 / n, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "u8", "data": "synthetic",
        "config": {"workload": a.config, "sampled_layers": n, "B": b.B, "T": b.T},
        "cpu_baseline": {"value": round(gbs, 3), "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(gbs, 3), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
