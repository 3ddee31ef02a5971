"""Full-size parity in the benchmark's launch configuration.

The benchmark's own workload object (same inputs, same CUDA-graph replay of
plan + ragged plan + 78 x (fill + gather)) is run once, then whole dense
layers and stagings are compared byte for byte with the oracle.  The oracle
receives a pool compacted to the pages the batch references (page ids
relabelled with their owner kept), which leaves every output byte unchanged.
"""
import gc

import numpy as np
import pytest
import torch

import bench
import oracle
import workloads as wl

pytestmark = pytest.mark.gpu


def _batch_order_rows(batch, rows_per_writer):
    tw = wl.token_writer(batch)
    g = np.empty((batch.T, batch.row_bytes), np.uint8)
    for w in range(batch.cp_size):
        g[tw == w] = rows_per_writer[w].cpu().numpy()
    return g


_COMPACT = {}


def _compact(work, layer):
    """The layer's pool compacted to the referenced pages (cached for a pool
    that all layers share)."""
    if not work.shared_pool:
        return bench.compact_pool(work.batch, work.pools_of(layer))
    key = id(work)
    if key not in _COMPACT:
        _COMPACT.clear()
        _COMPACT[key] = bench.compact_pool(work.batch, work.pools_of(layer))
    return _COMPACT[key]


def _check_layer(work, layer, got=None):
    """Layer ``layer``'s dense buffer (or the host copy ``got``) against the
    oracle's definition; returns the batch-ordered rows of row-major pages."""
    b = work.batch
    nb, slabs = _compact(work, layer)
    if b.planes:
        tw = wl.token_writer(b)
        planes = []
        for p, wp in enumerate(b.planes):
            g = np.empty((b.T, wp), np.uint8)
            for w in range(b.cp_size):
                g[tw == w] = work.rows[layer][p][w].cpu().numpy()
            planes.append(g)
        want = oracle.compose_dense_planes(nb.prefix_lens, nb.cur_lens, nb.prefix_pages,
                                           [s.reshape(s.shape[0], -1) for s in slabs], planes,
                                           page_size=b.page_size, cp_size=b.cp_size, plane_bytes=list(b.planes),
                                           dense_cap=work.plan.dense_cap_pages)
        got = (work.dense_of(layer) if got is None else got).cpu().numpy().reshape(work.plan.dense_cap_pages, -1)
        assert np.array_equal(got, want), f"layer {layer}"
        return None
    g = _batch_order_rows(b, work.rows[layer])
    want = oracle.compose_dense(nb.prefix_lens, nb.cur_lens, nb.prefix_pages, slabs, g, page_size=b.page_size,
                                cp_size=b.cp_size, dense_cap=work.plan.dense_cap_pages)
    got = (work.dense_of(layer) if got is None else got).cpu().numpy()
    assert np.array_equal(got, want), f"layer {layer}"
    return g


def _check_staging(work, g):
    b = work.batch
    stg = [s.cpu().numpy() for s in work.layers.staging]
    want = [s.copy() for s in stg]  # undefined pages: whatever is there
    oracle.staging(b.cur_lens, b.writer, g, want, page_size=b.page_size, cp_size=b.cp_size)
    for w in range(b.cp_size):
        assert np.array_equal(stg[w], want[w]), w


def _check_plan(work):
    b = work.batch
    want = oracle.compose_plan(b.prefix_lens, b.cur_lens, b.prefix_pages, b.cur_pages, b.writer,
                               page_size=b.page_size, cp_size=b.cp_size, num_pool_pages=b.num_pool_pages,
                               dense_cap=work.plan.dense_cap_pages)
    for k in ("owner", "src", "page_inverse", "staging_page_inverse", "mixed_locs", "staging_rows",
              "token_writer_row", "prefix_spans", "cur_spans"):
        assert np.array_equal(work.plan[k].cpu().numpy().reshape(want[k].shape), want[k]), k
    rb = work.rb
    wr = oracle.ragged_plan(rb.prefix_lens, rb.q_lens, work.cp_index, chunk=rb.chunk, k_align=rb.k_align)
    assert work.ragged_counts.cpu().tolist() == [wr["S"], wr["Q"]]
    for k in ("seg_req", "kv_lens", "q_starts", "q_lens", "k_bases", "q_bases", "current_bases"):
        assert np.array_equal(work.ragged_out[k].cpu().numpy()[:wr["S"]], wr[k]), k
    assert np.array_equal(work.ragged_out["topk_offsets"].cpu().numpy()[:wr["Q"]], wr["topk_offsets"])


@pytest.mark.parametrize("config,variant", [("traced_78", "staging"), ("fp8_nsa", "staging"),
                                            ("traced_78", "fused"), ("fp8_nsa", "fused"),
                                            ("traced_78", "prefetch"), ("index_k", "staging"),
                                            ("traced_78", "layer"), ("fp8_nsa", "layer"), ("index_k", "layer"),
                                            ("index_k", "fused"), ("traced_78", "staging-consume"),
                                            ("fp8_nsa", "staging-consume"), ("traced_78", "layer-consume"),
                                            ("index_k", "layer-consume"), ("traced_78_ps1", "staging"),
                                            ("traced_78_ps1", "fused"), ("traced_78_ps1", "staging-consume"),
                                            ("traced_78_ps1", "layer"), ("traced_78_ps1", "layer-consume")])
def test_benchmark_workload_matches_oracle(config, variant):
    consume = variant.endswith("-consume")  # plain variants keep their stagings, which are checked
    variant = variant.removesuffix("-consume")
    work = bench.ComposeWorkload(config, variant=variant, consume_staging=consume)
    try:
        for d in work.layers.dense:
            d.fill_(0xCD)
        work.capture()  # warm-up step + capture, as the benchmark does
        for d in work.layers.dense:
            d.fill_(0xCD)
        work.run()
        torch.cuda.synchronize()
        assert work.status() == 0
        _check_plan(work)
        _check_layer(work, work.num_layers - 2)
        g = _check_layer(work, work.num_layers - 1)
        if variant in ("staging", "prefetch", "layer") and g is not None and not consume:
            _check_staging(work, g)
    finally:
        _COMPACT.clear()
        del work
        gc.collect()
        torch.cuda.empty_cache()


@pytest.mark.parametrize("config,variant,early", [
    ("traced_78", "staging-consume", True), ("traced_78", "staging-consume", False), ("traced_78", "staging", True),
    ("traced_78", "fused", True), ("traced_78", "layer-consume", True), ("fp8_nsa", "staging-consume", True),
    ("traced_78_ps1", "layer-consume", True), ("traced_78_ps1", "fused", True)])
def test_every_layer_of_the_78_layer_graph_matches_oracle(config, variant, early):
    """The benchmark's 78-layer step over the traced batch, replayed from its
    CUDA graph, with one dense buffer per layer so that every layer's output
    survives the step: all 78 dense layers byte-exact against the oracle.
    With early launches (the benchmark's form) a layer's fill starts behind
    the previous layer's gather and its gather behind the fill; a store that
    ran ahead of its predecessor in any layer would show up here."""
    consume = variant.endswith("-consume")
    variant = variant.removesuffix("-consume")
    work = bench.ComposeWorkload(config, variant=variant, consume_staging=consume, num_dense=78, early=early)
    try:
        for d in work.layers.dense:
            d.fill_(0xCD)
        work.capture()
        for d in work.layers.dense:
            d.fill_(0xCD)
        work.run()
        torch.cuda.synchronize()
        assert work.status() == 0
        _check_plan(work)
        for layer in range(work.num_layers):
            _check_layer(work, layer)
    finally:
        _COMPACT.clear()
        del work
        gc.collect()
        torch.cuda.empty_cache()


@pytest.mark.parametrize("variant", ["staging", "fused", "layer"])
def test_end_to_end_graph_matches_oracle(variant):
    """The end-to-end step (rows uploaded from pinned host memory on a copy
    stream, each layer joined to its upload by an event wait, fills and
    one-launch composes launched early behind the previous kernel, the last
    layer's dense buffer read back to pinned host memory).  One dense buffer
    per layer, so every layer is checked.  The device rows are poisoned first,
    so a compose that read its rows before their upload landed would differ
    from the oracle."""
    work = bench.ComposeWorkload("traced_78", variant=variant, consume_staging=variant != "fused", num_dense=78)
    try:
        one, h2d, d2h, h_dense = bench.build_e2e(work)
        dense_bytes = work.dense_of(work.num_layers - 1).numel()
        assert h2d >= work.rows_all.numel() and d2h == 20 + dense_bytes
        work.rows_all.fill_(0xEE)
        for d in work.layers.dense:
            d.fill_(0xCD)
        h_dense.fill_(0xAB)
        one()
        assert work.status() == 0
        _check_plan(work)
        for layer in range(work.num_layers):
            _check_layer(work, layer)
        _check_layer(work, work.num_layers - 1, got=h_dense)
    finally:
        _COMPACT.clear()
        del work
        gc.collect()
        torch.cuda.empty_cache()


def test_traced_single_layer_full_pool():
    """The traced batch against its 200 000-page pool (one layer)."""
    from paged_kv_cache_compose_gb300.runtime import ComposeLayers, ComposePlan

    b = wl.traced_batch()
    plan = ComposePlan(b.prefix_lens, b.cur_lens, b.prefix_pages, b.cur_pages, b.writer, page_size=b.page_size,
                       cp_size=b.cp_size, num_pool_pages=b.num_pool_pages, dense_cap_pages=None)
    plan.build()
    layers = ComposeLayers(plan, b.row_bytes)
    pools = wl.device_pool(b, 0)
    g_dev = wl.device_current_rows(b, 0)
    rows = wl.device_split_rows_by_writer(b, g_dev)
    dense = layers.compose_layer(0, pools, rows)
    torch.cuda.synchronize()
    assert int(plan.d_status.item()) == 0
    nb, slabs = bench.compact_pool(b, pools)
    want = oracle.compose_dense(nb.prefix_lens, nb.cur_lens, nb.prefix_pages, slabs, g_dev.cpu().numpy(),
                                page_size=b.page_size, cp_size=b.cp_size)
    assert np.array_equal(dense.cpu().numpy(), want)
    del pools, rows, g_dev, layers, plan
    gc.collect()
    torch.cuda.empty_cache()
