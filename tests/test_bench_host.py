"""Host-side pieces of the benchmark (CPU only)."""
import numpy as np
import pytest

import bench
import oracle
import oracle_pins as pins
import workloads as wl


@pytest.mark.parametrize("batch", [b for b in pins.edge_batches() if b.B > 0], ids=lambda b: b.name)
def test_compact_pool_leaves_the_dense_kv_unchanged(batch):
    """Relabelling prefix pages onto a compact pool (owner kept) gives the
    oracle byte-identical dense KV."""
    slabs = wl.host_pool(batch)
    rows = wl.host_current_rows(batch)
    full = oracle.compose_dense(batch.prefix_lens, batch.cur_lens, batch.prefix_pages, slabs, rows,
                                page_size=batch.page_size, cp_size=batch.cp_size)
    nb, compact = bench.compact_pool(batch, slabs)
    got = oracle.compose_dense(nb.prefix_lens, nb.cur_lens, nb.prefix_pages, compact, rows,
                               page_size=batch.page_size, cp_size=batch.cp_size)
    assert np.array_equal(full, got)
    assert all(s.shape[0] <= batch.slab_pages + 1 for s in compact)
    plan = oracle.compose_plan(nb.prefix_lens, nb.cur_lens, nb.prefix_pages, nb.cur_pages, nb.writer,
                               page_size=nb.page_size, cp_size=nb.cp_size, num_pool_pages=nb.num_pool_pages)
    assert plan["status"] == 0


def test_oracle_step_counts_bytes():
    b = wl.tiny_batch()
    nb, pools, rows = bench.oracle_sample(b, 2)
    moved = bench.oracle_step(nb, pools, rows)
    lb = bench.layer_bytes(b.prefix_lens, b.cur_lens, b.page_size, b.row_bytes,
                           oracle.sizes(b.prefix_lens, b.cur_lens, b.page_size)[2])
    assert moved == 2 * lb["total"]


def test_read_peaks_fallback(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.read_peaks()[:2] == (bench.FALLBACK_HBM_GBS, "fallback")
    (tmp_path / "MEASURED_PEAKS.json").write_text('{"hbm_gbs": 7100.5, "bf16_tflops": 1900}')
    assert bench.read_peaks()[:2] == (7100.5, "measured")
