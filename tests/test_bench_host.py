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


def test_layer_bytes_hand_counted():
    """ps=4, R=16, prefix [4, 0], current [3, 5], dense_cap 5: T=8 rows, 4 pad
    rows (1 + 3), D=4 pages (1 prefix + 1 + 2 current)."""
    lb = bench.layer_bytes([4, 0], [3, 5], 4, 16, 5)
    assert (lb["T"], lb["D"], lb["pad_rows"]) == (8, 4, 4)
    assert lb["fill"] == 8 * 16 + 12 * 16
    assert lb["gather"] == 4 * 4 * 16 + 5 * 4 * 16
    assert lb["total"] == 896
    assert lb["layer"] == 896 - 4 * 16      # pad rows zeroed in the dense page, not read back
    assert lb["fused"] == 8 * 16 + 4 * 16 + 5 * 4 * 16


def test_layer_bytes_planar_unstaged_planes():
    """Planes (128, 4) at ps=4: the 4-byte scale plane is not staged; planes
    (16, 4, 16) at ps=3: the third plane starts at byte 60, not staged."""
    lb = bench.layer_bytes([4, 0], [3, 5], 4, 132, 5, planes=(128, 4))
    assert lb["layer"] == lb["total"] - 4 * 132 - 8 * 4
    lb = bench.layer_bytes([3], [4], 3, 36, 3, planes=(16, 4, 16))
    # T=4, pad=2; plane offsets 0, 48, 60: planes 2 (width 4) and 3 (offset 60) unstaged
    assert lb["layer"] == lb["total"] - 2 * 36 - 4 * (4 + 16)


def test_pool_pages_only_for_shared_pool_workloads():
    with pytest.raises(ValueError):
        bench.ComposeWorkload("traced_78", device="cpu", pool_pages=4096)


def test_all_cores_oracle_baseline_runs_and_aggregates():
    got, why = bench.time_oracle_all_cores("tiny", 1, seconds=0.3, workers=2)
    assert why is None
    gbs, procs, secs, steps = got
    assert procs == 2 and gbs > 0 and secs >= 0.3 and steps >= 2


def test_all_cores_oracle_baseline_reports_a_failed_worker():
    got, why = bench.time_oracle_all_cores("no such workload", 1, seconds=0.1, workers=2)
    assert got is None and "KeyError" in why


def test_reference_arm_prints_the_contract_line():
    """`bench.py --impl reference` (the CPU oracle arm) runs without a GPU and
    prints one JSON line with the keys the contract asks for."""
    import json
    import subprocess
    import sys

    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--config", "traced", "--steps", "1",
                          "--cpu-layers", "1"], cwd=bench.ROOT, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC and line["unit"] == "GB/s"
    assert line["value"] > 0 and line["higher_is_better"] is True and line["warmup"] >= 3
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] == 1
    assert line["e2e"] == {"value": line["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
