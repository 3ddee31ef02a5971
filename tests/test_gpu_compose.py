"""GPU parity of the compose path (plan, fill, gather) against the CPU oracle.

Every comparison is byte-exact (tolerance 0: the path is integer indexing and
byte copies).  Inputs are the seeded generators of ``workloads``; expected
values come only from ``oracle``.  All calls go through the C ABI binding.
"""
import numpy as np
import pytest
import torch

import oracle
import oracle_pins as pins
import workloads as wl
from paged_kv_cache_compose_gb300 import cpkv
from paged_kv_cache_compose_gb300.runtime import ComposeLayers, ComposePlan

pytestmark = pytest.mark.gpu

PLAN_KEYS = ("prefix_spans", "cur_spans", "owner", "src", "page_inverse", "staging_page_inverse", "mixed_locs",
             "staging_rows", "token_writer_row")


def _plan_pair(batch, dense_extra=0):
    T, C, D = oracle.sizes(batch.prefix_lens, batch.cur_lens, batch.page_size)
    cap = D + dense_extra
    want = oracle.compose_plan(batch.prefix_lens, batch.cur_lens, batch.prefix_pages, batch.cur_pages, batch.writer,
                               page_size=batch.page_size, cp_size=batch.cp_size,
                               num_pool_pages=batch.num_pool_pages, dense_cap=cap)
    plan = ComposePlan(batch.prefix_lens, batch.cur_lens, batch.prefix_pages, batch.cur_pages, batch.writer,
                       page_size=batch.page_size, cp_size=batch.cp_size, num_pool_pages=batch.num_pool_pages,
                       dense_cap_pages=cap)
    # poison outputs so that unwritten entries show up
    for t in plan.bufs.values():
        if t.numel():
            t.fill_(-7)
    plan.build()
    torch.cuda.synchronize()
    return plan, want


def _assert_plan_equal(plan, want):
    assert int(plan.d_status.item()) == want["status"] == 0
    for k in PLAN_KEYS:
        got = plan[k].cpu().numpy()
        assert got.dtype == want[k].dtype, k
        assert np.array_equal(got.reshape(want[k].shape), want[k]), k


@pytest.mark.parametrize("batch", pins.edge_batches(), ids=lambda b: b.name)
def test_plan_matches_oracle_edge_cases(batch):
    plan, want = _plan_pair(batch, dense_extra=3)
    _assert_plan_equal(plan, want)


def test_plan_matches_oracle_traced_full_size():
    plan, want = _plan_pair(wl.traced_batch(), dense_extra=0)
    _assert_plan_equal(plan, want)


def test_plan_matches_oracle_fp8_full_size():
    plan, want = _plan_pair(wl.fp8_nsa_batch(), dense_extra=5)
    _assert_plan_equal(plan, want)


def _many_pages_batch(name, seed, ps, cp, B, cur_hi, writers="random"):
    rng = np.random.default_rng(seed)
    cur = rng.integers(1, cur_hi, B)
    pfx = (rng.integers(0, 4 * cur_hi, B) // ps) * ps
    C = int(((cur + ps - 1) // ps).sum())
    writer = rng.integers(0, cp, C) if writers == "random" else None
    P = int((pfx // ps).sum() + C + 10)
    return wl.make_compose_batch(name, seed, page_size=ps, cp_size=cp, num_pool_pages=P, row_bytes=16,
                                 prefix_lens=pfx, cur_lens=cur, writer=writer, row_kind="bytes", rng=rng)


def _exact_pages_batch(C, ps=1, cp=5, seed=9):
    """A batch of exactly C current pages (the workspace threshold sits at 4096)."""
    rng = np.random.default_rng(seed)
    cur = np.full(4, (C // 4) * ps)
    cur[0] += (C - int(cur.sum()) // ps) * ps
    return wl.make_compose_batch(f"C{C}", seed, page_size=ps, cp_size=cp, num_pool_pages=C + 64, row_bytes=16,
                                 prefix_lens=np.array([0, ps, 0, 2 * ps]), cur_lens=cur,
                                 writer=rng.integers(0, cp, C), row_kind="bytes", rng=rng)


@pytest.mark.parametrize("batch", [
    _exact_pages_batch(4096), _exact_pages_batch(4097), _exact_pages_batch(5000, ps=2),
    _many_pages_batch("ps1-random", 31, 1, 8, 12, 7000),
    _many_pages_batch("ps3-random", 32, 3, 7, 40, 2000),
    _many_pages_batch("ps16-b300", 33, 16, 5, 300, 600),
    _many_pages_batch("ps1-b1000-rr", 34, 1, 12, 1000, 60, writers="round-robin"),
], ids=lambda b: b.name)
def test_plan_matches_oracle_many_current_pages(batch):
    """Batches of thousands of current pages in many token blocks: per-writer
    row bases from per-block totals in the workspace (random and round-robin
    writers, partial pages, blocks of 1024 one-token pages, the B > 64
    parameter block)."""
    plan, want = _plan_pair(batch, dense_extra=2)
    _assert_plan_equal(plan, want)


def test_plan_large_batch_template():
    """B > 64 takes the 1024-request parameter block."""
    rng = np.random.default_rng(5)
    B, ps = 300, 16
    batch = wl.make_compose_batch("b300", 5, page_size=ps, cp_size=5, num_pool_pages=20000, row_bytes=64,
                                  prefix_lens=(rng.integers(0, 100, B) // ps) * ps, cur_lens=rng.integers(0, 70, B),
                                  writer=None, row_kind="bytes")
    plan, want = _plan_pair(batch, dense_extra=1)
    _assert_plan_equal(plan, want)


def _run_compose(batch, dense_extra=1, guard=0xA5, num_layers=1, page_runs=True):
    """Plan + fill + gather on the GPU with host-generated inputs; returns
    (dense [host], staging list [host], plan, slabs, rows) for the last layer.
    ``page_runs``: the fill moves pages as runs (pages of 4 KB and more) or
    takes the row-by-row index copy."""
    plan, want = _plan_pair(batch, dense_extra)
    _assert_plan_equal(plan, want)
    layers = ComposeLayers(plan, batch.row_bytes)
    for s in layers.staging:
        s.fill_(guard)
    for d in layers.dense:
        d.fill_(0xCD)
    out = None
    for layer in range(num_layers):
        slabs = wl.host_pool(batch, layer)
        rows = wl.host_current_rows(batch, layer)
        d_slabs = [torch.from_numpy(s).cuda() for s in slabs]
        d_rows = [torch.from_numpy(r).cuda() for r in wl.split_rows_by_writer(batch, rows)]
        dense = layers.compose_layer(layer, d_slabs, d_rows, page_runs=page_runs)
        out = (dense, slabs, rows)
    torch.cuda.synchronize()
    assert int(plan.d_status.item()) == 0
    dense, slabs, rows = out
    return dense.cpu().numpy(), [s.cpu().numpy() for s in layers.staging], plan, slabs, rows


@pytest.mark.parametrize("page_runs", [True, False], ids=["page-runs", "rows"])
@pytest.mark.parametrize("batch", pins.edge_batches(), ids=lambda b: b.name)
def test_compose_matches_oracle_edge_cases(batch, page_runs):
    dense, staging, plan, slabs, rows = _run_compose(batch, dense_extra=2, page_runs=page_runs)
    want = oracle.compose_dense(batch.prefix_lens, batch.cur_lens, batch.prefix_pages, slabs, rows,
                                page_size=batch.page_size, cp_size=batch.cp_size, dense_cap=plan.dense_cap_pages)
    assert np.array_equal(dense, want)
    # staging: defined pages equal the oracle's, every other page keeps its guard bytes
    ps, R = batch.page_size, batch.row_bytes
    stg_want = [np.full_like(s, 0xA5) for s in staging]
    oracle.staging(batch.cur_lens, batch.writer, rows, stg_want, page_size=ps, cp_size=batch.cp_size)
    for w in range(batch.cp_size):
        assert np.array_equal(staging[w], stg_want[w]), w


@pytest.mark.parametrize("ps,R", [(64, 656), (5, 1024), (64, 64), (16, 1152), (4, 1152), (3, 1152), (128, 48),
                                  (2, 4096), (1, 8192)])
def test_page_run_fill_geometries(ps, R):
    """The page-run fill on pages of one, several and partial 4 KB chunks
    (41 984-byte fp8 pages end in a 1024-byte chunk; 5 x 1024 = 4 KB + 1 KB;
    exactly one chunk; 18 chunks; one-token pages of 4 and 8 KB) and below
    one chunk (the row fill), three layers each with short pages: stagings
    (guard bytes elsewhere) and dense against the oracle."""
    rng = np.random.default_rng(ps * 7 + R)
    B = 9
    pfx = (rng.integers(0, 6 * ps, B) // ps) * ps
    cur = rng.integers(1, 5 * ps + 3, B)
    batch = wl.make_compose_batch("geo-runs", 53, page_size=ps, cp_size=3, num_pool_pages=400, row_bytes=R,
                                  prefix_lens=pfx, cur_lens=cur, row_kind="bytes")
    dense, staging, plan, slabs, rows = _run_compose(batch, dense_extra=1, num_layers=3)
    want = oracle.compose_dense(batch.prefix_lens, batch.cur_lens, batch.prefix_pages, slabs, rows,
                                page_size=ps, cp_size=batch.cp_size, dense_cap=plan.dense_cap_pages)
    assert np.array_equal(dense, want)
    stg_want = [np.full_like(s, 0xA5) for s in staging]
    oracle.staging(batch.cur_lens, batch.writer, rows, stg_want, page_size=ps, cp_size=batch.cp_size)
    for w in range(batch.cp_size):
        assert np.array_equal(staging[w], stg_want[w]), w


def test_page_run_fill_flags_indices_that_are_not_runs():
    """With FILL_PAGE_RUNS, a page whose source rows are reversed, or whose
    first staging row is moved, breaks the promised run: that page raises
    ROW_OOB and keeps its guard bytes; every other page is filled."""
    batch = wl.make_compose_batch("runs-check", 57, page_size=8, cp_size=4, num_pool_pages=64, row_bytes=1152,
                                  prefix_lens=np.array([16, 0]), cur_lens=np.array([20, 13]), row_kind="bytes")
    ps, R = batch.page_size, batch.row_bytes
    plan, _ = _plan_pair(batch)
    layers = ComposeLayers(plan, R)
    rows = wl.host_current_rows(batch, 0)
    d_rows = [torch.from_numpy(r).cuda() for r in wl.split_rows_by_writer(batch, rows)]
    tw = plan["token_writer_row"].cpu().numpy().copy()
    sr = plan["staging_rows"].cpu().numpy().copy()
    assert plan.C >= 3 and ps * R >= 4096
    tw[0:ps] = tw[0:ps][::-1]  # page 0: reversed source rows
    sr[ps] += 1                 # page 1: first staging row moved
    for s_ in layers.staging:
        s_.fill_(0xA5)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    cpkv.cpkv_fill_current(plan.cur_lens, d_rows, layers.staging, page_size=ps, cp_size=plan.cp_size, row_bytes=R,
                           staging_cap_pages=plan.staging_cap_pages, d_staging_rows=torch.from_numpy(sr).cuda(),
                           d_token_writer_row=torch.from_numpy(tw).cuda(), d_writer=plan.d_writer,
                           num_cur_pages=plan.C, d_status=status, page_runs=True)
    torch.cuda.synchronize()
    assert int(status.item()) == cpkv.STATUS_ROW_OOB
    stg_want = [np.full(((plan.C + 1) * ps, R), 0xA5, np.uint8) for _ in range(plan.cp_size)]
    oracle.staging(batch.cur_lens, batch.writer, rows, stg_want, page_size=ps, cp_size=plan.cp_size)
    for i in (0, 1):  # the broken pages keep their guard bytes
        w = int(batch.writer[i])
        stg_want[w][(i + 1) * ps:(i + 2) * ps] = 0xA5
    for w in range(plan.cp_size):
        assert np.array_equal(layers.staging[w].cpu().numpy(), stg_want[w]), w


def test_compose_tiny_78_layers():
    """The tiny batch through 78 layers with distinct pools and rows; the two
    parity buffers hold layers 76 and 77."""
    batch = wl.tiny_batch()
    batch.num_layers = 78
    plan, want = _plan_pair(batch, dense_extra=1)
    layers = ComposeLayers(plan, batch.row_bytes)
    kept = {}
    for layer in range(78):
        slabs = wl.host_pool(batch, layer)
        rows = wl.host_current_rows(batch, layer)
        d_slabs = [torch.from_numpy(s).cuda() for s in slabs]
        d_rows = [torch.from_numpy(r).cuda() for r in wl.split_rows_by_writer(batch, rows)]
        layers.compose_layer(layer, d_slabs, d_rows)
        if layer >= 76:
            kept[layer] = (slabs, rows)
    torch.cuda.synchronize()
    assert int(plan.d_status.item()) == 0
    for layer in (76, 77):
        slabs, rows = kept[layer]
        want_dense = oracle.compose_dense(batch.prefix_lens, batch.cur_lens, batch.prefix_pages, slabs, rows,
                                          page_size=batch.page_size, cp_size=batch.cp_size,
                                          dense_cap=plan.dense_cap_pages)
        assert np.array_equal(layers.dense[layer % 2].cpu().numpy(), want_dense), layer


def test_gather_random_descriptors_and_sentinels():
    rng = np.random.default_rng(9)
    ps, R, cp = 8, 1152, 3
    caps = [int(x) for x in rng.integers(4, 40, size=2 * cp)]
    host_tbl = [np.frombuffer(rng.bytes(c * ps * R), np.uint8).copy() for c in caps]
    n = 500
    owner = rng.integers(-1, 2 * cp, size=n).astype(np.int32)
    src = np.array([rng.integers(0, caps[o]) if o >= 0 else 0 for o in owner], np.int32)
    # a few invalid descriptors
    owner[7], src[7] = 2 * cp, 0
    owner[11], src[11] = 1, caps[1]
    owner[13], src[13] = -3, 0
    want, st = oracle.gather(host_tbl, caps, owner, src, page_size=ps, row_bytes=R, dense_cap=n)
    assert st == oracle.DESC_OOB
    d_tbl = [torch.from_numpy(t).cuda() for t in host_tbl]
    dense = torch.full((n * ps, R), 0xCD, dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    cpkv.cpkv_compose_gather(d_tbl, caps, torch.from_numpy(owner).cuda(), torch.from_numpy(src).cuda(), dense,
                             page_size=ps, cp_size=cp, row_bytes=R, dense_cap_pages=n, d_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == cpkv.STATUS_DESC_OOB
    assert np.array_equal(dense.cpu().numpy(), want)


@pytest.mark.parametrize("ps,R", [(64, 656), (16, 1152), (1, 16), (3, 48), (128, 1152), (64, 4096),
                                  (1, 1152), (2, 2048), (1, 4096), (5, 64)])
def test_gather_page_geometries(ps, R):
    """Pages that split into one or several bulk-copy pieces, odd page sizes,
    and the 656-byte fp8 row; pages of at most 4 KB in groups (7 of 1152 B,
    2 of 4096 B, 25 of 320 B, 32 of 16 B)."""
    rng = np.random.default_rng(ps * 1000 + R)
    cp = 2
    caps = [9, 7, 5, 6]
    host_tbl = [np.frombuffer(rng.bytes(c * ps * R), np.uint8).copy() for c in caps]
    n = 41
    owner = rng.integers(-1, 2 * cp, size=n).astype(np.int32)
    src = np.array([rng.integers(0, caps[o]) if o >= 0 else 0 for o in owner], np.int32)
    want, _ = oracle.gather(host_tbl, caps, owner, src, page_size=ps, row_bytes=R, dense_cap=n)
    d_tbl = [torch.from_numpy(t).cuda() for t in host_tbl]
    dense = torch.full((n * ps, R), 0xCD, dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    cpkv.cpkv_compose_gather(d_tbl, caps, torch.from_numpy(owner).cuda(), torch.from_numpy(src).cuda(), dense,
                             page_size=ps, cp_size=cp, row_bytes=R, dense_cap_pages=n, d_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.array_equal(dense.cpu().numpy(), want)


@pytest.mark.parametrize("case", ["dup_current", "current_in_prefix", "page_oob", "writer_oob", "page_zero"])
def test_plan_status_matches_oracle(case):
    mk = dict(page_size=4, cp_size=2, num_pool_pages=32)
    if case == "dup_current":
        args = ([0, 0], [3, 4], [], [5, 5], [0, 1])
    elif case == "current_in_prefix":
        args = ([4, 0], [3, 4], [6], [9, 6], [0, 1])
    elif case == "page_oob":
        args = ([4, 0], [3, 4], [40], [9, 6], [0, 1])
    elif case == "writer_oob":
        args = ([4, 0], [3, 4], [3], [9, 6], [0, 5])
    else:
        args = ([4, 0], [3, 4], [0], [9, 6], [0, 1])
    want = oracle.compose_plan(*args, **mk)
    plan = ComposePlan(*args, page_size=4, cp_size=2, num_pool_pages=32)
    plan.build()
    torch.cuda.synchronize()
    assert want["status"] != 0
    assert int(plan.d_status.item()) == want["status"]
    # descriptors agree too (the offending slot gets owner -1)
    assert np.array_equal(plan["owner"].cpu().numpy(), want["owner"])


def test_fill_row_out_of_range_is_skipped_and_flagged():
    batch = wl.tiny_batch()
    plan, _ = _plan_pair(batch)
    layers = ComposeLayers(plan, batch.row_bytes)
    rows = wl.host_current_rows(batch)
    d_rows = [torch.from_numpy(r).cuda() for r in wl.split_rows_by_writer(batch, rows)]
    # writer 0's buffer claims one row fewer than it holds -> its last token is out of range
    caps = [d_rows[0].shape[0] - 1, d_rows[1].shape[0]]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    cpkv.cpkv_fill_current(batch.cur_lens, d_rows, layers.staging, page_size=batch.page_size,
                           cp_size=batch.cp_size, row_bytes=batch.row_bytes, staging_cap_pages=plan.staging_cap_pages,
                           d_staging_rows=plan["staging_rows"], d_token_writer_row=plan["token_writer_row"],
                           d_writer=plan.d_writer, num_cur_pages=plan.C, d_status=status, cur_rows_cap=caps)
    torch.cuda.synchronize()
    assert int(status.item()) == cpkv.STATUS_ROW_OOB


def test_host_argument_errors_raise():
    batch = wl.tiny_batch()
    plan, _ = _plan_pair(batch)
    with pytest.raises(cpkv.CpkvError) as e:
        cpkv.cpkv_compose_gather([None] * 4, [1, 1, 1, 1], plan["owner"], plan["src"],
                                 torch.empty(plan.dense_cap_pages * 16, 1152, dtype=torch.uint8, device="cuda"),
                                 page_size=16, cp_size=2, row_bytes=1152, dense_cap_pages=plan.dense_cap_pages,
                                 d_status=plan.d_status)
    assert e.value.code == cpkv.CPKV_ERR_ARG
    with pytest.raises(cpkv.CpkvError) as e:
        cpkv.cpkv_fill_current(batch.cur_lens, [None, None], [None, None], page_size=16, cp_size=2, row_bytes=1000,
                               staging_cap_pages=10, d_staging_rows=None, d_token_writer_row=None, d_writer=None,
                               num_cur_pages=plan.C, d_status=plan.d_status, cur_rows_cap=[0, 0])
    assert e.value.code == cpkv.CPKV_ERR_ARG
    layers = ComposeLayers(plan, batch.row_bytes)
    with pytest.raises(cpkv.CpkvError) as e:
        cpkv.cpkv_fill_current(batch.cur_lens, [None, None], layers.staging, page_size=16, cp_size=2,
                               row_bytes=1152, staging_cap_pages=plan.C, d_staging_rows=plan["staging_rows"],
                               d_token_writer_row=plan["token_writer_row"], d_writer=plan.d_writer,
                               num_cur_pages=plan.C, d_status=plan.d_status, cur_rows_cap=[0, 0])
    assert e.value.code == cpkv.CPKV_ERR_CAPACITY


# ---------------------------------------------------------------------------
# fused single-GPU compose (no staging round trip): same output as fill + gather
# ---------------------------------------------------------------------------

def _run_fused(batch, dense_extra=2, layer=0, early=False):
    plan, want = _plan_pair(batch, dense_extra)
    layers = ComposeLayers(plan, batch.row_bytes)
    slabs = wl.host_pool(batch, layer)
    rows = wl.host_current_rows(batch, layer)
    d_slabs = [torch.from_numpy(s).cuda() for s in slabs]
    d_rows = [torch.from_numpy(r).cuda() for r in wl.split_rows_by_writer(batch, rows)]
    dense = torch.full((plan.dense_cap_pages * batch.page_size, batch.row_bytes), 0xCD, dtype=torch.uint8,
                       device="cuda")
    layers.compose_fused(d_slabs, d_rows, dense, early_inputs=early)
    if early:  # a second, dependent launch right behind the first (its inputs were complete before either)
        layers.compose_fused(d_slabs, d_rows, dense, early_inputs=True)
    torch.cuda.synchronize()
    assert int(plan.d_status.item()) == 0
    return dense.cpu().numpy(), plan, slabs, rows


@pytest.mark.parametrize("early", [False, True], ids=["plain", "early-inputs"])
@pytest.mark.parametrize("batch", pins.edge_batches(), ids=lambda b: b.name)
def test_fused_matches_oracle_edge_cases(batch, early):
    dense, plan, slabs, rows = _run_fused(batch, early=early)
    want = oracle.compose_dense(batch.prefix_lens, batch.cur_lens, batch.prefix_pages, slabs, rows,
                                page_size=batch.page_size, cp_size=batch.cp_size, dense_cap=plan.dense_cap_pages)
    assert np.array_equal(dense, want)


@pytest.mark.parametrize("ps,R", [(64, 656), (16, 1152), (3, 48), (128, 1152), (64, 4096), (7, 16),
                                  (1, 1152), (2, 2048), (1, 4096), (5, 64)])
def test_fused_page_geometries(ps, R):
    """Pieces that straddle the end of a partial page's rows, several pieces
    per page; pages of at most 4 KB in groups of consecutive dense pages."""
    rng = np.random.default_rng(ps * 7 + R)
    B = 6
    pfx = (rng.integers(0, 6 * ps, B) // ps) * ps
    cur = rng.integers(0, 5 * ps, B)
    batch = wl.make_compose_batch("geo", 31, page_size=ps, cp_size=3, num_pool_pages=400, row_bytes=R,
                                  prefix_lens=pfx, cur_lens=cur, row_kind="bytes")
    dense, plan, slabs, rows = _run_fused(batch, dense_extra=1)
    want = oracle.compose_dense(batch.prefix_lens, batch.cur_lens, batch.prefix_pages, slabs, rows,
                                page_size=batch.page_size, cp_size=batch.cp_size, dense_cap=plan.dense_cap_pages)
    assert np.array_equal(dense, want)


def test_fused_large_batch_template():
    rng = np.random.default_rng(8)
    B, ps = 150, 16
    batch = wl.make_compose_batch("b150", 8, page_size=ps, cp_size=4, num_pool_pages=20000, row_bytes=64,
                                  prefix_lens=(rng.integers(0, 90, B) // ps) * ps, cur_lens=rng.integers(0, 50, B),
                                  row_kind="bytes")
    dense, plan, slabs, rows = _run_fused(batch, dense_extra=0)
    want = oracle.compose_dense(batch.prefix_lens, batch.cur_lens, batch.prefix_pages, slabs, rows,
                                page_size=batch.page_size, cp_size=batch.cp_size, dense_cap=plan.dense_cap_pages)
    assert np.array_equal(dense, want)


def test_fused_bad_descriptor_is_zeroed_and_flagged():
    batch = wl.tiny_batch()
    plan, _ = _plan_pair(batch, dense_extra=0)
    layers = ComposeLayers(plan, batch.row_bytes)
    slabs = [torch.from_numpy(s).cuda() for s in wl.host_pool(batch)]
    rows = [torch.from_numpy(r).cuda() for r in wl.split_rows_by_writer(batch, wl.host_current_rows(batch))]
    owner = plan["owner"].clone()
    src = plan["src"].clone()
    owner[0] = 2 * batch.cp_size  # outside the table
    src[1] = 10_000               # beyond the slab / current page range
    dense = torch.full((plan.dense_cap_pages * batch.page_size, batch.row_bytes), 0xCD, dtype=torch.uint8,
                       device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    cpkv.cpkv_compose_fused(batch.cur_lens, slabs, rows, owner, src, plan["token_writer_row"], dense,
                            page_size=batch.page_size, cp_size=batch.cp_size, row_bytes=batch.row_bytes,
                            dense_cap_pages=plan.dense_cap_pages, d_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == cpkv.STATUS_DESC_OOB
    page = batch.page_size
    assert torch.all(dense[:page] == 0) and torch.all(dense[page:2 * page] == 0)


# ---------------------------------------------------------------------------
# one-launch layer compose: fill + gather in one kernel, same stagings and dense
# ---------------------------------------------------------------------------

def _run_one_launch(batch, dense_extra=2, layer=0, guard=0x5A, early=False):
    plan, want_plan = _plan_pair(batch, dense_extra)
    layers = ComposeLayers(plan, batch.row_bytes)
    slabs = wl.host_pool(batch, layer)
    rows = wl.host_current_rows(batch, layer)
    d_slabs = [torch.from_numpy(s).cuda() for s in slabs]
    d_rows = [torch.from_numpy(r).cuda() for r in wl.split_rows_by_writer(batch, rows)]
    for s in layers.staging:
        s.fill_(guard)
    dense = torch.full((plan.dense_cap_pages * batch.page_size, batch.row_bytes), 0xCD, dtype=torch.uint8,
                       device="cuda")
    layers.compose_one_launch(d_slabs, d_rows, dense, early_inputs=early)
    if early:  # a second, dependent launch right behind the first (its inputs were complete before either)
        layers.compose_one_launch(d_slabs, d_rows, dense, early_inputs=True)
    torch.cuda.synchronize()
    assert int(plan.d_status.item()) == 0
    want = oracle.compose_dense(batch.prefix_lens, batch.cur_lens, batch.prefix_pages, slabs, rows,
                                page_size=batch.page_size, cp_size=batch.cp_size, dense_cap=plan.dense_cap_pages)
    assert np.array_equal(dense.cpu().numpy(), want)
    want_stg = [np.full(tuple(s.shape), guard, np.uint8) for s in layers.staging]
    oracle.staging(batch.cur_lens, batch.writer, rows, want_stg, page_size=batch.page_size, cp_size=batch.cp_size)
    for w, s in enumerate(layers.staging):
        assert np.array_equal(s.cpu().numpy(), want_stg[w]), w


@pytest.mark.parametrize("early", [False, True], ids=["plain", "early-inputs"])
@pytest.mark.parametrize("batch", pins.edge_batches(), ids=lambda b: b.name)
def test_one_launch_matches_oracle_edge_cases(batch, early):
    _run_one_launch(batch, early=early)


@pytest.mark.parametrize("ps,R", [(64, 656), (16, 1152), (3, 48), (128, 1152), (64, 4096), (7, 16), (1, 16),
                                  (1, 1152), (2, 2048), (5, 64), (1, 4096)])
def test_one_launch_page_geometries(ps, R):
    """Pieces that straddle the end of a partial page's rows, several pieces
    per page; pages of at most 4 KB go in groups of consecutive dense pages
    (32 pages of 16 bytes, 7 of 1152, 25 of 320, 2 of 4096)."""
    rng = np.random.default_rng(ps * 11 + R)
    B = 7
    pfx = (rng.integers(0, 6 * ps, B) // ps) * ps
    cur = rng.integers(0, 5 * ps, B)
    batch = wl.make_compose_batch("geo1", 37, page_size=ps, cp_size=3, num_pool_pages=400, row_bytes=R,
                                  prefix_lens=pfx, cur_lens=cur, row_kind="bytes")
    _run_one_launch(batch, dense_extra=1)


def test_one_launch_large_batch_template():
    rng = np.random.default_rng(9)
    B, ps = 200, 16
    batch = wl.make_compose_batch("b200", 9, page_size=ps, cp_size=5, num_pool_pages=20000, row_bytes=96,
                                  prefix_lens=(rng.integers(0, 90, B) // ps) * ps, cur_lens=rng.integers(0, 50, B),
                                  row_kind="bytes")
    _run_one_launch(batch, dense_extra=0)


def test_one_launch_bad_descriptor_and_rows_are_zeroed_and_flagged():
    batch = wl.tiny_batch()
    plan, _ = _plan_pair(batch, dense_extra=0)
    layers = ComposeLayers(plan, batch.row_bytes)
    slabs = [torch.from_numpy(s).cuda() for s in wl.host_pool(batch)]
    rows = [torch.from_numpy(r).cuda() for r in wl.split_rows_by_writer(batch, wl.host_current_rows(batch))]
    owner = plan["owner"].clone()
    src = plan["src"].clone()
    owner[0] = 2 * batch.cp_size  # outside the table
    src[1] = 10_000               # beyond the slab / current page range
    table = list(slabs) + list(layers.staging)
    caps = [t.shape[0] for t in slabs] + [plan.staging_cap_pages] * batch.cp_size
    dense = torch.full((plan.dense_cap_pages * batch.page_size, batch.row_bytes), 0xCD, dtype=torch.uint8,
                       device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    cpkv.cpkv_compose_layer(batch.cur_lens, rows, table, caps, owner, src, plan["token_writer_row"], dense,
                            page_size=batch.page_size, cp_size=batch.cp_size, row_bytes=batch.row_bytes,
                            dense_cap_pages=plan.dense_cap_pages, d_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == cpkv.STATUS_DESC_OOB
    page = batch.page_size
    assert torch.all(dense[:page] == 0) and torch.all(dense[page:2 * page] == 0)
    # a writer buffer one row short: that writer's last current page is zeroed, ROW_OOB
    caps_rows = [rows[0].shape[0] - 1] + [r.shape[0] for r in rows[1:]]
    status.zero_()
    cpkv.cpkv_compose_layer(batch.cur_lens, rows, table, caps, plan["owner"], plan["src"], plan["token_writer_row"],
                            dense, page_size=batch.page_size, cp_size=batch.cp_size, row_bytes=batch.row_bytes,
                            dense_cap_pages=plan.dense_cap_pages, d_status=status, cur_rows_cap=caps_rows)
    torch.cuda.synchronize()
    assert int(status.item()) == cpkv.STATUS_ROW_OOB


# ---------------------------------------------------------------------------
# fill with row indices that do not form page runs (row-by-row path)
# ---------------------------------------------------------------------------

def _fill_case(batch, mutate):
    plan, _ = _plan_pair(batch)
    ps, cp, R = batch.page_size, batch.cp_size, batch.row_bytes
    sr = plan["staging_rows"].cpu().numpy().copy()
    tw = plan["token_writer_row"].cpu().numpy().copy()
    mutate(batch, sr, tw)
    rows = wl.host_current_rows(batch)
    per_writer = wl.split_rows_by_writer(batch, rows)
    want = [np.full(((batch.C + 1) * ps, R), 0x77, np.uint8) for _ in range(cp)]
    st = oracle.fill_index_copy(batch.cur_lens, sr, tw, batch.writer, per_writer, want, page_size=ps, cp_size=cp,
                                row_bytes=R)
    assert st == 0
    staging = [torch.full(((batch.C + 1) * ps, R), 0x77, dtype=torch.uint8, device="cuda") for _ in range(cp)]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    cpkv.cpkv_fill_current(batch.cur_lens, [torch.from_numpy(r).cuda() for r in per_writer], staging, page_size=ps,
                           cp_size=cp, row_bytes=R, staging_cap_pages=batch.C + 1,
                           d_staging_rows=torch.from_numpy(sr).cuda(), d_token_writer_row=torch.from_numpy(tw).cuda(),
                           d_writer=plan.d_writer, num_cur_pages=batch.C, d_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for w in range(cp):
        assert np.array_equal(staging[w].cpu().numpy(), want[w]), w


def _pages(batch):
    """(first token, rows, is last page of its request) of every current page."""
    out, t = [], 0
    for n in batch.cur_lens.tolist():
        for k in range(0, n, batch.page_size):
            m = min(batch.page_size, n - k)
            out.append((t + k, m, k + m == n))
        t += n
    return out


@pytest.mark.parametrize("batch", [b for b in pins.edge_batches() if b.T > 0], ids=lambda b: b.name)
def test_fill_reversed_source_rows(batch):
    """Source rows reversed inside every page: no page is a run."""
    def mutate(b, sr, tw):
        for t0, n, _ in _pages(b):
            tw[t0:t0 + n] = tw[t0:t0 + n][::-1]
    _fill_case(batch, mutate)


@pytest.mark.parametrize("batch", [b for b in pins.edge_batches() if b.T > 0], ids=lambda b: b.name)
def test_fill_mixed_runs_and_shuffled_pages(batch):
    """Staging rows shuffled inside every other full page that is not a
    request's last page; all other pages stay runs."""
    rng = np.random.default_rng(3)

    def mutate(b, sr, tw):
        for j, (t0, n, last) in enumerate(_pages(b)):
            if j % 2 == 0 and n == b.page_size and not last:
                sr[t0:t0 + n] = sr[t0:t0 + n][rng.permutation(n)]
    _fill_case(batch, mutate)


def test_fill_traced_full_size_runs():
    """The traced batch (every page a run) against the index-copy oracle."""
    _fill_case(wl.traced_batch(), lambda b, sr, tw: None)


# ---------------------------------------------------------------------------
# layer-ahead split: prefix/zero slots early, current slots at consume
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("batch", pins.edge_batches(), ids=lambda b: b.name)
def test_prefetch_then_consume_equals_compose(batch):
    plan, _ = _plan_pair(batch, dense_extra=2)
    layers = ComposeLayers(plan, batch.row_bytes)
    slabs = wl.host_pool(batch)
    rows = wl.host_current_rows(batch)
    d_slabs = [torch.from_numpy(s).cuda() for s in slabs]
    d_rows = [torch.from_numpy(r).cuda() for r in wl.split_rows_by_writer(batch, rows)]
    ps = batch.page_size
    dense = torch.full((plan.dense_cap_pages * ps, batch.row_bytes), 0xCD, dtype=torch.uint8, device="cuda")
    want = oracle.compose_dense(batch.prefix_lens, batch.cur_lens, batch.prefix_pages, slabs, rows, page_size=ps,
                                cp_size=batch.cp_size, dense_cap=plan.dense_cap_pages)
    layers.prefetch(d_slabs, dense)
    torch.cuda.synchronize()
    # after the prefetch: prefix and zero slots final, current slots untouched
    got = dense.cpu().numpy().reshape(plan.dense_cap_pages, ps, batch.row_bytes)
    owner = plan["owner"].cpu().numpy()
    w3 = want.reshape(plan.dense_cap_pages, ps, batch.row_bytes)
    for d in range(plan.dense_cap_pages):
        if owner[d] >= batch.cp_size:
            assert np.all(got[d] == 0xCD), d
        else:
            assert np.array_equal(got[d], w3[d]), d
    layers.consume(d_rows, dense)
    torch.cuda.synchronize()
    assert int(plan.d_status.item()) == 0
    assert np.array_equal(dense.cpu().numpy(), want)


@pytest.mark.parametrize("ps,R", [(16, 1152), (64, 1152), (64, 656), (3, 48)])
def test_gather_early_behind_fill_page_geometries(ps, R):
    """Early gathers (several pieces per page, and one piece: launched
    plainly) behind early fills, three layers, every layer checked."""
    rng = np.random.default_rng(ps * 13 + R)
    B = 7
    pfx = (rng.integers(0, 8 * ps, B) // ps) * ps
    cur = rng.integers(1, 6 * ps, B)
    batch = wl.make_compose_batch("geo-early", 41, page_size=ps, cp_size=3, num_pool_pages=500, row_bytes=R,
                                  prefix_lens=pfx, cur_lens=cur, row_kind="bytes")
    plan, _ = _plan_pair(batch, dense_extra=1)
    layers = ComposeLayers(plan, batch.row_bytes)
    host = [(wl.host_pool(batch, l), wl.host_current_rows(batch, l)) for l in range(3)]
    dev = [([torch.from_numpy(s).cuda() for s in slabs],
            [torch.from_numpy(r).cuda() for r in wl.split_rows_by_writer(batch, rows)]) for slabs, rows in host]
    dense = [torch.full((plan.dense_cap_pages * ps, R), 0xCD, dtype=torch.uint8, device="cuda") for _ in range(3)]
    torch.cuda.synchronize()
    for l in range(3):
        layers.fill(dev[l][1], early_inputs=True)
        layers.gather(dev[l][0], dense[l], consume_staging=True, early_inputs=True)
    torch.cuda.synchronize()
    assert int(plan.d_status.item()) == 0
    for l, (slabs, rows) in enumerate(host):
        want = oracle.compose_dense(batch.prefix_lens, batch.cur_lens, batch.prefix_pages, slabs, rows,
                                    page_size=ps, cp_size=batch.cp_size, dense_cap=plan.dense_cap_pages)
        assert np.array_equal(dense[l].cpu().numpy(), want), l


@pytest.mark.parametrize("batch", pins.edge_batches(), ids=lambda b: b.name)
def test_consumed_stagings_are_rewritten_before_every_read(batch):
    """After a consuming gather a staging holds whatever DRAM last saw (here a
    0xA5 poison written before the first layer): three layers of row fill +
    consuming gather with distinct inputs, each dense buffer against the
    oracle.  Exact only if every fill rewrites every staged row and every pad
    row that the gather reads."""
    plan, _ = _plan_pair(batch, dense_extra=2)
    layers = ComposeLayers(plan, batch.row_bytes)
    for st in layers.staging:
        st.fill_(0xA5)
    ps = batch.page_size
    host = [(wl.host_pool(batch, l), wl.host_current_rows(batch, l)) for l in range(3)]
    dense = [torch.full((plan.dense_cap_pages * ps, batch.row_bytes), 0xCD, dtype=torch.uint8, device="cuda")
             for _ in range(3)]
    torch.cuda.synchronize()
    for l, (slabs, rows) in enumerate(host):
        layers.fill([torch.from_numpy(r).cuda() for r in wl.split_rows_by_writer(batch, rows)])
        layers.gather([torch.from_numpy(s).cuda() for s in slabs], dense[l], consume_staging=True)
    torch.cuda.synchronize()
    assert int(plan.d_status.item()) == 0
    for l, (slabs, rows) in enumerate(host):
        want = oracle.compose_dense(batch.prefix_lens, batch.cur_lens, batch.prefix_pages, slabs, rows,
                                    page_size=ps, cp_size=batch.cp_size, dense_cap=plan.dense_cap_pages)
        assert np.array_equal(dense[l].cpu().numpy(), want), l


def _page_run_batch(seed=77, cp=4, ps=1, R=1152, B=5):
    """Small pages whose sources form runs: each request's prefix pages are
    consecutive local pages of one owner (ids r + cp * k for consecutive k),
    and its current pages go to contiguous writers, so consecutive dense
    current pages have consecutive staging slots of one writer."""
    rng = np.random.default_rng(seed)
    pfx = rng.integers(5, 40, B) * ps
    cur = rng.integers(3, 30, B)
    next_local = [1] * cp
    prefix_pages = []
    for b in range(B):
        r = int(rng.integers(0, cp))
        n = int(pfx[b] // ps)
        prefix_pages += [r + cp * (next_local[r] + k) for k in range(n)]
        next_local[r] += n + int(rng.integers(0, 3))  # a gap between requests now and then
    first_cur = cp * (max(next_local) + 1)
    C = int(((cur + ps - 1) // ps).sum())
    cur_pages = first_cur + np.arange(C)
    P = int(first_cur + C + 1)
    return wl.make_compose_batch("page-runs", seed, page_size=ps, cp_size=cp, num_pool_pages=P, row_bytes=R,
                                 prefix_lens=pfx, cur_lens=cur, prefix_pages=np.array(prefix_pages),
                                 cur_pages=cur_pages, writer=wl.contiguous_writers(cur, ps, cp),
                                 row_kind="bytes")


@pytest.mark.parametrize("early", [False, True], ids=["plain", "early"])
@pytest.mark.parametrize("consume", [False, True], ids=["kept", "consumed"])
@pytest.mark.parametrize("ps,R", [(1, 1152), (4, 272), (2, 16)])
def test_gather_merges_page_runs(ps, R, consume, early):
    """Page-run merging in the grouped small-page gather: pool and staging
    runs are loaded as single copies, zero slots fill the group's tail; two
    layers of distinct inputs, each checked."""
    batch = _page_run_batch(ps=ps, R=R)
    plan, _ = _plan_pair(batch, dense_extra=9)
    layers = ComposeLayers(plan, batch.row_bytes)
    host = [(wl.host_pool(batch, l), wl.host_current_rows(batch, l)) for l in range(2)]
    dev = [([torch.from_numpy(s).cuda() for s in slabs],
            [torch.from_numpy(r).cuda() for r in wl.split_rows_by_writer(batch, rows)]) for slabs, rows in host]
    dense = [torch.full((plan.dense_cap_pages * ps, R), 0xCD, dtype=torch.uint8, device="cuda") for _ in range(2)]
    torch.cuda.synchronize()
    for l in range(2):
        layers.fill(dev[l][1], early_inputs=early)
        layers.gather(dev[l][0], dense[l], consume_staging=consume, early_inputs=early)
    torch.cuda.synchronize()
    assert int(plan.d_status.item()) == 0
    for l, (slabs, rows) in enumerate(host):
        want = oracle.compose_dense(batch.prefix_lens, batch.cur_lens, batch.prefix_pages, slabs, rows,
                                    page_size=ps, cp_size=batch.cp_size, dense_cap=plan.dense_cap_pages)
        assert np.array_equal(dense[l].cpu().numpy(), want), l


def test_gather_kinds_rejects_bad_mask():
    batch = wl.tiny_batch()
    plan, _ = _plan_pair(batch)
    layers = ComposeLayers(plan, batch.row_bytes)
    for bad in (-1, 32, 63):
        with pytest.raises(cpkv.CpkvError):
            layers.gather_kinds([torch.from_numpy(s).cuda() for s in wl.host_pool(batch)], layers.dense[0], bad)


# ---------------------------------------------------------------------------
# gather that consumes the stagings: same dense buffer (staging bytes undefined)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("batch", pins.edge_batches(), ids=lambda b: b.name)
def test_gather_consuming_staging_matches_oracle(batch):
    plan, _ = _plan_pair(batch, dense_extra=2)
    layers = ComposeLayers(plan, batch.row_bytes)
    slabs = wl.host_pool(batch)
    rows = wl.host_current_rows(batch)
    d_slabs = [torch.from_numpy(s).cuda() for s in slabs]
    d_rows = [torch.from_numpy(r).cuda() for r in wl.split_rows_by_writer(batch, rows)]
    dense = torch.full((plan.dense_cap_pages * batch.page_size, batch.row_bytes), 0xCD, dtype=torch.uint8,
                       device="cuda")
    for _ in range(2):  # the second layer refills the consumed stagings
        layers.fill(d_rows)
        layers.gather(d_slabs, dense, consume_staging=True)
    torch.cuda.synchronize()
    assert int(plan.d_status.item()) == 0
    want = oracle.compose_dense(batch.prefix_lens, batch.cur_lens, batch.prefix_pages, slabs, rows,
                                page_size=batch.page_size, cp_size=batch.cp_size, dense_cap=plan.dense_cap_pages)
    assert np.array_equal(dense.cpu().numpy(), want)


@pytest.mark.parametrize("batch", pins.edge_batches(), ids=lambda b: b.name)
def test_one_launch_consuming_staging_matches_oracle(batch):
    plan, _ = _plan_pair(batch, dense_extra=1)
    layers = ComposeLayers(plan, batch.row_bytes)
    slabs = wl.host_pool(batch)
    rows = wl.host_current_rows(batch)
    d_slabs = [torch.from_numpy(s).cuda() for s in slabs]
    d_rows = [torch.from_numpy(r).cuda() for r in wl.split_rows_by_writer(batch, rows)]
    dense = torch.full((plan.dense_cap_pages * batch.page_size, batch.row_bytes), 0xCD, dtype=torch.uint8,
                       device="cuda")
    for _ in range(2):  # the second layer restages what the first consumed
        layers.compose_one_launch(d_slabs, d_rows, dense, consume_staging=True, early_inputs=True)
    torch.cuda.synchronize()
    assert int(plan.d_status.item()) == 0
    want = oracle.compose_dense(batch.prefix_lens, batch.cur_lens, batch.prefix_pages, slabs, rows,
                                page_size=batch.page_size, cp_size=batch.cp_size, dense_cap=plan.dense_cap_pages)
    assert np.array_equal(dense.cpu().numpy(), want)


# ---------------------------------------------------------------------------
# fill launched early behind the previous layer's gather (FLAG_EARLY_INPUTS)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("early_gather", [False, True], ids=["gather-plain", "gather-early"])
@pytest.mark.parametrize("consume", [False, True], ids=["kept", "consumed"])
@pytest.mark.parametrize("batch", pins.edge_batches(), ids=lambda b: b.name)
def test_fill_early_behind_gather_matches_oracle(batch, consume, early_gather):
    """Three layers of distinct rows and pools, uploaded before the loop; each
    fill starts while the previous layer's gather still reads the stagings it
    overwrites, and (gather-early) each gather starts while its fill still
    writes them.  Every layer has its own dense buffer and is checked, so a
    store or a staging read that ran ahead would show."""
    n_layers = 3
    plan, _ = _plan_pair(batch, dense_extra=1)
    layers = ComposeLayers(plan, batch.row_bytes)
    for s in layers.staging:
        s.fill_(0xA5)
    host = [(wl.host_pool(batch, l), wl.host_current_rows(batch, l)) for l in range(n_layers)]
    dev = [([torch.from_numpy(s).cuda() for s in slabs],
            [torch.from_numpy(r).cuda() for r in wl.split_rows_by_writer(batch, rows)]) for slabs, rows in host]
    dense = [torch.full((plan.dense_cap_pages * batch.page_size, batch.row_bytes), 0xCD, dtype=torch.uint8,
                        device="cuda") for _ in range(n_layers)]
    torch.cuda.synchronize()
    for l in range(n_layers):
        layers.fill(dev[l][1], early_inputs=True)
        layers.gather(dev[l][0], dense[l], consume_staging=consume, early_inputs=early_gather)
    torch.cuda.synchronize()
    assert int(plan.d_status.item()) == 0
    for l, (slabs, rows) in enumerate(host):
        want = oracle.compose_dense(batch.prefix_lens, batch.cur_lens, batch.prefix_pages, slabs, rows,
                                    page_size=batch.page_size, cp_size=batch.cp_size, dense_cap=plan.dense_cap_pages)
        assert np.array_equal(dense[l].cpu().numpy(), want), l
    if not consume:
        stg_want = [np.full(tuple(s.shape), 0xA5, np.uint8) for s in layers.staging]
        oracle.staging(batch.cur_lens, batch.writer, host[-1][1], stg_want, page_size=batch.page_size,
                       cp_size=batch.cp_size)
        for w, s in enumerate(layers.staging):
            assert np.array_equal(s.cpu().numpy(), stg_want[w]), w


# ---------------------------------------------------------------------------
# failure detection on the GPU without a fault: a copy that never lands
# ---------------------------------------------------------------------------

def test_ring_wait_times_out_and_the_context_stays_usable():
    """The bulk ring's bounded wait gives up on a load that never arrives
    (an mbarrier phase that nothing completes): TIMEOUT is raised, nothing is
    stored, and the next compose on the same context is still byte-exact."""
    import time

    dst = torch.full((16,), 0x77, dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.perf_counter()
    cpkv.cpkv_selftest_ring_timeout(dst, status)
    torch.cuda.synchronize()
    waited = time.perf_counter() - t0
    assert int(status.item()) == cpkv.STATUS_TIMEOUT
    assert torch.all(dst == 0x77)
    assert 1.5 < waited < 30.0  # the ring's 2 s limit, not a hang
    batch = wl.tiny_batch()        # the context is fine: a compose right after is byte-exact
    dense, plan, slabs, rows = _run_fused(batch)
    want = oracle.compose_dense(batch.prefix_lens, batch.cur_lens, batch.prefix_pages, slabs, rows,
                                page_size=batch.page_size, cp_size=batch.cp_size, dense_cap=plan.dense_cap_pages)
    assert np.array_equal(dense, want)
