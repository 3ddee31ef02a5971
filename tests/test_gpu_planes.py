"""GPU parity of the planar-page (NSA indexer key) fill and compose against
the oracle's planar definitions, byte-exact."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import oracle_pins as pins
import workloads as wl
from paged_kv_cache_compose_gb300 import cpkv
from paged_kv_cache_compose_gb300.runtime import ComposeLayers, ComposePlan

pytestmark = pytest.mark.gpu


def _planar(batch, planes=wl.INDEX_K_PLANES):
    return dataclasses.replace(batch, row_bytes=sum(planes), planes=tuple(planes), row_kind="bytes")


def _inputs(batch, seed=0):
    rng = np.random.default_rng(batch.seed + 1000 + seed)
    pbytes = batch.page_size * batch.row_bytes
    slabs = [np.frombuffer(rng.bytes(batch.slab_pages * pbytes), np.uint8).reshape(batch.slab_pages, pbytes).copy()
             for _ in range(batch.cp_size)]
    rows = np.frombuffer(rng.bytes(batch.T * batch.row_bytes), np.uint8).reshape(batch.T, batch.row_bytes).copy()
    planes = wl.split_planes(rows, batch.planes)
    tw = wl.token_writer(batch)
    per_writer = [[np.ascontiguousarray(pl[tw == w]) for w in range(batch.cp_size)] for pl in planes]
    return slabs, planes, per_writer


def _edge_planar():
    return [_planar(b) for b in pins.edge_batches() if (b.page_size * 132) % 16 == 0]


def _compose(batch, per_writer_mut=None, reverse_rows=False, page_runs=False):
    ps, cp = batch.page_size, batch.cp_size
    plan = ComposePlan(batch.prefix_lens, batch.cur_lens, batch.prefix_pages, batch.cur_pages, batch.writer,
                       page_size=ps, cp_size=cp, num_pool_pages=batch.num_pool_pages,
                       dense_cap_pages=None).build()
    layers = ComposeLayers(plan, batch.row_bytes)
    slabs, planes, per_writer = _inputs(batch)
    for st in layers.staging:
        st.fill_(0x6B)
    d_planes = [[torch.from_numpy(x).cuda() for x in pw] for pw in per_writer]
    tw = plan["token_writer_row"]
    if reverse_rows:  # source rows reversed inside every page: the index copy must still hold
        h = tw.cpu().numpy().copy()
        t = 0
        for n in batch.cur_lens.tolist():
            for k in range(0, n, ps):
                m = min(ps, n - k)
                h[t + k:t + k + m] = h[t + k:t + k + m][::-1]
            t += n
        tw = torch.from_numpy(h).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    cpkv.cpkv_fill_current_planes(batch.cur_lens, d_planes, layers.staging, page_size=ps, cp_size=cp,
                                  plane_bytes=list(batch.planes), staging_cap_pages=plan.staging_cap_pages,
                                  d_staging_rows=plan["staging_rows"], d_token_writer_row=tw, d_writer=plan.d_writer,
                                  num_cur_pages=plan.C, d_status=status, page_runs=page_runs)
    dense = torch.full((plan.dense_cap_pages * ps, batch.row_bytes), 0xCD, dtype=torch.uint8, device="cuda")
    layers.gather([torch.from_numpy(s).cuda() for s in slabs], dense)
    torch.cuda.synchronize()
    assert int(status.item()) == 0 and int(plan.d_status.item()) == 0
    # staging against the planar index copy
    want_stg = [np.full((plan.staging_cap_pages, ps * batch.row_bytes), 0x6B, np.uint8) for _ in range(cp)]
    st = oracle.fill_planes(batch.cur_lens, plan["staging_rows"].cpu().numpy(), tw.cpu().numpy(), batch.writer,
                            per_writer, want_stg, page_size=ps, cp_size=cp, plane_bytes=list(batch.planes))
    assert st == 0
    for w in range(cp):
        assert np.array_equal(layers.staging[w].cpu().numpy().reshape(plan.staging_cap_pages, ps * batch.row_bytes), want_stg[w]), w
    return dense, plan, slabs, planes


@pytest.mark.parametrize("page_runs", [False, True], ids=["rows", "page-runs"])
@pytest.mark.parametrize("batch", _edge_planar(), ids=lambda b: b.name)
def test_planar_compose_matches_oracle(batch, page_runs):
    dense, plan, slabs, planes = _compose(batch, page_runs=page_runs)
    want = oracle.compose_dense_planes(batch.prefix_lens, batch.cur_lens, batch.prefix_pages, slabs, planes,
                                       page_size=batch.page_size, cp_size=batch.cp_size,
                                       plane_bytes=list(batch.planes))
    assert np.array_equal(dense.cpu().numpy().reshape(plan.dense_cap_pages, batch.page_size * batch.row_bytes), want)


@pytest.mark.parametrize("batch", _edge_planar(), ids=lambda b: b.name)
def test_planar_fill_early_behind_gather(batch):
    """Three layers of distinct planar rows and pools, uploaded first; each
    planar fill starts while the previous gather still reads the stagings.
    Every layer has its own dense buffer and is checked."""
    ps, cp, n_layers = batch.page_size, batch.cp_size, 3
    plan = ComposePlan(batch.prefix_lens, batch.cur_lens, batch.prefix_pages, batch.cur_pages, batch.writer,
                       page_size=ps, cp_size=cp, num_pool_pages=batch.num_pool_pages, dense_cap_pages=None).build()
    layers = ComposeLayers(plan, batch.row_bytes)
    host = [_inputs(batch, seed=l) for l in range(n_layers)]
    dev = [([torch.from_numpy(s).cuda() for s in slabs], [[torch.from_numpy(x).cuda() for x in pw] for pw in per_writer])
           for slabs, _, per_writer in host]
    dense = [torch.full((plan.dense_cap_pages * ps, batch.row_bytes), 0xCD, dtype=torch.uint8, device="cuda")
             for _ in range(n_layers)]
    torch.cuda.synchronize()
    for l in range(n_layers):
        layers.fill_planes(dev[l][1], list(batch.planes), early_inputs=True)
        layers.gather(dev[l][0], dense[l])
    torch.cuda.synchronize()
    assert int(plan.d_status.item()) == 0
    for l, (slabs, planes, _) in enumerate(host):
        want = oracle.compose_dense_planes(batch.prefix_lens, batch.cur_lens, batch.prefix_pages, slabs, planes,
                                           page_size=ps, cp_size=cp, plane_bytes=list(batch.planes))
        assert np.array_equal(dense[l].cpu().numpy().reshape(plan.dense_cap_pages, ps * batch.row_bytes), want), l


@pytest.mark.parametrize("batch", _edge_planar()[:4], ids=lambda b: b.name)
def test_planar_fill_reversed_rows(batch):
    _compose(batch, reverse_rows=True)


@pytest.mark.parametrize("page_runs", [False, True], ids=["rows", "page-runs"])
@pytest.mark.parametrize("planes", [(16,), (64, 4), (4, 4, 8), (128, 4), (32, 16, 4, 12), (4096, 4), (4, 260)])
def test_planar_plane_shapes(planes, page_runs):
    """Plane widths 4 to 4096 bytes (a plane of several 4 KB chunks per page;
    4-byte planes at offsets that are not 16-byte multiples), tiny batch
    (ps 16, short pages), both fills."""
    b = _planar(wl.tiny_batch(), planes)
    dense, plan, slabs, cur = _compose(b, page_runs=page_runs)
    want = oracle.compose_dense_planes(b.prefix_lens, b.cur_lens, b.prefix_pages, slabs, cur, page_size=b.page_size,
                                       cp_size=b.cp_size, plane_bytes=list(planes))
    assert np.array_equal(dense.cpu().numpy().reshape(plan.dense_cap_pages, b.page_size * b.row_bytes), want)


def test_planar_rejects_bad_planes():
    b = _planar(wl.tiny_batch())
    plan = ComposePlan(b.prefix_lens, b.cur_lens, b.prefix_pages, b.cur_pages, b.writer, page_size=b.page_size,
                       cp_size=b.cp_size, num_pool_pages=b.num_pool_pages).build()
    layers = ComposeLayers(plan, b.row_bytes)
    with pytest.raises(cpkv.CpkvError):
        cpkv.cpkv_fill_current_planes(b.cur_lens, [[None] * 2, [None] * 2], layers.staging, page_size=16, cp_size=2,
                                      plane_bytes=[130, 2], staging_cap_pages=plan.staging_cap_pages,
                                      d_staging_rows=plan["staging_rows"], d_token_writer_row=plan["token_writer_row"],
                                      d_writer=plan.d_writer, num_cur_pages=plan.C, d_status=plan.d_status,
                                      cur_rows_cap=[0, 0])


# ---------------------------------------------------------------------------
# one-launch layer compose of planar pages: same stagings and dense buffer
# ---------------------------------------------------------------------------

def _one_launch(batch, dense_extra=1, guard=0x3C, fused=False, early=False):
    """The one-launch layer compose (fused=False: the stagings are checked
    too) or the planar fused compose (fused=True: the stagings must keep
    their guard bytes)."""
    ps, cp = batch.page_size, batch.cp_size
    T, C, D = oracle.sizes(batch.prefix_lens, batch.cur_lens, ps)
    plan = ComposePlan(batch.prefix_lens, batch.cur_lens, batch.prefix_pages, batch.cur_pages, batch.writer,
                       page_size=ps, cp_size=cp, num_pool_pages=batch.num_pool_pages,
                       dense_cap_pages=D + dense_extra).build()
    layers = ComposeLayers(plan, batch.row_bytes)
    slabs, planes, per_writer = _inputs(batch)
    for st in layers.staging:
        st.fill_(guard)
    d_planes = [[torch.from_numpy(x).cuda() for x in pw] for pw in per_writer]
    dense = torch.full((plan.dense_cap_pages * ps, batch.row_bytes), 0xCD, dtype=torch.uint8, device="cuda")
    pools = [torch.from_numpy(s).cuda() for s in slabs]
    for _ in range(2 if early else 1):  # early: a second, dependent launch right behind the first
        if fused:
            layers.compose_fused(pools, d_planes, dense, plane_bytes=list(batch.planes), early_inputs=early)
        else:
            layers.compose_one_launch(pools, d_planes, dense, plane_bytes=list(batch.planes), early_inputs=early)
    torch.cuda.synchronize()
    assert int(plan.d_status.item()) == 0
    want = oracle.compose_dense_planes(batch.prefix_lens, batch.cur_lens, batch.prefix_pages, slabs, planes,
                                       page_size=ps, cp_size=cp, plane_bytes=list(batch.planes),
                                       dense_cap=plan.dense_cap_pages)
    assert np.array_equal(dense.cpu().numpy().reshape(plan.dense_cap_pages, ps * batch.row_bytes), want)
    want_stg = [np.full((plan.staging_cap_pages, ps * batch.row_bytes), guard, np.uint8) for _ in range(cp)]
    if not fused:
        st = oracle.fill_planes(batch.cur_lens, plan["staging_rows"].cpu().numpy(),
                                plan["token_writer_row"].cpu().numpy(), batch.writer, per_writer, want_stg,
                                page_size=ps, cp_size=cp, plane_bytes=list(batch.planes))
        assert st == 0
    for w in range(cp):
        got = layers.staging[w].cpu().numpy().reshape(plan.staging_cap_pages, ps * batch.row_bytes)
        assert np.array_equal(got, want_stg[w]), w


@pytest.mark.parametrize("early", [False, True], ids=["plain", "early-inputs"])
@pytest.mark.parametrize("batch", _edge_planar(), ids=lambda b: b.name)
def test_planar_one_launch_matches_oracle(batch, early):
    _one_launch(batch, early=early)


@pytest.mark.parametrize("ps,planes", [(16, (16,)), (16, (64, 4)), (16, (4, 4, 8)), (16, (128, 4)),
                                       (16, (32, 16, 4, 12)), (3, (4, 16, 12)), (64, (512, 16)), (64, (384, 4, 12)),
                                       (1, (4, 12)), (64, (128, 4))])
def test_planar_one_launch_plane_shapes(ps, planes):
    """Staged and lane-copied planes, a 16-byte plane at an unaligned offset
    (ps=3), and pages of several pieces whose boundaries cut a plane."""
    rng = np.random.default_rng(ps * 100 + sum(planes))
    B = 6
    pfx = (rng.integers(0, 5 * ps, B) // ps) * ps
    cur = rng.integers(0, 4 * ps, B)
    b = wl.make_compose_batch("pl", 77, page_size=ps, cp_size=3, num_pool_pages=300, row_bytes=sum(planes),
                              prefix_lens=pfx, cur_lens=cur, row_kind="bytes")
    _one_launch(_planar(b, planes))


@pytest.mark.parametrize("seed", range(16))
def test_planar_one_launch_fuzz(seed):
    rng = np.random.default_rng(50_000 + seed)
    ps = int(rng.choice([1, 2, 3, 4, 8, 16, 64]))
    while True:
        planes = tuple(int(4 * rng.integers(1, 40)) for _ in range(int(rng.integers(1, 5))))
        if (ps * sum(planes)) % 16 == 0:
            break
    cp = int(rng.integers(1, 9))
    B = int(rng.integers(0, 20))
    pfx = rng.integers(0, 5, size=B) * ps
    cur = rng.integers(0, 4 * ps + 1, size=B)
    mode = int(rng.integers(0, 3))
    C = int(((cur + ps - 1) // ps).sum())
    writer = (wl.round_robin_writers(C, cp) if mode == 0 else wl.contiguous_writers(cur, ps, cp) if mode == 1
              else rng.integers(0, cp, size=C).astype(np.int32))
    b = wl.make_compose_batch(f"plf{seed}", seed, page_size=ps, cp_size=cp, num_pool_pages=int(pfx.sum() // ps) + C + 9,
                              row_bytes=sum(planes), prefix_lens=pfx, cur_lens=cur, writer=writer, row_kind="bytes")
    extra = int(rng.integers(0, 3))
    _one_launch(_planar(b, planes), dense_extra=extra)
    _one_launch(_planar(b, planes), dense_extra=extra, fused=True)


# ---------------------------------------------------------------------------
# planar fused compose (no stagings): same dense buffer, stagings untouched
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("early", [False, True], ids=["plain", "early-inputs"])
@pytest.mark.parametrize("batch", _edge_planar(), ids=lambda b: b.name)
def test_planar_fused_matches_oracle(batch, early):
    _one_launch(batch, fused=True, early=early)


@pytest.mark.parametrize("ps,planes", [(16, (64, 4)), (16, (4, 4, 8)), (16, (128, 4)), (16, (32, 16, 4, 12)),
                                       (3, (4, 16, 12)), (64, (512, 16)), (64, (384, 4, 12)), (1, (4, 12)),
                                       (64, (128, 4)), (16, (16,))])
def test_planar_fused_plane_shapes(ps, planes):
    rng = np.random.default_rng(ps * 101 + sum(planes))
    B = 6
    pfx = (rng.integers(0, 5 * ps, B) // ps) * ps
    cur = rng.integers(0, 4 * ps, B)
    b = wl.make_compose_batch("plF", 78, page_size=ps, cp_size=3, num_pool_pages=300, row_bytes=sum(planes),
                              prefix_lens=pfx, cur_lens=cur, row_kind="bytes")
    _one_launch(_planar(b, planes), fused=True)


def test_planar_fused_bad_descriptor_and_rows_are_zeroed_and_flagged():
    b = _planar(wl.tiny_batch())
    ps, cp = b.page_size, b.cp_size
    plan = ComposePlan(b.prefix_lens, b.cur_lens, b.prefix_pages, b.cur_pages, b.writer, page_size=ps, cp_size=cp,
                       num_pool_pages=b.num_pool_pages).build()
    slabs, planes, per_writer = _inputs(b)
    pools = [torch.from_numpy(s).cuda() for s in slabs]
    d_planes = [[torch.from_numpy(x).cuda() for x in pw] for pw in per_writer]
    owner, src = plan["owner"].clone(), plan["src"].clone()
    owner[0] = 2 * cp           # outside the table
    src[1] = 10_000             # beyond the slab / current page range
    dense = torch.full((plan.dense_cap_pages * ps, b.row_bytes), 0xCD, dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    cpkv.cpkv_compose_fused_planes(b.cur_lens, pools, d_planes, owner, src, plan["token_writer_row"], dense,
                                   page_size=ps, cp_size=cp, plane_bytes=list(b.planes),
                                   dense_cap_pages=plan.dense_cap_pages, d_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == cpkv.STATUS_DESC_OOB
    assert torch.all(dense[:2 * ps] == 0)
    # writer 0's buffers one row short: its last current page is zeroed, ROW_OOB
    caps = [per_writer[0][0].shape[0] - 1] + [per_writer[0][w].shape[0] for w in range(1, cp)]
    status.zero_()
    cpkv.cpkv_compose_fused_planes(b.cur_lens, pools, d_planes, plan["owner"], plan["src"], plan["token_writer_row"],
                                   dense, page_size=ps, cp_size=cp, plane_bytes=list(b.planes),
                                   dense_cap_pages=plan.dense_cap_pages, d_status=status, cur_rows_cap=caps)
    torch.cuda.synchronize()
    assert int(status.item()) == cpkv.STATUS_ROW_OOB


@pytest.mark.parametrize("batch", _edge_planar(), ids=lambda b: b.name)
def test_consumed_stagings_are_rewritten_before_every_read(batch):
    """A consuming gather drops the stagings' L2 lines, so afterwards a
    staging holds whatever DRAM last saw (here a 0xA5 poison).  The dense
    output stays exact only if the next fill rewrites every staging byte the
    gather reads, pad slices included.  Stagings poisoned, then three layers
    of planar fill + consuming gather with distinct inputs; every layer's
    dense buffer against the oracle."""
    ps, cp = batch.page_size, batch.cp_size
    plan = ComposePlan(batch.prefix_lens, batch.cur_lens, batch.prefix_pages, batch.cur_pages, batch.writer,
                       page_size=ps, cp_size=cp, num_pool_pages=batch.num_pool_pages, dense_cap_pages=None).build()
    layers = ComposeLayers(plan, batch.row_bytes)
    for st in layers.staging:
        st.fill_(0xA5)
    torch.cuda.synchronize()
    dense, wants = [], []
    for layer in range(3):
        slabs, planes, per_writer = _inputs(batch, seed=layer)
        d = torch.full((plan.dense_cap_pages * ps, batch.row_bytes), 0xCD, dtype=torch.uint8, device="cuda")
        layers.fill_planes([[torch.from_numpy(x).cuda() for x in pw] for pw in per_writer], list(batch.planes))
        layers.gather([torch.from_numpy(s).cuda() for s in slabs], d, consume_staging=True)
        dense.append(d)
        wants.append(oracle.compose_dense_planes(batch.prefix_lens, batch.cur_lens, batch.prefix_pages, slabs,
                                                 planes, page_size=ps, cp_size=cp, plane_bytes=list(batch.planes)))
    torch.cuda.synchronize()
    assert int(plan.d_status.item()) == 0
    for layer, (d, want) in enumerate(zip(dense, wants)):
        assert np.array_equal(d.cpu().numpy().reshape(plan.dense_cap_pages, ps * batch.row_bytes), want), layer
