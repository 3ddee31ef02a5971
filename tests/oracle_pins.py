"""Pins of the CPU oracle to facts other than itself.

Each ``pin_*`` function takes a loaded oracle library and raises
``AssertionError`` when the oracle disagrees with:
  * a hand-worked example (tests/golden/*.json, each with its derivation),
  * a library routine the method reduces to in a special case
    (cp = 1: the dense KV is ``torch.cat`` of ``index_select`` per request),
  * brute force on small inputs (inverting a map by enumeration, counting
    writers, tiling q tokens),
  * closed forms (exclusive cumsum, ``np.repeat``).
They are shared by tests/test_oracle_pins.py (the real oracle) and
tests/test_oracle_mutants.py (copies of the oracle with a planted mistake,
each of which must fail at least one pin).
"""
from __future__ import annotations

import json
import os

import numpy as np
import torch

import oracle
import workloads as wl

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _load_golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _labelled_pool(cp, slab_pages, ps, R):
    """Pool whose every row is distinct and decodable: bytes 0..5 hold
    (owner, local page, offset) and the rest is a fixed pattern."""
    slabs = []
    for o in range(cp):
        s = np.zeros((slab_pages, ps, R), np.uint8)
        for p in range(slab_pages):
            for r in range(ps):
                s[p, r, 0] = 1  # tag: pool row
                s[p, r, 1] = o
                s[p, r, 2:4] = np.frombuffer(np.uint16(p).tobytes(), np.uint8)
                s[p, r, 4] = r
                s[p, r, 5:] = (o * 31 + p * 7 + r * 3) % 251
        slabs.append(s)
    return slabs


def _labelled_rows(T, R):
    rows = np.zeros((T, R), np.uint8)
    for t in range(T):
        rows[t, 0] = 2  # tag: current row
        rows[t, 1:3] = np.frombuffer(np.uint16(t).tobytes(), np.uint8)
        rows[t, 3:] = (t * 13 + 5) % 253
    return rows


def _label_row(kind_row, slabs, rows):
    kind = kind_row[0]
    if kind == "pool":
        return slabs[kind_row[1]][kind_row[2], kind_row[3]]
    if kind == "cur":
        return rows[kind_row[1]]
    return np.zeros(rows.shape[1] if rows.size else slabs[0].shape[-1], np.uint8)


# ---------------------------------------------------------------------------
# golden, hand-worked
# ---------------------------------------------------------------------------

def pin_golden_compose(lib):
    g = _load_golden("compose_worked_example.json")
    inp, exp = g["input"], g["expected"]
    ps, cp, P, cap = inp["page_size"], inp["cp_size"], inp["num_pool_pages"], inp["dense_cap"]
    plan = oracle.compose_plan(inp["prefix_lens"], inp["cur_lens"], inp["prefix_pages"], inp["cur_pages"],
                               inp["writer"], page_size=ps, cp_size=cp, num_pool_pages=P, dense_cap=cap, lib=lib)
    assert plan["status"] == 0
    assert (plan["T"], plan["C"], plan["D"]) == (exp["T"], exp["C"], exp["D"])
    for k in ("prefix_spans", "cur_spans", "owner", "src", "mixed_locs", "staging_rows", "token_writer_row"):
        assert plan[k].tolist() == exp[k], k
    pi = np.full(P, -1, np.int32)
    for k, v in exp["page_inverse_nonneg"].items():
        pi[int(k)] = v
    spi = np.zeros(P, np.int32)
    for k, v in exp["staging_page_inverse_nonzero"].items():
        spi[int(k)] = v
    assert np.array_equal(plan["page_inverse"], pi)
    assert np.array_equal(plan["staging_page_inverse"], spi)

    R = 16
    slab_pages = -(-P // cp)
    slabs = _labelled_pool(cp, slab_pages, ps, R)
    rows = _labelled_rows(exp["T"], R)
    dense = oracle.compose_dense(inp["prefix_lens"], inp["cur_lens"], inp["prefix_pages"], slabs, rows,
                                 page_size=ps, cp_size=cp, dense_cap=cap, lib=lib)
    want = np.stack([_label_row(x, slabs, rows) for x in exp["dense_rows"]])
    assert np.array_equal(dense, want)

    # staging: defined pages only; everything else keeps its guard byte
    stg = [np.full(((exp["C"] + 1) * ps, R), 0xA5, np.uint8) for _ in range(cp)]
    oracle.staging(inp["cur_lens"], inp["writer"], rows, stg, page_size=ps, cp_size=cp, lib=lib)
    defined = set()
    for w, pages in exp["staging_defined"].items():
        for p, prow in pages.items():
            got = stg[int(w)][int(p) * ps:(int(p) + 1) * ps]
            assert np.array_equal(got, np.stack([_label_row(x, slabs, rows) for x in prow]))
            defined.add((int(w), int(p)))
    for w in range(cp):
        for p in range(exp["C"] + 1):
            if (w, p) not in defined:
                assert np.all(stg[w][p * ps:(p + 1) * ps] == 0xA5), (w, p)

    # gather through the plan's descriptors reproduces the dense rows
    table = slabs + [s.reshape(-1, ps, R) for s in stg]
    caps = [slab_pages] * cp + [exp["C"] + 1] * cp
    g_dense, st = oracle.gather([t.reshape(-1) for t in table], caps, plan["owner"], plan["src"],
                                page_size=ps, row_bytes=R, dense_cap=cap, lib=lib)
    assert st == 0
    assert np.array_equal(g_dense, want)


def pin_golden_ragged(lib):
    g = _load_golden("ragged_worked_example.json")
    inp = g["input"]
    for case in g["cases"]:
        got = oracle.ragged_plan(inp["prefix_lens"], inp["q_lens"], case["cp_index"], chunk=inp["chunk"],
                                 k_align=case["k_align"], lib=lib)
        exp = case["expected"]
        assert got["status"] == 0
        assert (got["S"], got["Q"]) == (exp["S"], exp["Q"]), case["cp_index"]
        for k in ("seg_req", "q_starts", "q_lens", "kv_lens", "k_bases", "current_bases", "q_bases",
                  "topk_offsets"):
            assert got[k].tolist() == exp[k], (k, case["cp_index"], case["k_align"])


# ---------------------------------------------------------------------------
# brute force and library reductions on seeded batches
# ---------------------------------------------------------------------------

def _dense_page_sequence(batch):
    """(kind, logical page, current index) of every dense page, by enumeration
    of each request's page table: prefix pages, then current pages."""
    seq = []
    pp = 0
    i = 0
    ps = batch.page_size
    for b in range(batch.B):
        npp = int(batch.prefix_lens[b]) // ps
        ncp = -(-int(batch.cur_lens[b]) // ps)
        for k in range(npp):
            seq.append(("p", int(batch.prefix_pages[pp + k]), -1))
        for k in range(ncp):
            seq.append(("c", int(batch.cur_pages[i + k]), i + k))
        pp += npp
        i += ncp
    return seq


def pin_plan_brute_force(lib, batch, dense_extra=0):
    ps, cp, P = batch.page_size, batch.cp_size, batch.num_pool_pages
    seq = _dense_page_sequence(batch)
    D = len(seq)
    cap = D + dense_extra
    plan = oracle.compose_plan(batch.prefix_lens, batch.cur_lens, batch.prefix_pages, batch.cur_pages,
                               batch.writer, page_size=ps, cp_size=cp, num_pool_pages=P, dense_cap=cap, lib=lib)
    assert plan["status"] == 0
    assert plan["D"] == D and plan["C"] == batch.C and plan["T"] == batch.T

    # page_inverse: inverse of the dense-slot -> logical-page map (smallest slot)
    want_pi = np.full(P, -1, np.int32)
    for d in range(D - 1, -1, -1):
        want_pi[seq[d][1]] = d
    assert np.array_equal(plan["page_inverse"], want_pi)
    for d, (_, lp, _) in enumerate(seq):
        assert seq[plan["page_inverse"][lp]][1] == lp

    # staging inverse: current page i -> i + 1 (row 0 reserved)
    want_spi = np.zeros(P, np.int32)
    for kind, lp, i in seq:
        if kind == "c":
            want_spi[lp] = i + 1
    assert np.array_equal(plan["staging_page_inverse"], want_spi)

    # descriptors: modulo owner for prefix, cp + writer / staging slot for current
    for d, (kind, lp, i) in enumerate(seq):
        if kind == "p":
            assert (plan["owner"][d], plan["src"][d]) == (lp % cp, lp // cp), d
        else:
            assert (plan["owner"][d], plan["src"][d]) == (cp + int(batch.writer[i]), i + 1), d
    assert np.all(plan["owner"][D:] == -1) and np.all(plan["src"][D:] == 0)

    # spans tile the dense slots in request order
    nxt = 0
    for b in range(batch.B):
        ds, npp = plan["prefix_spans"][b]
        cs, ncp = plan["cur_spans"][b]
        assert ds == nxt and cs == ds + npp
        assert npp == batch.prefix_lens[b] // ps and ncp == -(-batch.cur_lens[b] // ps)
        assert all(seq[d][0] == "p" for d in range(ds, ds + npp))
        assert all(seq[d][0] == "c" for d in range(cs, cs + ncp))
        nxt = cs + ncp
    assert nxt == D

    # per-token locations agree with the inverses (the pages' fill derives its
    # destinations from the page inverse)
    cur_lp = np.repeat(np.asarray(batch.cur_pages, np.int64), ps)
    offs = np.tile(np.arange(ps, dtype=np.int64), batch.C)
    keep = []
    for b in range(batch.B):
        ncp = -(-int(batch.cur_lens[b]) // ps)
        m = np.zeros(ncp * ps, bool)
        m[:int(batch.cur_lens[b])] = True
        keep.append(m)
    keep = np.concatenate(keep) if keep else np.zeros(0, bool)
    cur_lp, offs = cur_lp[keep], offs[keep]
    assert np.array_equal(plan["mixed_locs"], plan["page_inverse"][cur_lp].astype(np.int64) * ps + offs)
    assert np.array_equal(plan["staging_rows"], plan["staging_page_inverse"][cur_lp].astype(np.int64) * ps + offs)

    # token_writer_row: each writer's tokens, in batch order, are rows 0..T_w-1
    tw = wl.token_writer(batch)
    for w in range(cp):
        assert np.array_equal(plan["token_writer_row"][tw == w], np.arange(int((tw == w).sum())))

    # every current page has exactly one writer, and it is in range
    assert np.all((batch.writer >= 0) & (batch.writer < cp))
    return plan


def pin_dense_token_level(lib, batch, dense_extra=0):
    """Dense KV from logical token locations (lp * ps + off), vectorised with
    numpy fancy indexing, must equal the oracle's row walk."""
    ps, cp, R = batch.page_size, batch.cp_size, batch.row_bytes
    slabs = wl.host_pool(batch)
    rows = wl.host_current_rows(batch)
    flat = np.concatenate([s.reshape(-1, R) for s in slabs])  # owner-major flat pool
    slab_rows = slabs[0].shape[0] * ps
    D = len(_dense_page_sequence(batch))
    cap = D + dense_extra
    want = np.zeros((cap * ps, R), np.uint8)
    row, pp, tok = 0, 0, 0
    for b in range(batch.B):
        npp = int(batch.prefix_lens[b]) // ps
        locs = np.repeat(np.asarray(batch.prefix_pages[pp:pp + npp], np.int64), ps) * ps + np.tile(np.arange(ps), npp)
        lp, off = locs // ps, locs % ps
        want[row:row + len(locs)] = flat[(lp % cp) * slab_rows + (lp // cp) * ps + off]
        row += len(locs)
        n = int(batch.cur_lens[b])
        want[row:row + n] = rows[tok:tok + n]
        row += -(-n // ps) * ps
        pp += npp
        tok += n
    got = oracle.compose_dense(batch.prefix_lens, batch.cur_lens, batch.prefix_pages, slabs, rows,
                               page_size=ps, cp_size=cp, dense_cap=cap, lib=lib)
    assert np.array_equal(got, want)
    return got, slabs, rows


def pin_cp1_index_select_cat(lib, seed=7):
    """cp = 1: the whole pool is one slab and the dense KV of a request is
    ``cat(pool_rows.index_select(prefix rows), current rows, zeros)``."""
    rng = np.random.default_rng(seed)
    ps, R = 8, 32
    pfx = (rng.integers(0, 40, size=5) // ps) * ps
    cur = rng.integers(0, 30, size=5)
    batch = wl.make_compose_batch("cp1", seed, page_size=ps, cp_size=1, num_pool_pages=64, row_bytes=R,
                                  prefix_lens=pfx, cur_lens=cur, row_kind="bytes")
    slabs = wl.host_pool(batch)
    rows = wl.host_current_rows(batch)
    pool = torch.from_numpy(slabs[0].reshape(-1, R))
    parts = []
    pp, tok = 0, 0
    for b in range(batch.B):
        npp = int(pfx[b]) // ps
        pages = torch.from_numpy(np.asarray(batch.prefix_pages[pp:pp + npp], np.int64))
        idx = (pages[:, None] * ps + torch.arange(ps)[None, :]).reshape(-1)
        n = int(cur[b])
        pad = (-n) % ps
        parts += [pool.index_select(0, idx), torch.from_numpy(rows[tok:tok + n]), torch.zeros(pad, R, dtype=torch.uint8)]
        pp += npp
        tok += n
    want = torch.cat(parts).numpy()
    got = oracle.compose_dense(pfx, cur, batch.prefix_pages, slabs, rows, page_size=ps, cp_size=1, lib=lib)
    assert np.array_equal(got, want)


def pin_staging_gather_roundtrip(lib, batch, dense_extra=0):
    """Plan + staging + descriptor gather reproduces the plain dense KV, and
    the current slots of the dense KV give back every current row."""
    ps, cp, R = batch.page_size, batch.cp_size, batch.row_bytes
    plan = oracle.compose_plan(batch.prefix_lens, batch.cur_lens, batch.prefix_pages, batch.cur_pages,
                               batch.writer, page_size=ps, cp_size=cp, num_pool_pages=batch.num_pool_pages,
                               dense_cap=None, lib=lib)
    cap = plan["D"] + dense_extra
    plan = oracle.compose_plan(batch.prefix_lens, batch.cur_lens, batch.prefix_pages, batch.cur_pages,
                               batch.writer, page_size=ps, cp_size=cp, num_pool_pages=batch.num_pool_pages,
                               dense_cap=cap, lib=lib)
    slabs = wl.host_pool(batch)
    rows = wl.host_current_rows(batch)
    stg = [np.full(((batch.C + 1) * ps, R), 0x5A, np.uint8) for _ in range(cp)]
    oracle.staging(batch.cur_lens, batch.writer, rows, stg, page_size=ps, cp_size=cp, lib=lib)
    # page 0 of every staging is reserved and never written
    for s in stg:
        assert np.all(s[:ps] == 0x5A)
    table = [s.reshape(-1) for s in slabs] + [s.reshape(-1) for s in stg]
    caps = [batch.slab_pages] * cp + [batch.C + 1] * cp
    dense_g, st = oracle.gather(table, caps, plan["owner"], plan["src"], page_size=ps, row_bytes=R,
                                dense_cap=cap, lib=lib)
    assert st == 0
    dense = oracle.compose_dense(batch.prefix_lens, batch.cur_lens, batch.prefix_pages, slabs, rows,
                                 page_size=ps, cp_size=cp, dense_cap=cap, lib=lib)
    assert np.array_equal(dense_g, dense)
    assert np.array_equal(dense[plan["mixed_locs"]], rows)
    # the staging rows written by the fill are the current rows, writer by writer
    tw = wl.token_writer(batch)
    for t in range(0, batch.T, max(1, batch.T // 64)):
        assert np.array_equal(stg[tw[t]][plan["staging_rows"][t]], rows[t])


def pin_fill_index_copy(lib, batch):
    """The general index copy agrees with the staging definition on
    plan-built indices (pad rows zeroed, other pages untouched)."""
    ps, cp, R = batch.page_size, batch.cp_size, batch.row_bytes
    plan = oracle.compose_plan(batch.prefix_lens, batch.cur_lens, batch.prefix_pages, batch.cur_pages, batch.writer,
                               page_size=ps, cp_size=cp, num_pool_pages=batch.num_pool_pages, lib=lib)
    rows = wl.host_current_rows(batch)
    per_writer = wl.split_rows_by_writer(batch, rows)
    a = [np.full(((batch.C + 1) * ps, R), 0x3C, np.uint8) for _ in range(cp)]
    b = [x.copy() for x in a]
    st = oracle.fill_index_copy(batch.cur_lens, plan["staging_rows"], plan["token_writer_row"], batch.writer,
                                per_writer, a, page_size=ps, cp_size=cp, row_bytes=R, lib=lib)
    assert st == 0
    oracle.staging(batch.cur_lens, batch.writer, rows, b, page_size=ps, cp_size=cp, lib=lib)
    for w in range(cp):
        assert np.array_equal(a[w], b[w]), w


def pin_fill_index_copy_permuted(lib):
    """Hand-worked: ps=2, cp=1, one request of 3 tokens on current pages 0, 1
    (staging slots 1, 2).  Source rows of the first page swapped: token 0 <-
    row 1, token 1 <- row 0, token 2 <- row 2; staging rows 2, 3, 4; row 5 is
    the pad after the last token and becomes zero; rows 0, 1 (slot 0) keep
    their guard bytes."""
    R = 16
    rows = np.stack([np.full(R, 10 + i, np.uint8) for i in range(3)])
    stg = [np.full((3 * 2, R), 0xEE, np.uint8)]
    st = oracle.fill_index_copy([3], [2, 3, 4], [1, 0, 2], [0, 0], [rows], stg, page_size=2, cp_size=1,
                                row_bytes=R, lib=lib)
    assert st == 0
    want = np.stack([np.full(R, v, np.uint8) for v in (0xEE, 0xEE, 11, 10, 12, 0)])
    assert np.array_equal(stg[0], want)
    # an out-of-range source row is skipped and flagged
    stg = [np.full((3 * 2, R), 0xEE, np.uint8)]
    st = oracle.fill_index_copy([3], [2, 3, 4], [1, 7, 2], [0, 0], [rows], stg, page_size=2, cp_size=1,
                                row_bytes=R, lib=lib)
    assert st == oracle.ROW_OOB
    assert np.all(stg[0][3] == 0xEE)


def pin_planes_golden(lib):
    """Hand-worked two-plane page: ps=2, planes of 8 and 4 bytes, cp=1, one
    request with a 2-token prefix on logical page 3 and 1 current token on
    page 5 (writer 0).  Pool page 3 = [0x11 x8][0x12 x8][0x21 x4][0x22 x4]
    (plane 0 rows 0,1 then plane 1 rows 0,1); the current token is 0x31 x8 /
    0x41 x4.  Dense page 0 is the pool page; dense page 1 is
    [0x31 x8][0 x8][0x41 x4][0 x4]; staging slot 1 holds the same bytes and
    slot 0 keeps its guard bytes."""
    ps, pb = 2, [8, 4]
    page = bytes([0x11] * 8 + [0x12] * 8 + [0x21] * 4 + [0x22] * 4)
    slab = np.zeros((6, 24), np.uint8)
    slab[3] = np.frombuffer(page, np.uint8)
    cur = [np.full((1, 8), 0x31, np.uint8), np.full((1, 4), 0x41, np.uint8)]
    dense = oracle.compose_dense_planes([2], [1], [3], [slab], cur, page_size=ps, cp_size=1, plane_bytes=pb, lib=lib)
    want1 = np.frombuffer(bytes([0x31] * 8 + [0] * 8 + [0x41] * 4 + [0] * 4), np.uint8)
    assert np.array_equal(dense[0], slab[3]) and np.array_equal(dense[1], want1)
    stg = [np.full((2, 24), 0xEE, np.uint8)]
    st = oracle.fill_planes([1], [2], [0], [0], [[cur[0]], [cur[1]]], stg, page_size=ps, cp_size=1, plane_bytes=pb,
                            lib=lib)
    assert st == 0
    assert np.all(stg[0][0] == 0xEE) and np.array_equal(stg[0][1], want1)


def _split_planes(pages, ps, pb):
    """[n, ps*sum(pb)] planar pages -> list over planes of [n, ps, w_p] row pages."""
    out, start = [], 0
    for w in pb:
        out.append(pages[:, start:start + ps * w].reshape(pages.shape[0], ps, w))
        start += ps * w
    return out


def pin_planes_reduce_to_rows(lib, batch, pb=(128, 4)):
    """Plane p of the planar compose equals the row compose (width w_p) of
    plane p of every input; one plane of width R equals the row layout."""
    ps, cp = batch.page_size, batch.cp_size
    rng = np.random.default_rng(batch.seed + 77)
    pbytes = ps * sum(pb)
    slabs = [np.frombuffer(rng.bytes(batch.slab_pages * pbytes), np.uint8).reshape(batch.slab_pages, pbytes).copy()
             for _ in range(cp)]
    planes = [np.frombuffer(rng.bytes(batch.T * w), np.uint8).reshape(batch.T, w).copy() for w in pb]
    dense = oracle.compose_dense_planes(batch.prefix_lens, batch.cur_lens, batch.prefix_pages, slabs, planes,
                                        page_size=ps, cp_size=cp, plane_bytes=list(pb), lib=lib)
    dense_planes = _split_planes(dense, ps, pb)
    slab_planes = [_split_planes(s, ps, pb) for s in slabs]
    for p, w in enumerate(pb):
        want = oracle.compose_dense(batch.prefix_lens, batch.cur_lens, batch.prefix_pages,
                                    [np.ascontiguousarray(sp[p]) for sp in slab_planes], planes[p], page_size=ps,
                                    cp_size=cp, lib=lib)
        assert np.array_equal(dense_planes[p].reshape(-1, w), want), p
    # fill: plane by plane equals the row index copy
    plan = oracle.compose_plan(batch.prefix_lens, batch.cur_lens, batch.prefix_pages, batch.cur_pages, batch.writer,
                               page_size=ps, cp_size=cp, num_pool_pages=batch.num_pool_pages, lib=lib)
    tw = wl.token_writer(batch)
    per_writer = [[np.ascontiguousarray(pl[tw == w]) for w in range(cp)] for pl in planes]
    stg = [np.full((batch.C + 1, pbytes), 0x5D, np.uint8) for _ in range(cp)]
    st = oracle.fill_planes(batch.cur_lens, plan["staging_rows"], plan["token_writer_row"], batch.writer, per_writer,
                            stg, page_size=ps, cp_size=cp, plane_bytes=list(pb), lib=lib)
    assert st == 0
    for p, w in enumerate(pb):
        rows_stg = [np.ascontiguousarray(_split_planes(x, ps, pb)[p]).reshape(-1, w) for x in stg]
        ref = [np.full(((batch.C + 1) * ps, w), 0x5D, np.uint8) for _ in range(cp)]
        oracle.fill_index_copy(batch.cur_lens, plan["staging_rows"], plan["token_writer_row"], batch.writer,
                               per_writer[p], ref, page_size=ps, cp_size=cp, row_bytes=w, lib=lib)
        for x in range(cp):
            assert np.array_equal(rows_stg[x], ref[x]), (p, x)
    # one plane of width R: the row layout itself
    one = oracle.compose_dense_planes(batch.prefix_lens, batch.cur_lens, batch.prefix_pages,
                                      [s.reshape(batch.slab_pages, -1)[:, :ps * pb[0]].copy() for s in slabs],
                                      [planes[0]], page_size=ps, cp_size=cp, plane_bytes=[pb[0]], lib=lib)
    assert np.array_equal(one.reshape(-1, pb[0]), dense_planes[0].reshape(-1, pb[0]))


def pin_gather_sentinel_and_oob(lib):
    rng = np.random.default_rng(3)
    ps, R = 4, 16
    table = [np.frombuffer(rng.bytes(5 * ps * R), np.uint8).copy() for _ in range(3)]
    caps = [5, 5, 5]
    owner = np.array([0, -1, 2, 1, 3, 1, -2], np.int32)
    src = np.array([4, 9, 0, 5, 0, 2, 0], np.int32)
    dense, st = oracle.gather(table, caps, owner, src, page_size=ps, row_bytes=R, dense_cap=7, lib=lib)
    pb = ps * R
    d = dense.reshape(7, pb)
    assert np.array_equal(d[0], table[0][4 * pb:5 * pb])
    assert np.all(d[1] == 0)  # owner -1 zero-fills
    assert np.array_equal(d[2], table[2][0:pb])
    assert np.all(d[3] == 0)  # src beyond capacity
    assert np.all(d[4] == 0)  # owner beyond the table
    assert np.array_equal(d[5], table[1][2 * pb:3 * pb])
    assert np.all(d[6] == 0)
    assert st == oracle.DESC_OOB


def pin_ragged_closed_forms(lib, rb, ranks=None):
    """q_bases is the exclusive cumsum of q_lens; topk offsets are
    ``np.repeat(k_bases, q_lens)``; kv_lens / current_bases follow from the
    request; the ranks' segments tile every request's q tokens once."""
    B = rb.B
    pfx = rb.prefix_lens.astype(np.int64)
    q = rb.q_lens.astype(np.int64)
    kv_aligned = -(-(pfx + q) // rb.k_align) * rb.k_align
    kbase_req = np.concatenate([[0], np.cumsum(kv_aligned)[:-1]]) if B else np.zeros(0, np.int64)
    cover = [np.zeros(int(n), np.int32) for n in q]
    total_Q = 0
    ranks = range(rb.cp_size) if ranks is None else ranks
    for r in ranks:
        ci = rb.cp_index(r)
        got = oracle.ragged_plan(rb.prefix_lens, rb.q_lens, ci, chunk=rb.chunk, k_align=rb.k_align, lib=lib)
        assert got["status"] == 0
        S, Q = got["S"], got["Q"]
        ql = got["q_lens"].astype(np.int64)
        assert np.array_equal(got["q_bases"], np.concatenate([[0], np.cumsum(ql)[:-1]]).astype(np.int32)[:S])
        assert np.array_equal(got["topk_offsets"], np.repeat(got["k_bases"], got["q_lens"]))
        assert Q == int(ql.sum())
        req = got["seg_req"]
        assert np.array_equal(got["k_bases"], kbase_req[req])
        assert np.array_equal(got["current_bases"], kbase_req[req] + pfx[req])
        assert np.array_equal(got["kv_lens"], pfx[req] + got["q_starts"] + got["q_lens"])
        for s in range(S):
            b = int(req[s])
            cover[b][got["q_starts"][s]:got["q_starts"][s] + got["q_lens"][s]] += 1
        # segments are maximal: two adjacent segments of one request do not abut
        for s in range(1, S):
            if req[s] == req[s - 1]:
                assert got["q_starts"][s] > got["q_starts"][s - 1] + got["q_lens"][s - 1]
        total_Q += Q
    if ranks == range(rb.cp_size):
        assert total_Q == int(q.sum())
        for b in range(B):
            assert np.all(cover[b] == 1), b


def pin_ragged_cp1(lib, rb):
    """cp = 1 owns every chunk: one segment per non-empty request, starting at
    0 and ending at the request's full kv length."""
    n = rb.num_chunks
    got = oracle.ragged_plan(rb.prefix_lens, rb.q_lens, np.arange(n, dtype=np.int32), chunk=rb.chunk,
                             k_align=rb.k_align, lib=lib)
    nz = np.nonzero(rb.q_lens > 0)[0]
    assert got["S"] == len(nz)
    assert np.array_equal(got["seg_req"], nz)
    assert np.all(got["q_starts"] == 0)
    assert np.array_equal(got["q_lens"], rb.q_lens[nz])
    assert np.array_equal(got["kv_lens"], rb.prefix_lens[nz] + rb.q_lens[nz])


def pin_errors(lib):
    # unaligned prefix -> error code, capacity -> error code
    try:
        oracle.compose_plan([3], [4], [1], [2], [0], page_size=2, cp_size=1, num_pool_pages=8, lib=lib)
        raise AssertionError("unaligned prefix accepted")
    except oracle.OracleError as e:
        assert "-2" in str(e)
    try:
        oracle.compose_plan([2], [4], [1], [2, 3], [0, 0], page_size=2, cp_size=1, num_pool_pages=8,
                            dense_cap=2, lib=lib)
        raise AssertionError("capacity accepted")
    except oracle.OracleError as e:
        assert "-3" in str(e)
    # data violations -> status bits
    p = oracle.compose_plan([0, 0], [2, 2], [], [3, 3], [0, 1], page_size=2, cp_size=2, num_pool_pages=8, lib=lib)
    assert p["status"] & oracle.DUP_CURRENT_PAGE
    p = oracle.compose_plan([2], [2], [5], [5], [0], page_size=2, cp_size=1, num_pool_pages=8, lib=lib)
    assert p["status"] & oracle.CURRENT_IN_PREFIX
    p = oracle.compose_plan([2], [2], [0], [5], [0], page_size=2, cp_size=1, num_pool_pages=8, lib=lib)
    assert p["status"] & oracle.PAGE_OOB
    p = oracle.compose_plan([0], [2], [], [5], [3], page_size=2, cp_size=2, num_pool_pages=8, lib=lib)
    assert p["status"] & oracle.WRITER_OOB
    # shared prefix page across two requests is allowed; the inverse keeps the smaller slot
    p = oracle.compose_plan([2, 2], [1, 1], [4, 4], [5, 6], [0, 0], page_size=2, cp_size=1, num_pool_pages=8, lib=lib)
    assert p["status"] == 0 and p["page_inverse"][4] == 0
    # ragged: unsorted cp_index -> status bit
    r = oracle.ragged_plan([0, 0], [8, 8], [2, 1], chunk=4, lib=lib)
    assert r["status"] & oracle.CHUNK_OOB


# ---------------------------------------------------------------------------
# edge-case batches
# ---------------------------------------------------------------------------

def edge_batches():
    """Seeded small batches covering the degenerate cases of the method."""
    out = [wl.tiny_batch()]
    R = 64
    mk = wl.make_compose_batch
    out.append(mk("no_prefix", 11, page_size=4, cp_size=2, num_pool_pages=64, row_bytes=R,
                  prefix_lens=[0, 0, 0], cur_lens=[5, 8, 1], row_kind="bytes"))
    out.append(mk("no_current", 12, page_size=4, cp_size=3, num_pool_pages=64, row_bytes=R,
                  prefix_lens=[8, 4, 0], cur_lens=[0, 0, 0], row_kind="bytes"))
    out.append(mk("exact_multiple", 13, page_size=4, cp_size=2, num_pool_pages=64, row_bytes=R,
                  prefix_lens=[4, 12], cur_lens=[8, 4], row_kind="bytes"))
    out.append(mk("one_request", 14, page_size=8, cp_size=4, num_pool_pages=64, row_bytes=R,
                  prefix_lens=[16], cur_lens=[21], row_kind="bytes"))
    out.append(mk("cp1", 15, page_size=4, cp_size=1, num_pool_pages=64, row_bytes=R,
                  prefix_lens=[8, 0, 4], cur_lens=[3, 9, 4], row_kind="bytes"))
    out.append(mk("empty_batch", 16, page_size=4, cp_size=2, num_pool_pages=16, row_bytes=R,
                  prefix_lens=[], cur_lens=[], row_kind="bytes"))
    # shared radix prefix: both requests reuse logical pages 9 and 17
    out.append(mk("shared_prefix", 17, page_size=4, cp_size=2, num_pool_pages=64, row_bytes=R,
                  prefix_lens=[8, 12], cur_lens=[3, 6], prefix_pages=[9, 17, 9, 17, 30],
                  cur_pages=[40, 41, 42], row_kind="bytes"))
    # a request shaped like a chunked-prefill chunk (2048 prefix tokens, 512 new tokens) beside a short one
    out.append(mk("chunk_shaped", 18, page_size=64, cp_size=8, num_pool_pages=256, row_bytes=R,
                  prefix_lens=[2048, 64], cur_lens=[512, 37], row_kind="bytes"))
    # writers not round-robin: all current pages on one rank, others idle
    out.append(mk("one_writer", 19, page_size=4, cp_size=4, num_pool_pages=64, row_bytes=R,
                  prefix_lens=[4, 8], cur_lens=[7, 6], writer=[2, 2, 2, 2], row_kind="bytes"))
    # contiguous in-seq split of each request's current pages over the writers
    cur = [37, 9, 64, 20]
    out.append(mk("contiguous_writers", 20, page_size=8, cp_size=3, num_pool_pages=128, row_bytes=R,
                  prefix_lens=[16, 0, 8, 24], cur_lens=cur, writer=wl.contiguous_writers(cur, 8, 3),
                  row_kind="bytes"))
    return out


def ragged_edge_batches():
    out = []
    rng = np.random.default_rng(21)
    for cp, chunk, B, k_align in ((2, 4, 5, 1), (3, 8, 7, 1), (4, 16, 9, 16), (8, 64, 12, 64), (1, 4, 4, 1)):
        q = rng.integers(0, 5 * chunk, size=B).astype(np.int32)
        pfx = rng.integers(0, 100, size=B).astype(np.int32)
        out.append(wl.RaggedBatch(f"ragged_cp{cp}", 21, cp, chunk, k_align, pfx, q))
    # the other CP splits: contiguous in-seq blocks and zigzag (2*cp slots per request)
    for split in ("contiguous", "zigzag"):
        for cp, chunk, B in ((2, 4, 6), (4, 8, 9), (8, 64, 12)):
            q = rng.integers(0, 20 * chunk, size=B).astype(np.int32)
            pfx = rng.integers(0, 300, size=B).astype(np.int32)
            out.append(wl.RaggedBatch(f"ragged_{split}_cp{cp}", 22, cp, chunk, 1, pfx, q, split=split))
    return out


ALL_PINS = [
    ("golden_compose", lambda lib: pin_golden_compose(lib)),
    ("golden_ragged", lambda lib: pin_golden_ragged(lib)),
    ("cp1_index_select_cat", lambda lib: pin_cp1_index_select_cat(lib)),
    ("gather_sentinel", lambda lib: pin_gather_sentinel_and_oob(lib)),
    ("fill_index_copy_permuted", lambda lib: pin_fill_index_copy_permuted(lib)),
    ("planes_golden", lambda lib: pin_planes_golden(lib)),
    ("planes_reduce_to_rows", lambda lib: [pin_planes_reduce_to_rows(lib, b) for b in edge_batches() if b.B > 0]),
    ("fill_index_copy", lambda lib: [pin_fill_index_copy(lib, b) for b in edge_batches()]),
    ("errors", lambda lib: pin_errors(lib)),
    ("plan_brute_force", lambda lib: [pin_plan_brute_force(lib, b, 2) for b in edge_batches()]),
    ("dense_token_level", lambda lib: [pin_dense_token_level(lib, b, 1) for b in edge_batches()]),
    ("roundtrip", lambda lib: [pin_staging_gather_roundtrip(lib, b, 1) for b in edge_batches()]),
    ("ragged_closed_forms", lambda lib: [pin_ragged_closed_forms(lib, rb) for rb in ragged_edge_batches()]),
    ("ragged_cp1", lambda lib: [pin_ragged_cp1(lib, rb) for rb in ragged_edge_batches()]),
]
