"""CPU model of the compose plan's two-level per-writer row bases.

The plan kernel takes each current page's row base (the row of its first
token in its writer's current-row buffer) from per-block writer totals in a
workspace (an exclusive sum over the blocks before it) plus a scan over the
warps of its block plus the lanes below it in its warp.  This model runs the
same decomposition in numpy, with the block size the library uses, and
compares every token's row with the oracle's ``token_writer_row``.  It also
checks the workspace size that the library reports and that a short
workspace is refused before any launch."""
import numpy as np
import pytest

import oracle
import oracle_pins as pins
import workloads as wl
from paged_kv_cache_compose_gb300 import build as cuda_build
from paged_kv_cache_compose_gb300 import cpkv


def pages_per_block(ps):
    k = 2048 // ps
    k = (k + 31) // 32 * 32
    return int(min(max(k, 32), 1024))


def model_token_writer_row(batch):
    ps, cp = batch.page_size, batch.cp_size
    cur = np.asarray(batch.cur_lens, np.int64)
    ncp = (cur + ps - 1) // ps
    C = int(ncp.sum())
    n = np.empty(C, np.int64)  # rows of each current page
    tok0 = np.empty(C, np.int64)
    i, t = 0, 0
    for b in range(batch.B):
        for k in range(int(ncp[b])):
            n[i] = min(ps, int(cur[b]) - k * ps)
            tok0[i] = t + k * ps
            i += 1
        t += int(cur[b])
    w = np.asarray(batch.writer, np.int64)
    K = pages_per_block(ps)
    NB = -(-C // K)
    block_rows = np.zeros((NB, cp), np.int64)  # first kernel: totals per block
    for j in range(NB):
        for q in range(j * K, min(C, (j + 1) * K)):
            block_rows[j, w[q]] += n[q]
    out = np.full(int(cur.sum()), -1, np.int64)
    for j in range(NB):  # second kernel, one block
        base = block_rows[:j].sum(axis=0)  # blocks before this one
        pages = range(j * K, min(C, (j + 1) * K))
        warp_rows = np.zeros((32, cp), np.int64)
        before = {}
        for q in pages:
            t_ = q - j * K
            warp, lane = t_ // 32, t_ % 32
            first = j * K + warp * 32
            before[q] = sum(int(n[r]) for r in range(first, q) if w[r] == w[q])
            warp_rows[warp, w[q]] += n[q]
        scanned = np.cumsum(warp_rows, axis=0) - warp_rows + base  # exclusive over warps
        for q in pages:
            warp = (q - j * K) // 32
            rb = scanned[warp, w[q]] + before[q]
            out[tok0[q]:tok0[q] + n[q]] = rb + np.arange(n[q])
    return out, NB


def _batches():
    out = list(pins.edge_batches())
    out.append(wl.traced_batch())
    tb = wl.traced_batch()
    rng = np.random.default_rng(5)
    out.append(wl.make_compose_batch("ps1", 5, page_size=1, cp_size=8, num_pool_pages=1 << 18, row_bytes=16,
                                     prefix_lens=tb.prefix_lens, cur_lens=tb.cur_lens, rng=rng))
    rng = np.random.default_rng(6)
    cur = rng.integers(1, 400, 40)
    out.append(wl.make_compose_batch("ps3-random-writers", 6, page_size=3, cp_size=7, num_pool_pages=20000,
                                     row_bytes=16, prefix_lens=np.zeros(40, np.int64), cur_lens=cur,
                                     writer=rng.integers(0, 7, int(((cur + 2) // 3).sum())), rng=rng))
    return out


@pytest.mark.parametrize("batch", _batches(), ids=lambda b: b.name)
def test_two_level_row_bases_match_oracle(batch):
    want = oracle.compose_plan(batch.prefix_lens, batch.cur_lens, batch.prefix_pages, batch.cur_pages,
                               batch.writer, page_size=batch.page_size, cp_size=batch.cp_size,
                               num_pool_pages=batch.num_pool_pages)["token_writer_row"]
    got, NB = model_token_writer_row(batch)
    assert np.array_equal(got, want)
    cuda_build.build()
    assert cpkv.cpkv_plan_workspace_bytes(batch.cur_lens, batch.page_size, batch.cp_size) == NB * batch.cp_size * 4


def test_short_workspace_is_refused_before_any_launch():
    cuda_build.build()
    lib = cpkv.load()
    b = wl.traced_78_token_pages_batch()  # 44 600 current pages in 44 blocks
    need = cpkv.cpkv_plan_workspace_bytes(b.cur_lens, b.page_size, b.cp_size)
    assert need > 0
    pl = np.ascontiguousarray(b.prefix_lens, np.int32)
    cl = np.ascontiguousarray(b.cur_lens, np.int32)
    fake = 256  # never dereferenced: the call returns before launching
    args = [b.B, b.page_size, b.cp_size, b.num_pool_pages, pl.ctypes.data, cl.ctypes.data, fake, fake, fake,
            1_000_000] + [fake] * 9
    assert lib.cpkv_plan_build(*args, fake, need - 4, fake, None) == cpkv.CPKV_ERR_CAPACITY
    assert lib.cpkv_plan_build(*args, None, need, fake, None) == cpkv.CPKV_ERR_ARG
    assert lib.cpkv_plan_build(*args, fake + 2, need, fake, None) == cpkv.CPKV_ERR_ARG


def test_workspace_is_small():
    cuda_build.build()
    # traced: 703 pages in blocks of 32; fp8: 2065 in blocks of 32; one-token
    # pages: 44 600 in blocks of 1024; 8 writers, 4 bytes each
    for batch, blocks in ((wl.traced_batch(), 22), (wl.fp8_nsa_batch(), 65), (wl.traced_78_token_pages_batch(), 44)):
        assert cpkv.cpkv_plan_workspace_bytes(batch.cur_lens, batch.page_size, batch.cp_size) == blocks * 8 * 4
    assert cpkv.cpkv_plan_workspace_bytes([0, 0], 16, 4) == 0
    assert cpkv.cpkv_plan_workspace_bytes([4097], 1, 4) == 5 * 4 * 4
