"""The compose plan for callers that cannot allocate device memory.

``cpkv_plan_build_noalloc`` builds the same plan as ``cpkv_plan_build`` but
takes no workspace from the caller: it uses a fixed array in device memory
that the library owns (for plugins inside a framework whose allocator owns
all device memory, or servers that reserved all of HBM up front).  These
checks call it through the C ABI twice in a row, on batches that need its
workspace (many blocks of current pages), and compare every output array
with what ``cpkv_plan_build`` writes for the same batch, byte for byte.  The
file is named to be collected last, so a run that stops at its first failure
has run every other test before this one; it also passes alone in a fresh
process (its first call sets the array up).
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads as wl
from paged_kv_cache_compose_gb300 import cpkv
from paged_kv_cache_compose_gb300.runtime import ComposePlan

pytestmark = pytest.mark.gpu

PLAN_KEYS = ("prefix_spans", "cur_spans", "owner", "src", "page_inverse", "staging_page_inverse", "mixed_locs",
             "staging_rows", "token_writer_row")


def _random_writer_batch(seed=21, ps=3, cp=7, B=40):
    rng = np.random.default_rng(seed)
    cur = rng.integers(1, 2000, B)
    pfx = (rng.integers(0, 6000, B) // ps) * ps
    C = int(((cur + ps - 1) // ps).sum())
    P = int((pfx // ps).sum() + C + 10)
    return wl.make_compose_batch("ps3-random", seed, page_size=ps, cp_size=cp, num_pool_pages=P, row_bytes=16,
                                 prefix_lens=pfx, cur_lens=cur, writer=rng.integers(0, cp, C), row_kind="bytes",
                                 rng=rng)


def _noalloc_plan(batch):
    """Output buffers (poisoned) for a no-allocation build of ``batch``, and
    the call that fills them."""
    ref = ComposePlan(batch.prefix_lens, batch.cur_lens, batch.prefix_pages, batch.cur_pages, batch.writer,
                      page_size=batch.page_size, cp_size=batch.cp_size, num_pool_pages=batch.num_pool_pages)
    out = cpkv.plan_buffers(ref.B, ref.T, ref.dense_cap_pages, batch.num_pool_pages, "cuda")
    for t in out.values():
        if t.numel():
            t.fill_(-7)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")

    def call():
        cpkv.cpkv_plan_build_noalloc(batch.prefix_lens, batch.cur_lens, ref.d_prefix_pages, ref.d_cur_pages,
                                     ref.d_writer, page_size=batch.page_size, cp_size=batch.cp_size,
                                     num_pool_pages=batch.num_pool_pages, dense_cap_pages=ref.dense_cap_pages,
                                     out=out, d_status=status)
    return ref, out, status, call


def test_noalloc_plan_matches_the_workspace_plan_twice_in_a_row():
    batches = [wl.traced_78_token_pages_batch(), _random_writer_batch()]
    for b in batches:  # both need the fixed array: 44 and 22 blocks of current pages
        assert 0 < cpkv.cpkv_plan_workspace_bytes(b.cur_lens, b.page_size, b.cp_size) <= 64 * 1024
    runs = [_noalloc_plan(b) for b in batches]
    torch.cuda.synchronize()
    for _, _, _, call in runs:  # two calls in a row on one stream, sharing the array
        call()
    for ref, _, _, _ in runs:  # the existing entry point, with a caller workspace
        ref.build()
    torch.cuda.synchronize()
    for b, (ref, out, status, _) in zip(batches, runs):
        assert int(status.item()) == 0 and int(ref.d_status.item()) == 0, b.name
        for k in PLAN_KEYS:
            assert torch.equal(out[k], ref[k]), (b.name, k)


def test_noalloc_plan_refuses_a_batch_beyond_its_array():
    """A batch whose workspace exceeds the fixed 64 KiB gets CPKV_ERR_LIMIT
    before anything is launched (host lengths only; the device pointers are
    never used)."""
    lib = cpkv.load()
    ps, cp = 64, 64
    cl = np.array([600_000], np.int32)  # 9375 current pages, 293 blocks x 64 writers x 4 B > 64 KiB
    pl = np.zeros(1, np.int32)
    assert cpkv.cpkv_plan_workspace_bytes(cl, ps, cp) > 64 * 1024
    fake = ctypes.c_void_p(256)
    rc = lib.cpkv_plan_build_noalloc(1, ps, cp, 20_000, pl.ctypes.data, cl.ctypes.data, fake, fake, fake, 10_000,
                                     *([fake] * 10), None)
    assert rc == cpkv.CPKV_ERR_LIMIT
