"""Seeded random shapes through every entry point, byte-exact against the oracle.

Each case draws a batch (requests, page size, cp, row width, prefix/current
lengths, writer assignment, shared prefix pages, capacity padding) from a
fixed seed, runs the plan, the fill + gather, the one-launch layer compose, the fused
compose and the prefix/current split on the GPU, plain and as chains of early launches,
and the ragged plan for every rank, and compares everything with the CPU oracle.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from paged_kv_cache_compose_gb300 import cpkv
from paged_kv_cache_compose_gb300.runtime import ComposeLayers, ComposePlan

pytestmark = pytest.mark.gpu

PLAN_KEYS = ("prefix_spans", "cur_spans", "owner", "src", "page_inverse", "staging_page_inverse", "mixed_locs",
             "staging_rows", "token_writer_row")


def random_batch(seed):
    rng = np.random.default_rng(seed)
    ps = int(rng.choice([1, 2, 3, 4, 8, 16, 32, 64, 128]))
    cp = int(rng.integers(1, 13))
    R = 16 * int(rng.integers(1, 90))
    B = int(rng.integers(0, 33))
    pfx = rng.integers(0, 6, size=B) * ps
    cur = rng.integers(0, 5 * ps + 1, size=B)
    n_pfx = int((pfx // ps).sum())
    C = int(((cur + ps - 1) // ps).sum())
    P = n_pfx + C + int(rng.integers(2, 40))
    ids = rng.permutation(np.arange(1, P))
    prefix_pages = ids[:n_pfx].copy()
    if n_pfx > 2 and rng.random() < 0.5:  # a shared radix prefix: one page repeated
        prefix_pages[rng.integers(0, n_pfx)] = prefix_pages[0]
    cur_pages = ids[n_pfx:n_pfx + C]
    mode = rng.integers(0, 3)
    if mode == 0:
        writer = wl.round_robin_writers(C, cp)
    elif mode == 1:
        writer = wl.contiguous_writers(cur, ps, cp)
    else:
        writer = rng.integers(0, cp, size=C).astype(np.int32)
    return wl.make_compose_batch(f"fuzz{seed}", seed, page_size=ps, cp_size=cp, num_pool_pages=P, row_bytes=R,
                                 prefix_lens=pfx, cur_lens=cur, prefix_pages=prefix_pages, cur_pages=cur_pages,
                                 writer=writer, row_kind="bytes"), int(rng.integers(0, 4))


@pytest.mark.parametrize("seed", range(40))
def test_fuzz_compose(seed):
    batch, extra = random_batch(seed)
    ps, cp, R = batch.page_size, batch.cp_size, batch.row_bytes
    T, C, D = oracle.sizes(batch.prefix_lens, batch.cur_lens, ps)
    cap = D + extra
    want_plan = oracle.compose_plan(batch.prefix_lens, batch.cur_lens, batch.prefix_pages, batch.cur_pages,
                                    batch.writer, page_size=ps, cp_size=cp, num_pool_pages=batch.num_pool_pages,
                                    dense_cap=cap)
    plan = ComposePlan(batch.prefix_lens, batch.cur_lens, batch.prefix_pages, batch.cur_pages, batch.writer,
                       page_size=ps, cp_size=cp, num_pool_pages=batch.num_pool_pages, dense_cap_pages=cap)
    for t in plan.bufs.values():
        if t.numel():
            t.fill_(-3)
    plan.build()
    layers = ComposeLayers(plan, R)
    slabs = wl.host_pool(batch)
    rows = wl.host_current_rows(batch)
    d_slabs = [torch.from_numpy(s).cuda() for s in slabs]
    d_rows = [torch.from_numpy(r).cuda() for r in wl.split_rows_by_writer(batch, rows)]
    for s in layers.staging:
        s.fill_(0x42)
    dense = torch.full((cap * ps, R), 0xCD, dtype=torch.uint8, device="cuda")
    fused = torch.full((cap * ps, R), 0xCE, dtype=torch.uint8, device="cuda")
    split = torch.full((cap * ps, R), 0xCF, dtype=torch.uint8, device="cuda")
    layers.fill(d_rows)
    layers.gather(d_slabs, dense)
    layers.compose_fused(d_slabs, d_rows, fused)
    layers.prefetch(d_slabs, split)
    layers.consume(d_rows, split)
    torch.cuda.synchronize()
    assert int(plan.d_status.item()) == want_plan["status"] == 0
    for k in PLAN_KEYS:
        assert np.array_equal(plan[k].cpu().numpy().reshape(want_plan[k].shape), want_plan[k]), k
    want = oracle.compose_dense(batch.prefix_lens, batch.cur_lens, batch.prefix_pages, slabs, rows, page_size=ps,
                                cp_size=cp, dense_cap=cap)
    assert np.array_equal(dense.cpu().numpy(), want)
    assert np.array_equal(fused.cpu().numpy(), want)
    assert np.array_equal(split.cpu().numpy(), want)
    stg = [s.cpu().numpy() for s in layers.staging]
    want_stg = [np.full_like(s, 0x42) for s in stg]
    oracle.staging(batch.cur_lens, batch.writer, rows, want_stg, page_size=ps, cp_size=cp)
    for w in range(cp):
        assert np.array_equal(stg[w], want_stg[w]), w
    # the one-launch layer compose: same dense buffer, same stagings
    for s in layers.staging:
        s.fill_(0x42)
    one = torch.full((cap * ps, R), 0xD1, dtype=torch.uint8, device="cuda")
    layers.compose_one_launch(d_slabs, d_rows, one)
    torch.cuda.synchronize()
    assert int(plan.d_status.item()) == 0
    assert np.array_equal(one.cpu().numpy(), want)
    for w in range(cp):
        assert np.array_equal(layers.staging[w].cpu().numpy(), want_stg[w]), w


@pytest.mark.parametrize("seed", range(100, 120))
def test_fuzz_early_launch_chains(seed):
    """Three layers of distinct inputs, uploaded first, through each chain of
    early launches (CPKV_FLAG_EARLY_INPUTS, CPKV_GATHER_EARLY_INPUTS): fill +
    gather, the fused compose and the one-launch layer compose.  Every
    layer has its own dense buffer and is checked against the oracle.  Odd
    seeds widen the rows to pages of about 40 KB, several pieces for every
    kernel, so the early launches are taken (one-piece pages launch the
    gather and the one-launch kernels plainly)."""
    batch, extra = random_batch(seed)
    if seed % 2:
        batch = dataclasses.replace(batch, row_bytes=16 * -(-40960 // (batch.page_size * 16)))
    ps, cp, R = batch.page_size, batch.cp_size, batch.row_bytes
    T, C, D = oracle.sizes(batch.prefix_lens, batch.cur_lens, ps)
    cap = D + extra
    plan = ComposePlan(batch.prefix_lens, batch.cur_lens, batch.prefix_pages, batch.cur_pages, batch.writer,
                       page_size=ps, cp_size=cp, num_pool_pages=batch.num_pool_pages, dense_cap_pages=cap).build()
    layers = ComposeLayers(plan, R)
    n_layers, consume = 3, seed % 2 == 0
    host = [(wl.host_pool(batch, l), wl.host_current_rows(batch, l)) for l in range(n_layers)]
    dev = [([torch.from_numpy(s).cuda() for s in slabs],
            [torch.from_numpy(r).cuda() for r in wl.split_rows_by_writer(batch, rows)]) for slabs, rows in host]
    out = {k: [torch.full((cap * ps, R), 0xCD, dtype=torch.uint8, device="cuda") for _ in range(n_layers)]
           for k in ("staging", "fused", "layer")}
    torch.cuda.synchronize()
    for l in range(n_layers):
        layers.fill(dev[l][1], early_inputs=True)
        layers.gather(dev[l][0], out["staging"][l], consume_staging=consume, early_inputs=True)
    for l in range(n_layers):
        layers.compose_fused(dev[l][0], dev[l][1], out["fused"][l], early_inputs=True)
    for l in range(n_layers):
        layers.compose_one_launch(dev[l][0], dev[l][1], out["layer"][l], consume_staging=consume,
                                  early_inputs=True)
    torch.cuda.synchronize()
    assert int(plan.d_status.item()) == 0
    for l, (slabs, rows) in enumerate(host):
        want = oracle.compose_dense(batch.prefix_lens, batch.cur_lens, batch.prefix_pages, slabs, rows,
                                    page_size=ps, cp_size=cp, dense_cap=cap)
        for k, bufs in out.items():
            assert np.array_equal(bufs[l].cpu().numpy(), want), (k, l)


def small_pages_large_batch(seed):
    """B in [65, 300] (the 1024-request parameter block), pages of 1-3
    tokens and at most 4 KB (the grouped kernels), random writers."""
    rng = np.random.default_rng(20_000 + seed)
    ps = int(rng.choice([1, 2, 3]))
    cp = int(rng.integers(1, 9))
    R = 16 * int(rng.integers(1, 4096 // (16 * ps) + 1))
    B = int(rng.integers(65, 301))
    pfx = rng.integers(0, 8, size=B) * ps
    cur = rng.integers(0, 6 * ps + 1, size=B)
    n_pfx = int((pfx // ps).sum())
    C = int(((cur + ps - 1) // ps).sum())
    P = n_pfx + C + 8
    ids = rng.permutation(np.arange(1, P))
    writer = rng.integers(0, cp, size=C).astype(np.int32)
    return wl.make_compose_batch(f"big{seed}", seed, page_size=ps, cp_size=cp, num_pool_pages=P, row_bytes=R,
                                 prefix_lens=pfx, cur_lens=cur, prefix_pages=ids[:n_pfx].copy(),
                                 cur_pages=ids[n_pfx:n_pfx + C], writer=writer, row_kind="bytes")


@pytest.mark.parametrize("seed", range(8))
def test_fuzz_early_chains_small_pages_large_batch(seed):
    """Three layers through each chain of early launches on pages of at most
    4 KB with more than 64 requests: the row fill + group gather, the grouped
    fused compose and the grouped one-launch compose (stagings consumed on
    even seeds), every layer against the oracle."""
    batch = small_pages_large_batch(seed)
    ps, cp, R = batch.page_size, batch.cp_size, batch.row_bytes
    assert ps * R <= 4096 and batch.B > 64
    T, C, D = oracle.sizes(batch.prefix_lens, batch.cur_lens, ps)
    cap = D + 3
    plan = ComposePlan(batch.prefix_lens, batch.cur_lens, batch.prefix_pages, batch.cur_pages, batch.writer,
                       page_size=ps, cp_size=cp, num_pool_pages=batch.num_pool_pages, dense_cap_pages=cap).build()
    layers = ComposeLayers(plan, R)
    n_layers, consume = 3, seed % 2 == 0
    host = [(wl.host_pool(batch, l), wl.host_current_rows(batch, l)) for l in range(n_layers)]
    dev = [([torch.from_numpy(s).cuda() for s in slabs],
            [torch.from_numpy(r).cuda() for r in wl.split_rows_by_writer(batch, rows)]) for slabs, rows in host]
    out = {k: [torch.full((cap * ps, R), 0xCD, dtype=torch.uint8, device="cuda") for _ in range(n_layers)]
           for k in ("staging", "fused", "layer")}
    torch.cuda.synchronize()
    for l in range(n_layers):
        layers.fill(dev[l][1], early_inputs=True)
        layers.gather(dev[l][0], out["staging"][l], consume_staging=consume, early_inputs=True)
    for l in range(n_layers):
        layers.compose_fused(dev[l][0], dev[l][1], out["fused"][l], early_inputs=True)
    for l in range(n_layers):
        layers.compose_one_launch(dev[l][0], dev[l][1], out["layer"][l], consume_staging=consume,
                                  early_inputs=True)
    torch.cuda.synchronize()
    assert int(plan.d_status.item()) == 0
    for l, (slabs, rows) in enumerate(host):
        want = oracle.compose_dense(batch.prefix_lens, batch.cur_lens, batch.prefix_pages, slabs, rows,
                                    page_size=ps, cp_size=cp, dense_cap=cap)
        for k, bufs in out.items():
            assert np.array_equal(bufs[l].cpu().numpy(), want), (k, l)


@pytest.mark.parametrize("seed", range(30))
def test_fuzz_ragged(seed):
    rng = np.random.default_rng(10_000 + seed)
    cp = int(rng.integers(1, 9))
    chunk = int(rng.choice([1, 4, 16, 64, 128]))
    B = int(rng.integers(0, 80))
    split = str(rng.choice(["interleaved", "contiguous", "zigzag"]))
    rb = wl.RaggedBatch(f"r{seed}", seed, cp, chunk, int(rng.choice([1, 8, 64])),
                        rng.integers(0, 3000, size=B).astype(np.int32),
                        rng.integers(0, 40 * chunk, size=B).astype(np.int32), split=split)
    for rank in range(cp):
        ci = rb.cp_index(rank)
        want = oracle.ragged_plan(rb.prefix_lens, rb.q_lens, ci, chunk=chunk, k_align=rb.k_align)
        S, Q = cpkv.cpkv_ragged_plan_sizes(rb.q_lens, ci, chunk)
        assert (S, Q) == (want["S"], want["Q"])
        out = cpkv.ragged_buffers(S + 1, Q + 1)
        counts = torch.zeros(2, dtype=torch.int64, device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        cpkv.cpkv_ragged_plan_build(rb.prefix_lens, rb.q_lens, torch.from_numpy(ci).cuda(), len(ci), chunk=chunk,
                                    k_align=rb.k_align, topk=rb.topk, out=out, d_counts=counts, d_status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == want["status"] == 0
        assert counts.cpu().tolist() == [S, Q]
        for k in ("seg_req", "kv_lens", "q_starts", "q_lens", "k_bases", "q_bases", "current_bases"):
            assert np.array_equal(out[k].cpu().numpy()[:S], want[k]), (k, rank)
        assert np.array_equal(out["topk_offsets"].cpu().numpy()[:Q], want["topk_offsets"])
