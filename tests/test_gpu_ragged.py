"""GPU parity of the ragged index plan against the CPU oracle (byte-exact)."""
import numpy as np
import pytest
import torch

import oracle
import oracle_pins as pins
import workloads as wl
from paged_kv_cache_compose_gb300 import cpkv

pytestmark = pytest.mark.gpu

KEYS = ("seg_req", "kv_lens", "q_starts", "q_lens", "k_bases", "q_bases", "current_bases")


def _gpu_ragged(rb, rank, cp_index=None, seg_extra=3, topk_extra=5):
    ci = rb.cp_index(rank) if cp_index is None else np.asarray(cp_index, np.int32)
    S, Q = cpkv.cpkv_ragged_plan_sizes(rb.q_lens, ci, rb.chunk)
    out = cpkv.ragged_buffers(S + seg_extra, Q + topk_extra)
    for t in out.values():
        t.fill_(-9)
    counts = torch.full((2,), -1, dtype=torch.int64, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    d_ci = torch.from_numpy(ci.astype(np.int32)).cuda()
    cpkv.cpkv_ragged_plan_build(rb.prefix_lens, rb.q_lens, d_ci, len(ci), chunk=rb.chunk, k_align=rb.k_align, topk=rb.topk,
                                out=out, d_counts=counts, d_status=status)
    torch.cuda.synchronize()
    return out, counts.cpu().numpy(), int(status.item()), (S, Q)


def _check_rank(rb, rank):
    want = oracle.ragged_plan(rb.prefix_lens, rb.q_lens, rb.cp_index(rank), chunk=rb.chunk, k_align=rb.k_align)
    out, counts, status, (S, Q) = _gpu_ragged(rb, rank)
    assert status == 0
    assert (S, Q) == (want["S"], want["Q"])
    assert counts.tolist() == [want["S"], want["Q"]]
    for k in KEYS:
        got = out[k].cpu().numpy()
        assert np.array_equal(got[:S], want[k]), k
        assert np.all(got[S:] == -9), k  # nothing written past S
    got = out["topk_offsets"].cpu().numpy()
    assert np.array_equal(got[:Q], want["topk_offsets"])
    assert np.all(got[Q:] == -9)


@pytest.mark.parametrize("rank", range(8))
def test_ragged_config_all_ranks(rank):
    _check_rank(wl.ragged_batch(), rank)


@pytest.mark.parametrize("rb", pins.ragged_edge_batches(), ids=lambda r: r.name)
def test_ragged_edge_cases(rb):
    for rank in range(rb.cp_size):
        _check_rank(rb, rank)


def test_ragged_cp1_many_tiles():
    """cp = 1 owns every chunk: more than one 1024-chunk tile, several CTAs."""
    rb = wl.ragged_batch()
    rb = wl.RaggedBatch("cp1", rb.seed, 1, rb.chunk, 1, rb.prefix_lens, rb.q_lens)
    assert rb.num_chunks > 2048
    _check_rank(rb, 0)


def test_ragged_traced_batch_view():
    rb = wl.ragged_from_compose(wl.traced_batch())
    for rank in range(rb.cp_size):
        _check_rank(rb, rank)


def test_ragged_large_batch_and_alignment():
    rng = np.random.default_rng(77)
    B = 200
    rb = wl.RaggedBatch("b200", 77, 4, 32, 64, rng.integers(0, 3000, B).astype(np.int32),
                        rng.integers(0, 400, B).astype(np.int32))
    for rank in range(4):
        _check_rank(rb, rank)


def test_ragged_empty_rank_and_bad_index():
    rb = wl.RaggedBatch("tiny", 1, 4, 8, 1, np.array([3, 5], np.int32), np.array([4, 2], np.int32))
    # 2 chunks in total: ranks 2 and 3 own nothing
    out, counts, status, (S, Q) = _gpu_ragged(rb, 3)
    assert status == 0 and counts.tolist() == [0, 0] and (S, Q) == (0, 0)
    # a descending cp_index is flagged on the device
    out, counts, status, _ = _gpu_ragged(rb, 0, cp_index=[0, 1], seg_extra=2, topk_extra=8)
    assert status == 0
    bad = torch.from_numpy(np.array([1, 0], np.int32)).cuda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    cnt = torch.zeros(2, dtype=torch.int64, device="cuda")
    cpkv.cpkv_ragged_plan_build(rb.prefix_lens, rb.q_lens, bad, 2, chunk=8, k_align=1, topk=2048, out=out, d_counts=cnt,
                                d_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & cpkv.STATUS_CHUNK_OOB
