"""Multi-process aggregation of bench.py's replicas (world size 2, gloo, CPU).

The compose path does not shard: N GPUs run N independent replicas.  The only
cross-rank step is timing: the slowest rank's time and the sum of all ranks'
bytes."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, ws, port, q):
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    import bench

    ms, units = bench.aggregate(10.0 + 5.0 * rank, 1000 * (rank + 1), ws)
    q.put((rank, ms, units))
    dist.destroy_process_group()


def test_aggregate_max_time_sum_units():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get() for _ in range(2))
    for _, ms, units in res:
        assert ms == 15.0 and units == 3000.0


def test_bench_single_process_aggregate_is_identity():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.aggregate(7.5, 42, 1) == (7.5, 42.0)


def test_layer_bytes_accounting():
    sys.path.insert(0, ROOT)
    import bench
    import workloads as wl

    b = wl.traced_batch()
    lb = bench.layer_bytes(b.prefix_lens, b.cur_lens, b.page_size, b.row_bytes, 2091)
    assert lb["T"] == 44600 and lb["D"] == 2091
    assert lb["gather"] == 2 * 2091 * 64 * 1152
    assert lb["fill_read"] == 44600 * 1152
    assert lb["total"] == lb["fill"] + lb["gather"]
