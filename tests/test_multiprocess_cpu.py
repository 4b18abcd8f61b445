"""The N > 1 path of bench.py on CPU: world_size-2 gloo ranks.

The hot path shards by independent problems (sequences, heads), so ranks run
their own replicas with no data-path collective; the only cross-rank steps are
the barrier and the max-over-ranks timing reduction checked here."""
import multiprocessing as mp
import os
import socket

import pytest


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    out = bench.reduce_max([1.0 + rank, 10.0 - rank, 3.5])
    dist.barrier()
    q.put((rank, out, bench.rank_seed(2, rank)))
    dist.destroy_process_group()


def test_two_rank_timing_reduction_and_sharding():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for pr in procs:
        pr.start()
    res = [q.get(timeout=120) for _ in procs]
    for pr in procs:
        pr.join(timeout=60)
        assert pr.exitcode == 0
    res.sort()
    for rank, out, seed in res:
        assert out == [2.0, 10.0, 3.5]           # element-wise max over both ranks
    assert res[0][2] != res[1][2]                # ranks draw different problems


def test_single_process_helpers():
    import bench
    assert bench.reduce_max([1.0, 2.0]) == [1.0, 2.0]
    # weak scaling: 2 ranks x 1000 tokens in 4 ms (slowest rank) = 500k tokens/s
    assert bench.whole_job_rate(1000, 2, 4.0) == pytest.approx(500_000.0)
    assert bench.prefill_algorithmic_bytes(64, 1) == 1538 * 64 * 32 + 65536 * 32 * 3
    # final state + 5 checkpoints of 32 heads x 128 x 128 fp32 (the T=145408 prompt)
    assert bench.kv_state_bytes(5) == 6 * 32 * 128 * 128 * 4
