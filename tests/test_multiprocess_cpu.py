"""The N > 1 path of bench.py on CPU: world_size-2 gloo ranks.

The hot path shards by independent problems (sequences, heads), so ranks run
their own replicas, or their own heads of one prompt, with no data-path
collective; the only cross-rank steps are the barrier and the max-over-ranks
timing reduction checked here.  The head split is checked end to end on the
fp64 oracle: each rank runs the recurrence on its head range only, and the
gathered outputs, final states and checkpoints equal one run over all heads."""
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


def _split_worker(rank, world, port, q):
    import torch
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    import oracle
    from kimi_delta_attention_06_gb300 import workloads
    (h0, h1), off = bench.rank_problem("heads", world, rank)
    # one prompt of two ragged sequences with initial states and checkpoints, H = 4 for speed
    full = workloads.prefill_case([150, 90], H=4, D=64, seed=11 + off, ckpt_stride=64)
    hs = bench.head_range(full.H, world, rank)
    mine = workloads.head_slice(full, *hs)
    o, fin, ck = oracle.prefill(mine.q, mine.k, mine.v, mine.log_alpha, mine.beta, mine.cu_seqlens,
                                mine.init_state, ckpt_stride=64, threads=1)
    parts = []
    for x in (o, fin, ck):
        t = torch.from_numpy(x).contiguous()
        g = [torch.empty_like(t) for _ in range(world)]
        dist.all_gather(g, t)
        parts.append(torch.cat(g, dim=1).numpy())     # heads are dim 1 of all three
    dist.barrier()
    q.put((rank, (h0, h1), hs, parts if rank == 0 else None))
    dist.destroy_process_group()


def test_two_rank_head_split_is_one_prompt():
    import numpy as np
    import oracle
    from kimi_delta_attention_06_gb300 import workloads
    oracle.build()                               # built once, before the ranks load it
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_split_worker, args=(r, 2, port, q)) for r in range(2)]
    for pr in procs:
        pr.start()
    res = [q.get(timeout=180) for _ in procs]
    for pr in procs:
        pr.join(timeout=60)
        assert pr.exitcode == 0
    res.sort(key=lambda r: r[0])
    assert [r[1] for r in res] == [(0, 16), (16, 32)]     # the bench's 32 heads, halved
    assert [r[2] for r in res] == [(0, 2), (2, 4)]
    full = workloads.prefill_case([150, 90], H=4, D=64, seed=11, ckpt_stride=64)
    ref = oracle.prefill(full.q, full.k, full.v, full.log_alpha, full.beta, full.cu_seqlens, full.init_state,
                         ckpt_stride=64, threads=1)
    for got, want in zip(res[0][3], ref):
        assert got.shape == want.shape
        assert np.array_equal(got, want)          # heads are independent: bit-identical


def test_single_process_helpers():
    import bench
    assert bench.reduce_max([1.0, 2.0]) == [1.0, 2.0]
    # weak scaling: 2 ranks x 1000 tokens in 4 ms (slowest rank) = 500k tokens/s
    assert bench.whole_job_rate(1000, 2, 4.0) == pytest.approx(500_000.0)
    assert bench.prefill_algorithmic_bytes(64, 1) == 1538 * 64 * 32 + 65536 * 32 * 3
    # final state + 5 checkpoints of 32 heads x 128 x 128 fp32 (the T=145408 prompt)
    assert bench.kv_state_bytes(5) == 6 * 32 * 128 * 128 * 4
    # per-rank byte counts of a head split add up to the whole problem's
    assert bench.prefill_algorithmic_bytes(64, 1, 16) * 2 == bench.prefill_algorithmic_bytes(64, 1)
    assert bench.decode_algorithmic_bytes(512, 8) * 4 == bench.decode_algorithmic_bytes(512)
    # strong scaling: 2 ranks share one 1000-token prompt finished in 4 ms = 250k tokens/s
    assert bench.job_rate(1000, 2, 4.0, "heads") == pytest.approx(250_000.0)
    assert bench.job_rate(1000, 2, 4.0, "replicas") == pytest.approx(500_000.0)
    assert [bench.head_range(32, 4, r) for r in range(4)] == [(0, 8), (8, 16), (16, 24), (24, 32)]
    with pytest.raises(ValueError):
        bench.head_range(32, 3, 0)                # 32 heads do not split over 3 ranks
    with pytest.raises(ValueError):
        bench.head_range(32, 2, 2)
    assert bench.rank_problem("replicas", 2, 1) == ((0, 32), 1000)
    assert bench.rank_problem("heads", 2, 1) == ((16, 32), 0)
    assert bench.bench_config(4, "heads")["global_batch"] == 1
