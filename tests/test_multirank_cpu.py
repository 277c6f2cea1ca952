"""The multi-GPU bench logic on CPU: two gloo ranks on 127.0.0.1.

Rows are independent, so a run on N GPUs gives each rank its own batch of the
same shape (its own seed) and uses no collective on the data path; the only
exchange is the max over ranks of the timed region.  These tests run that
logic with world size 2 on the gloo backend, without a GPU.
"""
from __future__ import annotations

import os
import socket
import subprocess
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, q):
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # each rank "timed" a different total; every rank must see the slowest
        slowest = bench.max_over_ranks(10.0 + 5.0 * rank, world, "cpu")
        wl = bench.build_workload("tiny", shard=rank)
        shard_wl = bench.workloads.decode(batch=3, seq_len=64, shard=rank)
        dist.barrier()
        q.put((rank, slowest, shard_wl.scores.tobytes(), wl.name))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_draw_distinct_batches():
    import torch.multiprocessing as mp

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert [g[1] for g in got] == [15.0, 15.0]
    assert got[0][2] != got[1][2]  # each rank draws its own batch
    from sparse_attention_indexer_uint32_gb300 import workloads

    # shard 0 is the single-GPU workload itself
    assert got[0][2] == workloads.decode(batch=3, seq_len=64).scores.tobytes()


def test_job_throughput_counts_every_rank():
    sys.path.insert(0, ROOT)
    import bench

    # 2 ranks x 3 steps x 1e9 bytes in 2 ms (slowest rank) = 3000 GB/s
    assert bench.job_gbs(10**9, 2, 3, 2.0) == pytest.approx(3000.0)
    assert bench.max_over_ranks(4.5, 1) == 4.5


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1", MASTER_ADDR="127.0.0.1")
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                          "--steps", "1", "--warmup", "0"], capture_output=True, text=True, env=env, timeout=120,
                         cwd=ROOT)
    assert res.returncode == 0, res.stderr
    assert res.stdout.strip() == ""


def test_shards_have_the_same_shape():
    from sparse_attention_indexer_uint32_gb300 import workloads

    a = workloads.ragged(batch=6, max_len=4096, min_len=1024, shard=0)
    b = workloads.ragged(batch=6, max_len=4096, min_len=1024, shard=1)
    assert a.scores.shape == b.scores.shape and a.k == b.k and a.page_size == b.page_size
    assert not np.array_equal(a.seq_lens, b.seq_lens)
