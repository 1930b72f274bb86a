"""The N > 1 bench path on CPU: two gloo ranks run as independent replicas
(no data-path collective); the timing is the max over ranks and the whole-job
rate sums the ranks' tokens over that time."""

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, results):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import bench
    r, w = bench.dist_setup("gloo")
    assert (r, w) == (rank, world)
    bench.barrier()
    local_ms = 10.0 * (rank + 1)          # rank 1 is the slow one
    worst = bench.max_over_ranks(local_ms)
    results[rank] = worst
    import torch.distributed as dist
    dist.destroy_process_group()


def test_max_over_two_gloo_ranks():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    results = manager.dict()
    procs = [ctx.Process(target=_worker, args=(r, world, port, results)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert dict(results) == {0: 20.0, 1: 20.0}


def test_single_process_is_identity():
    import bench
    for key in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        os.environ.pop(key, None)
    assert bench.dist_env() == (0, 1, 0)
    assert bench.max_over_ranks(3.5) == 3.5


def test_algorithmic_work_of_the_prefill_workload():
    import bench
    from hashed_gram_embedding_gb300 import workloads as wl
    work = bench.algorithmic_work(wl.WORKLOADS["prefill8k"])
    # 8192 tokens x (16 ids x 8 B + 16 rows x 256 B read + written)
    assert work["lookup"] == ("hbm", 8192 * (128 + 4096 + 4096))
    assert work["kv_proj"] == ("tensor", 2.0 * 8192 * 2048 * 8192)
    assert work["gate_conv"] == ("hbm", 8192 * (8192 + 16384 + 8192))


def test_algorithmic_work_counts_the_decode_conv_state():
    import bench
    from hashed_gram_embedding_gb300 import workloads as wl
    w = wl.WORKLOADS["decode256x4"]
    work = bench.algorithmic_work(w)
    # 1024 tokens x (v 8 KB + g 4 B + y 8 KB) + 256 requests x 9 rows x 4096 x 2 B, in and out
    assert work["conv"] == ("hbm", 1024 * (8192 + 4 + 8192) + 2 * 256 * 9 * 4096 * 2)
