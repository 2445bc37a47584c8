"""Multi-rank host logic of the benchmark on CPU (gloo, world size 2): each
rank gets disjoint micro-batches (and so different synthetic data), and the
step time reported is the maximum over ranks."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mbs = bench.rank_micro_batches(rank, 3)
        t = bench.max_over_ranks(10.0 + rank, world, torch.device("cpu"))
        bench.barrier(world)
        q.put((rank, mbs, t))
    finally:
        dist.destroy_process_group()


def test_two_rank_sharding_and_max_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = {}
    try:
        for _ in range(2):
            r, mbs, t = q.get(timeout=120)
            out[r] = (mbs, t)
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.terminate()
    assert set(out) == {0, 1}
    assert out[0][0] == [0, 1, 2] and out[1][0] == [3, 4, 5]   # disjoint micro-batches
    assert out[0][1] == 11.0 and out[1][1] == 11.0             # max over ranks


def test_rank_micro_batches_give_distinct_data():
    import bench
    from synth import CONFIGS, make_workload
    cfg = CONFIGS[2]
    a = make_workload(cfg, micro_batch=bench.rank_micro_batches(0, 1)[0], with_weight=False)
    b = make_workload(cfg, micro_batch=bench.rank_micro_batches(1, 1)[0], with_weight=False)
    assert not (a["H"] == b["H"]).all()
