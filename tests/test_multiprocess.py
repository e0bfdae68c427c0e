"""The multi-process (one replica per GPU) host logic of bench.py, run as
two gloo ranks on the CPU: the slowest rank's time is what every rank
reports, and each replica draws its own batch."""
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    from lora_mixture_experts_gb300.inputs import CONFIGS, make_routing
    got = bench.reduce_max(1.5 + rank, world, torch.device("cpu"))
    ids, _, lo = make_routing(CONFIGS["tiny"], seed=bench.rank_seed(rank))
    dist.barrier()
    q.put((rank, got, int(ids.sum()), int(lo.sum())))
    dist.destroy_process_group()


def test_two_gloo_ranks_take_max_and_distinct_batches():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [2.5, 2.5]
    assert (res[0][2], res[0][3]) != (res[1][2], res[1][3])


def test_single_rank_is_identity():
    import bench
    assert bench.reduce_max(3.25, 1, torch.device("cpu")) == 3.25
