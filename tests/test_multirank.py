"""Multi-rank host logic on the CPU: two gloo ranks (world size 2) draw
different data shards, agree on the max-over-ranks elapsed time, and report
the whole-job rate over both ranks' blocks."""
import os
import socket

import numpy as np
import torch.distributed as dist
import torch.multiprocessing as mp

from draft_selection_dflash2_gb300 import replicas, synth


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    shard = synth.normal_bits(replicas.rank_seed(7, rank), (4, 8))
    elapsed = 1.5 + rank            # rank 1 is the slow one
    worst = replicas.max_over_ranks(elapsed, dist)
    out[rank] = (shard.tobytes(), worst, replicas.whole_job_rate(128, world, worst))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] != res[1][0]                      # distinct data shards
    assert res[0][1] == res[1][1] == 2.5               # max over ranks
    assert res[0][2] == res[1][2] == 128 * 2 / 2.5     # whole-job blocks/s


def test_single_process_fallbacks():
    assert replicas.max_over_ranks(3.0) == 3.0
    assert replicas.rank_seed(5, 0) == 5
    assert np.isclose(replicas.whole_job_rate(10, 1, 2.0), 5.0)
