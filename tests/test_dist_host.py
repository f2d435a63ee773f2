"""Host logic of the multi-GPU bench path, on CPU with two gloo ranks: every
rank gets its own batch (different seeds, no shared data), the job time is the
slowest rank's, and the job throughput counts every rank's sequences."""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import workloads


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, ws, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        assert bench._dist() == (ws, rank, rank)
        local_time = 1.0 + 0.25 * rank  # rank 1 is slower
        total = bench._max_over_ranks(local_time, ws, torch.device("cpu"))
        w = workloads.make("gqa8k", B=2, Hkv=1, Hq=8, seq_lens=[64, 64], seed=bench._rank_seed(rank))
        k, _ = w.kv(0, 0, 16)
        out[rank] = (total, bench._job_throughput(ws, 8, 100, total), float(k.float().sum()))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks():
    ws, port = 2, _free_port()
    with mp.Manager() as man:
        out = man.dict()
        mp.spawn(_worker, args=(ws, port, out), nprocs=ws, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 1.25                       # max over ranks
    assert res[0][1] == res[1][1] == ws * 8 * 100 / 1.25          # whole-job tokens/s
    assert res[0][2] != res[1][2]                                # different data per rank
    assert bench._max_over_ranks(3.0, 1, torch.device("cpu")) == 3.0
