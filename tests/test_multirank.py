"""Host logic of the N>1 bench path: replicas meet only at a barrier and a max-over-ranks
reduction of their timings. World size 2 on gloo, CPU only."""
import os
import socket
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank), MLA_BENCH_BACKEND="gloo")
    sys.path.insert(0, ROOT)
    import torch
    import bench
    w, r, _ = bench._dist_init()
    assert (w, r) == (world, rank)
    bench._barrier(w)
    t = bench._max_over_ranks(1.5 + rank, w, torch.device("cpu"))
    out[rank] = t
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_replicas_agree_on_max_time():
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(2, port, out), nprocs=2, join=True, start_method="spawn")
    assert dict(out) == {0: 2.5, 1: 2.5}
