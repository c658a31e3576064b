"""The multi-GPU bookkeeping (replicas, no data-path collective) on CPU:
two gloo ranks, each with its own units and time, agree on the whole-job
throughput = all ranks' units / the slowest rank's time."""

import os
import socket

import torch.multiprocessing as mp

from bwd_flashattention_fwd_gb300 import replicas


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank(rank, world, port, out):
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    replicas.init("gloo")
    assert replicas.world() == (rank, rank, world)
    replicas.barrier()
    units = 10.0 * (rank + 1)      # 10 and 20
    seconds = 1.0 + rank           # 1 s and 2 s
    out[rank] = replicas.aggregate_throughput(units, seconds)
    replicas.shutdown()


def test_two_gloo_ranks_aggregate():
    world, port = 2, _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        value, total, tmax = res[r]
        assert total == 30.0 and tmax == 2.0 and value == 15.0


def test_single_process_is_identity(monkeypatch):
    for k in ("RANK", "LOCAL_RANK", "WORLD_SIZE"):
        monkeypatch.delenv(k, raising=False)
    replicas.init("gloo")
    assert replicas.aggregate_throughput(7.0, 2.0) == (3.5, 7.0, 2.0)
