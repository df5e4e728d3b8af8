"""Host logic of the multi-process benchmark on CPU (gloo, world size 2): every rank gets
its own independent batches (weak scaling, no collective on the data path), and the
reported time is the maximum over ranks."""
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    import synth

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = bench.shard_workload(synth.WORKLOADS["c1"], rank)
        lg = synth.logits(w, 0, batches=[0])
        t = bench.max_over_ranks(1.0 + rank, world)
        bench.barrier(world)
        out[rank] = (w.seed, float(lg.sum()), t, bench.dist_env())
    finally:
        dist.destroy_process_group()


def test_two_rank_sharding_and_max_time():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_worker, args=(world, port, out), nprocs=world, join=True, start_method="spawn")
        res = dict(out)
    assert set(res) == {0, 1}
    seeds = [res[r][0] for r in range(world)]
    assert seeds[0] != seeds[1]                      # independent batches per rank
    assert not np.isclose(res[0][1], res[1][1])     # ... so different logits
    assert res[0][2] == res[1][2] == 2.0            # max over ranks
    assert res[1][3] == (2, 1, 1)
