"""The multi-rank path of the benchmark on CPU (gloo, world size 2): every rank runs its own
replica of the workload, the job's time per step is the slowest rank's, and its tokens are
the sum over ranks.  Also checks that ranks draw different seeded data."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    from mesa_layer_gb300 import synth
    step_ms = 1.0 + rank          # rank 1 is the slower one
    ms, tokens, value = bench.aggregate(step_ms, 4096, world, torch, dist, device="cpu")
    w = synth.workload("fwd_fp32_d64", B=1, H=1, T=32)
    q_first = float(synth.forward_inputs(w, seed=rank)["q"][0, 0, 0, 0])
    dist.barrier()
    q.put((rank, ms, tokens, value, q_first))
    dist.destroy_process_group()


def test_two_rank_aggregation_and_replica_seeds():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, tokens, value, _ in out:
        assert ms == 2.0                       # max over ranks
        assert tokens == 2 * 4096              # whole-job tokens
        assert value == pytest.approx(8192 / 2e-3)
    assert out[0][4] != out[1][4]              # each replica has its own seeded data
