"""The multi-process path of bench.py on CPU (world size 2, gloo, 127.0.0.1): problems are
sharded across ranks with no collective on the data path, each rank plans its own, and the
plans gathered from the ranks equal the single-process plans bit for bit (the planning page:
a given seed yields the same plan whatever the number of GPUs). The planner here is the oracle, so
the test needs no GPU; the timing reduction is the one bench.py uses."""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from cem_search_transformer_gb300 import synthetic
from oracle import cem

PC = synthetic.TINY
B_PER_RANK, N, K, R, H, SEED = 2, 16, 4, 2, 1, 42


def _plans(z0, goal, s0):
    w = synthetic.make_weights(PC)
    mu0, sg0 = synthetic.make_gaussian(PC, 1, H)
    return np.stack([cem.plan(w, PC, z0[b], s0[b], goal[b], mu0[0], sg0[0], N, K, R, SEED)["action"]
                     for b in range(z0.shape[0])])


def _rank(rank, world, port, out_path):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    z0, goal, s0 = bench.rank_problems(PC, B_PER_RANK, rank)
    actions = torch.from_numpy(_plans(z0, goal, s0))
    gathered = [torch.zeros_like(actions) for _ in range(world)]
    dist.all_gather(gathered, actions)
    slowest = bench.reduce_max(float(rank + 1) * 0.25, world, "cpu")
    if rank == 0:
        np.save(out_path, np.concatenate([g.numpy() for g in gathered]))
        with open(out_path + ".max", "w") as f:
            f.write(repr(slowest))
    dist.destroy_process_group()


def test_two_ranks_reproduce_single_process_plans(tmp_path):
    with socket.socket() as sck:
        sck.bind(("127.0.0.1", 0))
        port = sck.getsockname()[1]
    out = str(tmp_path / "gathered.npy")
    mp.start_processes(_rank, args=(2, port, out), nprocs=2, join=True, start_method="spawn")
    gathered = np.load(out)
    z0, goal, s0 = synthetic.make_problems(PC, 2 * B_PER_RANK)      # one process, all problems
    assert np.array_equal(gathered, _plans(z0, goal, s0))
    assert float(open(out + ".max").read()) == 0.5                   # max over the two ranks
