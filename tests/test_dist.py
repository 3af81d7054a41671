"""Multi-process host logic of the replica benchmark, on CPU with gloo.

Decode batches are independent problems, so N GPUs run N replicas with no
collective on the data path; the only cross-rank steps are the barrier around
the timed region and the max over ranks of the timings.  Both are exercised
here with two gloo ranks (no GPU)."""

import os
import socket
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    import msa_synth as ms
    base = ms.make_workload("fp8_decode", seq_lens=(300, 200), seed=5)
    seed = bench.replica_seed(base.seed, rank)
    w = ms.make_workload("fp8_decode", seq_lens=(300, 200), seed=seed)
    case = ms.make_case(w)
    dist.barrier()
    timings = [1.0 + rank, 5.0 - rank, 2.0]
    mx = bench.max_over_ranks(timings, world, dist)
    out[rank] = (seed, float(case["q"].float().sum()), mx)
    dist.destroy_process_group()


def test_two_replicas_with_gloo():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] != res[1][0]                # independent replicas
    assert res[0][1] != res[1][1]                # different data
    assert res[0][2] == res[1][2] == [2.0, 5.0, 2.0]  # max over ranks seen by every rank
