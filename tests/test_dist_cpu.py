"""Multi-rank host logic on CPU (gloo, world size 2).

The benchmark shards by batch (each rank draws its own sequences) and sums
the per-layer dL/dtheta over ranks with one all-reduce.  Here two gloo ranks
run the fp64 oracle on their own shards and reduce with the benchmark's
function; the result must equal the single-process oracle over both shards
(dtheta is a sum over the batch).
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ALPHAS = [0.5 + 3 / 15, 0.5 + 11 / 15]  # two layers of the linear schedule
SHAPE = dict(B=1, T=40, Hq=4, Hkv=2, D=8)
W = 3


def _shard_dtheta(rank):
    import bench
    import oracle as o
    import sfa_inputs as si

    out = []
    for l, a in enumerate(ALPHAS):
        x = si.make_qkvdo(SHAPE["B"], SHAPE["T"], SHAPE["Hq"], SHAPE["Hkv"], SHAPE["D"], "f32",
                          bench.rank_seed(rank), layer=l)
        g = o.backward(x["q"], x["k"], x["v"], x["do"], o.interp_slots(o.fib_offsets(10), a, W),
                       1e4, alpha=a)
        out.append(torch.tensor([g["dalpha"], g["dtheta"]], dtype=torch.float64))
    return out


def _worker(rank, world, port, result_path):
    import sys

    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    reduced = bench.allreduce_dtheta(_shard_dtheta(rank), torch.zeros(len(ALPHAS), dtype=torch.float64))
    if rank == 0:
        np.save(result_path, reduced.numpy())
    dist.barrier()
    dist.destroy_process_group()


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_rank_dtheta_allreduce(tmp_path):
    path = str(tmp_path / "dtheta.npy")
    mp.start_processes(_worker, args=(2, _free_port(), path), nprocs=2, start_method="spawn")
    got = np.load(path)
    want = sum(np.array([d[1].item() for d in _shard_dtheta(r)]) for r in range(2))
    assert np.allclose(got, want, rtol=1e-12, atol=1e-12)
    # the shards are different data: neither rank alone gives the sum
    assert not np.allclose(got, np.array([d[1].item() for d in _shard_dtheta(0)]))
