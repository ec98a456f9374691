"""Multi-rank host logic on CPU with gloo, world size 2.

1. A long sequence sharded across ranks: each rank reduces its slice of the
   tokens to a split-K partial state (m, l, o) with the oracle, the states are
   all-gathered and merged with the rescaling identity; the result must equal
   dense attention over the whole sequence.  This is the exchange a
   sequence-sharded decode would need (the only collective the path admits).
2. bench.py's timing reduction takes the maximum over ranks.
"""

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


def _init(rank, world, port):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)


def _split_merge_worker(rank, world, port, errfile):
    try:
        import oracle
        _init(rank, world, port)
        rng = np.random.default_rng(17)           # same data on every rank
        L, D = 1000, 16
        q = rng.standard_normal(D)
        K = rng.standard_normal((L, D)) * 1.5
        V = rng.standard_normal((L, D))
        bounds = np.linspace(0, L, world + 1).astype(int)
        a, b = bounds[rank], bounds[rank + 1]
        m, l, o = oracle.partial_state(q, K[a:b], V[a:b], 0.25)
        mine = torch.tensor([m, l, *o], dtype=torch.float64)
        got = [torch.empty_like(mine) for _ in range(world)]
        dist.all_gather(got, mine)
        ms = [g[0].item() for g in got]
        ls = [g[1].item() for g in got]
        os_ = [g[2:].numpy() for g in got]
        merged = oracle.merge_partials(ms, ls, os_)
        ref = oracle.dense_attention(q, K, V, 0.25)
        assert np.abs(merged - ref).max() < 1e-12
        dist.destroy_process_group()
    except BaseException as e:  # report to the parent
        with open(errfile, "a") as f:
            f.write(f"rank {rank}: {e!r}\n")
        raise


def _max_worker(rank, world, port, errfile):
    try:
        import sys
        sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
        import bench
        _init(rank, world, port)
        vals = [1.0 + rank, 5.0 - rank, 3.0]
        got = bench.max_over_ranks(vals, torch.device("cpu"))
        assert got == [2.0, 5.0, 3.0], got
        assert bench.rank_seed(7, rank) == 7 + rank
        dist.destroy_process_group()
    except BaseException as e:
        with open(errfile, "a") as f:
            f.write(f"rank {rank}: {e!r}\n")
        raise


@pytest.mark.parametrize("worker", [_split_merge_worker, _max_worker])
def test_two_gloo_ranks(tmp_path, worker):
    err = tmp_path / "err.txt"
    mp.start_processes(worker, args=(2, _free_port(), str(err)), nprocs=2, join=True,
                       start_method="spawn")
    assert not err.exists() or err.read_text() == ""


def test_max_over_ranks_single_process():
    import bench
    assert bench.max_over_ranks([1, 2.5], torch.device("cpu")) == [1.0, 2.5]
