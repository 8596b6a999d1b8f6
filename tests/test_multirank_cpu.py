"""The N > 1 path of bench.py on CPU: two processes with the gloo backend.

The convolution path shards over the batch with no exchange on the forward and
input-gradient side; bench.py runs independent replicas (one per GPU), takes the
job's step time as the slowest rank's, and reports the whole job's rate as
world x per-rank units over that time (weak scaling).  These tests run the
cross-rank reduction and the rate on two gloo ranks (no GPU): every rank must
see the same maximum, and the rate must count both ranks' work.
"""
import os
import socket

import pytest

torch = pytest.importorskip("torch")


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    import sys
    import torch.distributed as dist
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local_ms = [3.25, 5.5][rank]                 # rank 1 is the slower replica
    ms = bench.max_over_ranks(local_ms, dist)
    rate = bench.job_rate(1000, ms, world)
    # the same max seen everywhere (a second reduction of the results)
    both = torch.tensor([ms, rate], dtype=torch.float64)
    gathered = [torch.zeros(2, dtype=torch.float64) for _ in range(world)]
    dist.all_gather(gathered, both)
    out[rank] = [g.tolist() for g in gathered]
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time_and_the_job_rate():
    import torch.multiprocessing as mp
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    for rank in (0, 1):
        for ms, rate in res[rank]:
            assert ms == 5.5                      # the slowest rank's time, on both ranks
            assert rate == pytest.approx(2 * 1000 / 5.5e-3)


def test_single_process_path():
    import bench
    assert bench.max_over_ranks(4.0, None) == 4.0
    assert bench.job_rate(64, 0.2, 1) == pytest.approx(320000.0)
