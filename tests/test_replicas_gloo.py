"""Multi-GPU mode is replicas only (one encode shares nothing across GPUs): the
bench's whole-job throughput is the units of all ranks over the slowest rank's
time.  Checked with two gloo ranks on CPU."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = 100.0 if rank == 0 else 250.0     # rank 1 is the slow one
        value, ms = bench.job_throughput(local_ms, units_per_rank=1024, steps=4, dist=dist, device="cpu")
        out[rank] = (value, ms)
    finally:
        dist.destroy_process_group()


def test_two_replica_ranks_report_max_time_and_total_units():
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.start_processes(_rank, args=(2, port, out), nprocs=2, join=True, start_method="spawn")
        res = dict(out)
    for rank in (0, 1):
        value, ms = res[rank]
        assert ms == 250.0
        assert value == pytest.approx(2 * 1024 * 4 / 0.25)


def test_single_process_needs_no_process_group():
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    value, ms = bench.job_throughput(50.0, units_per_rank=1000, steps=5)
    assert ms == 50.0 and value == pytest.approx(1000 * 5 / 0.05)
