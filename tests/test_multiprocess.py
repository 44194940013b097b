"""The bench's multi-replica path on the CPU: two processes with the gloo
backend (rendezvous on 127.0.0.1) agree on the slowest replica's time, and
the job-wide figure divides the step time by the replica count (weak
scaling).  No GPU is involved."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        got = bench.max_over_ranks(1.5 + rank, dist, "cpu")
        dist.barrier()
    finally:
        dist.destroy_process_group()
    with open(os.path.join(out_dir, f"r{rank}.txt"), "w") as f:
        f.write(repr(got))


def test_max_over_ranks_gloo_two_ranks(tmp_path):
    port = _free_port()
    mp.spawn(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True)
    for r in range(2):
        assert float((tmp_path / f"r{r}.txt").read_text()) == 2.5


def test_single_process_and_job_figure():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.25) == 3.25
    assert bench.job_us_per_layer(0.2, 1) == pytest.approx(200.0)
    assert bench.job_us_per_layer(0.2, 4) == pytest.approx(50.0)
