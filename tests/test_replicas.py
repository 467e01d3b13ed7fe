"""Replica timing for `bench.py --gpus N` on CPU: two gloo ranks, each with
its own step time, must both see the slowest rank's time, and the whole-job
throughput counts every replica's bytes.  The path has no data exchange, so
this host logic is all there is to the N > 1 case."""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    mine = [1.0 + rank, 10.0 - 3.0 * rank]          # rank 0: (1, 10); rank 1: (2, 7)
    got = bench.max_over_ranks(dist, mine)
    dist.barrier()
    dist.destroy_process_group()
    with open(os.path.join(out_dir, f"r{rank}.txt"), "w") as f:
        f.write(" ".join(repr(v) for v in got))


def test_max_over_ranks_two_gloo_ranks(tmp_path):
    import torch.multiprocessing as mp
    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True,
                       start_method="spawn")
    for r in range(2):
        vals = [float(v) for v in (tmp_path / f"r{r}.txt").read_text().split()]
        assert vals == [2.0, 10.0]


def test_single_process_is_identity_and_throughput_counts_replicas():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(None, [3, 4.5]) == [3.0, 4.5]
    # 1.66e9 bytes per step per replica, 2 replicas, 0.5 ms -> 6640 GB/s
    assert bench.job_throughput(1.66e9, 2, 0.5) == pytest.approx(6640.0)
