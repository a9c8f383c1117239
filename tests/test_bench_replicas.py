"""The multi-GPU path of bench.py is replicas only: every rank runs the whole
layer on its own data, the job time is the slowest rank's and the job's
throughput counts every rank's tokens. These checks run that host logic as two
gloo ranks on the CPU."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    r, w, local = bench.dist_env()
    assert (r, w, local) == (rank, world, rank)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    # rank 1 is the slow replica for the timed loop, rank 0 for end to end
    mine = [10.0 + 5.0 * rank, 7.0 - 2.0 * rank]
    got = bench.reduce_max_over_ranks(dist, mine, "cpu")
    with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
        f.write(" ".join(str(v) for v in got))
    dist.barrier()
    dist.destroy_process_group()


def test_replicas_take_the_slowest_rank(tmp_path):
    port = _free_port()
    mp.spawn(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True)
    for rank in range(2):
        vals = [float(v) for v in (tmp_path / f"rank{rank}.txt").read_text().split()]
        assert vals == [15.0, 7.0]


def test_single_rank_needs_no_collective():
    assert bench.reduce_max_over_ranks(None, [3.0, 4.0], "cpu") == [3.0, 4.0]


def test_job_throughput_counts_every_replica():
    # 2 replicas x 64 tokens x 100 steps in 50 ms (slowest rank) -> 256k tokens/s
    assert bench.job_tokens_per_s(2, 64, 100, 50.0) == pytest.approx(256000.0)
    assert bench.job_tokens_per_s(1, 64, 1, 0.2) == pytest.approx(320000.0)
