"""The N > 1 path of the benchmark on CPU: two gloo ranks run replicas, the
timing is the max over ranks and the throughput sums the ranks' FLOPs."""

import os
import socket

import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = [10.0, 25.0][rank]                    # rank 1 is the slow one
    slow = bench.slowest_rank_ms(ms, world)
    value = bench.replica_throughput(2.0e12, 4, world, slow)
    out[rank] = (slow, value)
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_sum_flops():
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 25.0
    # 2 ranks x 4 steps x 2 TFLOP in 25 ms -> 640 TFLOP/s, on every rank
    assert res[0][1] == res[1][1] == 2.0e12 * 4 * 2 / 0.025 / 1e12


def test_single_rank_needs_no_collective():
    assert bench.slowest_rank_ms(7.5, 1) == 7.5
    assert bench.replica_throughput(1e12, 10, 1, 5.0) == 1e12 * 10 / 0.005 / 1e12
