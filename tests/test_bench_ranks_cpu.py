"""The replicas (N > 1) path of the bench's aggregation on CPU: two gloo
ranks, the max-over-ranks time and the whole-job throughput, and the
reference arm doing nothing on ranks other than 0."""
import argparse
import os
import socket

import torch.multiprocessing as mp

import bench
from int4_routed_expert_06_b300 import synth


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = [12.5, 20.0][rank]          # this rank's timed region
        ms_max = bench.max_over_ranks(ms, dist, "cpu")
        q.put((rank, ms_max, bench.job_tokens_per_s(1000, world, ms_max)))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_throughput_with_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in procs)
    for rank, ms_max, v in got:
        assert ms_max == 20.0                     # the slowest replica's time
        assert abs(v - 2 * 1000 / 0.020) < 1e-6   # all ranks' tokens over it


def test_single_process_aggregation_is_the_identity():
    assert bench.max_over_ranks(7.0) == 7.0
    assert bench.job_tokens_per_s(500, 1, 10.0) == 50000.0


def test_reference_arm_other_ranks_do_nothing(capsys):
    args = argparse.Namespace(steps=1, warmup=0)
    assert bench.run_reference(args, synth.DEC_80B, 1) is None
    assert capsys.readouterr().out == ""
