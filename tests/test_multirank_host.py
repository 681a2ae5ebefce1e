"""The N > 1 host logic of bench.py on CPU: two gloo ranks, no GPU.

Rows are independent, so each rank runs its own replica of the workload with
no data-path collective; the only exchange is the max over ranks of the step
time. These tests run that exchange and the whole-job value under a real
two-process gloo group.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import seeded_inputs as si


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = bench.replica_workload(si.WORKLOADS["s1000_b12"], rank)
        lens = si.seq_lens(w)
        fb, bb = bench.required_bytes(w, lens)
        local_ms = 1.0 + rank            # rank 1 is the slow one
        ms = bench.max_over_ranks(local_ms, dist, torch.device("cpu"))
        total = bench.sum_over_ranks(fb + bb, dist, torch.device("cpu"))
        value = bench.whole_job_gbs(total, ms)
        out[rank] = (w.seed, tuple(int(v) for v in lens), fb + bb, ms, value)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_step_time_and_keep_replicas_independent():
    world, port = 2, _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_rank_main, args=(world, port, out), nprocs=world, start_method="spawn", join=True)
        res = dict(out)
    assert set(res) == {0, 1}
    (s0, l0, b0, ms0, v0), (s1, l1, b1, ms1, v1) = res[0], res[1]
    assert s0 != s1 and l0 != l1                 # each rank draws its own replica
    assert ms0 == ms1 == 2.0                     # everyone reports the slowest rank's time
    # the whole-job value is the bytes of both replicas over the slowest step
    assert v0 == v1 == pytest.approx((b0 + b1) / 2e-3 / 1e9, rel=1e-12)


def test_single_rank_needs_no_group():
    assert bench.max_over_ranks(3.5, None, torch.device("cpu")) == 3.5
    assert bench.sum_over_ranks(7.0, None, torch.device("cpu")) == 7.0
    w = si.WORKLOADS["s1000_b12"]
    assert bench.replica_workload(w, 0) is w
