"""The N > 1 host logic of bench.py on CPU: two gloo ranks, no GPU.

Rows are independent, so each rank runs either its own replica of the workload
(weak scaling) or a contiguous range of one workload's (batch, head) slices
(--split, strong scaling), with no data-path collective; the only exchanges are
the max over ranks of the step time and the sum of the bytes moved. These tests
run those exchanges and the whole-job value under a real two-process gloo group.
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


def _split_rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = si.WORKLOADS["s1000_b12"]
        lens = si.seq_lens(w)
        ws = bench.shard_workload(w, lens, rank, world)
        fb, bb = bench.required_bytes(ws, si.seq_lens(ws))
        total = bench.sum_over_ranks(fb + bb, dist, torch.device("cpu"))
        out[rank] = (bench.shard_slices(w.B * w.M, rank, world), ws.B, ws.M, tuple(si.seq_lens(ws)), total)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_split_one_workload_exactly():
    world, port = 2, _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_split_rank_main, args=(world, port, out), nprocs=world, start_method="spawn", join=True)
        res = dict(out)
    w = si.WORKLOADS["s1000_b12"]
    lens = si.seq_lens(w)
    (r0, b0, m0, l0, t0), (r1, b1, m1, l1, t1) = res[0], res[1]
    # the two ranges tile the B*M slices, each slice once, and carry its batch's length
    assert r0 == (0, w.B * w.M // 2) and r1 == (w.B * w.M // 2, w.B * w.M)
    assert (b0, m0, b1, m1) == (r0[1] - r0[0], 1, r1[1] - r1[0], 1)
    assert l0 + l1 == tuple(int(lens[s // w.M]) for s in range(w.B * w.M))
    # the whole job moves exactly the bytes of the unsplit workload
    fb, bb = bench.required_bytes(w, lens)
    assert t0 == t1 == fb + bb


@pytest.mark.parametrize("n", [0, 1, 5, 12, 768, 1001])
@pytest.mark.parametrize("world", [1, 2, 3, 8])
def test_shard_slices_tile_the_slices(n, world):
    ranges = [bench.shard_slices(n, r, world) for r in range(world)]
    assert ranges[0][0] == 0 and ranges[-1][1] == n
    for (a0, a1), (b0, b1) in zip(ranges, ranges[1:]):
        assert a1 == b0
    sizes = [b - a for a, b in ranges]
    assert max(sizes) - min(sizes) <= 1 and min(sizes) >= 0
