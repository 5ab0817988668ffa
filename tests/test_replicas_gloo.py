"""Host-side logic of the N-GPU benchmark (independent replicas, no exchange
step): the slowest rank's time and the whole-job throughput, on two gloo
ranks on the CPU."""

import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", init_method="env://", rank=rank, world_size=world)
    import bench
    my_ms = 10.0 + 5.0 * rank                      # rank 1 is the slow one
    got = bench.max_over_ranks(my_ms)
    dist.barrier()
    tok = bench.whole_job_tokens_per_s(world, 16, 100, got)
    out[rank] = (got, tok)
    dist.destroy_process_group()


def test_two_replica_ranks_agree_on_slowest_time_and_throughput():
    world, port = 2, _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank, args=(world, port, out), nprocs=world, start_method="spawn")
    assert out[0][0] == out[1][0] == 15.0
    # 2 ranks x 16 tokens x 100 steps over 15 ms
    assert out[0][1] == out[1][1] == pytest.approx(2 * 16 * 100 / 0.015)


def test_single_process_is_its_own_maximum():
    import bench
    assert bench.max_over_ranks(3.5) == 3.5


def test_end_to_end_reports_the_faster_host_buffer_mode_and_both_figures():
    import bench
    few = bench.e2e_line(1, 1, 2048, 1000, zero_copy_ms=31.0, copies_ms=45.0)
    assert few["mode"] == "zero_copy" and few["us_per_call"] == 31.0
    assert few["h2d_bytes_per_step"] == few["d2h_bytes_per_step"] == 2048 * 2
    assert few["with_copies"]["us_per_call"] == 45.0
    many = bench.e2e_line(2, 256, 2048, 100, zero_copy_ms=36.0, copies_ms=30.0)
    assert many["mode"] == "with_copies" and many["us_per_call"] == 300.0
    # whole-job tokens/s over both ranks, from the chosen mode's time
    assert abs(many["value"] - 2 * 256 * 100 / 30e-3) < 1e-6 * many["value"]
