"""Host logic of the N-GPU bench (independent replicas, no data-path collective),
run as two gloo ranks on the CPU.

The only collective is the max over ranks of the timed region; whole-job
throughput is the rows all ranks processed divided by the slowest rank's time.
Replicas draw disjoint input sets, and the reference arm does its work on
rank 0 only."""
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


def _worker(rank, ws, port, times, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        ms, value = bench.job_throughput(times[rank], 10, 576, ws, "cpu")
        q.put((rank, ms, value))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("ws", [2])
def test_job_time_is_the_slowest_rank_and_value_counts_all_ranks(ws):
    times = [120.0, 95.5, 130.0, 80.0][:ws]          # total ms of each rank's 10 timed steps
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, ws, port, times, q)) for r in range(ws)]
    for p in procs:
        p.start()
    got = [q.get(timeout=120) for _ in range(ws)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    slowest = max(times)
    for rank, ms, value in got:
        assert ms == pytest.approx(slowest / 10)
        # 576 rows per step per rank, 10 steps, ws ranks, over the slowest rank's time
        assert value == pytest.approx(576 * 10 * ws / (slowest / 1e3))


def test_single_rank_needs_no_process_group():
    ms, value = bench.job_throughput(50.0, 5, 100, 1, "cpu")
    assert ms == 10.0 and value == pytest.approx(100 * 5 / 0.05)


def test_replicas_draw_disjoint_input_sets():
    from speculative_decoding_verification_30_gb300.workloads import WORKLOADS, make_batch
    w = WORKLOADS["tiny"]
    steps = {bench.replica_input_step(r, s) for r in range(8) for s in range(64)}
    assert len(steps) == 8 * 64
    a = make_batch(w, bench.replica_input_step(0, 0))
    b = make_batch(w, bench.replica_input_step(1, 0))
    assert not torch.equal(a.target, b.target)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")

    class A:
        workload, steps, warmup = "tiny", 1, 0
    assert bench.bench_reference(A()) is None
    assert capsys.readouterr().out == ""
