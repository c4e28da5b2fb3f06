"""The N > 1 host path of the benchmark, on CPU with two gloo ranks.

The forward does not shard (one weight fits one GPU): N GPUs run N
independent replicas, the step time is the slowest rank's, and the job's
throughput counts every rank's bytes.  These tests run the rendezvous,
barrier and max-over-ranks helpers of bench.py as two processes, and the
reference arm's rule that only rank 0 works.
"""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    r, local, ws = bench.dist_setup(0)  # no GPU: gloo
    assert (r, local, ws) == (rank, rank, world)
    bench.barrier(ws)
    t = bench.max_over_ranks(1.5 + rank, ws, torch.device("cpu"))  # rank r took 1.5 + r ms
    out[rank] = t
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_step():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        port = _free_port()
        procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        assert dict(out) == {0: 2.5, 1: 2.5}


def test_job_throughput_counts_every_replica():
    # two replicas of 724,172,800 bytes each in a 2.5 ms step
    assert bench.job_gbs(2, 724_172_800, 2.5) == pytest.approx(2 * 724_172_800 / 2.5e-3 / 1e9)
    assert bench.job_gbs(1, 10**9, 1000.0) == pytest.approx(1.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    monkeypatch.setenv("RANK", "1")
    called = []
    monkeypatch.setattr(bench, "oracle_sample", lambda *a, **k: called.append(1) or (1, 1.0, 1))

    class Args:
        steps, warmup, gpus = 2, 1, 2
    assert bench.run_reference(Args()) == 0
    assert not called
