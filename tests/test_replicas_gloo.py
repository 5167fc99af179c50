"""The multi-rank host logic of bench.py on CPU: two gloo ranks run independent
replicas (no data-path collective), the job time is the max over ranks, and the
whole-job throughput counts every rank's work."""

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench

    w, r, local = bench.dist_env()
    dist = bench.dist_init(w, "gloo")
    bench.barrier(dist)
    my_ms = 10.0 * (rank + 1)          # rank 1 is the slow one
    worst = bench.reduce_max(dist, my_ms)
    value = bench.job_throughput(w, 1_000_000_000, 4, worst)
    bench.barrier(dist)
    dist.destroy_process_group()
    q.put((rank, w, local, worst, value))


def test_two_gloo_replicas():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, world, local, worst, value in res:
        assert world == 2 and local == rank
        assert worst == 20.0                            # max over ranks
        assert value == pytest.approx(2 * 1e9 * 4 / 0.020 / 1e12)


def test_single_process_env_defaults(monkeypatch):
    import bench

    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_env() == (1, 0, 0)
    assert bench.dist_init(1, "gloo") is None
    assert bench.reduce_max(None, 3.5) == 3.5


def test_flop_accounting_matches_closed_forms():
    # 4 B H L^2 d for standard attention, 2 maps x 2 (d + d_v) per pair for the differential
    # form, and the window's allowed pairs sum_i (min(L - 1, i + w) - max(0, i - w) + 1)
    import bench
    import synth

    W = synth.WORKLOADS
    assert bench.flops(W["dit_l1292"]) == 6_837_305_344
    assert bench.flops(W["dit_l4096_outliers"]) == 103_079_215_104
    assert bench.flops(W["diff_l4096"]) == 206_158_430_208
    assert bench.allowed_pairs_per_head(W["swa_diff_l8192"]) == 4_136_704
    assert bench.flops(W["tiny"]) == 2 * 64 * 64 * 256
