"""Host-side logic of bench.py that needs no GPU: the multi-rank (replica)
reduction over a world_size-2 gloo process group, the job-throughput
arithmetic, the algorithmic byte and FLOP counts, and the reference arm's
behaviour on ranks other than 0."""

from __future__ import annotations

import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench as b
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        got = b.max_over_ranks(10.0 + 5.0 * rank, "cpu")
        out.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world_size_2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = dict(q.get(timeout=10) for _ in range(2))
    assert got == {0: 15.0, 1: 15.0}  # every rank reports the slowest


def test_max_over_ranks_without_process_group_is_identity():
    assert bench.max_over_ranks(3.25, "cpu") == 3.25


def test_job_throughput_is_weak_scaling_aggregate():
    # 2 replicas, each 32768 tokens per 0.5 ms step
    assert bench.job_tokens_per_s(2, 32768, 0.5) == pytest.approx(2 * 32768 / 0.5e-3)


def test_algorithmic_counts_of_the_headline_workload():
    b, f = bench.algorithmic(bench.WORKLOAD)
    # Q, K, V, Y once (bf16) and sigma (int32)
    n, hq, hkv, d = 32768, 32, 8, 128
    assert b == 2 * n * d * (hq + 2 * hkv + hq) + 4 * n == 671219712
    # causal SA pairs n(1+h) - h(h+1)/2 with h = 64, two d-length dot products each
    h = 64
    assert f == 4.0 * d * hq * (n * (1 + h) - h * (h + 1) // 2)


def test_reference_arm_other_ranks_exit_without_work(monkeypatch):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class Args:
        steps, warmup = 1, 3

    assert bench.run_reference(Args()) == 0
