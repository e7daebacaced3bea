"""Host-side logic of bench.py that needs no GPU: the multi-rank (replica)
reduction over a world_size-2 gloo process group, the job-throughput
arithmetic, the algorithmic byte and FLOP counts, and the reference arm's
behaviour on ranks other than 0."""

from __future__ import annotations

import json

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


@pytest.mark.parametrize("n,w", [(1, 1), (5, 2), (64, 9), (256, 32), (100, 300), (2048, 128),
                                 (32768, 128)])
def test_pair_counts_agree_with_the_oracle_closed_forms(n, w):
    """The bench's pair counts are the oracle's closed forms, which the oracle
    pins check against brute-force adjacency counts."""
    from oracle import graph
    assert bench.causal_sa_pairs(n, w) == graph.attended_pairs_closed_form(n, w, "sa", True)
    assert bench.swa_pairs(n, w) == graph.attended_pairs_closed_form(n, w, "swa")


@pytest.mark.parametrize("name,window,seq_len,mb,gflop", [
    # algorithmic bytes (MB) and FLOPs (GF) per step, as tabulated for each shape
    ("pretrain_layer", 0, 0, 68.2, 6.31),
    ("long_prefill_gqa", 32, 0, 671.2, 9.12),
    ("long_prefill_gqa", 64, 0, 671.2, 17.71),
    ("long_prefill_gqa", 256, 0, 671.2, 69.12),
    ("very_long_context", 0, 0, 2450.0, 3290.0),
    ("very_long_context", 2048, 0, 2450.0, 6556.0),
    ("length_sweep", 0, 0, 4300.0, 139.6),
    ("length_sweep", 0, 2048, 33.6, 1.07),
])
def test_algorithmic_counts_of_every_workload(name, window, seq_len, mb, gflop):
    wl = dict(bench.WORKLOADS[name])
    if window:
        wl["window"] = window
    if seq_len:
        wl["seq_len"] = seq_len
    b, f = bench.algorithmic(wl)
    assert b / 1e6 == pytest.approx(mb, rel=5e-3)
    assert f / 1e9 == pytest.approx(gflop, rel=5e-3)


def test_reference_arm_other_ranks_exit_without_work(monkeypatch):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class Args:
        steps, warmup = 1, 3

    assert bench.run_reference(Args()) == 0


def test_reference_arm_prints_the_contract_line(monkeypatch, capsys):
    """Rank 0 of the reference arm times the oracle and prints one JSON line
    with the keys the bench contract names (checked on a tiny workload)."""
    monkeypatch.delenv("RANK", raising=False)
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    monkeypatch.setattr(bench.os, "sched_getaffinity", lambda pid: {0, 1})
    wl = dict(workload="tiny", batch=1, seq_len=256, num_q_heads=2, num_kv_heads=2, head_dim=64,
              window=32, causal=True, path="sa", seed=0, std=None)

    class Args:
        steps, warmup = 1, 0

    assert bench.run_reference(Args(), wl) == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e", "gpu_launches"):
        assert key in line, key
    assert line["impl"] == "reference" and line["value"] > 0 and line["unit"] == "tokens/s"
    assert line["n_gpus"] == 1 and line["steps"] == 1 and line["higher_is_better"] is True
    assert line["config"]["workload"] == "tiny" and line["vs_baseline"] is None
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] == 2 and cb["value"] == line["value"]
    assert cb["unit"] == "tokens/s" and cb["sample"]
    assert line["e2e"] == dict(value=line["value"], unit="tokens/s", h2d_bytes_per_step=0,
                               d2h_bytes_per_step=0)


def test_profiled_traffic_follows_the_kernel_source_hash(tmp_path, monkeypatch):
    """roofline.traffic comes from the committed ncu record only while the
    kernel sources hash to the value recorded with it; otherwise it is null."""
    rec = {"traffic_bytes_per_launch": 643352832,
           "kernel_source_sha256": bench.kernel_source_sha256()}
    p = tmp_path / "rec.json"
    p.write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "PROFILE", str(p))
    assert bench.profiled_traffic() == 643352832
    rec["kernel_source_sha256"] = "0" * 64
    p.write_text(json.dumps(rec))
    assert bench.profiled_traffic() is None
    monkeypatch.setattr(bench, "PROFILE", str(tmp_path / "missing.json"))
    assert bench.profiled_traffic() is None


def test_committed_traffic_record_is_plausible():
    """The committed record names the headline kernel and a DRAM byte count
    within 10% of the algorithmic bytes (no operand re-read)."""
    with open(bench.PROFILE) as f:
        rec = json.load(f)
    assert rec["kernel"].startswith("sa::ring::sa_ring_kernel<128")
    alg = 671219712
    assert 0.9 * alg <= rec["traffic_bytes_per_launch"] <= 1.1 * alg
    assert rec["traffic_bytes_per_launch"] == rec["dram_bytes_read"] + rec["dram_bytes_write"]
