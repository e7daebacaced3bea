"""sigma-routed sequence sharding, host side (CPU only): the library's
routing plan, the exactness of running the local problem in place of the
whole sequence, and the two all-to-all exchanges on gloo ranks (world sizes 2
and 3), with the fp64 oracle as each rank's local attention."""

from __future__ import annotations

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from stochastic_sliding_window_gb300 import shard


@pytest.mark.parametrize("n,w,world", [(1000, 64, 4), (37, 9, 5), (10, 4, 16), (513, 600, 3),
                                       (32768, 128, 8)])
def test_plan_invariants(n, w, world):
    perm = oracle.make_perm(7, 1, 0, n).astype(np.int32)
    ps = shard.plans(perm, w, world)
    c = -(-n // world)
    owned = np.concatenate([np.arange(p.own_begin, p.own_end) for p in ps])
    assert np.array_equal(owned, np.arange(n))  # the ranks' positions partition the sequence
    h = w // 2
    for r, p in enumerate(ps):
        assert p.chunk == c and p.own_begin == min(r * c, n)
        m = len(p.tokens)
        if p.own_end > p.own_begin:
            assert p.span_begin == max(0, p.own_begin - h)
            assert p.span_begin + m == min(n, p.own_end + h)
        assert (np.diff(p.tokens) > 0).all()
        assert np.array_equal(np.sort(p.local_perm), np.arange(m))
        assert np.array_equal(p.tokens[p.local_perm], perm[p.span_begin:p.span_begin + m])
        assert np.array_equal(p.own_tokens, perm[p.own_begin:p.own_end])
        assert sum(p.counts_from()) == m


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("n,w,world", [(300, 32, 3), (128, 40, 4), (64, 200, 2)])
def test_local_problems_give_the_global_rows_exactly(causal, n, w, world):
    """The local problem (span tokens in original order, local sigma) gives
    each owned position's row bit for bit as the whole sequence does: same
    keys, same order, same fp64 arithmetic."""
    rng = np.random.default_rng(n)
    q = rng.standard_normal((1, n, 4, 8))
    k = rng.standard_normal((1, n, 2, 8))
    v = rng.standard_normal((1, n, 2, 8))
    perm = oracle.make_perm(3, 0, 0, n)
    full = oracle.sa_forward(q, k, v, perm[None], w, causal)
    for p in shard.plans(perm.astype(np.int32), w, world):
        t = p.tokens
        loc = oracle.sa_rows(q[:, t], k[:, t], v[:, t], p.local_perm[None].astype(np.int64), w,
                             causal, rows=[(0, int(i)) for i in p.own_local])
        assert np.array_equal(loc, full[0, p.own_tokens])


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, n, w, causal, q, k, v, perm, want, q_out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        c = -(-n // world)
        lo, hi = min(rank * c, n), min(rank * c + c, n)
        ps = shard.plans(perm.astype(np.int32), w, world)
        me = ps[rank]
        loc = [shard.gather_local(torch.from_numpy(x[lo:hi]), ps, rank) for x in (q, k, v)]
        for got, x in zip(loc, (q, k, v)):  # each rank holds exactly its span's rows
            assert np.array_equal(got.numpy(), x[me.tokens])
        y = oracle.sa_rows(loc[0].numpy()[None], loc[1].numpy()[None], loc[2].numpy()[None],
                           me.local_perm[None].astype(np.int64), w, causal,
                           rows=[(0, int(i)) for i in me.own_local])
        mine = shard.scatter_back(torch.from_numpy(np.ascontiguousarray(y)), ps, rank, hi - lo)
        q_out.put((rank, bool(np.array_equal(mine.numpy(), want[lo:hi]))))
    except Exception as e:  # report, never hang the other ranks
        q_out.put((rank, repr(e)))
        raise
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world,n,w,causal", [(2, 200, 16, True), (3, 301, 40, False),
                                              (3, 50, 200, True)])
def test_gloo_ranks_exchange_and_reassemble(world, n, w, causal):
    rng = np.random.default_rng(world * 100 + n)
    q = rng.standard_normal((n, 4, 8))
    k = rng.standard_normal((n, 2, 8))
    v = rng.standard_normal((n, 2, 8))
    perm = oracle.make_perm(11, 0, 0, n)
    want = oracle.sa_forward(q[None], k[None], v[None], perm[None], w, causal)[0]
    ctx = mp.get_context("spawn")
    q_out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, n, w, causal, q, k, v, perm, want,
                                               q_out)) for r in range(world)]
    for p in procs:
        p.start()
    results = dict(q_out.get(timeout=180) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
    assert all(results[r] is True for r in range(world)), results
