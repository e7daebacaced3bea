"""sigma-routed sequence sharding of SA over several GPUs (one rank each).

One sequence is split twice with the same chunk c = ceil(n / world): rank r
holds the original tokens [r c, (r+1) c) of Q, K, V and of the output, and
computes the SA rows of the permuted positions [r c, (r+1) c) (the "Core
mechanism" of the Stochastic Attention summary runs sliding-window attention
over the permuted order).  The routing plan comes from the library
(sa_shard_plan): the span of positions rank r works on (its own plus the
window halo), that span's tokens in ascending original order (the local rows)
and the local permutation.  Two all-to-all exchanges move the rows:
gather_local brings each rank the Q/K/V rows of its span's tokens from their
owners, scatter_back returns each owned position's output row to its token's
owner.  Because the local rows keep the original order, the causal rule holds
unchanged and sa_forward runs the local problem as is (sharded_sa_forward).

Every rank computes every rank's plan (sigma is replicated; a plan costs
O(n + span log span) on the host), which fixes the order of every send and
receive without an extra exchange of requests.
"""

from __future__ import annotations

import ctypes
from dataclasses import dataclass

import numpy as np

from ._libsa import _check, load


@dataclass
class ShardPlan:
    n: int
    window: int
    world: int
    rank: int
    chunk: int           # c: tokens and positions per rank
    tokens: np.ndarray   # int32 [span]: local rows' tokens, ascending
    local_perm: np.ndarray  # int32 [span]: local row of each span position
    span_begin: int
    own_begin: int
    own_end: int

    @property
    def own_local(self) -> np.ndarray:
        """Local rows of the owned positions, in permuted order."""
        return self.local_perm[self.own_begin - self.span_begin:self.own_end - self.span_begin]

    @property
    def own_tokens(self) -> np.ndarray:
        """Tokens of the owned positions (where their rows go)."""
        return self.tokens[self.own_local]

    def counts_from(self) -> list[int]:
        """Rows this rank receives from each rank in gather_local."""
        edges = np.arange(self.world + 1) * self.chunk
        return np.diff(np.searchsorted(self.tokens, edges)).tolist()


def plan(perm: np.ndarray, window: int, world: int, rank: int) -> ShardPlan:
    """The library's routing plan of one rank (perm: sigma of the sequence)."""
    lib = load()
    perm = np.ascontiguousarray(perm, dtype=np.int32)
    n = perm.shape[0]
    cap = int(lib.sa_shard_span(n, int(window), int(world), int(rank)))
    tok = np.zeros(max(cap, 1), dtype=np.int32)
    lp = np.zeros(max(cap, 1), dtype=np.int32)
    s0, o0, o1 = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
    ip = ctypes.POINTER(ctypes.c_int32)
    _check(lib.sa_shard_plan(perm.ctypes.data_as(ip), n, int(window), int(world), int(rank),
                             tok.ctypes.data_as(ip), lp.ctypes.data_as(ip), max(cap, 1),
                             ctypes.byref(s0), ctypes.byref(o0), ctypes.byref(o1)))
    return ShardPlan(n, int(window), int(world), int(rank), -(-n // world), tok[:cap], lp[:cap],
                     s0.value, o0.value, o1.value)


def plans(perm: np.ndarray, window: int, world: int) -> list[ShardPlan]:
    return [plan(perm, window, world, r) for r in range(world)]


def gather_local(x_shard, all_plans: list[ShardPlan], rank: int, group=None):
    """Rows of this rank's span tokens, [span, ...] in ascending token order,
    from the token shards x_shard ([rows of tokens rank*c ..., ...]) of every
    rank: one all-to-all."""
    import torch
    import torch.distributed as dist
    me = all_plans[rank]
    lo = rank * me.chunk
    send_idx, send_counts = [], []
    for p in all_plans:  # what each rank needs of my tokens, in its order
        a, b = np.searchsorted(p.tokens, [lo, lo + me.chunk])
        send_idx.append(p.tokens[a:b] - lo)
        send_counts.append(int(b - a))
    idx = torch.from_numpy(np.concatenate(send_idx).astype(np.int64)).to(x_shard.device)
    send = x_shard.index_select(0, idx).contiguous()
    recv_counts = me.counts_from()
    out = torch.empty((sum(recv_counts),) + tuple(x_shard.shape[1:]), dtype=x_shard.dtype,
                      device=x_shard.device)
    dist.all_to_all_single(out, send, recv_counts, send_counts, group=group)
    return out


def scatter_back(y_own, all_plans: list[ShardPlan], rank: int, rows: int, group=None):
    """Owned positions' output rows (y_own [own, ...], in permuted order) to
    their tokens' owners; returns this rank's token shard [rows, ...]: one
    all-to-all."""
    import torch
    import torch.distributed as dist
    me = all_plans[rank]
    c = me.chunk
    dest = me.own_tokens // c
    order = np.lexsort((me.own_tokens, dest))  # by owner, then by token
    send = y_own.index_select(0, torch.from_numpy(order.astype(np.int64)).to(y_own.device))
    send_counts = np.bincount(dest, minlength=me.world).tolist()
    recv_tok = []
    for p in all_plans:  # what each rank sends me: my tokens among its owned ones
        t = p.own_tokens
        recv_tok.append(np.sort(t[(t >= rank * c) & (t < rank * c + c)]))
    recv_counts = [len(t) for t in recv_tok]
    buf = torch.empty((sum(recv_counts),) + tuple(y_own.shape[1:]), dtype=y_own.dtype,
                      device=y_own.device)
    dist.all_to_all_single(buf, send.contiguous(), recv_counts, send_counts, group=group)
    out = torch.empty((rows,) + tuple(y_own.shape[1:]), dtype=y_own.dtype, device=y_own.device)
    place = torch.from_numpy((np.concatenate(recv_tok) - rank * c).astype(np.int64)).to(y_own.device)
    out.index_copy_(0, place, buf)
    return out


def sharded_sa_forward(q_shard, k_shard, v_shard, perm: np.ndarray, window: int,
                       causal: bool = True, group=None, err=None):
    """SA of one sequence split over the ranks of `group`: q_shard [c_r, Hq, d]
    and k_shard, v_shard [c_r, Hkv, d] hold this rank's tokens (bf16, on its
    GPU); returns this rank's output rows [c_r, Hq, d]."""
    import torch
    import torch.distributed as dist
    from ._libsa import sa_forward
    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    ps = plans(perm, window, world)
    me = ps[rank]
    ql = gather_local(q_shard, ps, rank, group)
    kl = gather_local(k_shard, ps, rank, group)
    vl = gather_local(v_shard, ps, rank, group)
    lp = torch.from_numpy(me.local_perm[None, :].copy()).to(q_shard.device)
    y = sa_forward(ql[None], kl[None], vl[None], lp, window, causal=causal, err=err)[0]
    own = torch.from_numpy(me.own_local.astype(np.int64)).to(q_shard.device)
    return scatter_back(y.index_select(0, own), ps, rank, q_shard.shape[0], group)
