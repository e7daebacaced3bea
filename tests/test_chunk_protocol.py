"""Model check of the chunk kernel's synchronisation protocol (no GPU).

The same model as tests/test_ring_protocol.py (mbarriers with counts,
transaction-free cp.async arrivals and parity waits; the tensor pipe; every
buffer handed between roles), restated for csrc/sa_tc_chunk.cu: producers
loading each tile's Q rows and tokens into a Q stage and each 128-key chunk's
K, V rows and key tokens into one of two chunk stages; one thread issuing S
= Q K^T per half and chunk as soon as the chunk has landed and the half's
previous O MMA has read P out of the S buffer; per half, four softmax
warps (each its own actor, on its own TMEM lane quarter) that read the
tile's query tokens, build each chunk's masks from its key tokens, correct
O when a reference rises, write P and read O out after the tile's last
chunk, warp 0's first lane issuing O += P V.  Geometries with one chunk per tile and one Q stage are
included: there the tile's only S MMA can finish before the softmax has read
the tile's tokens, so the Q stage must also wait for those reads.
"""

from __future__ import annotations

from dataclasses import dataclass

import pytest

from protocol_model import (Accumulator, Barrier, Buffer, ProtocolError, arrive, copy, mma,
                            simulate, wait)
from protocol_model import call as do


@dataclass
class ChunkGeometry:
    ntiles: int
    nch: int       # 128-key chunks per tile
    qstages: int   # 1 at d = 128, 2 at d = 64


@dataclass
class ChunkMutation:
    softmax_releases_q_stage: bool = True  # the Q stage also waits for the token reads
    qk_waits_previous_pv: bool = True
    producers_wait_chunk_free: bool = True


class ChunkModel:
    def __init__(self, geo: ChunkGeometry, mut: ChunkMutation | None = None):
        self.geo, self.mut = geo, mut or ChunkMutation()
        B = Barrier
        qfree_count = 2 + (8 if self.mut.softmax_releases_q_stage else 0)
        self.q_full = [B(f"Qfull{s}", 1) for s in range(geo.qstages)]
        self.q_free = [B(f"Qfree{s}", qfree_count) for s in range(geo.qstages)]
        self.c_full = [B(f"Cfull{s}", 1) for s in range(2)]
        self.c_free = [B(f"Cfree{s}", 2) for s in range(2)]
        self.s_full = [B(f"Sfull{h}", 1) for h in range(2)]
        self.p_full = [B(f"Pfull{h}", 4) for h in range(2)]
        self.pv_done = [B(f"PVdone{h}", 1) for h in range(2)]
        self.o_full = [B(f"Ofull{h}", 1) for h in range(2)]
        self.qrows = [Buffer(f"Qrows{s}") for s in range(geo.qstages)]
        self.qtok = [Buffer(f"qtok{s}") for s in range(geo.qstages)]
        self.kv = [Buffer(f"KV{s}") for s in range(2)]
        self.csig = [Buffer(f"csig{s}") for s in range(2)]
        # per TMEM lane quarter (warp q of a half's warpgroup owns quarter q)
        self.s_buf = [[Buffer(f"S/P{h}.{q}") for q in range(4)] for h in range(2)]
        self.o_buf = [[Accumulator(f"O{h}.{q}") for q in range(4)] for h in range(2)]

    # ------------------------------------------------------------ roles
    def producers(self):
        g = self.geo
        for x in range(g.ntiles):
            qs = x % g.qstages
            if x >= g.qstages:
                z = x // g.qstages - 1
                yield wait(self.q_free[qs], z & 1, z)
            yield copy([(self.qrows[qs], x), (self.qtok[qs], x)], f"loadQ{x}", self.q_full[qs],
                       "arrive")
            for c in range(g.nch):
                call = x * g.nch + c
                s = call & 1
                if call >= 2 and self.mut.producers_wait_chunk_free:
                    z = (call >> 1) - 1
                    yield wait(self.c_free[s], z & 1, z)
                yield copy([(self.kv[s], call), (self.csig[s], call)], f"loadC{call}",
                           self.c_full[s], "arrive")

    def mma(self):
        """One thread polls both halves; modelled as one actor per half, which
        allows every interleaving the polling loop allows."""
        g = self.geo
        total = g.ntiles * g.nch

        def half(h):
            for call in range(total):
                x, c = divmod(call, g.nch)
                qs = x % g.qstages
                yield wait(self.c_full[call & 1], (call >> 1) & 1, call >> 1)
                if self.mut.qk_waits_previous_pv:
                    yield wait(self.pv_done[h], (call & 1) ^ 1, call - 1)
                if c == 0:
                    z = x // g.qstages
                    yield wait(self.q_full[qs], z & 1, z)
                commits = [self.s_full[h]] + ([self.q_free[qs]] if c == g.nch - 1 else [])
                yield mma([(self.qrows[qs], x), (self.kv[call & 1], call)],
                          [(b, ("S", call)) for b in self.s_buf[h]], f"QK{h}.{call}", commits)
        return half(0), half(1)

    def softmax_warp(self, h, q):
        """Warp q of half h's softmax warpgroup; warp 0's first lane issues the
        half's O MMAs.  A warp corrects O (after the previous O MMA) only on
        chunks where one of its rows raised its reference: here on a fixed
        pattern that differs between warps."""
        g = self.geo
        who = f"softmax{h}.{q}"
        sb, ob = self.s_buf[h][q], self.o_buf[h][q]
        for x in range(g.ntiles):
            qs = x % g.qstages
            z = x // g.qstages
            yield wait(self.q_full[qs], z & 1, z)
            yield do(lambda qs=qs, x=x: self.qtok[qs].read(who, x))
            if self.mut.softmax_releases_q_stage:
                yield arrive(self.q_free[qs])
            for c in range(g.nch):
                call = x * g.nch + c
                b = call & 1
                yield wait(self.c_full[b], (call >> 1) & 1, call >> 1)
                yield do(lambda b=b, call=call: self.csig[b].read(who, call))
                yield wait(self.s_full[h], call & 1, call)
                if c > 0 and (call + q) % 3 == 0:  # O correction
                    yield wait(self.pv_done[h], (call - 1) & 1, call - 1)
                    yield do(lambda x=x: ob.read(who, ("O", x)))

                def passes(call=call):
                    sb.read(who, ("S", call))
                    sb.write(who, ("P", call))
                yield do(passes)
                yield arrive(self.p_full[h])
                if q == 0:  # the half's issuer
                    yield wait(self.p_full[h], call & 1, call)
                    commits = [self.pv_done[h], self.c_free[b]] + \
                              ([self.o_full[h]] if c == g.nch - 1 else [])
                    yield mma([(bb, ("P", call)) for bb in self.s_buf[h]] + [(self.kv[b], call)],
                              [(ab, ("O", x), c == 0) for ab in self.o_buf[h]],
                              f"PV{h}.{call}", commits)
            yield wait(self.o_full[h], x & 1, x)
            yield do(lambda x=x: ob.read(who + "epi", ("O", x)))

    def run(self, seed: int):
        m0, m1 = self.mma()
        roles = {"producers": self.producers(), "qk0": m0, "qk1": m1}
        for h in range(2):
            for q in range(4):
                roles[f"softmax{h}.{q}"] = self.softmax_warp(h, q)
        return simulate(roles, seed)


GEOMETRIES = {
    "one_chunk_one_qstage": ChunkGeometry(ntiles=8, nch=1, qstages=1),
    "three_chunks_one_qstage": ChunkGeometry(ntiles=5, nch=3, qstages=1),
    "one_chunk_two_qstages": ChunkGeometry(ntiles=8, nch=1, qstages=2),
    "eight_chunks_two_qstages": ChunkGeometry(ntiles=3, nch=8, qstages=2),
}


@pytest.mark.parametrize("geo", sorted(GEOMETRIES))
def test_chunk_protocol_has_no_race_deadlock_or_parity_alias(geo):
    for seed in range(150):
        ChunkModel(GEOMETRIES[geo]).run(seed)


MUTANTS = {
    "Q stage refilled before the softmax read its tokens":
        (ChunkMutation(softmax_releases_q_stage=False), "one_chunk_one_qstage"),
    "S MMA does not wait for the half's previous O MMA":
        (ChunkMutation(qk_waits_previous_pv=False), "three_chunks_one_qstage"),
    "chunk stage refilled before both halves' O MMAs":
        (ChunkMutation(producers_wait_chunk_free=False), "three_chunks_one_qstage"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_chunk_protocol_mistakes_are_caught(name):
    mut, geo = MUTANTS[name]
    for seed in range(600):
        try:
            ChunkModel(GEOMETRIES[geo], mut).run(seed)
        except ProtocolError:
            return
    pytest.fail(f"the model did not catch: {name}")
