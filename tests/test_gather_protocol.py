"""Model check of the gather kernel's synchronisation protocol (no GPU).

The model of tests/protocol_model.py restated for csrc/sa_tc.cu: one
producer warp gathering a tile's sigma, Q, K and V rows into shared-memory
stage it % S (the copies complete transaction bytes on the stage's full
barrier); one thread issuing S = Q K^T into TMEM stage it % T and, one tile
behind, O = P V into the same columns; softmax warpgroups taking tiles it %
num_wg, each warp its own actor on its TMEM lane quarter, reading S,
writing P over the stage's dead Q and K bytes, and reading O out.  Every stage count the host picks (S in {1, 2}, T in 1..4,
two warpgroups only with S and T even) must be free of deadlock, phase
aliasing and buffer races; planted mistakes must be caught, among them one
of the kind behind the GPU fault of an early version (two warpgroups sharing
one shared-memory stage, each waiting for the stage's sigma before its S: the
parity wait can pass on the previous tile's phase and read stale sigma).
"""

from __future__ import annotations

from dataclasses import dataclass

import pytest

from protocol_model import Barrier, Buffer, ProtocolError, arrive, copy, mma, simulate, wait
from protocol_model import call as do


@dataclass
class GatherConfig:
    ntiles: int
    s_stages: int
    t_stages: int
    num_wg: int
    producer_waits_empty: bool = True
    qk_waits_tempty: bool = True
    sigma_wait_after_s: bool = True  # the softmax waits for its S before the stage's sigma


class GatherModel:
    def __init__(self, cfg: GatherConfig):
        self.cfg = cfg
        S, T = cfg.s_stages, cfg.t_stages
        self.full = [Barrier(f"full{s}", 1) for s in range(S)]
        self.empty = [Barrier(f"empty{s}", 1) for s in range(S)]
        self.pfull = [Barrier(f"pfull{s}", 4) for s in range(S)]
        self.sfull = [Barrier(f"sfull{t}", 1) for t in range(T)]
        self.ofull = [Barrier(f"ofull{t}", 1) for t in range(T)]
        self.tempty = [Barrier(f"tempty{t}", 4) for t in range(T)]
        self.sig = [Buffer(f"sigma{s}") for s in range(S)]
        # Q and K rows, then P over them (per quarter of the 128 rows)
        self.qk = [[Buffer(f"QK/P{s}.{q}") for q in range(4)] for s in range(S)]
        self.v = [Buffer(f"V{s}") for s in range(S)]
        # S, then O in the same columns, per TMEM lane quarter
        self.tm = [[Buffer(f"TMEM{t}.{q}") for q in range(4)] for t in range(T)]

    def producer(self):
        c = self.cfg
        for it in range(c.ntiles):
            s = it % c.s_stages
            z = it // c.s_stages
            if c.producer_waits_empty:
                yield wait(self.empty[s], (z & 1) ^ 1, z - 1)
            yield do(lambda s=s, it=it: self.sig[s].write("producer", it))
            yield arrive(self.full[s], tx=2)
            yield do(lambda s=s, it=it: self.sig[s].read("producer", it))  # the gathers' rows
            yield copy([(b, ("QK", it)) for b in self.qk[s]], f"gatherQK{it}", self.full[s], "tx")
            yield copy([(self.v[s], it)], f"gatherV{it}", self.full[s], "tx")

    def mma_thread(self):
        c = self.cfg
        S, T = c.s_stages, c.t_stages

        def qk(it):
            s, ts = it % S, it % T
            yield wait(self.full[s], (it // S) & 1, it // S)
            if c.qk_waits_tempty:
                yield wait(self.tempty[ts], ((it // T) & 1) ^ 1, it // T - 1)
            yield mma([(b, ("QK", it)) for b in self.qk[s]], [(b, ("S", it)) for b in self.tm[ts]],
                      f"QK{it}", [self.sfull[ts]])

        def pv(it):
            s, ts = it % S, it % T
            yield wait(self.pfull[s], (it // S) & 1, it // S)
            yield mma([(b, ("P", it)) for b in self.qk[s]] + [(self.v[s], it)],
                      [(b, ("O", it)) for b in self.tm[ts]], f"PV{it}", [self.ofull[ts], self.empty[s]])

        overlap = S >= 2 and T >= 2
        for it in range(c.ntiles):
            if not overlap and it > 0:
                yield from pv(it - 1)
            yield from qk(it)
            if overlap and it > 0:
                yield from pv(it - 1)
        if c.ntiles > 0:
            yield from pv(c.ntiles - 1)

    def softmax_warp(self, wg, q):
        """Warp q of softmax warpgroup wg: TMEM lane quarter q, rows 32q..."""
        c = self.cfg
        S, T = c.s_stages, c.t_stages
        who = f"softmax{wg}.{q}"
        for it in range(c.ntiles):
            if it % c.num_wg != wg:
                continue
            s, ts = it % S, it % T
            if c.sigma_wait_after_s:
                yield wait(self.sfull[ts], (it // T) & 1, it // T)
                yield wait(self.full[s], (it // S) & 1, it // S)
            else:
                yield wait(self.full[s], (it // S) & 1, it // S)
                yield wait(self.sfull[ts], (it // T) & 1, it // T)

            def passes(s=s, ts=ts, it=it):
                self.sig[s].read(who, it)
                self.tm[ts][q].read(who, ("S", it))
                self.qk[s][q].write(who, ("P", it))  # over the dead Q and K bytes
            yield do(passes)
            yield arrive(self.pfull[s])
            yield wait(self.ofull[ts], (it // T) & 1, it // T)
            yield do(lambda ts=ts, it=it: self.tm[ts][q].read(who + "epi", ("O", it)))
            yield arrive(self.tempty[ts])

    def run(self, seed: int):
        roles = {"producer": self.producer(), "mma": self.mma_thread()}
        for wg in range(self.cfg.num_wg):
            for q in range(4):
                roles[f"softmax{wg}.{q}"] = self.softmax_warp(wg, q)
        return simulate(roles, seed)


CONFIGS = {  # the stage counts the host can pick
    "S2_T2_two_wg": GatherConfig(ntiles=14, s_stages=2, t_stages=2, num_wg=2),
    "S2_T4_two_wg": GatherConfig(ntiles=14, s_stages=2, t_stages=4, num_wg=2),
    "S2_T1_one_wg": GatherConfig(ntiles=10, s_stages=2, t_stages=1, num_wg=1),
    "S1_T4_one_wg": GatherConfig(ntiles=10, s_stages=1, t_stages=4, num_wg=1),
    "S1_T1_one_wg": GatherConfig(ntiles=8, s_stages=1, t_stages=1, num_wg=1),
    "S1_T3_one_wg": GatherConfig(ntiles=10, s_stages=1, t_stages=3, num_wg=1),
}


@pytest.mark.parametrize("name", sorted(CONFIGS))
def test_gather_protocol_has_no_race_deadlock_or_parity_alias(name):
    for seed in range(150):
        GatherModel(CONFIGS[name]).run(seed)


MUTANTS = {
    "two warpgroups on one smem stage, sigma waited for before S":
        GatherConfig(ntiles=14, s_stages=1, t_stages=2, num_wg=2, sigma_wait_after_s=False),
    "producer refills a stage before its O MMA":
        GatherConfig(ntiles=14, s_stages=2, t_stages=2, num_wg=2, producer_waits_empty=False),
    "S MMA into a TMEM stage before its read-out":
        GatherConfig(ntiles=14, s_stages=2, t_stages=2, num_wg=2, qk_waits_tempty=False),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_gather_protocol_mistakes_are_caught(name):
    for seed in range(600):
        try:
            GatherModel(MUTANTS[name]).run(seed)
        except ProtocolError:
            return
    pytest.fail(f"the model did not catch: {name}")
