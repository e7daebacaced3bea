"""Model check of the backward kernels' operand pipelines (no GPU).

The model of tests/protocol_model.py restated for sa_bwd_dq_kernel in
csrc/sa_bwd.cu.  The kernel's threads meet at CTA barriers, so they are one
actor here; what runs beside them is the copy engine (cp.async gathers, seen
to land only by cp.async.wait_all) and the tensor pipe.  Per tile: the span
tokens go to one of two buffers; Q, dY, K and V rows are gathered; S = Q K^T
and dP = dY V^T run into TMEM; the next tile's tokens are written and its Q,
dY and V rows gathered once those MMAs are done; three passes over TMEM
write dS over S; dQ = dS K runs into the dP columns; the next tile's K rows
are gathered once it is done; dQ is read out.  The key-tile kernel
(sa_bwd_dkv_kernel) keeps a tile's K and V rows and walks its query chunks
through two stages: chunk c + 1's tokens, Q and dY rows, lse2' and D are
prepared into the other stage while chunk c is computed (S^T and dP^T into
TMEM, the elementwise pass over them, dV and dK accumulated in TMEM).
Planted mistakes (a gather issued before the MMA that reads its buffer is
done, one token buffer, the wait for the copies left out, a chunk's second
MMAs not waited for) must be caught.
"""

from __future__ import annotations

from dataclasses import dataclass

import pytest

from protocol_model import (Accumulator, Barrier, Buffer, ProtocolError, commit_group, copy,
                            mma, simulate, wait, wait_copies)
from protocol_model import call as do


@dataclass
class DqConfig:
    ntiles: int
    v_after_s_mma: bool = True    # next V gathered after the S / dP MMAs
    k_after_dq_mma: bool = True   # next K gathered after the dQ MMA
    token_buffers: int = 2
    waits_copies: bool = True


class DqModel:
    def __init__(self, cfg: DqConfig):
        self.cfg = cfg
        self.mma_bar = Barrier("mma", 1)
        self.sig = [Buffer(f"tokens{b}") for b in range(cfg.token_buffers)]
        self.q, self.dy = Buffer("Q"), Buffer("dY")
        self.k, self.v = Buffer("K"), Buffer("V")
        self.ts = Buffer("TMEM.S")     # S, then dS over it
        self.tp = Buffer("TMEM.dP")    # dP, then dQ over it

    def gathers(self, x, which):
        sg = self.sig[x % len(self.sig)]
        for name in which:
            buf = {"Q": self.q, "dY": self.dy, "K": self.k, "V": self.v}[name]
            yield do(lambda sg=sg, x=x: sg.read("gather", x))   # rows from the tokens
            yield copy([(buf, x)], f"gather{name}{x}", None, "")

    def cta(self):
        c = self.cfg
        phase = 0
        if c.ntiles:
            yield do(lambda: self.sig[0].write("cta", 0))
            yield from self.gathers(0, ["Q", "dY", "K", "V"])
        for x in range(c.ntiles):
            cur = self.sig[x % len(self.sig)]
            nxt_sig = self.sig[(x + 1) % len(self.sig)]
            has_next = x + 1 < c.ntiles
            if c.waits_copies:
                yield wait_copies()
            yield mma([(self.q, x), (self.k, x), (self.dy, x), (self.v, x)],
                      [(self.ts, ("S", x)), (self.tp, ("dP", x))], f"SdP{x}", [self.mma_bar])
            if has_next:
                yield do(lambda x=x, nb=nxt_sig: nb.write("cta", x + 1))
            if not c.v_after_s_mma and has_next:
                yield from self.gathers(x + 1, ["V"])
            yield wait(self.mma_bar, phase & 1, phase)
            phase += 1
            if has_next:
                yield from self.gathers(x + 1, ["Q", "dY"] + (["V"] if c.v_after_s_mma else []))
            if not c.k_after_dq_mma and has_next:
                yield from self.gathers(x + 1, ["K"])

            def passes(x=x, cur=cur):
                cur.read("passes", x)
                self.ts.read("passes", ("S", x))
                self.tp.read("passes", ("dP", x))
                self.ts.write("passes", ("dS", x))
            yield do(passes)
            yield mma([(self.ts, ("dS", x)), (self.k, x)], [(self.tp, ("dQ", x))], f"dQ{x}",
                      [self.mma_bar])
            yield wait(self.mma_bar, phase & 1, phase)
            phase += 1
            if c.k_after_dq_mma and has_next:
                yield from self.gathers(x + 1, ["K"])
            yield do(lambda x=x: self.tp.read("write-out", ("dQ", x)))

    def run(self, seed: int):
        return simulate({"cta": self.cta()}, seed)


def test_dq_pipeline_has_no_race_or_deadlock():
    for ntiles in (1, 2, 7):
        for seed in range(200):
            DqModel(DqConfig(ntiles=ntiles)).run(seed)


MUTANTS = {
    "next V gathered before the S and dP MMAs are done": DqConfig(ntiles=5, v_after_s_mma=False),
    "next K gathered before the dQ MMA is done": DqConfig(ntiles=5, k_after_dq_mma=False),
    "one token buffer": DqConfig(ntiles=5, token_buffers=1),
    "MMAs issued without waiting for the copies": DqConfig(ntiles=5, waits_copies=False),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_dq_pipeline_mistakes_are_caught(name):
    for seed in range(600):
        try:
            DqModel(MUTANTS[name]).run(seed)
        except ProtocolError:
            return
    pytest.fail(f"the model did not catch: {name}")


@dataclass
class DkvConfig:
    ntiles: int
    nchunks: int
    waits_second_mmas: bool = True   # a chunk's dV / dK MMAs done before the next chunk


class DkvModel:
    def __init__(self, cfg: DkvConfig):
        self.cfg = cfg
        self.mma_bar = Barrier("mma", 1)
        self.ktok = Buffer("ktok")
        self.k, self.v = Buffer("K"), Buffer("V")
        self.qtok = [Buffer(f"qtok{s}") for s in range(2)]
        self.q = [Buffer(f"Q{s}") for s in range(2)]
        self.dy = [Buffer(f"dY{s}") for s in range(2)]
        self.col = [Buffer(f"lse/D{s}") for s in range(2)]
        self.ts, self.tp = Buffer("TMEM.S^T"), Buffer("TMEM.dP^T")  # then P' and dS^T over them
        self.dv, self.dk = Accumulator("TMEM.dV"), Accumulator("TMEM.dK")

    def cta(self):
        c = self.cfg
        phase = 0
        for x in range(c.ntiles):
            yield do(lambda x=x: self.ktok.write("cta", x))
            yield do(lambda x=x: self.ktok.read("gather", x))
            yield copy([(self.k, x)], f"K{x}", None, "")
            yield copy([(self.v, x)], f"V{x}", None, "")

            def prepare(ch, x=x):
                st = ch & 1
                tag = (x, ch)
                yield do(lambda: self.qtok[st].write("prepare", tag))
                yield do(lambda: self.qtok[st].read("gather", tag))
                yield copy([(self.q[st], tag)], f"Q{tag}", None, "")
                yield copy([(self.dy[st], tag)], f"dY{tag}", None, "")
                yield commit_group()
                yield do(lambda: self.col[st].write("prepare", tag))
            yield from prepare(0)
            for ch in range(c.nchunks):
                st, tag = ch & 1, (x, ch)
                yield wait_copies()
                if ch + 1 < c.nchunks:
                    yield from prepare(ch + 1)
                yield mma([(self.k, x), (self.q[st], tag), (self.v, x), (self.dy[st], tag)],
                          [(self.ts, ("S", tag)), (self.tp, ("dP", tag))], f"SdP{tag}",
                          [self.mma_bar])
                yield wait(self.mma_bar, phase & 1, phase)
                phase += 1

                def elementwise(st=st, tag=tag):
                    self.qtok[st].read("elementwise", tag)
                    self.col[st].read("elementwise", tag)
                    self.ts.read("elementwise", ("S", tag))
                    self.tp.read("elementwise", ("dP", tag))
                    self.ts.write("elementwise", ("P", tag))
                    self.tp.write("elementwise", ("dS", tag))
                yield do(elementwise)
                yield mma([(self.ts, ("P", tag)), (self.dy[st], tag), (self.tp, ("dS", tag)),
                           (self.q[st], tag)],
                          [(self.dv, ("dV", x), ch == 0), (self.dk, ("dK", x), ch == 0)],
                          f"dVdK{tag}", [self.mma_bar])
                if c.waits_second_mmas:
                    yield wait(self.mma_bar, phase & 1, phase)
                phase += 1
            if not c.waits_second_mmas:  # the last chunk's MMAs, at least
                yield wait(self.mma_bar, (phase - 1) & 1, phase - 1)
            yield do(lambda x=x: (self.dv.read("write-out", ("dV", x)),
                                  self.dk.read("write-out", ("dK", x))))

    def run(self, seed: int):
        return simulate({"cta": self.cta()}, seed)


def test_dkv_pipeline_has_no_race_or_deadlock():
    for ntiles, nch in ((1, 1), (2, 3), (3, 9)):
        for seed in range(200):
            DkvModel(DkvConfig(ntiles=ntiles, nchunks=nch)).run(seed)


def test_dkv_planted_mistake_is_caught():
    """A chunk's dV / dK MMAs not waited for before the next chunk's S^T and
    dP^T overwrite the TMEM columns they read."""
    for seed in range(600):
        try:
            DkvModel(DkvConfig(ntiles=2, nchunks=4, waits_second_mmas=False)).run(seed)
        except ProtocolError:
            return
    pytest.fail("the model did not catch the missing wait")
