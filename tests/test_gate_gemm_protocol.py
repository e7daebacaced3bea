"""Model check of the gate-projection GEMM's stage pipeline (no GPU).

The model of tests/protocol_model.py restated for sa_gate_proj_kernel in
csrc/sa_prologue.cu.  Its threads meet at CTA barriers, so they are one
actor; beside them run the copy engine (cp.async, one commit group per
64-column block, cp.async.wait_group) and the tensor pipe.  Blocks are
numbered over all of the CTA's tiles; block g uses stage g mod S (S = 2 or
4), and its MMA commit completes phase g / S of that stage's barrier.  Per
tile: the first S - 1 blocks are loaded (their stages were last read by the
previous tile's MMAs, which its final wait covers); block kb + S - 1 is
loaded into the stage block kb - 1 used once that block's MMA is done;
wait_group(S - 1) lands block kb, whose MMA accumulates into TMEM; the last
block's barrier is waited for and the accumulator read out.  Planted
mistakes (a stage reloaded before its MMA is done, a wait_group one too
lax, a tile's read-out before its last MMA) must be caught.
"""

from __future__ import annotations

from dataclasses import dataclass

import pytest

from protocol_model import (Accumulator, Barrier, Buffer, ProtocolError, commit_group, copy, mma,
                            simulate, wait, wait_group)
from protocol_model import call as do


@dataclass
class GemmConfig:
    ntiles: int
    nkb: int          # 64-column blocks per tile
    stages: int       # 2 or 4
    reload_waits: bool = True
    group_slack: int = 0      # extra groups wait_group lets through (a mistake when > 0)
    final_wait: bool = True


class GemmModel:
    def __init__(self, cfg: GemmConfig):
        self.cfg = cfg
        S = cfg.stages
        self.bars = [Barrier(f"stage{s}", 1) for s in range(S)]
        self.stage = [Buffer(f"x/w{s}") for s in range(S)]
        self.acc = Accumulator("TMEM")

    def cta(self):
        c = self.cfg
        S = c.stages
        g0 = 0
        for tile in range(c.ntiles):
            def load(kb, g0=g0):
                g = g0 + kb
                return copy([(self.stage[g % S], g)], f"load{g}", None, "")
            for j in range(S - 1):
                if j < c.nkb:
                    yield load(j)
                yield commit_group()
            for kb in range(c.nkb):
                gb = g0 + kb
                nk = kb + S - 1
                if nk < c.nkb:
                    if kb >= 1 and c.reload_waits:
                        gp = gb - 1
                        yield wait(self.bars[gp % S], (gp // S) & 1, gp // S)
                    yield load(nk)
                yield commit_group()
                yield wait_group(S - 1 + c.group_slack)
                yield mma([(self.stage[gb % S], gb)], [(self.acc, ("tile", tile), kb == 0)],
                          f"mma{gb}", [self.bars[gb % S]])
            gl = g0 + c.nkb - 1
            if c.final_wait:
                yield wait(self.bars[gl % S], (gl // S) & 1, gl // S)
            yield do(lambda tile=tile: self.acc.read("epilogue", ("tile", tile)))
            g0 += c.nkb

    def run(self, seed: int):
        return simulate({"cta": self.cta()}, seed)


CONFIGS = {
    "four_stages": GemmConfig(ntiles=4, nkb=9, stages=4),
    "two_stages": GemmConfig(ntiles=4, nkb=7, stages=2),
    "four_stages_short_tiles": GemmConfig(ntiles=6, nkb=2, stages=4),
    "two_stages_one_block": GemmConfig(ntiles=5, nkb=1, stages=2),
}


@pytest.mark.parametrize("name", sorted(CONFIGS))
def test_gate_gemm_pipeline_has_no_race_deadlock_or_parity_alias(name):
    for seed in range(200):
        GemmModel(CONFIGS[name]).run(seed)


MUTANTS = {
    "a stage reloaded before its MMA is done": GemmConfig(ntiles=3, nkb=9, stages=4,
                                                          reload_waits=False),
    "wait_group one group too lax": GemmConfig(ntiles=3, nkb=9, stages=4, group_slack=1),
    "read-out before the tile's last MMA": GemmConfig(ntiles=3, nkb=5, stages=2,
                                                      final_wait=False),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_gate_gemm_mistakes_are_caught(name):
    for seed in range(600):
        try:
            GemmModel(MUTANTS[name]).run(seed)
        except ProtocolError:
            return
    pytest.fail(f"the model did not catch: {name}")
