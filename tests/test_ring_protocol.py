"""Model check of the ring kernel's synchronisation protocol (no GPU).

compute-sanitizer is closed on this machine, so the hand-over protocol of the
tcgen05 ring kernel (csrc/sa_tc_ring.cu) is restated here as a model and run
under many random interleavings.  The model has
  - every mbarrier of the kernel with its arrival count, its transaction
    count and its phase, and the hardware's parity wait (a wait for parity
    P passes while the barrier's current phase has the other parity);
  - the copy engine: a TMA copy lands at any later time, in any order, and
    completes its transaction on its barrier;
  - the tensor pipe: MMAs complete in issue order, and a commit arrives on
    its barrier once the MMAs issued before it are done;
  - the buffers the roles hand to one another: the Q stages, the K, V and
    sigma ring slots, the mask-word buffers and each TMEM stage (its S/P
    columns and the columns O shares with S), per TMEM lane quarter;
  - each softmax warp as its own actor (the warps of a warpgroup meet only
    at the kernel's barriers), warp 0's first lane issuing the O MMAs.
The roles issue the kernel's waits and arrivals in the kernel's order
(copy_role, mask_role, mma_role, softmax_role).  Each run checks that
  - no role is left waiting forever;
  - every wait is released by exactly the phase it means: never a phase
    early through parity aliasing, never overrun by a later phase;
  - no buffer is written while a reader of its previous contents is still
    reading, and every read sees the contents the reader expects.
Planted mistakes (a retire distance one short, a hand-over without its
release wait, too few word buffers or sigma barriers, an S MMA that does not
wait for the read-out, an O MMA that does not wait for the previous tile's)
must each be caught.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import pytest

from protocol_model import (Buffer, Barrier, ProtocolError, arrive, call, copy, mma, simulate,
                            wait)

K_QSTAGES = 2  # Q stages
K_VDEPTH = 3   # V (and K) rows of tile x overwrite those of tile x - 3


@dataclass
class Tile:
    run: int
    p0: int
    new_seg: bool
    slot_a: int
    ld_pos: list[int]    # positions it loads
    ld_slots: list[int]  # and their ring slots


@dataclass
class Geometry:
    bt: int        # positions per tile
    left: int
    right: int
    tiles_per_seq: int
    first_tile: int  # this CTA's first tile (a run may start before it)
    ntiles: int
    span_pad: int = 0
    ring: int = 0

    def __post_init__(self):
        span = self.bt + self.left + self.right
        self.span_pad = -(-span // 32) * 32
        self.ring = -(-(self.span_pad + 2 * self.bt) // 16) * 16

    def tiles(self) -> list[Tile]:
        """The CTA's tiles in order with the ring mapping of TileWalk."""
        out, slot_a, prev_run = [], 0, None
        for i in range(self.ntiles):
            t = self.first_tile + i
            run, p0 = divmod(t, self.tiles_per_seq)
            p0 *= self.bt
            new_seg = run != prev_run
            prev_run = run
            if new_seg:
                slot_a = 0
                ld_pos = [p0 - self.left + x for x in range(self.span_pad)]
                ld_slots = list(range(self.span_pad))
            else:
                slot_a = (slot_a + self.bt) % self.ring
                first = p0 - self.left + self.span_pad - self.bt
                ld_pos = [first + x for x in range(self.bt)]
                ld_slots = [(slot_a + self.span_pad - self.bt + x) % self.ring
                            for x in range(self.bt)]
            out.append(Tile(run, p0, new_seg, slot_a, ld_pos, ld_slots))
        return out

    def span_slots(self, t: Tile):
        return [((t.slot_a + x) % self.ring, (t.run, t.p0 - self.left + x))
                for x in range(self.span_pad)]

    def row_slots(self, t: Tile):
        """The ring slots of the tile's own positions (sigma of its rows)."""
        return [((t.slot_a + self.left + x) % self.ring, (t.run, t.p0 + x))
                for x in range(self.bt)]


@dataclass
class Mutation:
    """A planted mistake (all off: the kernel's protocol)."""
    qk_retire_lag: int = K_QSTAGES   # Q stage reused after the S MMA this many tiles back
    pv_retire_lag: int = K_VDEPTH    # ring rows reused after the O MMA this many tiles back
    word_buffers: int = 4
    sigw_slots: int = 4
    masker_waits_release: bool = True
    mma_waits_readout: bool = True
    pv_waits_previous: bool = True   # O MMA of tile it after that of tile it - 1


@dataclass
class Model:
    geo: Geometry
    mut: Mutation = field(default_factory=Mutation)

    def __post_init__(self):
        g = self.geo
        self.tiles = g.tiles()
        B = Barrier
        self.full_qk = [B(f"FullQK{s}", 1) for s in range(K_QSTAGES)]
        self.qk_done = [B(f"QKdone{s}", 1) for s in range(K_QSTAGES)]
        self.full_v = [B(f"FullV{s}", 1) for s in range(K_VDEPTH)]
        self.pv_done = [B(f"PVdone{s}", 1) for s in range(K_VDEPTH)]
        self.s_ready = [B(f"Sready{w}", 1) for w in range(2)]
        self.s_free = [B(f"Sfree{w}", 4) for w in range(2)]
        self.s_full = [B(f"Sfull{w}", 1) for w in range(2)]
        self.p_full = [B(f"Pfull{w}", 4) for w in range(2)]
        self.o_full = [B(f"Ofull{w}", 1) for w in range(2)]
        self.t_empty = [B(f"Tempty{w}", 4) for w in range(2)]
        self.sig_w = [B(f"SigW{x}", 1) for x in range(self.mut.sigw_slots)]
        self.q = [Buffer(f"Q{s}") for s in range(K_QSTAGES)]
        self.kr = [Buffer(f"K[{x}]") for x in range(g.ring)]
        self.vr = [Buffer(f"V[{x}]") for x in range(g.ring)]
        self.sg = [Buffer(f"sigma[{x}]") for x in range(g.ring)]
        # per TMEM lane quarter (warp q of a warpgroup reads and writes only its
        # quarter): the words of its rows, its S/P columns and its O columns
        # (S spills into the O columns)
        self.words = [[Buffer(f"words{b}.{q}") for q in range(4)]
                      for b in range(self.mut.word_buffers)]
        self.tp = [[Buffer(f"TMEM{w}.{q}.S/P") for q in range(4)] for w in range(2)]
        self.to = [[Buffer(f"TMEM{w}.{q}.O") for q in range(4)] for w in range(2)]

    def word_buf(self, it):
        if self.mut.word_buffers == 4:
            return self.words[(it & 1) * 2 + ((it >> 1) & 1)]
        return self.words[it % self.mut.word_buffers]

    # ------------------------------------------------------------ roles
    def copier(self):
        g, m = self.geo, self.mut
        qk_seen = pv_seen = -1
        for it, t in enumerate(self.tiles):
            s = it % K_QSTAGES
            upto = it - 1 if t.new_seg else it - m.qk_retire_lag
            for z in range(qk_seen + 1, upto + 1):
                yield wait(self.qk_done[z % K_QSTAGES], (z // K_QSTAGES) & 1, z // K_QSTAGES)
            qk_seen = max(qk_seen, upto)
            upto = it - 1 if t.new_seg else it - m.pv_retire_lag
            for z in range(pv_seen + 1, upto + 1):
                yield wait(self.pv_done[z % K_VDEPTH], (z // K_VDEPTH) & 1, z // K_VDEPTH)
            pv_seen = max(pv_seen, upto)

            def put_sigma(t=t, it=it):
                for slot, pos in zip(t.ld_slots, t.ld_pos):
                    self.sg[slot].begin_write(f"copier{it}")
                    self.sg[slot].end_write((t.run, pos))
            yield call(put_sigma)
            yield arrive(self.full_qk[s], tx=2)        # Q rows and new K rows
            yield arrive(self.full_v[it % K_VDEPTH], tx=1)
            sw = self.sig_w[it % m.sigw_slots]
            yield arrive(sw)

            def read_rows(t=t, it=it):  # the Q gathers read the tile's sigma
                for slot, tag in g.row_slots(t):
                    self.sg[slot].begin_read(f"copierQ{it}", tag)
                    self.sg[slot].end_read(f"copierQ{it}")
            yield call(read_rows)
            yield copy([(self.q[s], it)], f"tmaQ{it}", self.full_qk[s], "tx")
            yield copy([(self.kr[x], (t.run, p)) for x, p in zip(t.ld_slots, t.ld_pos)],
                       f"tmaK{it}", self.full_qk[s], "tx")
            yield copy([(self.vr[x], (t.run, p)) for x, p in zip(t.ld_slots, t.ld_pos)],
                       f"tmaV{it}", self.full_v[it % K_VDEPTH], "tx")
        n = len(self.tiles)
        for x in range(max(0, n - K_QSTAGES), n):  # the last copies land before exit
            yield wait(self.full_qk[x % K_QSTAGES], (x // K_QSTAGES) & 1, x // K_QSTAGES)
        for x in range(max(0, n - K_VDEPTH), n):
            yield wait(self.full_v[x % K_VDEPTH], (x // K_VDEPTH) & 1, x // K_VDEPTH)

    def masker(self):
        g, m = self.geo, self.mut
        for it, t in enumerate(self.tiles):
            slots = m.sigw_slots
            yield wait(self.sig_w[it % slots], (it // slots) & 1, it // slots)
            who = f"masker{it}"
            wb = self.word_buf(it)

            def start(t=t, who=who, wb=wb):
                for slot, tag in g.span_slots(t):
                    self.sg[slot].begin_read(who, tag)
                for quarter in wb:
                    quarter.begin_write(who)
            yield call(start)

            def finish(t=t, it=it, who=who, wb=wb):
                for quarter in wb:
                    quarter.end_write(it)
                for slot, _ in g.span_slots(t):
                    self.sg[slot].end_read(who)
            yield call(finish)
            wg = it & 1
            if m.masker_waits_release:
                yield wait(self.s_free[wg], ((it >> 1) & 1) ^ 1, (it >> 1) - 1)
            yield arrive(self.s_ready[wg])

    def mma_warp(self):
        g, m = self.geo, self.mut
        for it, t in enumerate(self.tiles):
            s, st = it % K_QSTAGES, it & 1
            yield wait(self.full_qk[s], (it // K_QSTAGES) & 1, it // K_QSTAGES)
            if m.mma_waits_readout:
                yield wait(self.t_empty[st], ((it >> 1) & 1) ^ 1, (it >> 1) - 1)
            reads = [(self.q[s], it)] + [(self.kr[x], tag) for x, tag in g.span_slots(t)]
            writes = [(b, ("S", it)) for b in self.tp[st] + self.to[st]]
            yield mma(reads, writes, f"QK{it}", [self.s_full[st], self.qk_done[s]])

    def softmax_warp(self, wg: int, q: int):
        """Warp q of softmax warpgroup wg; warp 0's first lane issues the
        warpgroup's O MMAs (its other lanes wait for it)."""
        g = self.geo
        for it, t in enumerate(self.tiles):
            if (it & 1) != wg:
                continue
            ph, meant = (it >> 1) & 1, it >> 1
            who = f"softmax{it}.{q}"
            yield wait(self.s_ready[wg], ph, meant)
            wb = self.word_buf(it)[q]

            def read_words(t=t, who=who, wb=wb, it=it):
                wb.begin_read(who, it)
                for slot, tag in g.row_slots(t):
                    self.sg[slot].begin_read(who, tag)
            yield call(read_words)

            def words_done(t=t, who=who, wb=wb):
                wb.end_read(who)
                for slot, _ in g.row_slots(t):
                    self.sg[slot].end_read(who)
            yield call(words_done)
            yield arrive(self.s_free[wg])
            yield wait(self.s_full[wg], ph, meant)
            tp, to = self.tp[wg][q], self.to[wg][q]

            def passes(who=who, it=it, tp=tp, to=to):
                tp.read(who, ("S", it))
                to.read(who, ("S", it))
                tp.write(who, ("P", it))
            yield call(passes)
            yield arrive(self.p_full[wg])
            if q == 0:  # the warpgroup's issuer
                yield wait(self.p_full[wg], ph, meant)
                yield wait(self.full_v[it % K_VDEPTH], (it // K_VDEPTH) & 1, it // K_VDEPTH)
                if self.mut.pv_waits_previous and it > 0:
                    # the span's older V rows came with earlier tiles, whose own
                    # waits this chain of O MMAs inherits
                    z = it - 1
                    yield wait(self.pv_done[z % K_VDEPTH], (z // K_VDEPTH) & 1, z // K_VDEPTH)
                reads = [(b, ("P", it)) for b in self.tp[wg]] + \
                        [(self.vr[x], tag) for x, tag in g.span_slots(t)]
                yield mma(reads, [(b, ("O", it)) for b in self.to[wg]], f"PV{it}",
                          [self.o_full[wg], self.pv_done[it % K_VDEPTH]])
            # epilogue
            yield wait(self.o_full[wg], ph, meant)
            yield call(lambda who=who, it=it, to=to: to.read(who + "epi", ("O", it)))
            yield arrive(self.t_empty[wg])

    def run(self, seed: int):
        roles = {"copier": self.copier(), "masker": self.masker(), "mma": self.mma_warp()}
        for wg in range(2):
            for q in range(4):
                roles[f"wg{wg}.warp{q}"] = self.softmax_warp(wg, q)
        return simulate(roles, seed)


GEOMETRIES = {
    # positions per tile, window halves, tiles per sequence, first tile, tiles of this CTA
    "gqa_w128": Geometry(bt=32, left=64, right=64, tiles_per_seq=6, first_tile=3, ntiles=14),
    "gqa_w32": Geometry(bt=32, left=16, right=16, tiles_per_seq=5, first_tile=0, ntiles=12),
    "mha_w128": Geometry(bt=128, left=64, right=64, tiles_per_seq=3, first_tile=1, ntiles=9),
    "swa_w96": Geometry(bt=16, left=95, right=0, tiles_per_seq=40, first_tile=7, ntiles=16),
    "one_tile_runs": Geometry(bt=32, left=64, right=64, tiles_per_seq=1, first_tile=0, ntiles=7),
}


@pytest.mark.parametrize("geo", sorted(GEOMETRIES))
def test_ring_protocol_has_no_race_deadlock_or_parity_alias(geo):
    for seed in range(60):
        Model(GEOMETRIES[geo]).run(seed)


MUTANTS = {
    "Q stage reused one tile early": Mutation(qk_retire_lag=K_QSTAGES + 1),
    "ring rows reused one tile early": Mutation(pv_retire_lag=K_VDEPTH + 1),
    "masker hands over without the release wait": Mutation(masker_waits_release=False),
    "two mask-word buffers": Mutation(word_buffers=2),
    "two sigma barriers": Mutation(sigw_slots=2),
    "S MMA does not wait for the O read-out": Mutation(mma_waits_readout=False),
    "O MMA does not wait for the previous tile's": Mutation(pv_waits_previous=False),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_protocol_mistakes_are_caught(name):
    geo = GEOMETRIES["gqa_w128"]
    for seed in range(400):
        try:
            Model(geo, MUTANTS[name]).run(seed)
        except ProtocolError:
            return
    pytest.fail(f"the model did not catch: {name}")
