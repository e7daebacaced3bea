"""A small model of the tcgen05 kernels' synchronisation, for CPU model checks
of their hand-over protocols (compute-sanitizer is closed on this machine).

What is modelled:
  - mbarriers: an arrival count and transaction units complete a phase; the
    parity wait passes while the current phase has the other parity, as the
    hardware's try_wait.parity does;
  - the copy engine: a copy (TMA or cp.async) lands at any later time, in any
    order, and then completes transaction units on its barrier or arrives on
    it;
  - the tensor pipe: MMAs complete in issue order, and a commit arrives on its
    barrier once the MMAs issued before it are done;
  - buffers handed between roles: a write may not start while a reader of the
    previous contents still reads, and a read must see the contents the
    reader expects; accumulators take a tile's first MMA as a replacement and
    its later ones as additions.

Roles are generators of actions; `simulate` runs them under a random
interleaving in which every actor has its own random speed, and raises
ProtocolError on a deadlock, on a wait released by any phase but the one it
is for, or on a buffer race.
"""

from __future__ import annotations

import random


class ProtocolError(AssertionError):
    pass


class Barrier:
    """mbarrier: `count` arrivals plus all expected transaction units
    complete a phase; `k` phases have completed."""

    def __init__(self, name: str, count: int):
        self.name, self.count = name, count
        self.pending, self.tx, self.k = count, 0, 0

    def _maybe_complete(self):
        if self.pending == 0 and self.tx == 0:
            self.k += 1
            self.pending = self.count

    def arrive(self, expect_tx: int = 0):
        if self.pending <= 0:
            raise ProtocolError(f"{self.name}: arrival beyond the count")
        self.tx += expect_tx
        self.pending -= 1
        self._maybe_complete()

    def complete_tx(self, units: int = 1):
        self.tx -= units
        if self.tx < 0:
            raise ProtocolError(f"{self.name}: transaction bytes before they were expected")
        self._maybe_complete()

    def passes(self, parity: int) -> bool:
        return (self.k & 1) != parity


class Buffer:
    def __init__(self, name: str):
        self.name = name
        self.content = None
        self.readers: dict[str, object] = {}
        self.writer = None

    def begin_write(self, who: str):
        if self.readers:
            raise ProtocolError(f"{who} writes {self.name} while {sorted(self.readers)} read "
                                f"{self.content}")
        if self.writer is not None:
            raise ProtocolError(f"{who} writes {self.name} during {self.writer}'s write")
        self.writer = who
        self.content = None

    def end_write(self, tag):
        self.writer = None
        self.content = tag

    def begin_read(self, who: str, want):
        if self.writer is not None:
            raise ProtocolError(f"{who} reads {self.name} during {self.writer}'s write")
        if self.content != want:
            raise ProtocolError(f"{who} reads {self.name}: holds {self.content}, wants {want}")
        self.readers[who] = want

    def end_read(self, who: str):
        del self.readers[who]

    def read(self, who: str, want):
        self.begin_read(who, want)
        self.end_read(who)

    def write(self, who: str, tag):
        self.begin_write(who)
        self.end_write(tag)


class Accumulator(Buffer):
    """A TMEM accumulator: a tile's first MMA replaces it, the tile's later
    ones add to it (MMAs into one accumulator run in issue order)."""

    def __init__(self, name):
        super().__init__(name)
        self.inflight = 0

    def begin_mma(self, who, tag, replace):
        if replace:
            if self.readers:
                raise ProtocolError(f"{who} replaces {self.name} while {sorted(self.readers)} "
                                    f"read {self.content}")
            if self.inflight:
                raise ProtocolError(f"{who} replaces {self.name} under earlier MMAs")
        elif self.content != tag:
            raise ProtocolError(f"{who} adds to {self.name} holding {self.content}, not {tag}")
        self.content = tag
        self.inflight += 1

    def end_mma(self):
        self.inflight -= 1

    def begin_read(self, who, want):
        if self.inflight:
            raise ProtocolError(f"{who} reads {self.name} under MMAs in flight")
        super().begin_read(who, want)


# ---------------------------------------------------------------- actions
def wait(bar: Barrier, parity: int, meant: int):
    """A parity wait for phase index `meant` (-1: the phase before the first)."""
    return ("wait", bar, parity, meant)


def arrive(bar: Barrier, n: int = 1, tx: int = 0):
    """n arrivals; the first also expects `tx` transaction units."""
    return ("arrive", bar, n, tx)


def call(fn):
    return ("call", fn)


def copy(writes, who: str, bar: Barrier, completes: str):
    """An asynchronous copy into `writes` [(buffer, tag)]; on landing it
    completes one transaction unit on `bar` ("tx") or arrives on it
    ("arrive"); with no barrier, only wait_copies sees it land."""
    return ("copy", writes, who, bar, completes)


def wait_copies():
    """cp.async.wait_all: passes once every copy issued so far has landed."""
    return ("wait_copies",)


def commit_group():
    """cp.async.commit_group: closes the group the copies since the last
    commit belong to (a group may be empty)."""
    return ("commit_group",)


def wait_group(n: int):
    """cp.async.wait_group n: passes once at most the n newest committed
    groups still have copies in flight."""
    return ("wait_group", n)


def mma(reads, writes, who: str, commits):
    """An MMA reading [(buffer, tag)] and writing [(buffer, tag)] or
    [(accumulator, tag, replace)], followed by commits to `commits`."""
    return ("mma", reads, writes, who, commits)


# ---------------------------------------------------------------- scheduler
def simulate(roles: dict, seed: int, max_steps: int = 400000) -> int:
    rng = random.Random(seed)
    speed = {n: rng.choice([0.02, 0.2, 1.0, 5.0]) for n in list(roles) + ["copy", "pipe"]}
    nxt = {}
    for name, gen in roles.items():
        try:
            nxt[name] = next(gen)
        except StopIteration:
            pass
    copies, pipe = [], []
    groups = 0  # cp.async groups committed so far (copies carry their group)
    steps = 0

    def runnable(name):
        a = nxt[name]
        if a[0] == "wait_copies":
            return not copies
        if a[0] == "wait_group":
            return all(cp[4] >= groups - a[1] for cp in copies)
        return a[0] != "wait" or a[1].passes(a[2])

    while nxt or copies or pipe:
        steps += 1
        if steps > max_steps:
            raise ProtocolError("no progress bound reached")
        for name, a in nxt.items():  # a wait overrun by a later phase means nothing
            if a[0] == "wait" and a[1].k - 1 > a[3]:
                raise ProtocolError(f"{name}: {a[1].name} is {a[1].k - 1 - a[3]} phases past "
                                    f"the phase {a[3]} it waits for")
        choices = [("role", n) for n in nxt if runnable(n)]
        choices += [("copy", i) for i in range(len(copies))]
        if pipe:
            choices.append(("pipe", 0))
        if not choices:
            raise ProtocolError("deadlock: " + ", ".join(
                f"{n} waits {a[1].name} parity {a[2]}" if a[0] == "wait" else f"{n}: {a[0]}"
                for n, a in nxt.items()))
        weights = [speed[n] if k == "role" else speed[k] for k, n in choices]
        kind, key = rng.choices(choices, weights=weights)[0]
        if kind == "copy":
            writes, who, bar, completes, _ = copies.pop(key)
            for buf, tag in writes:
                buf.end_write(tag)
            if bar is None:  # a cp.async waited for with wait_copies
                pass
            elif completes == "tx":
                bar.complete_tx(1)
            else:
                bar.arrive()
            continue
        if kind == "pipe":
            reads, writes, who, commits = pipe.pop(0)
            for buf, _ in reads:
                buf.end_read(who)
            for w in writes:
                if isinstance(w[0], Accumulator):
                    w[0].end_mma()
                else:
                    w[0].end_write(w[1])
            for bar in commits:
                bar.arrive()
            continue
        a = nxt[key]
        if a[0] == "wait":
            if a[1].k - 1 != a[3]:
                raise ProtocolError(f"{key}: {a[1].name} released at phase {a[1].k - 1}, the "
                                    f"wait is for phase {a[3]}")
        elif a[0] == "arrive":
            _, bar, n, tx = a
            bar.arrive(expect_tx=tx)
            for _ in range(n - 1):
                bar.arrive()
        elif a[0] == "call":
            a[1]()
        elif a[0] == "copy":
            _, writes, who, bar, completes = a
            for buf, _ in writes:
                buf.begin_write(who)
            copies.append((writes, who, bar, completes, groups))
        elif a[0] == "commit_group":
            groups += 1
        elif a[0] == "mma":
            _, reads, writes, who, commits = a
            for buf, tag in reads:
                buf.begin_read(who, tag)
            for w in writes:
                if isinstance(w[0], Accumulator):
                    w[0].begin_mma(who, w[1], w[2])
                else:
                    w[0].begin_write(who)
            pipe.append((reads, writes, who, commits))
        try:
            nxt[key] = next(roles[key])
        except StopIteration:
            del nxt[key]
    return steps
