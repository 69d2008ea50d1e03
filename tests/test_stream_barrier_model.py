"""A model of the stream kernel's barrier protocol, explored over random
interleavings on the CPU.

The kernel's roles (one TMA producer, or for candidate tiles one per tile
parity; two converter groups, two MMA issuers and two epilogue groups, one
of each per tile parity) hand tiles to
each other through mbarriers waited on by phase parity. A parity wait cannot
tell phase n from phase n-2: if a waiter can ever reach a barrier two phases
early, it passes on a stale phase. The model tracks every barrier's count of
completed phases and checks, at each successful wait, that the completed
phase is exactly the one the waiter means. It also checks the data hazards
the waits are there for: a K stage, an A (operand) slot, an accumulator slot
and a weight/scale slot are never rewritten while a reader still needs them.

The slot counts are read from the kernel source, so the model follows the
code; a second test gives the model the odd counts an earlier build had
(five A slots, three accumulator slots) and checks that it finds the stale
phase that build hit.
"""
import os
import random
import re

import pytest

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "sparse_attention_indexer_qli_gb300", "csrc", "qli_score.cu")


def kernel_constants():
    txt = open(SRC).read()

    def const(name):
        m = re.search(r"constexpr int %s = (\d+);" % name, txt)
        if m:
            return int(m.group(1))
        m = re.search(r"\b%s = (\d+)[,;]" % name, txt)
        assert m, name
        return int(m.group(1))
    return {"S": const("kKStages"), "A": const("kASlots"), "D": const("kDSlots"),
            "SL": const("kSlots")}


class Stale(AssertionError):
    pass


class Barrier:
    """count arrivals complete one phase; `done` = phases completed."""

    def __init__(self, count):
        self.count, self.pending, self.done = count, count, 0

    def arrive(self):
        self.pending -= 1
        if self.pending == 0:
            self.done += 1
            self.pending = self.count

    def ready(self, phase):
        # try_wait.parity(phase & 1) succeeds once the barrier's current phase
        # has the other parity
        return (self.done & 1) != (phase & 1)

    def check(self, phase, what):
        if self.done != phase + 1:
            raise Stale("%s: waited for phase %d, barrier has completed %d" % (what, phase, self.done))


def run(c, nk, seed, token_every, producers=1):
    S, A, D, SL = c["S"], c["A"], c["D"], c["SL"]
    rng = random.Random(seed)
    full = [Barrier(1) for _ in range(S)]
    empty = [Barrier(1) for _ in range(S)]        # the converting group (one arrival)
    afull = [Barrier(1) for _ in range(A)]
    afree = [Barrier(1) for _ in range(A)]
    dfull = [Barrier(1) for _ in range(D)]
    dfree = [Barrier(1) for _ in range(D)]
    kready = [Barrier(1) for _ in range(SL)]
    # who holds what (tile numbers), for the data-hazard checks
    stage_tile = [None] * S          # K tile in a stage, until its converter read it
    aslot_tile = [None] * A          # converted tile in an A slot, until its MMA finished
    dslot_tile = [None] * D          # MMA tile in an accumulator, until its epilogue read it
    wslot_tile = [None] * SL         # tile whose weights / scales a slot holds until read
    mma_done = set()
    token_change = {k for k in range(nk) if k < 2 or (token_every and k % token_every == 0)}

    # role programs: lists of steps; each step = (ready(), act())
    def producer(p):
        for k in range(p, nk, producers):
            s = k % S
            if k >= S:
                yield ("wait", empty[s], k // S - 1, "empty")
            if stage_tile[s] is not None:
                raise Stale("stage %d rewritten while tile %d unread" % (s, stage_tile[s]))
            stage_tile[s] = k
            inflight.append(("tma", k))
            yield ("step",)

    def converter(g):
        for k in range(g, nk, 2):
            a, s, sl = k % A, k % S, k % SL
            if k >= A:
                yield ("wait", afree[a], k // A - 1, "afree")
            if k in token_change and k >= 2:
                yield ("wait", afree[(k - 2) % A], (k - 2) // A, "afree(query buffer)")
            if wslot_tile[sl] is not None:
                raise Stale("weight slot %d rewritten before tile %d's epilogue read it"
                            % (sl, wslot_tile[sl]))
            wslot_tile[sl] = k
            yield ("wait", full[s], k // S, "full")
            assert stage_tile[s] == k
            stage_tile[s] = None
            empty[s].arrive()
            kready[sl].arrive()
            if aslot_tile[a] is not None:
                raise Stale("A slot %d rewritten while tile %d's MMA unfinished" % (a, aslot_tile[a]))
            aslot_tile[a] = k
            afull[a].arrive()
            yield ("step",)

    def mma(p):
        for k in range(p, nk, 2):
            a, d = k % A, k % D
            yield ("wait", afull[a], k // A, "afull")
            if k >= D:
                yield ("wait", dfree[d], k // D - 1, "dfree")
            if aslot_tile[a] != k:
                raise Stale("MMA %d found A slot %d holding %r" % (k, a, aslot_tile[a]))
            if dslot_tile[d] is not None:
                raise Stale("MMA %d overwrites accumulator %d of tile %d" % (k, d, dslot_tile[d]))
            dslot_tile[d] = k
            mmas.append(k)
            yield ("step",)

    def epilogue(g):
        for k in range(g, nk, 2):
            d, sl = k % D, k % SL
            yield ("wait", kready[sl], k // SL, "kready")
            yield ("wait", dfull[d], k // D, "dfull")
            if dslot_tile[d] != k or k not in mma_done:
                raise Stale("epilogue %d read accumulator %d holding %r" % (k, d, dslot_tile[d]))
            dslot_tile[d] = None
            dfree[d].arrive()
            yield ("step",)
            if wslot_tile[sl] != k:
                raise Stale("epilogue %d found weight slot %d holding %r" % (k, sl, wslot_tile[sl]))
            wslot_tile[sl] = None
            yield ("step",)

    inflight = []                   # copies in flight: they land in any order
    mmas = []                       # MMAs in flight: the tensor core finishes them in issue order
    roles = [producer(p) for p in range(producers)]
    roles += [converter(0), converter(1), mma(0), mma(1), epilogue(0), epilogue(1)]

    def advance(r):
        try:
            return next(r)
        except StopIteration:
            return None
    pending = [advance(r) for r in roles]
    while True:
        options = []
        for i, step in enumerate(pending):
            if step is None:
                continue
            if step[0] == "step" or step[1].ready(step[2]):
                options.append(("role", i))
        options += [("done", j) for j in range(len(inflight))]
        if mmas:
            options.append(("mma", 0))
        if not options:
            break
        kind, i = rng.choice(options)
        if kind == "done":
            _, k = inflight.pop(i)
            full[k % S].arrive()
            continue
        if kind == "mma":                           # the oldest MMA completes: both commits
            k = mmas.pop(0)
            mma_done.add(k)
            aslot_tile[k % A] = None
            afree[k % A].arrive()
            dfull[k % D].arrive()
            continue
        step = pending[i]
        if step[0] == "wait":
            step[1].check(step[2], step[3])
        pending[i] = advance(roles[i])
    if any(p is not None for p in pending) or inflight or mmas:
        raise Stale("deadlock: roles still waiting %r" % [p[3] if p and p[0] == "wait" else p
                                                         for p in pending])


@pytest.mark.parametrize("producers", [1, 2])
def test_kernel_slot_counts_never_meet_a_stale_phase(producers):
    # one producer for dense tiles; for candidate tiles two, each issuing
    # the tiles of one parity into the stages of that parity
    c = kernel_constants()
    assert c["A"] % 2 == 0 and c["D"] % 2 == 0 and c["S"] % 2 == 0
    for seed in range(400):
        for nk in (1, 2, 7, 33):
            run(c, nk, seed, token_every=1 + seed % 9, producers=producers)


def test_the_model_catches_odd_slot_counts():
    # five A slots and three accumulator slots: the configuration that once
    # produced timeouts and wrong scores on full-size runs
    c = dict(kernel_constants(), A=5, D=3)
    with pytest.raises(Stale):
        for seed in range(400):
            run(c, 40, seed, token_every=7)


@pytest.mark.parametrize("slots,safe", [(8, False), (10, True)])
def test_weight_slot_ring_needs_two_plus_a_plus_d(slots, safe):
    # a tile's weights and K scales are read by its epilogue after the
    # accumulator is released; the converter of tile k + slots rewrites them
    # only after the MMA of tile k + slots - A, whose accumulator the
    # epilogue of tile k + slots - A - D released: the ring needs
    # slots >= 2 + A + D (A = D = 4 in the kernel)
    c = dict(kernel_constants(), SL=slots)
    found = False
    for seed in range(300):
        try:
            run(c, 40, seed, token_every=5)
        except Stale:
            found = True
            break
    assert found != safe
