"""CPU models of the barrier protocols in csrc/attention.cu, run under random
interleavings of the warps' steps. No GPU: the hardware barriers of those
kernels cannot time out, so their protocols are checked here before they run.

1. The extend kernel's tensor-pipe turns: warp groups A (warps 0-3) and B
   (warps 4-7) hand the turn over with named barriers 1 (to A) and 2 (to B),
   `bar.arrive` by the group that ends a phase and `bar.sync` by the one that
   starts; two `__syncthreads` per chunk. Checked: no deadlock, every phase of
   a named barrier pairs one arrival from each group, nothing left over.

2. The decode kernel's slot ring: one loading warp per slot fills it item by
   item after the slot's "empty" barrier releases it; each (slot, consumer
   group) has its own "full" barrier with a transaction count the copies pay
   off asynchronously; waits are parity waits (true as soon as the barrier's
   phase parity differs). Checked: no deadlock, a consumer always finds its
   own item's data, no copy lands in a slot that is still being read. The
   earlier form (one "full" barrier per slot shared by both groups, two
   loading warps taking alternate items) is shown to break, which pins the
   model to a fault it must catch. (The one-item-per-CTA shape counts its V
   rows on a second "full" barrier; it fills its one slot once, so no phase
   of either barrier is reused.)
"""
import random

import pytest


# --------------------------------------------------------------- extend turns

def _extend_program(group, chunks):
    ops = []
    for c in range(chunks):
        ops += [("W", 0), ("W", 0)]                       # __syncthreads_or, __syncthreads
        if group == "A":
            if c > 0:
                ops.append(("W", 1))
            ops += [("P", 2), ("W", 1), ("P", 2)]         # after q.k; before p.V; after p.V
        else:
            ops += [("W", 2), ("P", 1), ("W", 2), ("P", 1)]
    if group == "A":
        ops.append(("W", 1))                              # B's hand-over after its last p.V
    return ops


def _run_turns(chunks, seed):
    rng = random.Random(seed)
    progs = {g: _extend_program(g, chunks) for g in "AB"}
    pc = {g: 0 for g in "AB"}
    waiting = {g: None for g in "AB"}
    arrived = {0: [], 1: [], 2: []}
    for _ in range(100000):
        live = [g for g in "AB" if pc[g] < len(progs[g])]
        if not live:
            return "ok" if not any(arrived.values()) else f"left over {arrived}"
        runnable = [g for g in live if waiting[g] is None]
        if not runnable:
            return "deadlock"
        g = rng.choice(runnable)
        kind, bar = progs[g][pc[g]]
        pc[g] += 1
        if g in arrived[bar]:
            return f"{g} arrived twice in one phase of barrier {bar}"
        arrived[bar].append(g)
        if kind == "W":
            waiting[g] = bar
        if len(arrived[bar]) == 2:                        # 256 threads: both groups
            arrived[bar] = []
            for x in "AB":
                if waiting[x] == bar:
                    waiting[x] = None
    return "stuck"


@pytest.mark.parametrize("chunks", [1, 2, 3, 9])
def test_extend_turns(chunks):
    for seed in range(400):
        assert _run_turns(chunks, seed) == "ok", f"chunks={chunks} seed={seed}"


# --------------------------------------------------------------- decode ring

class _Bar:
    """An mbarrier: expected arrivals, a transaction count, a phase counter."""

    def __init__(self, count):
        self.count, self.arr, self.tx, self.phase = count, 0, 0, 0

    def arrive(self, tx=0):
        self.arr += 1
        self.tx += tx
        self._step()

    def complete_tx(self, nbytes):
        self.tx -= nbytes
        self._step()

    def _step(self):
        if self.arr == self.count and self.tx == 0:
            self.arr = 0
            self.phase += 1

    def try_wait(self, parity):
        return (self.phase & 1) != parity


def _run_ring(slots, groups, items, seed, shared_full=False, loaders=None):
    """The ring as the kernel runs it (shared_full / loaders: the earlier form)."""
    rng = random.Random(seed)
    loaders = loaders or slots
    nfull = slots if shared_full else slots * groups
    full = [_Bar(1) for _ in range(nfull)]
    empty = [_Bar(1) for _ in range(slots)]
    data = [None] * slots
    reading = [None] * slots
    pending = []

    def full_of(k):
        return full[k % slots] if shared_full else full[(k % slots) * groups + k % groups]

    def full_parity(k):
        return ((k // slots) if shared_full else (k // (slots * groups))) & 1

    def loader(lw):
        for k in range(lw, items, loaders):
            s = k % slots
            if k >= slots:
                while not empty[s].try_wait(((k // slots) - 1) & 1):
                    yield
            full_of(k).arrive(tx=1)
            pending.append((s, k, full_of(k)))
            yield

    def consumer(g):
        for k in range(g, items, groups):
            s = k % slots
            while not full_of(k).try_wait(full_parity(k)):
                yield
            if data[s] != k:
                raise AssertionError(f"group {g} took item {k} from slot {s} holding {data[s]}")
            reading[s] = k
            for _ in range(rng.randint(0, 4)):
                yield
            reading[s] = None
            empty[s].arrive()

    progs = [loader(i) for i in range(loaders)] + [consumer(g) for g in range(groups)]
    live = list(range(len(progs)))
    for _ in range(200000):
        if not live and not pending:
            return "ok"
        if pending and (not live or rng.random() < 0.3):
            s, k, bar = pending.pop(rng.randrange(len(pending)))
            if reading[s] is not None:
                raise AssertionError(f"item {k} lands in slot {s} while item {reading[s]} is read")
            data[s] = k
            bar.complete_tx(1)
            continue
        j = rng.choice(live)
        try:
            next(progs[j])
        except StopIteration:
            live.remove(j)
    return "stuck"


@pytest.mark.parametrize("slots,groups", [(3, 2), (1, 1)])
@pytest.mark.parametrize("items", [1, 2, 5, 7, 13, 40])
def test_decode_ring(slots, groups, items):
    for seed in range(150):
        assert _run_ring(slots, groups, items, seed) == "ok", f"seed={seed}"


def test_decode_ring_model_catches_the_shared_barrier_form():
    """One "full" barrier per slot for both groups and two loading warps on
    alternate items: some interleaving must break it."""
    broke = 0
    for seed in range(400):
        try:
            _run_ring(3, 2, 24, seed, shared_full=True, loaders=2)
        except AssertionError:
            broke += 1
    assert broke > 0
